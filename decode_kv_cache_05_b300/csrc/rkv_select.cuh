// rkv_select: min-max normalisation, the lambda blend and windowed top-budget
// selection, one CTA per (layer, sequence, KV head) -- or per (layer,
// sequence) when the KV heads share one eviction set.
//
// The R-KV review page ("How R-KV decides what to drop") keeps kv_budget tokens
// with a protected local window of window_size tokens and blends the two
// scores with mix_lambda; the hotdry.top blog (R-KV section) keeps tokens of
// high importance and low redundancy. Here:
//     I^, R^ = min-max over the head's N tokens (constant -> 0),
//     S = lambda * I^ - (1 - lambda) * R^,
//     keep = window [N-w, N) + the (budget - w) largest S of [0, N-w),
//            equal S -> lower index, emitted ascending.
// The threshold is found by an 8-bit-digit radix select over order-preserving
// uint32 keys of S in shared memory (warp-aggregated histogram increments,
// double-buffered histograms so each digit costs two barriers, and an early
// stop once the threshold's bin is kept whole); one block-wide scan of packed
// (ties, others) counts places the kept indices.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

#ifndef RKV_SEL_THREADS
#define RKV_SEL_THREADS 256
#endif
// Test builds only (never the shipped library): with RKV_SELECT_WAIT_TEST
// the kernel, after its score rows have landed, also waits on a barrier that
// nothing ever arrives on, with a limit of RKV_SELECT_WAIT_TEST_NS, so that
// the bounded wait runs out and the kernel takes its timeout path: error word
// RKV_ERR_TIMEOUT, the bulk copies it issued drained, no kept index written.
#ifndef RKV_SELECT_WAIT_TEST
#define RKV_SELECT_WAIT_TEST 0
#endif
#ifndef RKV_SELECT_WAIT_TEST_NS
#define RKV_SELECT_WAIT_TEST_NS 2000000ull
#endif
constexpr int kSelThreads = RKV_SEL_THREADS;
constexpr int kSelWarps = kSelThreads / 32;

struct SelArgs {
    Geom g;
    const float *imp;
    const float *red;
    int32_t *keep;
    float *scores; // [3][L][B][Hkv][nmax] or null
};

// Shared memory of one CTA of `threads` threads: the S keys [npad], one or
// two staging buffers of the importance and redundancy rows [2][npad], two
// 256-bin histograms, reduction / scan scratch and three mbarriers (the third
// is used by test builds only).
__host__ __device__ constexpr size_t sel_smem_bytes(int npad, bool shared_heads, int threads = kSelThreads)
{
    return ((1 + (shared_heads ? 4 : 2)) * static_cast<size_t>(npad) + 2 * 256 + 5 * (threads / 32) + 2) * 4 + 24;
}

__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide {min, max, min, max} of per-thread partials v (all threads call;
// results broadcast).
template <int kWarps = kSelWarps>
__device__ __forceinline__ void block_minmax2(float (&v)[4], float *scratch)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        v[0] = fminf(v[0], __shfl_xor_sync(0xffffffffu, v[0], off));
        v[1] = fmaxf(v[1], __shfl_xor_sync(0xffffffffu, v[1], off));
        v[2] = fminf(v[2], __shfl_xor_sync(0xffffffffu, v[2], off));
        v[3] = fmaxf(v[3], __shfl_xor_sync(0xffffffffu, v[3], off));
    }
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
        for (int t = 0; t < 4; ++t)
            scratch[(threadIdx.x >> 5) * 4 + t] = v[t];
    }
    __syncthreads();
#pragma unroll
    for (int t = 0; t < 4; ++t)
        v[t] = scratch[t];
    for (int w = 1; w < kWarps; ++w) {
        v[0] = fminf(v[0], scratch[w * 4 + 0]);
        v[1] = fmaxf(v[1], scratch[w * 4 + 1]);
        v[2] = fminf(v[2], scratch[w * 4 + 2]);
        v[3] = fmaxf(v[3], scratch[w * 4 + 3]);
    }
}

// Exclusive prefix sum over the block (thread order).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, uint32_t *scratch)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    if (lane == 31)
        scratch[warp] = x;
    __syncthreads();
    uint32_t before = 0;
    for (int w = 0; w < warp; ++w)
        before += scratch[w];
    return before + x - v;
}

// The selection of one unit by the whole CTA (kSelThreads threads): a
// (layer, sequence, KV head) row of scores starting at head e0, or, with
// kShared (eviction shared by the KV heads of a layer), a (layer, sequence)
// event whose Hkv rows are normalised and blended per head and then summed
// over the heads (head order, fp32) into one score per token; that one keep
// set is written to every head's row. `sel_smem` is the CTA's selection
// scratch (sel_smem_bytes). If keep_s is not null (per-head units only), the
// kept indices are also written there: keep_s[0 .. budget), -1 past
// min(N, budget), visible to the CTA after the function returns. Returns
// false if a bounded wait gave up (kept indices then not written).
template <bool kShared, int kThreads = kSelThreads>
__device__ __forceinline__ bool select_unit(const SelArgs &a, int e0, uint32_t *sel_smem, int32_t *keep_s)
{
    constexpr int kSelThreads = kThreads; // this function's block size (shadows the namespace default)
    constexpr int kSelWarps = kThreads / 32;
    const Geom &g = a.g;
    constexpr int kBufs = kShared ? 2 : 1;
    uint32_t *key = sel_smem;                                       // [npad]
    float *ssum = reinterpret_cast<float *>(key);                   // shared mode: sum of S before keying
    float *stage = reinterpret_cast<float *>(key + g.npad);         // [kBufs][2][npad]: I, R
    uint32_t *hist = reinterpret_cast<uint32_t *>(stage + kBufs * 2 * g.npad); // [2][256]
    float *fscratch = reinterpret_cast<float *>(hist + 2 * 256);    // [4 * kSelWarps]
    uint32_t *uscratch = reinterpret_cast<uint32_t *>(fscratch + 4 * kSelWarps); // [kSelWarps]
    uint64_t *bars = reinterpret_cast<uint64_t *>(
        (reinterpret_cast<uintptr_t>(uscratch + kSelWarps + 1) + 7) & ~static_cast<uintptr_t>(7));
    __shared__ uint32_t sh_prefix[2], sh_remaining[2], sh_done[2], sh_abort;

    const int nh = kShared ? g.Hkv : 1;                // heads of this unit
    const HeadId id = head_id(g, e0);
    // ---- score rows into shared memory with bulk copies (one memory round
    // trip per head; the next head's rows load while this one is processed)
    auto stage_head = [&](int hh) {
        const int buf = hh & 1;
        const size_t sbase = static_cast<size_t>(e0 + hh) * g.npad;
        mbar_expect_tx(&bars[buf], 2u * g.npad * 4u);
        bulk_load(stage + (buf * 2) * g.npad, a.imp + sbase, g.npad * 4, &bars[buf]);
        bulk_load(stage + (buf * 2 + 1) * g.npad, a.red + sbase, g.npad * 4, &bars[buf]);
    };
    int n = g.seq_lens[id.b];
    if (n < 0 || n > g.nmax)
        n = 0; // recorded by rkv_importance / rkv_compact
    const int kb = min(n, g.budget);
    if (!triggered(g, n)) {
        // left for a later call: the identity prefix, nothing else
        for (int hh = 0; hh < nh; ++hh)
            for (int j = threadIdx.x; j < g.budget; j += kSelThreads)
                a.keep[static_cast<size_t>(e0 + hh) * g.budget + j] = j < kb ? j : -1;
        if (keep_s) {
            for (int j = threadIdx.x; j < g.budget; j += kSelThreads)
                keep_s[j] = j < kb ? j : -1;
            __syncthreads();
        }
        return true;
    }
    if (threadIdx.x == 0) {
        sh_abort = 0;
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1); // test builds: never arrived on
        fence_barrier_init();
        stage_head(0);
        if (kShared && nh > 1)
            stage_head(1);
    }
    for (int i = threadIdx.x; i < 256; i += kSelThreads)
        hist[i] = 0;
    if (kShared) {
        for (int j = threadIdx.x; j < n; j += kSelThreads)
            ssum[j] = 0.f;
    }
    __syncthreads(); // barriers initialised

    const float lam = g.lam;
    const size_t plane = static_cast<size_t>(g.L) * g.B * g.Hkv * g.nmax;
    for (int hh = 0; hh < nh; ++hh) {
        const int buf = hh & 1;
        bool landed = mbar_wait(&bars[buf], (hh >> 1) & 1, &sh_abort);
#if RKV_SELECT_WAIT_TEST
        landed = landed && mbar_wait(&bars[2], 0, &sh_abort, RKV_SELECT_WAIT_TEST_NS);
#endif
        if (__syncthreads_or(!landed)) {
            // copies that never complete are waited for (bounded) before leaving
            if (threadIdx.x == 0) {
                mbar_drain(&bars[hh & 1], (hh >> 1) & 1);
                if (hh + 1 < nh)
                    mbar_drain(&bars[(hh + 1) & 1], ((hh + 1) >> 1) & 1);
            }
            return false;
        }
        const float *is = stage + (buf * 2) * g.npad;
        const float *rs = stage + (buf * 2 + 1) * g.npad;
        // min-max over the head's n tokens
        float mm[4] = {INFINITY, -INFINITY, INFINITY, -INFINITY};
        for (int j = threadIdx.x; j < n; j += kSelThreads) {
            const float x = is[j], y = rs[j];
            mm[0] = fminf(mm[0], x);
            mm[1] = fmaxf(mm[1], x);
            mm[2] = fminf(mm[2], y);
            mm[3] = fmaxf(mm[3], y);
        }
        block_minmax2<kSelWarps>(mm, fscratch);
        const float imin = mm[0], rmin = mm[2];
        const float irange = mm[1] - mm[0], rrange = mm[3] - mm[2];
        // one division per head; a multiply per token (fp32 rounding differs
        // from a per-token division by at most an ulp, far inside tolerance)
        const float irc = irange > 0.f ? 1.f / irange : 0.f, rrc = rrange > 0.f ? 1.f / rrange : 0.f;
        // normalise, blend, then key (or add to the head sum); the optional
        // score planes get the per-head values
        for (int j = threadIdx.x; j < n; j += kSelThreads) {
            const float ih = (is[j] - imin) * irc;
            const float rh = (rs[j] - rmin) * rrc;
            const float sc = lam * ih - (1.f - lam) * rh;
            if (kShared)
                ssum[j] += sc;
            else
                key[j] = order_key(sc);
            if (a.scores) {
                const size_t o = static_cast<size_t>(e0 + hh) * g.nmax + j;
                a.scores[o] = ih;
                a.scores[plane + o] = rh;
                a.scores[2 * plane + o] = sc;
            }
        }
        __syncthreads(); // staging buffer and min-max scratch free again
        if (kShared && threadIdx.x == 0 && hh + 2 < nh)
            stage_head(hh + 2);
    }
    if (kShared) {
        for (int j = threadIdx.x; j < n; j += kSelThreads)
            key[j] = order_key(ssum[j]);
    }

    if (n <= g.budget) {
        for (int hh = 0; hh < nh; ++hh) {
            int32_t *keep = a.keep + static_cast<size_t>(e0 + hh) * g.budget;
            for (int j = threadIdx.x; j < g.budget; j += kSelThreads)
                keep[j] = j < n ? j : -1;
        }
        if (keep_s) {
            for (int j = threadIdx.x; j < g.budget; j += kSelThreads)
                keep_s[j] = j < n ? j : -1;
            __syncthreads();
        }
        return true;
    }
    __syncthreads(); // keys complete

    const int cand = n - g.w;      // candidates [0, cand); window [cand, n)
    const int take = g.budget - g.w;
    // kept candidates: key > thr, and the first need_eq (by index) with key == thr
    uint32_t thr = 0xFFFFFFFFu;
    uint32_t need_eq = 0;
    if (take > 0) {
        uint32_t prefix = 0, mask = 0;
        uint32_t remaining = static_cast<uint32_t>(take);
        const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
        for (int p = 0; p < 4; ++p) {
            const int shift = 24 - 8 * p;
            uint32_t *H = hist + (p & 1) * 256;
            // warp-aggregated increments: the digits of nearby scores mostly
            // coincide, and per-lane shared atomics on one bin serialise
            for (int base = 0; base < cand; base += kSelThreads) {
                const int j = base + static_cast<int>(threadIdx.x);
                const uint32_t k = j < cand ? key[j] : 0u;
                const bool act = j < cand && (k & mask) == prefix;
                const uint32_t d = act ? ((k >> shift) & 255u) : 256u;
                const uint32_t peers = __match_any_sync(0xffffffffu, d);
                if (act && lane == __ffs(peers) - 1)
                    atomicAdd(&H[d], static_cast<uint32_t>(__popc(peers)));
            }
            __syncthreads();
            if (warp == 0) {
                // lane L owns digits 255-8L .. 248-8L (descending)
                uint32_t c[8], tot = 0;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    c[t] = H[255 - 8 * lane - t];
                    tot += c[t];
                }
                uint32_t incl = tot;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off)
                        incl += y;
                }
                const uint32_t excl = incl - tot;
                // the lane whose range crosses `remaining`
                if (excl < remaining && incl >= remaining) {
                    uint32_t above = excl, digit = 0, rem = 0, done = 0;
                    bool found = false;
#pragma unroll
                    for (int t = 0; t < 8; ++t) {
                        if (!found && above + c[t] >= remaining) {
                            found = true;
                            digit = static_cast<uint32_t>(255 - 8 * lane - t);
                            rem = remaining - above;
                            // the threshold's bin is kept whole: no further digit needed
                            done = (above + c[t] == remaining) ? 1u : 0u;
                        } else if (!found) {
                            above += c[t];
                        }
                    }
                    sh_prefix[p & 1] = prefix | (digit << shift);
                    sh_remaining[p & 1] = rem;
                    sh_done[p & 1] = done;
                }
            } else {
                uint32_t *Hn = hist + ((p + 1) & 1) * 256;
                for (int i = threadIdx.x - 32; i < 256; i += kSelThreads - 32)
                    Hn[i] = 0;
            }
            __syncthreads();
            prefix = sh_prefix[p & 1];
            remaining = sh_remaining[p & 1];
            mask |= 255u << shift;
            if (sh_done[p & 1]) {
                // keep every candidate whose key is at least the bin's prefix
                thr = prefix;
                need_eq = 0xFFFFFFFFu;
                remaining = 0;
                break;
            }
        }
        if (remaining > 0) {
            thr = prefix;
            need_eq = remaining;
        }
    }

    // ---- ascending emission: per-thread contiguous chunks + one packed scan
    const int chunk = (n + kSelThreads - 1) / kSelThreads;
    const int j0 = min(n, static_cast<int>(threadIdx.x) * chunk), j1 = min(n, j0 + chunk);
    uint32_t eq = 0, other = 0; // ties on the threshold / all other kept
    for (int j = j0; j < j1; ++j) {
        if (j >= cand) {
            ++other;
        } else if (take > 0) {
            const uint32_t k = key[j];
            other += k > thr;
            eq += k == thr;
        }
    }
    // n <= 8192: both counts and their prefix sums fit 16 bits
    const uint32_t packed = block_exclusive_scan((eq << 16) | other, uscratch);
    uint32_t eq_seen = packed >> 16;
    int pos = static_cast<int>((packed & 0xFFFFu) + min(eq_seen, need_eq));
    for (int j = j0; j < j1; ++j) {
        bool kept;
        if (j >= cand) {
            kept = true;
        } else if (take > 0) {
            const uint32_t k = key[j];
            if (k > thr) {
                kept = true;
            } else if (k == thr) {
                kept = eq_seen < need_eq;
                ++eq_seen;
            } else {
                kept = false;
            }
        } else {
            kept = false;
        }
        if (kept && pos < g.budget) {
            for (int hh = 0; hh < nh; ++hh)
                a.keep[static_cast<size_t>(e0 + hh) * g.budget + pos] = j;
            if (keep_s)
                keep_s[pos] = j;
            ++pos;
        }
    }
    if (keep_s)
        __syncthreads(); // every kept slot of keep_s written (n > budget fills all budget slots)
    return true;
}

// One CTA per unit (per KV head, or per (layer, sequence) with kShared).
template <bool kShared>
__global__ void __launch_bounds__(kSelThreads) rkv_select_kernel(const SelArgs a)
{
    extern __shared__ uint32_t sel_smem[];
    pdl_wait();
    pdl_trigger();
    select_unit<kShared>(a, kShared ? blockIdx.x * a.g.Hkv : blockIdx.x, sel_smem, nullptr);
}

} // namespace rkv
