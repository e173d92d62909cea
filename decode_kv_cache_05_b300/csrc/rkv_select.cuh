// rkv_select: min-max normalisation, the lambda blend and windowed top-budget
// selection, one CTA per (layer, sequence, KV head).
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
// uint32 keys of S in shared memory; two block-wide scans place ties and the
// kept indices.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

constexpr int kSelThreads = 512;
constexpr int kSelWarps = kSelThreads / 32;

struct SelArgs {
    Geom g;
    const float *imp;
    const float *red;
    int32_t *keep;
    float *scores; // [3][L][B][Hkv][nmax] or null
};

__device__ __forceinline__ uint32_t order_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide reduction helpers (all threads call; result broadcast).
__device__ __forceinline__ float block_min(float v, float *scratch)
{
    for (int off = 16; off > 0; off >>= 1)
        v = fminf(v, __shfl_xor_sync(0xffffffffu, v, off));
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = scratch[0];
    for (int w = 1; w < kSelWarps; ++w)
        r = fminf(r, scratch[w]);
    return r;
}

__device__ __forceinline__ float block_max(float v, float *scratch)
{
    for (int off = 16; off > 0; off >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    __syncthreads();
    if ((threadIdx.x & 31) == 0)
        scratch[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = scratch[0];
    for (int w = 1; w < kSelWarps; ++w)
        r = fmaxf(r, scratch[w]);
    return r;
}

// Exclusive prefix sum over the block (thread order); also returns the total.
__device__ __forceinline__ int block_exclusive_scan(int v, int *scratch, int *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
    for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, off);
        if (lane >= off)
            x += y;
    }
    __syncthreads();
    if (lane == 31)
        scratch[warp] = x;
    __syncthreads();
    int before = 0, all = 0;
    for (int w = 0; w < kSelWarps; ++w) {
        const int s = scratch[w];
        before += w < warp ? s : 0;
        all += s;
    }
    *total = all;
    return before + x - v;
}

__global__ void __launch_bounds__(kSelThreads) rkv_select_kernel(const SelArgs a)
{
    extern __shared__ uint32_t sel_smem[];
    uint32_t *key = sel_smem;                               // [npad]
    uint32_t *hist = key + a.g.npad;                        // [256]
    float *fscratch = reinterpret_cast<float *>(hist + 256); // [kSelWarps]
    int *iscratch = reinterpret_cast<int *>(fscratch + kSelWarps);
    __shared__ uint32_t sh_prefix, sh_remaining;

    const Geom &g = a.g;
    const int e = blockIdx.x;
    const HeadId id = head_id(g, e);
    int n = g.seq_lens[id.b];
    if (n < 0 || n > g.nmax)
        n = 0; // recorded by rkv_importance / rkv_compact
    const int kb = min(n, g.budget);
    const size_t sbase = static_cast<size_t>(e) * g.npad;
    const float *I = a.imp + sbase;
    const float *R = a.red + sbase;
    int32_t *keep = a.keep + static_cast<size_t>(e) * g.budget;

    // ---- min-max of both scores over the head's n tokens
    float imin = INFINITY, imax = -INFINITY, rmin = INFINITY, rmax = -INFINITY;
    for (int j = threadIdx.x; j < n; j += kSelThreads) {
        const float x = I[j], y = R[j];
        imin = fminf(imin, x);
        imax = fmaxf(imax, x);
        rmin = fminf(rmin, y);
        rmax = fmaxf(rmax, y);
    }
    imin = block_min(imin, fscratch);
    imax = block_max(imax, fscratch);
    rmin = block_min(rmin, fscratch);
    rmax = block_max(rmax, fscratch);
    const float irange = imax - imin, rrange = rmax - rmin;
    const float lam = g.lam;

    // ---- normalise, blend, keys (and the optional score planes)
    const size_t plane = static_cast<size_t>(g.L) * g.B * g.Hkv * g.nmax;
    for (int j = threadIdx.x; j < n; j += kSelThreads) {
        const float ih = irange > 0.f ? (I[j] - imin) / irange : 0.f;
        const float rh = rrange > 0.f ? (R[j] - rmin) / rrange : 0.f;
        const float s = lam * ih - (1.f - lam) * rh;
        key[j] = order_key(s);
        if (a.scores) {
            const size_t o = static_cast<size_t>(e) * g.nmax + j;
            a.scores[o] = ih;
            a.scores[plane + o] = rh;
            a.scores[2 * plane + o] = s;
        }
    }

    if (n <= g.budget) {
        for (int j = threadIdx.x; j < g.budget; j += kSelThreads)
            keep[j] = j < n ? j : -1;
        return;
    }

    const int cand = n - g.w;      // candidates [0, cand); window [cand, n)
    const int take = g.budget - g.w;
    uint32_t thr = 0xFFFFFFFFu;    // keys > thr are kept; `need_eq` keys == thr by index
    int need_eq = 0;
    if (take > 0) {
        uint32_t prefix = 0, mask = 0;
        uint32_t remaining = static_cast<uint32_t>(take);
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = threadIdx.x; i < 256; i += kSelThreads)
                hist[i] = 0;
            __syncthreads();
            for (int j = threadIdx.x; j < cand; j += kSelThreads) {
                const uint32_t k = key[j];
                if ((k & mask) == prefix)
                    atomicAdd(&hist[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (threadIdx.x < 32) {
                // lane L owns digits 255-8L .. 248-8L (descending)
                const int lane = threadIdx.x;
                uint32_t c[8], tot = 0;
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    c[t] = hist[255 - 8 * lane - t];
                    tot += c[t];
                }
                uint32_t incl = tot;
                for (int off = 1; off < 32; off <<= 1) {
                    const uint32_t y = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off)
                        incl += y;
                }
                const uint32_t excl = incl - tot;
                // the lane whose range crosses `remaining`
                if (excl < remaining && incl >= remaining) {
                    uint32_t above = excl;
                    int t = 0;
                    for (; t < 8; ++t) {
                        if (above + c[t] >= remaining)
                            break;
                        above += c[t];
                    }
                    const uint32_t digit = static_cast<uint32_t>(255 - 8 * lane - t);
                    sh_prefix = prefix | (digit << shift);
                    sh_remaining = remaining - above;
                }
            }
            __syncthreads();
            prefix = sh_prefix;
            remaining = sh_remaining;
            mask |= 255u << shift;
            __syncthreads();
        }
        thr = prefix;
        need_eq = static_cast<int>(remaining);
    }

    // ---- ascending emission: per-thread contiguous chunks + two scans
    const int chunk = (n + kSelThreads - 1) / kSelThreads;
    const int j0 = min(n, threadIdx.x * chunk), j1 = min(n, j0 + chunk);
    int eq = 0, gt = 0, win = 0;
    for (int j = j0; j < j1; ++j) {
        if (j >= cand) {
            ++win;
        } else if (take > 0) {
            const uint32_t k = key[j];
            gt += k > thr;
            eq += k == thr;
        }
    }
    int tmp;
    const int eq_before = block_exclusive_scan(eq, iscratch, &tmp);
    const int eq_kept = max(0, min(eq, need_eq - eq_before));
    const int mine = gt + eq_kept + win;
    const int pos0 = block_exclusive_scan(mine, iscratch, &tmp);
    int pos = pos0, eq_seen = eq_before;
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
        if (kept && pos < g.budget)
            keep[pos++] = j;
    }
}

} // namespace rkv
