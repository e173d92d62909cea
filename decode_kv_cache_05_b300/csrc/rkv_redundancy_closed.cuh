// rkv_redundancy, closed form: the same mean pairwise key cosine as the dense
// Gram, from the exact rank-one identity
//     sum_{j != i} cos(k_i, k_j) = k^_i . (sum_j k^_j) - |k^_i|^2,
// with k^ = k / |k| (a zero key has k^ = 0, hence cosine 0 with every key), so
//     R_i = (inv_i * (k_i . S) - [k_i != 0]) / (N - 1),   S = sum_j inv_j k_j.
// R-KV scores redundancy by the cosine similarity of key vectors (hotdry.top
// blog, R-KV section); the identity turns the N x N x d contraction into two
// N x d passes over the keys, so the step becomes bound by HBM instead of by
// the tensor cores.
//
// Three kernels, a cluster of C CTAs per head, each CTA owning a contiguous
// range of key rows; the inverse norms come from rkv_importance.
//   rkv_redundancy_closed_pkernel (the default for heads of up to 8 x 160
//     keys): persistent clusters walking the heads, the rows of the next head
//     brought into shared memory by TMA while this head's passes run (below).
//   rkv_redundancy_closed_res_kernel (a build option): the CTA's rows stream in
//     once (16 threads per 256-byte row) and stay in shared memory; partial S
//     over them, the C partials summed through DSMEM after a cluster barrier,
//     then k_i . S from the resident rows (shuffle-reduced over the row's 16
//     threads) and R_i. HBM reads K once.
//   rkv_redundancy_closed_kernel (longer heads, whose share of rows does not
//     fit shared memory): the same two passes straight from global memory; the
//     second pass reads K again (measured on B300: from HBM, not L2, once many
//     heads are in flight).
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

constexpr int kCfThreads = 256;
constexpr int kCfRowsPerPass = kCfThreads / 16; // rows one sweep of the CTA covers
constexpr int kCfUnroll = 4;                    // sweeps with loads in flight together

struct CfArgs {
    Geom g;
    const uint8_t *k;
    const float *inv;
    float *out_red;
    int rows_per_cta; // a multiple of kCfRowsPerPass
};

__global__ void __launch_bounds__(kCfThreads) rkv_redundancy_closed_kernel(const CfArgs a)
{
    __shared__ float red_s[kCfRowsPerPass][kHeadDim]; // pass-1 partials per row group
    __shared__ float sw_part[kHeadDim];               // this CTA's partial S (read by peers)
    __shared__ float sw[kHeadDim];                    // S of the head
    __shared__ int32_t table_s[kMaxSeq / kBlock];

    const Geom &g = a.g;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int e = blockIdx.x / csize;
    const HeadId id = head_id(g, e);
    pdl_wait();
    pdl_trigger();
    int n = g.seq_lens[id.b];
    if (n < 0 || n > g.nmax)
        n = 0; // rkv_importance records the error
    if (!triggered(g, n))
        n = 0; // left for a later call
    const int r_begin = min(n, static_cast<int>(crank) * a.rows_per_cta);
    const int r_end = min(n, r_begin + a.rows_per_cta);
    const int cg = threadIdx.x & 15;  // 16-byte column group: columns [8 cg, 8 cg + 8)
    const int rg = threadIdx.x >> 4;  // row within a sweep
    const float *inv = a.inv + static_cast<size_t>(e) * g.npad;

    bool ok = true;
    if (g.paged) {
        const int nblk = (n + kBlock - 1) / kBlock;
        for (int i = threadIdx.x; i < nblk; i += kCfThreads) {
            const int p = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + i];
            ok = ok && p >= 0 && p < g.num_blocks; // rkv_importance records the error
            table_s[i] = p;
        }
    }
    ok = __syncthreads_and(ok);
    auto row_ptr = [&](int t) -> const uint4 * {
        size_t off;
        if (!g.paged)
            off = (static_cast<size_t>(e) * g.nmax + t) * (kHeadDim * 2);
        else
            off = ((((static_cast<size_t>(id.l) * g.num_blocks + table_s[t / kBlock]) * kBlock + (t % kBlock)) *
                        g.Hkv + id.h) * (kHeadDim * 2));
        return reinterpret_cast<const uint4 *>(a.k + off) + cg;
    };
    auto widen = [](const uint4 &v, float (&x)[8]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            x[2 * t] = __uint_as_float(w[t] << 16);
            x[2 * t + 1] = __uint_as_float(w[t] & 0xFFFF0000u);
        }
    };

    // ---- pass 1: partial S = sum_j inv_j k_j over this CTA's rows
    float acc[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        acc[c] = 0.f;
    if (ok) {
        for (int base = r_begin; base < r_end; base += kCfRowsPerPass * kCfUnroll) {
            uint4 v[kCfUnroll];
            float w[kCfUnroll];
#pragma unroll
            for (int u = 0; u < kCfUnroll; ++u) {
                const int j = base + u * kCfRowsPerPass + rg;
                w[u] = 0.f;
                if (j < r_end) {
                    v[u] = __ldg(row_ptr(j));
                    w[u] = __ldg(inv + j);
                }
            }
#pragma unroll
            for (int u = 0; u < kCfUnroll; ++u) {
                if (w[u] != 0.f) {
                    float x[8];
                    widen(v[u], x);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        acc[c] = fmaf(w[u], x[c], acc[c]);
                }
            }
        }
    }
#pragma unroll
    for (int c = 0; c < 8; ++c)
        red_s[rg][8 * cg + c] = acc[c];
    __syncthreads();
    if (threadIdx.x < kHeadDim) {
        float s = 0.f;
#pragma unroll
        for (int r = 0; r < kCfRowsPerPass; ++r)
            s += red_s[r][threadIdx.x];
        sw_part[threadIdx.x] = s;
    }
    cluster_sync(); // every CTA's partial S is visible
    if (threadIdx.x < kHeadDim) {
        float s = 0.f;
        for (uint32_t c = 0; c < csize; ++c)
            s += ld_dsmem_f32(&sw_part[threadIdx.x], c);
        sw[threadIdx.x] = s;
    }
    cluster_arrive(); // done reading the peers' partials
    __syncthreads();

    // ---- pass 2: R_j = (inv_j * (k_j . S) - [k_j != 0]) / (N - 1)
    float s8[8];
#pragma unroll
    for (int c = 0; c < 8; ++c)
        s8[c] = sw[8 * cg + c];
    const float denom = n > 1 ? 1.f / static_cast<float>(n - 1) : 0.f;
    if (ok) {
        for (int base = r_begin; base < r_end; base += kCfRowsPerPass * kCfUnroll) {
            uint4 v[kCfUnroll];
#pragma unroll
            for (int u = 0; u < kCfUnroll; ++u) {
                const int j = base + u * kCfRowsPerPass + rg;
                if (j < r_end)
                    v[u] = __ldg(row_ptr(j));
            }
#pragma unroll
            for (int u = 0; u < kCfUnroll; ++u) {
                const int j = base + u * kCfRowsPerPass + rg;
                float d = 0.f;
                if (j < r_end) {
                    float x[8];
                    widen(v[u], x);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        d = fmaf(x[c], s8[c], d);
                }
                // the 16 threads of a row are 16 consecutive lanes
#pragma unroll
                for (int off = 8; off > 0; off >>= 1)
                    d += __shfl_xor_sync(0xffffffffu, d, off);
                if (cg == 0 && j < r_end) {
                    const float iv = __ldg(inv + j);
                    a.out_red[static_cast<size_t>(e) * g.npad + j] =
                        (iv * d - (iv > 0.f ? 1.f : 0.f)) * denom;
                }
            }
        }
    }
    cluster_wait(); // peers are done reading this CTA's partial
}

// ---------------------------------------------------------------------------
// Resident-rows form. Pass 1 streams the CTA's rows from global memory with
// 16-byte loads (16 threads per 256-byte row, four row sweeps in flight per
// thread), adds inv_j k_j into the thread's part of S, and also stores each
// row into shared memory; pass 2 then reads the rows from shared memory, so
// HBM sees K once. Dynamic shared memory: rows [rows_per_cta][256 B], their
// inverse norms [rows_per_cta], per-warp partial S [8][128], this CTA's S
// [128] (read by the peers) and the head's S [128].
constexpr int kCfResThreads = 256;

__host__ __device__ constexpr size_t cf_res_smem_bytes(int rows_per_cta)
{
    return static_cast<size_t>(rows_per_cta) * (kHeadDim * 2 + 4) + (8 * 128 + 128 + 128) * 4 + 16;
}

__global__ void __launch_bounds__(kCfResThreads) rkv_redundancy_closed_res_kernel(const CfArgs a)
{
    extern __shared__ __align__(16) uint8_t cf_smem[];
    __shared__ int32_t table_s[kMaxSeq / kBlock];
    const Geom &g = a.g;
    const int R = a.rows_per_cta;
    uint8_t *rows_s = cf_smem;                                              // [R][256]
    float *inv_s = reinterpret_cast<float *>(cf_smem + static_cast<size_t>(R) * 256); // [R]
    float *part = inv_s + R;                                                // [8][128]
    float *s_cta = part + 8 * 128;                                          // [128]
    float *s_all = s_cta + 128;                                             // [128]

    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int e = blockIdx.x / csize;
    const HeadId id = head_id(g, e);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    int n = g.seq_lens[id.b];
    if (n < 0 || n > g.nmax)
        n = 0; // rkv_importance records the error
    if (!triggered(g, n))
        n = 0; // left for a later call
    const int r_begin = min(n, static_cast<int>(crank) * R);
    const int r_end = min(n, r_begin + R);
    const int nr = r_end - r_begin;
    const float *inv = a.inv + static_cast<size_t>(e) * g.npad;
    bool ok = true;
    if (g.paged) {
        const int nblk = (n + kBlock - 1) / kBlock;
        for (int i = threadIdx.x; i < nblk; i += kCfResThreads) {
            const int p = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + i];
            ok = ok && p >= 0 && p < g.num_blocks; // rkv_importance records the error
            table_s[i] = p;
        }
    }
    ok = __syncthreads_and(ok);
    auto row_ptr = [&](int j) -> const uint4 * {
        size_t off;
        if (!g.paged)
            off = (static_cast<size_t>(e) * g.nmax + j) * (kHeadDim * 2);
        else
            off = ((((static_cast<size_t>(id.l) * g.num_blocks + table_s[j / kBlock]) * kBlock + (j % kBlock)) *
                        g.Hkv + id.h) * (kHeadDim * 2));
        return reinterpret_cast<const uint4 *>(a.k + off);
    };

    // ---- pass 1: stream the rows in, keep them, and add inv_j k_j into S
    const int c = threadIdx.x & 15, rg = threadIdx.x >> 4; // column chunk, row within a sweep of 16
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        acc[q] = 0.f;
    if (ok) {
        for (int base = 0; base < nr; base += 16 * kCfUnroll) {
            uint4 v[kCfUnroll];
            float w[kCfUnroll];
#pragma unroll
            for (int u = 0; u < kCfUnroll; ++u) {
                const int t = base + u * 16 + rg;
                w[u] = 0.f;
                if (t < nr) {
                    v[u] = __ldg(row_ptr(r_begin + t) + c);
                    w[u] = __ldg(inv + r_begin + t);
                }
            }
#pragma unroll
            for (int u = 0; u < kCfUnroll; ++u) {
                const int t = base + u * 16 + rg;
                if (t < nr) {
                    *reinterpret_cast<uint4 *>(rows_s + static_cast<size_t>(t) * 256 + c * 16) = v[u];
                    if (c == 0)
                        inv_s[t] = w[u];
                    const uint32_t wd[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = fmaf(w[u], __uint_as_float(wd[q] << 16), acc[2 * q]);
                        acc[2 * q + 1] = fmaf(w[u], __uint_as_float(wd[q] & 0xFFFF0000u), acc[2 * q + 1]);
                    }
                }
            }
        }
    }
    // lanes l and l ^ 16 share a chunk; then the 8 warps, in warp order
#pragma unroll
    for (int q = 0; q < 8; ++q)
        acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], 16);
    if (lane < 16) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
            part[warp * 128 + c * 8 + q] = acc[q];
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        float sum = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8)
            sum += part[w8 * 128 + threadIdx.x];
        s_cta[threadIdx.x] = sum;
    }
    cluster_sync(); // every CTA's partial S is visible
    if (threadIdx.x < 128) {
        float sum = 0.f;
        for (uint32_t r = 0; r < csize; ++r)
            sum += ld_dsmem_f32(&s_cta[threadIdx.x], r);
        s_all[threadIdx.x] = sum;
    }
    cluster_arrive(); // done reading the peers' partials
    __syncthreads();

    // ---- pass 2: R_j = (inv_j * (k_j . S) - [k_j != 0]) / (N - 1), from the resident rows
    float s8[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        s8[q] = s_all[8 * c + q];
    const float denom = n > 1 ? 1.f / static_cast<float>(n - 1) : 0.f;
    if (ok) {
        for (int base = 0; base < nr; base += 16) {
            const int t = base + rg;
            float d = 0.f;
            if (t < nr) {
                const uint4 v = *reinterpret_cast<const uint4 *>(rows_s + static_cast<size_t>(t) * 256 + c * 16);
                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    d = fmaf(__uint_as_float(wd[q] << 16), s8[2 * q], d);
                    d = fmaf(__uint_as_float(wd[q] & 0xFFFF0000u), s8[2 * q + 1], d);
                }
            }
#pragma unroll
            for (int off = 8; off > 0; off >>= 1)
                d += __shfl_xor_sync(0xffffffffu, d, off);
            if (c == 0 && t < nr) {
                const float iv = inv_s[t];
                a.out_red[static_cast<size_t>(e) * g.npad + r_begin + t] = (iv * d - (iv > 0.f ? 1.f : 0.f)) * denom;
            }
        }
    }
    cluster_wait(); // peers are done reading this CTA's partial
}

// ---------------------------------------------------------------------------
// Persistent form of the resident-rows kernel. One cluster of C CTAs walks a
// sequence of heads (head = cluster id + k * clusters), each CTA owning the
// same R-row slice of every head. A producer warp brings the slice into one
// of two shared-memory buffers with TMA (one 2D box on the contiguous layout,
// one 4D box per 16-token block on the paged one; no swizzle: rows are 256
// contiguous bytes as the passes read them) together with its inverse norms
// (a bulk copy), so the next head's rows load while this head is computed.
// Eight compute warps run the two passes of the kernel above from the buffer;
// the CTAs' partial S travel by asynchronous remote stores that count their
// bytes on the receiver's mbarrier (two slots alternating by head, as the
// persistent importance kernel exchanges its statistics) instead of cluster
// barriers, which the producer warp, running ahead, could not join. A slot of
// head k is rewritten only for head k + 2, after its owner has received every
// CTA's head k + 1 partial, which each CTA sends only after reading head k's.
constexpr int kCfpThreads = 288;      // 8 compute warps + 1 producer warp
constexpr int kCfpMaxRows = 160;      // rows per CTA and head
constexpr int kCfpRowBuf = kCfpMaxRows * kHeadDim * 2;

struct CfpSmem {
    static constexpr int kRows = 0;                                      // [2][kCfpMaxRows][256 B]
    static constexpr int kInv = 2 * kCfpRowBuf;                          // float[2][kCfpMaxRows]
    static constexpr int kPart = kInv + 2 * kCfpMaxRows * 4;             // float[8][128]
    static constexpr int kSlots = kPart + 8 * 128 * 4;                   // float[2][8 ranks][128]
    static constexpr int kSAll = kSlots + 2 * 8 * 128 * 4;               // float[128]
    static constexpr int kBars = kSAll + 128 * 4;                        // full[2], empty[2], stat[2]
    static constexpr int kMisc = kBars + 8 * 6;                          // uint32[2]
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;
};

__global__ void __launch_bounds__(kCfpThreads, 2)
    rkv_redundancy_closed_pkernel(const __grid_constant__ CUtensorMap kmap, const CfArgs a)
{
    extern __shared__ uint8_t cfp_raw[];
    uint8_t *smem = align1024(cfp_raw);
    uint8_t *rows_s = smem + CfpSmem::kRows;
    float *inv_s = reinterpret_cast<float *>(smem + CfpSmem::kInv);
    float *part = reinterpret_cast<float *>(smem + CfpSmem::kPart);
    float *slots = reinterpret_cast<float *>(smem + CfpSmem::kSlots);
    float *s_all = reinterpret_cast<float *>(smem + CfpSmem::kSAll);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + CfpSmem::kBars);
    uint64_t *full = bars, *empty = bars + 2, *stat = bars + 4;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + CfpSmem::kMisc);
    volatile uint32_t *abort = misc;

    const Geom &g = a.g;
    const int R = a.rows_per_cta;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int cid = blockIdx.x / csize, nclusters = gridDim.x / csize;
    const long long heads = static_cast<long long>(g.L) * g.B * g.Hkv;
    const int r_begin = static_cast<int>(crank) * R;

    if (threadIdx.x == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(&full[b], 1);
            mbar_init(&empty[b], 8); // one arrival per compute warp
            mbar_init(&stat[b], 1);  // one local arrival announcing the bytes of every CTA's partial
        }
        misc[0] = 0;
        fence_barrier_init();
    }
    cluster_sync(); // every CTA's barriers are initialised before any remote arrival
    pdl_wait();
    pdl_trigger();

    // length of head e (0: nothing to do for this call); the same in every role and CTA
    auto head_len = [&](long long e) {
        const HeadId id = head_id(g, static_cast<int>(e));
        int n = __ldg(g.seq_lens + id.b);
        if (n < 0 || n > g.nmax)
            n = 0; // rkv_importance records the error
        if (!triggered(g, n))
            n = 0; // left for a later call
        return n;
    };

    if (warp == 8) {
        // ---------------------------------------------------------- producer
        if (lane == 0)
            prefetch_tmap(&kmap);
        int k = 0;
        bool ok = true;
        for (long long e = cid; ok && e < heads; e += nclusters) {
            const int n = head_len(e);
            if (n == 0)
                continue;
            const int b = k & 1;
            if (k >= 2 && !mbar_wait(&empty[b], ((k >> 1) - 1) & 1, abort)) {
                ok = false;
                break;
            }
            const int nr = max(0, min(R, n - r_begin)); // rows of this CTA's slice that hold keys
            const int nblk = (nr + kBlock - 1) / kBlock;
            const int ninv = nr > 0 ? min(R, g.npad - r_begin) : 0;
            const uint32_t kbytes = nr == 0 ? 0u : (g.paged ? nblk * kBlock * 256u : static_cast<uint32_t>(R) * 256u);
            if (lane == 0)
                mbar_expect_tx(&full[b], kbytes + ninv * 4u);
            __syncwarp();
            if (nr > 0) {
                uint8_t *dst = rows_s + b * kCfpRowBuf;
                const HeadId id = head_id(g, static_cast<int>(e));
                if (!g.paged) {
                    if (lane == 0)
                        tma_load_2d(dst, &kmap, 0, static_cast<int>(e) * g.nmax + r_begin, &full[b]);
                } else if (lane < nblk) {
                    int phys = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + r_begin / kBlock + lane];
                    if (phys < 0 || phys >= g.num_blocks)
                        phys = 0; // rkv_importance records the error; the head's results are unspecified
                    tma_load_4d(dst + lane * (kBlock * 256), &kmap, 0, id.h, 0, id.l * g.num_blocks + phys,
                                &full[b]);
                }
                if (lane == 0)
                    bulk_load(inv_s + b * kCfpMaxRows, a.inv + static_cast<size_t>(e) * g.npad + r_begin, ninv * 4u,
                              &full[b]);
            }
            __syncwarp();
            ++k;
        }
        if (*abort && lane == 0) {
            for (int c = max(0, k - 2); c < k; ++c)
                mbar_drain(&full[c & 1], (c >> 1) & 1);
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------------- compute
        const int c = threadIdx.x & 15, rg = threadIdx.x >> 4; // column chunk; row within a 16-row sweep
        int k = 0;
        for (long long e = cid; e < heads; e += nclusters) {
            const int n = head_len(e);
            if (n == 0)
                continue;
            const int b = k & 1, sb = k & 1;
            const int nr = max(0, min(R, n - r_begin));
            const bool landed = mbar_wait(&full[b], (k >> 1) & 1, abort);
            const uint8_t *rows = rows_s + b * kCfpRowBuf;
            const float *iv = inv_s + b * kCfpMaxRows;
            // ---- pass 1: this CTA's part of S = sum_j inv_j k_j
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                acc[q] = 0.f;
            if (landed) {
                for (int t = rg; t < nr; t += 16) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(rows + t * 256 + c * 16);
                    const float w = iv[t];
                    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[2 * q] = fmaf(w, __uint_as_float(wd[q] << 16), acc[2 * q]);
                        acc[2 * q + 1] = fmaf(w, __uint_as_float(wd[q] & 0xFFFF0000u), acc[2 * q + 1]);
                    }
                }
            }
            // lanes l and l ^ 16 share a chunk; then the 8 warps, in warp order
#pragma unroll
            for (int q = 0; q < 8; ++q)
                acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], 16);
            if (lane < 16) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    part[warp * 128 + c * 8 + q] = acc[q];
            }
            named_sync(1, 256);
            // ---- exchange: this CTA's partial into every CTA of the cluster (bytes counted there)
            if (threadIdx.x < 128) {
                float sum = 0.f;
#pragma unroll
                for (int w8 = 0; w8 < 8; ++w8)
                    sum += part[w8 * 128 + threadIdx.x];
                const float sum1 = __shfl_down_sync(0xffffffffu, sum, 1);
                if (threadIdx.x == 0)
                    mbar_expect_tx(&stat[sb], csize * 128u * 4u);
                if ((threadIdx.x & 1) == 0) {
                    const float *dst = slots + (sb * 8 + crank) * 128 + threadIdx.x;
                    for (uint32_t r = 0; r < csize; ++r)
                        st_async_v2(cluster_addr(dst, r), sum, sum1, cluster_addr(&stat[sb], r));
                }
                // S of the head: every CTA's partial, in rank order
                const bool got = mbar_wait(&stat[sb], (k >> 1) & 1, abort);
                float S = 0.f;
                if (got)
                    for (uint32_t r = 0; r < csize; ++r)
                        S += slots[(sb * 8 + r) * 128 + threadIdx.x];
                s_all[threadIdx.x] = S;
            }
            named_sync(1, 256);
            // ---- pass 2: R_j = (inv_j * (k_j . S) - [k_j != 0]) / (N - 1), from the buffer
            float s8[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                s8[q] = s_all[8 * c + q];
            const float denom = n > 1 ? 1.f / static_cast<float>(n - 1) : 0.f;
            if (landed && !*abort) {
                for (int base = 0; base < nr; base += 16) {
                    const int t = base + rg;
                    float d = 0.f;
                    if (t < nr) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(rows + t * 256 + c * 16);
                        const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            d = fmaf(__uint_as_float(wd[q] << 16), s8[2 * q], d);
                            d = fmaf(__uint_as_float(wd[q] & 0xFFFF0000u), s8[2 * q + 1], d);
                        }
                    }
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1)
                        d += __shfl_xor_sync(0xffffffffu, d, off);
                    if (c == 0 && t < nr) {
                        const float w = iv[t];
                        a.out_red[static_cast<size_t>(e) * g.npad + r_begin + t] =
                            (w * d - (w > 0.f ? 1.f : 0.f)) * denom;
                    }
                }
            }
            // the buffer goes back to the producer
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&empty[b]);
            ++k;
        }
    }
    cluster_sync(); // no remote store is still addressed to a CTA that exits
}

} // namespace rkv
