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
// Design: one cluster of C CTAs per head, each CTA owning a contiguous range
// of key rows. A 256-byte key row is read by 16 threads (16 bytes each).
//   pass 1  partial S over the CTA's rows (fp32), reduced in shared memory;
//           the C partials are summed through DSMEM after a cluster barrier;
//   pass 2  the same rows again (now mostly L2 hits): k_i . S per row, reduced
//           over the row's 16 threads with shuffles, then R_i.
// The inverse norms come from rkv_importance.
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

} // namespace rkv
