// rkv_importance: attention importance of every cached key.
//
// R-KV scores a token's importance from the attention that the most recent
// queries pay to it (hotdry.top blog, R-KV section, second step; the R-KV
// review page, "How R-KV decides what to drop": the local window supplies the
// queries). For a (layer, sequence, KV head) with N keys and the w*G window
// query rows of its GQA group:
//     I_j = (1 / (w*G)) * sum_r softmax_j(q_r . k_j / sqrt(d)).
//
// Design (one cluster of C CTAs per head, each CTA owns T key tiles of 128):
//   warp 0      TMA producer: the head's query block once, then K tiles through
//               a STAGES-deep shared-memory ring (128B-swizzled, K-major).
//   warp 1      TMEM owner and MMA issuer: S^T = K_tile . Q^T with
//               tcgen05.mma (M = 128 keys, N = NR query rows, K = d = 128),
//               each tile into its own NR TMEM columns; all logits of the
//               CTA's keys stay in TMEM.
//   warps 2..   epilogue, one warpgroup per 32 query rows, one key (TMEM
//               lane) per thread:
//               - while tiles stream in, computes 1/|k_j| from the staged tile
//                 (for rkv_redundancy) and, per query row, online softmax
//                 statistics of its keys (running max m, sum of 2^(s - m));
//               - combines them over the CTA, then over the cluster in one
//                 DSMEM exchange: row max M_r and row sum L_r;
//               - I_j = sum_r 2^(s_rj - M_r) / (L_r * rows), a thread-local
//                 sum over the logits still held in TMEM (log2-domain logits
//                 s = q.k * log2(e)/sqrt(d)).
// K is read from HBM exactly once; no logit leaves the SM. One cluster
// barrier publishes the statistics; a second, split around the last pass,
// keeps each CTA's shared memory alive until its peers have read it.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

// Threads: producer warp, MMA warp, then one epilogue warpgroup per 32 query
// rows (NR / 32 warpgroups).
__host__ __device__ constexpr int imp_threads(int nr) { return 64 + 4 * nr; }
constexpr int kImpMaxTiles = 16; // tiles per CTA (TMEM: T * NR <= 512)
constexpr int kMaxCluster = 8;   // CTAs per head

struct ImpArgs {
    Geom g;
    float *out_imp;
    float *out_inv;
    int tiles_per_cta;
    uint32_t tmem_cols;
    float scale_log2; // log2(e) / sqrt(d)
};

template <int NR, int STAGES>
struct ImpSmem {
    static constexpr int kQ = 0;
    static constexpr int kK = NR * 256;
    static constexpr int kBars = kK + STAGES * kTileBytes;
    static constexpr int kNumBars = 2 * STAGES + 1 + kImpMaxTiles;
    static constexpr int kRed = kBars + 8 * kNumBars;     // float[8][NR]: per-warp max, sum
    static constexpr int kPart = kRed + 8 * 4 * NR;       // float[kImpMaxTiles][128]: second half-row sums
    static constexpr int kCtaM = kPart + (NR > 32 ? kImpMaxTiles * 128 * 4 : 0); // float[NR]
    static constexpr int kCtaL = kCtaM + 4 * NR;          // float[NR]
    static constexpr int kVec = kCtaL + 4 * NR;           // float[NR]: row max (log2 domain)
    static constexpr int kWgt = kVec + 4 * NR;            // float[NR]: 1 / (row sum * rows)
    static constexpr int kMisc = kWgt + 4 * NR;           // uint32[2]
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;          // + alignment slack
};

// Inverse L2 norm (fp32) of row `r` of a 128-row K tile staged as two
// 128B-swizzled halves.
__device__ __forceinline__ float tile_row_inv_norm(const uint8_t *tile, int r)
{
    float ss = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint8_t *row = tile + half * kHalfBytes + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(row + ((c ^ (r & 7)) << 4));
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const float lo = __uint_as_float(w[t] << 16);
                const float hi = __uint_as_float(w[t] & 0xFFFF0000u);
                ss = fmaf(lo, lo, ss);
                ss = fmaf(hi, hi, ss);
            }
        }
    }
    return ss > 0.f ? rsqrtf(ss) : 0.f;
}

template <int NR, int STAGES>
__global__ void __launch_bounds__(imp_threads(NR), 1)
    rkv_importance_kernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                          const ImpArgs a)
{
    using SM = ImpSmem<NR, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *q_s = smem + SM::kQ;
    uint8_t *k_s = smem + SM::kK;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBars);
    uint64_t *full = bars;
    uint64_t *empty = bars + STAGES;
    uint64_t *qfull = bars + 2 * STAGES;
    uint64_t *done = qfull + 1;
    float *red = reinterpret_cast<float *>(smem + SM::kRed);
    float *cta_m = reinterpret_cast<float *>(smem + SM::kCtaM);
    float *cta_l = reinterpret_cast<float *>(smem + SM::kCtaL);
    float *vec = reinterpret_cast<float *>(smem + SM::kVec);
    float *wgt = reinterpret_cast<float *>(smem + SM::kWgt);
    float *part = reinterpret_cast<float *>(smem + SM::kPart);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + SM::kMisc);
    volatile uint32_t *abort = misc + 1;

    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int e = blockIdx.x / csize; // one cluster per head
    const HeadId id = head_id(g, e);

    pdl_wait();
    pdl_trigger();
    int n = g.seq_lens[id.b];
    if (n < 0 || n > g.nmax) {
        if (threadIdx.x == 0 && crank == 0 && id.l == 0 && id.h == 0)
            record_error(kErrDevice);
        n = 0;
    }
    if (!triggered(g, n))
        n = 0; // left for a later call
    const int tiles = (n + kTileKeys - 1) / kTileKeys;
    const int t0 = static_cast<int>(crank) * a.tiles_per_cta;
    const int my_tiles = max(0, min(t0 + a.tiles_per_cta, tiles) - t0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 4); // MMA commit + one arrival per epilogue warp
        }
        mbar_init(qfull, 1);
        for (int i = 0; i < kImpMaxTiles; ++i)
            mbar_init(&done[i], 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc[0], a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&qmap);
        }
        if (my_tiles > 0) {
            if (lane == 0) {
                const int qrow = ((id.l * g.B + id.b) * g.Hq + id.h * g.G) * g.w;
                mbar_expect_tx(qfull, NR * 256);
                tma_load_2d(q_s, &qmap, 0, qrow, qfull);
                tma_load_2d(q_s + NR * 128, &qmap, 64, qrow, qfull);
            }
            const int nblk_seq = (n + kBlock - 1) / kBlock;
            for (int i = 0; i < my_tiles; ++i) {
                const int s = i % STAGES;
                const int tile = t0 + i;
                // paged: this lane's pool block, looked up before the ring wait
                int phys = 0;
                if (g.paged && lane < 16) {
                    const int lb = min(tile * 8 + (lane >> 1), nblk_seq - 1);
                    phys = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + lb];
                    if (phys < 0 || phys >= g.num_blocks) {
                        record_error(kErrDevice);
                        phys = 0;
                    }
                }
                if (i >= STAGES && !mbar_wait(&empty[s], ((i / STAGES) - 1) & 1, abort))
                    break;
                if (lane == 0)
                    mbar_expect_tx(&full[s], kTileBytes);
                __syncwarp();
                uint8_t *dst = k_s + s * kTileBytes;
                if (!g.paged) {
                    if (lane < 2) {
                        const int row = e * g.nmax + tile * kTileKeys;
                        tma_load_2d(dst + lane * kHalfBytes, &kmap, lane * 64, row, &full[s]);
                    }
                } else if (lane < 16) {
                    const int blk8 = lane >> 1, half = lane & 1;
                    tma_load_4d(dst + half * kHalfBytes + blk8 * (kBlock * 128), &kmap, half * 64, id.h, 0,
                                id.l * g.num_blocks + phys, &full[s]);
                }
                __syncwarp();
            }
        }
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        if (lane == 0 && my_tiles > 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, NR);
            bool ok = mbar_wait(qfull, 0, abort);
            for (int i = 0; ok && i < my_tiles; ++i) {
                const int s = i % STAGES;
                if (!mbar_wait(&full[s], (i / STAGES) & 1, abort))
                    break;
                tc_fence_after();
                const uint32_t kbase = smem_u32(k_s + s * kTileBytes);
                const uint32_t qbase = smem_u32(q_s);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint64_t ad = sdesc_sw128(kbase + (k >> 2) * kHalfBytes + (k & 3) * 32);
                    const uint64_t bd = sdesc_sw128(qbase + (k >> 2) * (NR * 128) + (k & 3) * 32);
                    umma_bf16(tmem + i * NR, ad, bd, idesc, k > 0 ? 1u : 0u);
                }
                umma_commit(&empty[s]);
                umma_commit(&done[i]);
            }
        }
        __syncwarp();
    }

    // ------------------------------------------------------------ epilogue
    constexpr int kEpi = 4 * NR;              // epilogue threads
    const bool epi = warp >= 2;
    const int q4 = warp & 3;                  // TMEM lane quarter of this warp
    const int wg = (warp - 2) >> 2;           // epilogue warpgroup: query rows [32 wg, 32 wg + 32)
    const int key_in_tile = q4 * 32 + lane;   // = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
    const int et = threadIdx.x - 64;          // epilogue thread index
    const size_t obase = static_cast<size_t>(e) * g.npad;
    const float c2 = a.scale_log2;            // logits are handled in the log2 domain

    if (epi) {
        // Online softmax statistics of this thread's keys (one per tile), per
        // query row: running max m and sum l of 2^(s - m).
        float m[32], l[32];
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.f;
        }
        for (int i = 0; i < my_tiles; ++i) {
            const int s = i % STAGES;
            const int j = (t0 + i) * kTileKeys + key_in_tile;
            if (wg == 0) {
                // the first warpgroup also takes the inverse key norms from the staged tile
                if (!mbar_wait(&full[s], (i / STAGES) & 1, abort))
                    break;
                const float inv = tile_row_inv_norm(k_s + s * kTileBytes, key_in_tile);
                if (j < n)
                    a.out_inv[obase + j] = inv;
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&empty[s]);
            }
            if (!mbar_wait(&done[i], 0, abort))
                break;
            tc_fence_after();
            float v[32];
            tmem_ld32(tmem + lane_addr + i * NR + wg * 32, v);
            tmem_wait_ld();
            if (j < n) {
#pragma unroll
                for (int r = 0; r < 32; ++r) {
                    const float x = v[r] * c2;
                    const float d = x - m[r];
                    const float t = ex2_approx(-fabsf(d));
                    // d > 0: a new max (rescale the sum); else add 2^(x - m)
                    l[r] = d > 0.f ? fmaf(l[r], t, 1.f) : l[r] + t;
                    m[r] = fmaxf(m[r], x);
                }
            }
        }
        // combine the statistics of the warp's 32 keys of each row: the row
        // maxima by a reduce-scatter (lane r gets row r), then each sum
        // rescaled to its row's maximum and reduce-scattered the same way
        float mx[32];
#pragma unroll
        for (int r = 0; r < 32; ++r)
            mx[r] = m[r];
        const float mw = warp_reduce_scatter32<true>(mx, lane);
#pragma unroll
        for (int r = 0; r < 32; ++r) {
            const float M = __shfl_sync(0xffffffffu, mw, r);
            l[r] = M == -INFINITY ? 0.f : l[r] * ex2_approx(m[r] - M);
        }
        const float lw = warp_reduce_scatter32<false>(l, lane);
        red[q4 * NR + wg * 32 + lane] = mw;
        red[(4 + q4) * NR + wg * 32 + lane] = lw;
        named_sync(1, kEpi);
        if (et < NR) {
            float mm = -INFINITY;
#pragma unroll
            for (int w = 0; w < 4; ++w)
                mm = fmaxf(mm, red[w * NR + et]);
            float ll = 0.f;
            if (mm != -INFINITY) {
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    ll += red[(4 + w) * NR + et] * ex2_approx(red[w * NR + et] - mm);
            }
            cta_m[et] = mm;
            cta_l[et] = ll;
        }
    }
    cluster_sync(); // (1) every CTA's row statistics are visible
    if (epi && et < NR) {
        float mm = -INFINITY;
        float mc[kMaxCluster], lc[kMaxCluster];
#pragma unroll
        for (uint32_t c = 0; c < kMaxCluster; ++c) {
            if (c < csize) {
                mc[c] = ld_dsmem_f32(&cta_m[et], c);
                lc[c] = ld_dsmem_f32(&cta_l[et], c);
                mm = fmaxf(mm, mc[c]);
            }
        }
        float ll = 0.f;
        if (mm != -INFINITY) {
#pragma unroll
            for (uint32_t c = 0; c < kMaxCluster; ++c)
                if (c < csize)
                    ll += lc[c] * ex2_approx(mc[c] - mm);
        }
        vec[et] = mm;
        wgt[et] = (et < g.rows && ll > 0.f) ? 1.f / (ll * static_cast<float>(g.rows)) : 0.f;
    }
    cluster_arrive(); // (2) this CTA is done reading its peers' shared memory
    if (epi) {
        // one decision for all epilogue warps, so that none waits alone below
        const bool go = !named_sync_or(1, kEpi, *abort != 0);
        // the weighted sum over this warpgroup's 32 rows of key j of tile i
        auto half_row_sum = [&](int i) {
            float v[32];
            tmem_ld32(tmem + lane_addr + i * NR + wg * 32, v);
            tmem_wait_ld();
            float acc = 0.f;
#pragma unroll
            for (int r = 0; r < 32; ++r) {
                const float w = wgt[wg * 32 + r];
                const float p = ex2_approx(fmaf(v[r], c2, -vec[wg * 32 + r]));
                acc = w != 0.f ? fmaf(p, w, acc) : acc; // padding rows never reach the sum
            }
            return acc;
        };
        if (go && NR > 32 && wg == 1) {
            for (int i = 0; i < my_tiles; ++i)
                part[i * 128 + key_in_tile] = half_row_sum(i);
        }
        if (NR > 32)
            named_sync(1, kEpi);
        if (go && wg == 0) {
            for (int i = 0; i < my_tiles; ++i) {
                const int j = (t0 + i) * kTileKeys + key_in_tile;
                float acc = half_row_sum(i);
                if (NR > 32)
                    acc += part[i * 128 + key_in_tile];
                if (j < n)
                    a.out_imp[obase + j] = acc;
            }
        }
    }
    cluster_wait(); // (2) peers are done reading this CTA's shared memory
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

} // namespace rkv
