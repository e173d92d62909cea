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
//   warps 2..   epilogue, NR/16 warpgroups, one key (TMEM lane) per thread:
//               - while tiles stream in, each warpgroup keeps online softmax
//                 statistics of its 16 query rows: the first tile's logit is
//                 a row's reference and every later logit adds 2^(s - ref)
//                 (log2-domain logits s = q.k * log2(e)/sqrt(d)); a spread
//                 above 2^64 is redone exactly from the logits in TMEM;
//               - the warpgroups take turns, tile by tile, at the inverse key
//                 norms 1/|k_j| (for rkv_redundancy) from the staged tile;
//               - the statistics are combined over the CTA, then over the
//                 cluster in one DSMEM exchange: row max M_r and row sum L_r;
//               - I_j = sum_r 2^(s_rj - M_r - log2(L_r * rows)), again tile
//                 by tile in turns, over the logits still held in TMEM.
// K is read from HBM exactly once; no logit leaves the SM. One cluster
// barrier publishes the statistics; a second, split around the last pass,
// keeps each CTA's shared memory alive until its peers have read it.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

// Threads: producer warp, MMA warp, then one epilogue warpgroup per 16 query
// rows (NR / 16 warpgroups).
__host__ __device__ constexpr int imp_threads(int nr) { return 64 + 8 * nr; }
// Largest spread (log2 domain) between a row's reference logit and a later
// one that the one-pass statistics accept; a row sum then stays below 2^80.
constexpr float kImpSpread = 64.f;
constexpr int kImpMaxTiles = 16; // tiles per CTA (TMEM: T * NR <= 512)
constexpr int kMaxCluster = 8;   // CTAs per head

struct ImpArgs {
    Geom g;
    float *out_imp;
    float *out_inv;
    float *out_red;     // closed-form redundancy (persistent kernel with kClosed only)
    const uint8_t *k;   // the K cache itself (kClosed: key rows read again for k_i . S)
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
    static constexpr int kRed = (kBars + 8 * kNumBars + 15) & ~15; // float[8][NR]: per-warp max, sum
    static constexpr int kCtaM = kRed + 8 * 4 * NR;       // float[NR]
    static constexpr int kCtaL = kCtaM + 4 * NR;          // float[NR]
    static constexpr int kShift = kCtaL + 4 * NR;         // float[NR]: M_r + log2(L_r * rows)
    static constexpr int kMisc = kShift + 4 * NR;         // uint32[2]
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024;          // + alignment slack
    static_assert(kShift % 16 == 0, "shift[] is read as float4");
};

// Inverse L2 norm (fp32) of row `r` of a 128-row K tile staged as two
// 128B-swizzled halves.
// Four partial sums (one per 32-bit word of each 16-byte chunk), so that the
// 128 FMAs form four short dependency chains instead of one long one.
__device__ __forceinline__ float tile_row_inv_norm(const uint8_t *tile, int r)
{
    float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const uint8_t *row = tile + half * kHalfBytes + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint4 v = *reinterpret_cast<const uint4 *>(row + ((c ^ (r & 7)) << 4));
            s0 = fma_sq_bf16x2(v.x, s0);
            s1 = fma_sq_bf16x2(v.y, s1);
            s2 = fma_sq_bf16x2(v.z, s2);
            s3 = fma_sq_bf16x2(v.w, s3);
        }
    }
    const float ss = (s0 + s1) + (s2 + s3);
    return ss > 0.f ? rsqrtf(ss) : 0.f;
}

template <int NR, int STAGES>
__global__ void __launch_bounds__(imp_threads(NR), NR == 32 ? 2 : 1)
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
    float *shift = reinterpret_cast<float *>(smem + SM::kShift);
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
    constexpr int kEW = NR / 16;              // epilogue warpgroups
    constexpr int kEpi = 128 * kEW;           // epilogue threads
    const bool epi = warp >= 2;
    const int q4 = warp & 3;                  // TMEM lane quarter of this warp
    const int wg = (warp - 2) >> 2;           // statistics of query rows [16 wg, 16 wg + 16)
    const int key_in_tile = q4 * 32 + lane;   // = TMEM lane
    const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
    const int et = threadIdx.x - 64;          // epilogue thread index
    const size_t obase = static_cast<size_t>(e) * g.npad;
    const float c2 = a.scale_log2;            // logits are handled in the log2 domain

    if (epi) {
        // Statistics of this thread's key, per query row: the reference ref
        // (the row's logit in the CTA's first tile) and l = sum of 2^(s - ref).
        float ref[16], l[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            ref[r] = -INFINITY;
            l[r] = 0.f;
        }
        float spread = -INFINITY; // largest s - ref met
        int seen = 0;
        for (int i = 0; i < my_tiles; ++i) {
            const int s = i % STAGES;
            const int j = (t0 + i) * kTileKeys + key_in_tile;
            if (i % kEW == wg) {
                // this warpgroup's turn at the tile's inverse key norms
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
            float v[16];
            tmem_ld16(tmem + lane_addr + i * NR + wg * 16, v);
            tmem_wait_ld();
            if (j < n) {
                if (i == 0) {
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        ref[r] = v[r] * c2;
                        l[r] = 1.f;
                    }
                } else {
#pragma unroll
                    for (int r = 0; r < 16; ++r) {
                        const float d = fmaf(v[r], c2, -ref[r]);
                        l[r] += ex2_approx(d);
                        spread = fmaxf(spread, d);
                    }
                }
            }
            seen = i + 1;
        }
        if (__any_sync(0xffffffffu, spread > kImpSpread)) {
            // a logit far above its row's reference: exact two-pass
            // statistics over the warp's logits, still held in TMEM
            const int tiles_read = __reduce_min_sync(0xffffffffu, seen);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                ref[r] = -INFINITY;
                l[r] = 0.f;
            }
            for (int pass = 0; pass < 2; ++pass) {
                for (int i = 0; i < tiles_read; ++i) {
                    float v[16];
                    tmem_ld16(tmem + lane_addr + i * NR + wg * 16, v);
                    tmem_wait_ld();
                    if ((t0 + i) * kTileKeys + key_in_tile < n) {
#pragma unroll
                        for (int r = 0; r < 16; ++r) {
                            if (pass == 0)
                                ref[r] = fmaxf(ref[r], v[r] * c2);
                            else
                                l[r] += ex2_approx(fmaf(v[r], c2, -ref[r]));
                        }
                    }
                }
            }
        }
        // combine the warp's 32 keys of each row: the row maxima of the
        // references by a reduce-scatter (lanes r and r + 16 get row r), then
        // each sum rescaled to its row's maximum and reduce-scattered the same way
        float mx[16];
#pragma unroll
        for (int r = 0; r < 16; ++r)
            mx[r] = ref[r];
        const float mw = warp_reduce_scatter<16, true>(mx, lane);
#pragma unroll
        for (int r = 0; r < 16; ++r) {
            const float M = __shfl_sync(0xffffffffu, mw, r);
            l[r] = M == -INFINITY ? 0.f : l[r] * ex2_approx(ref[r] - M);
        }
        const float lw = warp_reduce_scatter<16, false>(l, lane);
        if (lane < 16) {
            red[q4 * NR + wg * 16 + lane] = mw;
            red[(4 + q4) * NR + wg * 16 + lane] = lw;
        }
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
        // p_rj / rows = 2^(s_rj - shift_r); padding rows get +inf (p = 0)
        shift[et] = (et < g.rows && ll > 0.f) ? mm + lg2_approx(ll * static_cast<float>(g.rows)) : INFINITY;
    }
    cluster_arrive(); // (2) this CTA is done reading its peers' shared memory
    if (epi) {
        // one decision for all epilogue warps, so that none waits alone below
        const bool go = !named_sync_or(1, kEpi, *abort != 0);
        if (go) {
            // I_j for the keys of every kEW-th tile, all NR rows in this thread
            for (int i = wg; i < my_tiles; i += kEW) {
                const int j = (t0 + i) * kTileKeys + key_in_tile;
                float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f; // four short add chains
#pragma unroll
                for (int c = 0; c < NR / 32; ++c) {
                    float v[32];
                    tmem_ld32(tmem + lane_addr + i * NR + c * 32, v);
                    tmem_wait_ld();
                    const float4 *sh4 = reinterpret_cast<const float4 *>(shift + c * 32);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 sh = sh4[q];
                        acc0 += ex2_approx(fmaf(v[4 * q + 0], c2, -sh.x));
                        acc1 += ex2_approx(fmaf(v[4 * q + 1], c2, -sh.y));
                        acc2 += ex2_approx(fmaf(v[4 * q + 2], c2, -sh.z));
                        acc3 += ex2_approx(fmaf(v[4 * q + 3], c2, -sh.w));
                    }
                }
                if (j < n)
                    a.out_imp[obase + j] = (acc0 + acc1) + (acc2 + acc3);
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

// ---------------------------------------------------------------------------
// Persistent form of the same computation. Each cluster of C CTAs walks a
// sequence of heads (head = cluster id + k * clusters); every CTA owns the same
// T-tile slice of each head. What the one-shot kernel above pays per head --
// CTA launch, TMEM allocation, the first memory round trip, and a ring that
// drains while softmax statistics cross the cluster -- is overlapped here:
//   - the producer keeps streaming K tiles (and the next head's queries)
//     through the ring while the epilogue finishes the previous head;
//   - logits of consecutive heads go to two TMEM halves (when 2 * T * NR <=
//     512), so the MMA of head k+1 runs during the epilogue of head k;
//   - the per-row (max, sum) statistics are exchanged by asynchronous remote
//     shared-memory stores that count their bytes on the receiver's mbarrier
//     (two slots, alternating by head) instead of cluster-wide barriers, so
//     the producer and MMA warps never stop for the exchange and no sender
//     waits on a memory fence.
// A slot of head k is rewritten only for head k + 2, after its owner has
// published head k + 1's statistics, which it does only after reading head
// k's: two slots suffice without a further handshake. The epilogue is the
// one-shot kernel's (statistics by row halves, inverse norms and the final
// pass by tile turns).
//
// With kClosed the same pass over K also yields the redundancy R, by the
// exact rank-one identity (the R-KV review page, "How R-KV decides what to
// drop", credits a fused redundancy kernel and batched scoring for keeping the
// cost low; the blog's R-KV section defines redundancy from key cosines):
//     R_i = (inv_i * (k_i . S) - [k_i != 0]) / (N - 1),   S = sum_j inv_j k_j.
//   - pass A: the warpgroup whose turn it is at a tile's inverse norms also
//     adds the tile's inv_j k_j into S, from the tile already staged in shared
//     memory (each thread one 16-byte column chunk of 16 rows);
//   - the CTAs' partial S travel with the softmax statistics (same slots
//     protocol, same mbarrier, 512 more bytes per CTA);
//   - pass C: next to I_j, each thread forms k_j . S from its key row read
//     again from global memory -- the CTA staged that row a few microseconds
//     earlier, so the read is served by L2 and HBM sees K once.
template <int NR, bool kClosed = false>
struct ImpPSmem {
    static constexpr int kEW = NR / 16;                                // epilogue warpgroups
    static constexpr int kStages = NR == 32 ? (kClosed ? 5 : 6) : 5;
    static constexpr int kQ = 0;                                       // 2 x [NR rows][128] bf16 (2 halves)
    static constexpr int kK = kQ + 2 * NR * 256;                       // ring
    static constexpr int kSlots = kK + kStages * kTileBytes;           // float[2][kMaxCluster][NR][2]: (m, l)
    static constexpr int kRed = kSlots + 2 * kMaxCluster * 2 * NR * 4; // float[8][NR]
    static constexpr int kShift = kRed + 8 * NR * 4;                   // float[NR]
    static constexpr int kSSlots = kShift + NR * 4;                    // kClosed: float[2][kMaxCluster][128]
    static constexpr int kSRed = kSSlots + (kClosed ? 2 * kMaxCluster * 128 * 4 : 0); // float[4 kEW][128]
    static constexpr int kInvS = kSRed + (kClosed ? 4 * kEW * 128 * 4 : 0);          // float[kEW][2][128]
    static constexpr int kSFin = kInvS + (kClosed ? kEW * 2 * 128 * 4 : 0);          // float[128]: S
    static constexpr int kBars = kSFin + (kClosed ? 128 * 4 : 0);
    // full, empty per stage; qfull, qempty, tfree, stat per buffer; done per buffer x tile
    static constexpr int kNumBars = 2 * kStages + 2 * 4 + 2 * kImpMaxTiles;
    static constexpr int kMisc = kBars + 8 * kNumBars;
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024; // + alignment slack
    static_assert(kShift % 16 == 0, "shift[] is read as float4");
    static_assert(kSFin % 16 == 0, "S is read as float4");
    static_assert(kAlloc <= 232448, "importance kernel exceeds 227 KB of shared memory");
};

template <int NR, bool kClosed = false>
__global__ void __launch_bounds__(imp_threads(NR), 1)
    rkv_importance_pkernel(const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap qmap,
                           const ImpArgs a)
{
    using SM = ImpPSmem<NR, kClosed>;
    constexpr int STAGES = SM::kStages;
    constexpr int kEW = NR / 16;    // epilogue warpgroups
    constexpr int kEpi = 128 * kEW; // epilogue threads
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    uint8_t *q_s = smem + SM::kQ;
    uint8_t *k_s = smem + SM::kK;
    float *slots = reinterpret_cast<float *>(smem + SM::kSlots);
    float *red = reinterpret_cast<float *>(smem + SM::kRed);
    float *shift = reinterpret_cast<float *>(smem + SM::kShift);
    float *sslots = reinterpret_cast<float *>(smem + SM::kSSlots); // kClosed only
    float *sred = reinterpret_cast<float *>(smem + SM::kSRed);
    float *invs = reinterpret_cast<float *>(smem + SM::kInvS);
    float *sfin = reinterpret_cast<float *>(smem + SM::kSFin);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + SM::kBars);
    uint64_t *full = bars;
    uint64_t *empty = full + STAGES;
    uint64_t *qfull = empty + STAGES;   // [2]
    uint64_t *qempty = qfull + 2;       // [2]
    uint64_t *tfree = qempty + 2;       // [2]: a TMEM half free again (epilogue done with it)
    uint64_t *stat = tfree + 2;         // [2]: every CTA's statistics of the head landed here
    uint64_t *done = stat + 2;          // [2][kImpMaxTiles]
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + SM::kMisc);
    volatile uint32_t *abort = misc + 1;

    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int cid = blockIdx.x / csize, nclusters = gridDim.x / csize;
    const long long heads = static_cast<long long>(g.L) * g.B * g.Hkv;
    const int T = a.tiles_per_cta;
    const int t0 = static_cast<int>(crank) * T;
    const bool dbl = a.tmem_cols >= static_cast<uint32_t>(2 * T * NR); // two TMEM halves

    // per-head geometry; every role derives it the same way
    auto head_len = [&](long long e, bool record) {
        const HeadId id = head_id(g, static_cast<int>(e));
        int n = __ldg(g.seq_lens + id.b);
        if (n < 0 || n > g.nmax) {
            if (record && crank == 0 && id.l == 0 && id.h == 0)
                record_error(kErrDevice);
            n = 0;
        }
        if (!triggered(g, n))
            n = 0; // left for a later call
        return n;
    };
    auto my_tiles_of = [&](int n) { return max(0, min(t0 + T, (n + kTileKeys - 1) / kTileKeys) - t0); };

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 4); // MMA commit + the warpgroup taking the tile's inverse norms
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&qfull[b], 1);
            mbar_init(&qempty[b], 1);
            mbar_init(&tfree[b], kEpi / 32);
            mbar_init(&stat[b], 1); // one local arrival announcing the bytes of every CTA's pairs
        }
        for (int i = 0; i < 2 * kImpMaxTiles; ++i)
            mbar_init(&done[i], 1);
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc[0], a.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    cluster_sync(); // every CTA's barriers are initialised before any remote arrival
    tc_fence_after();
    const uint32_t tmem = misc[0];
    pdl_wait();    // inputs of earlier work in the stream are complete from here on
    pdl_trigger();

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(&kmap);
            prefetch_tmap(&qmap);
        }
        int kcnt = 0, qk = 0; // K tiles issued; heads with tiles in this CTA
        bool ok = true;
        for (long long e = cid; ok && e < heads; e += nclusters) {
            const int n = head_len(e, false);
            const int mt = my_tiles_of(n);
            if (mt == 0)
                continue; // nothing of this head lives in this CTA
            const HeadId id = head_id(g, static_cast<int>(e));
            const int qb = qk & 1;
            if (qk >= 2 && !mbar_wait(&qempty[qb], ((qk >> 1) - 1) & 1, abort))
                break;
            ++qk;
            if (lane == 0) {
                const int qrow = ((id.l * g.B + id.b) * g.Hq + id.h * g.G) * g.w;
                uint8_t *qd = q_s + qb * NR * 256;
                mbar_expect_tx(&qfull[qb], NR * 256);
                tma_load_2d(qd, &qmap, 0, qrow, &qfull[qb]);
                tma_load_2d(qd + NR * 128, &qmap, 64, qrow, &qfull[qb]);
            }
            const int nblk_seq = (n + kBlock - 1) / kBlock;
            for (int i = 0; i < mt; ++i, ++kcnt) {
                const int s = kcnt % STAGES;
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
                if (kcnt >= STAGES && !mbar_wait(&empty[s], ((kcnt / STAGES) - 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                if (lane == 0)
                    mbar_expect_tx(&full[s], kTileBytes);
                __syncwarp();
                uint8_t *dst = k_s + s * kTileBytes;
                if (!g.paged) {
                    if (lane < 2)
                        tma_load_2d(dst + lane * kHalfBytes, &kmap, lane * 64,
                                    static_cast<int>(e) * g.nmax + tile * kTileKeys, &full[s]);
                } else if (lane < 16) {
                    const int blk8 = lane >> 1, half = lane & 1;
                    tma_load_4d(dst + half * kHalfBytes + blk8 * (kBlock * 128), &kmap, half * 64, id.h, 0,
                                id.l * g.num_blocks + phys, &full[s]);
                }
                __syncwarp();
            }
        }
        if (*abort && lane == 0) {
            for (int c = max(0, kcnt - STAGES); c < kcnt; ++c)
                mbar_drain(&full[c % STAGES], (c / STAGES) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, NR);
            int kcnt = 0, qk = 0, issued = 0;
            bool ok = true;
            for (long long e = cid; ok && e < heads; e += nclusters) {
                const int n = head_len(e, false);
                const int mt = my_tiles_of(n);
                if (mt == 0)
                    continue;
                const int qb = qk & 1, hb = dbl ? (qk & 1) : 0;
                // the TMEM half of head qk - 2 (qk - 1 when single-buffered), released by the epilogue
                const int back = dbl ? 2 : 1;
                if (qk >= back && !mbar_wait(&tfree[hb], ((qk - back) / back) & 1, abort))
                    break;
                if (!mbar_wait(&qfull[qb], (qk >> 1) & 1, abort))
                    break;
                ++qk;
                tc_fence_after();
                const uint32_t qbase = smem_u32(q_s + qb * NR * 256);
                for (int i = 0; i < mt; ++i, ++kcnt) {
                    const int s = kcnt % STAGES;
                    if (!mbar_wait(&full[s], (kcnt / STAGES) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t kbase = smem_u32(k_s + s * kTileBytes);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint64_t ad = sdesc_sw128(kbase + (k >> 2) * kHalfBytes + (k & 3) * 32);
                        const uint64_t bd = sdesc_sw128(qbase + (k >> 2) * (NR * 128) + (k & 3) * 32);
                        umma_bf16(tmem + (hb * T + i) * NR, ad, bd, idesc, k > 0 ? 1u : 0u);
                    }
                    umma_commit(&empty[s]);
                    umma_commit(&done[hb * kImpMaxTiles + i]);
                    issued = 1;
                }
                if (ok)
                    umma_commit(&qempty[qb]);
            }
            if (*abort && issued) {
                // wait (bounded) for the last MMAs before TMEM is freed
                const int s = (kcnt - 1) % STAGES;
                mbar_drain(&empty[s], ((kcnt - 1) / STAGES) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int q4 = warp & 3;                  // TMEM lane quarter of this warp
        const int wg = (warp - 2) >> 2;           // statistics of query rows [16 wg, 16 wg + 16)
        const int key_in_tile = q4 * 32 + lane;   // = TMEM lane
        const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
        const int et = threadIdx.x - 64;
        const float c2 = a.scale_log2;
        int kcnt = 0, qk = 0, hk = 0; // K tiles consumed; heads with tiles here; heads exchanged
        bool ok = true;
        for (long long e = cid; ok && e < heads; e += nclusters) {
            const int n = head_len(e, true);
            if (n == 0)
                continue; // no CTA of the cluster has work on this head
            // a CTA without tiles of the head still takes part in the exchange
            const int mt = my_tiles_of(n);
            const int hb = dbl ? (qk & 1) : 0, par = dbl ? ((qk >> 1) & 1) : (qk & 1);
            const uint32_t cols = tmem + lane_addr + hb * T * NR; // this head's logits
            const size_t obase = static_cast<size_t>(e) * g.npad;
            // ---- pass A: inverse norms (by turns), statistics of 16 rows per thread
            float ref[16], l[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                ref[r] = -INFINITY;
                l[r] = 0.f;
            }
            float spread = -INFINITY;
            int seen = 0;
            // kClosed: this thread's part of S = sum_j inv_j k_j -- the dims of
            // column chunk (key_in_tile & 15), over rows (key_in_tile >> 4) + 8m
            float sacc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                sacc[q] = 0.f;
            int turn = 0;
            for (int i = 0; i < mt; ++i) {
                const int kc = kcnt + i;
                const int s = kc % STAGES;
                const int j = (t0 + i) * kTileKeys + key_in_tile;
                if (i % kEW == wg) {
                    bool landed = mbar_wait(&full[s], (kc / STAGES) & 1, abort);
                    if (kClosed) // one decision for the warpgroup, which meets at a barrier below
                        landed = !named_sync_or(2 + wg, 128, !landed);
                    if (!landed) {
                        ok = false;
                        break;
                    }
                    const float inv = tile_row_inv_norm(k_s + s * kTileBytes, key_in_tile);
                    if (j < n)
                        a.out_inv[obase + j] = inv;
                    if (kClosed) {
                        // the tile's inv_j k_j into S, from the staged tile (keys past n excluded)
                        float *ib = invs + (wg * 2 + (turn & 1)) * 128;
                        ib[key_in_tile] = inv;
                        named_sync(2 + wg, 128);
                        const int c = key_in_tile & 15, rg = key_in_tile >> 4;
                        const uint8_t *half = k_s + s * kTileBytes + (c >> 3) * kHalfBytes;
                        const int off = ((c & 7) ^ rg) << 4; // 128-byte swizzle: rows rg + 8m share r & 7 = rg
                        const int rows = min(kTileKeys, n - (t0 + i) * kTileKeys);
#pragma unroll 4
                        for (int m = 0; m < 16; ++m) {
                            const int r = rg + 8 * m;
                            if (r < rows) {
                                const uint4 v = *reinterpret_cast<const uint4 *>(half + r * 128 + off);
                                const float w = ib[r];
                                const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                                for (int t = 0; t < 4; ++t) {
                                    sacc[2 * t] = fmaf(w, __uint_as_float(wd[t] << 16), sacc[2 * t]);
                                    sacc[2 * t + 1] = fmaf(w, __uint_as_float(wd[t] & 0xFFFF0000u), sacc[2 * t + 1]);
                                }
                            }
                        }
                        ++turn;
                    }
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&empty[s]);
                }
                if (!mbar_wait(&done[hb * kImpMaxTiles + i], par, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                float v[16];
                tmem_ld16(cols + i * NR + wg * 16, v);
                tmem_wait_ld();
                if (j < n) {
                    if (i == 0) {
#pragma unroll
                        for (int r = 0; r < 16; ++r) {
                            ref[r] = v[r] * c2;
                            l[r] = 1.f;
                        }
                    } else {
#pragma unroll
                        for (int r = 0; r < 16; ++r) {
                            const float d = fmaf(v[r], c2, -ref[r]);
                            l[r] += ex2_approx(d);
                            spread = fmaxf(spread, d);
                        }
                    }
                }
                seen = i + 1;
            }
            kcnt += mt;
            // every epilogue warp takes the same decision to go on
            ok = !named_sync_or(1, kEpi, !ok || *abort);
            if (!ok)
                break;
            if (__any_sync(0xffffffffu, spread > kImpSpread)) {
                // a logit far above its row's reference: exact two-pass statistics
                const int tiles_read = __reduce_min_sync(0xffffffffu, seen);
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    ref[r] = -INFINITY;
                    l[r] = 0.f;
                }
                for (int pass = 0; pass < 2; ++pass) {
                    for (int i = 0; i < tiles_read; ++i) {
                        float v[16];
                        tmem_ld16(cols + i * NR + wg * 16, v);
                        tmem_wait_ld();
                        if ((t0 + i) * kTileKeys + key_in_tile < n) {
#pragma unroll
                            for (int r = 0; r < 16; ++r) {
                                if (pass == 0)
                                    ref[r] = fmaxf(ref[r], v[r] * c2);
                                else
                                    l[r] += ex2_approx(fmaf(v[r], c2, -ref[r]));
                            }
                        }
                    }
                }
            }
            // the warp's 32 keys of each row: reduce-scatters (lanes r and r + 16 get row r)
            float mx[16];
#pragma unroll
            for (int r = 0; r < 16; ++r)
                mx[r] = ref[r];
            const float mw = warp_reduce_scatter<16, true>(mx, lane);
#pragma unroll
            for (int r = 0; r < 16; ++r) {
                const float M = __shfl_sync(0xffffffffu, mw, r);
                l[r] = M == -INFINITY ? 0.f : l[r] * ex2_approx(ref[r] - M);
            }
            const float lw = warp_reduce_scatter<16, false>(l, lane);
            if (lane < 16) {
                red[q4 * NR + wg * 16 + lane] = mw;
                red[(4 + q4) * NR + wg * 16 + lane] = lw;
            }
            if (kClosed) {
                // lanes l and l ^ 16 hold the same column chunk (chunk = lane & 15)
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    sacc[q] += __shfl_xor_sync(0xffffffffu, sacc[q], 16);
                if (lane < 16) {
                    float4 *dst = reinterpret_cast<float4 *>(sred + (warp - 2) * 128 + 8 * lane);
                    dst[0] = make_float4(sacc[0], sacc[1], sacc[2], sacc[3]);
                    dst[1] = make_float4(sacc[4], sacc[5], sacc[6], sacc[7]);
                }
            }
            named_sync(1, kEpi);
            const int sb = hk & 1; // exchange slot of this head
            constexpr int kExThreads = kClosed ? (NR > 128 ? NR : 128) : NR;
            if (et < kExThreads) {
                float mm = -INFINITY, ll = 0.f;
                if (et < NR) {
#pragma unroll
                    for (int w = 0; w < 4; ++w)
                        mm = fmaxf(mm, red[w * NR + et]);
                    if (mm != -INFINITY) {
#pragma unroll
                        for (int w = 0; w < 4; ++w)
                            ll += red[(4 + w) * NR + et] * ex2_approx(red[w * NR + et] - mm);
                    }
                }
                // this CTA's part of S, dim et (the epilogue warps' partials in warp order)
                float sc = 0.f;
                if (kClosed) {
#pragma unroll
                    for (int w = 0; w < 4 * kEW; ++w)
                        sc += sred[w * 128 + et];
                }
                // publish (m, l) of row et, and S, into every CTA of the cluster (bytes counted there)
                if (et == 0)
                    mbar_expect_tx(&stat[sb], csize * (NR * 8 + (kClosed ? 128 * 4 : 0)));
                if (et < NR) {
                    const float *pair = slots + ((sb * kMaxCluster + crank) * NR + et) * 2;
                    for (uint32_t c = 0; c < csize; ++c)
                        st_async_v2(cluster_addr(pair, c), mm, ll, cluster_addr(&stat[sb], c));
                }
                if (kClosed) {
                    const float sc1 = __shfl_down_sync(0xffffffffu, sc, 1);
                    if ((et & 1) == 0) {
                        const float *sp = sslots + (sb * kMaxCluster + crank) * 128 + et;
                        for (uint32_t c = 0; c < csize; ++c)
                            st_async_v2(cluster_addr(sp, c), sc, sc1, cluster_addr(&stat[sb], c));
                    }
                }
                // combine the cluster's statistics of row et once they have all landed here
                const bool landed = mbar_wait(&stat[sb], (hk >> 1) & 1, abort);
                if (et < NR) {
                    float gm = -INFINITY, gl = 0.f;
                    if (landed) {
                        const float *got = slots + (sb * kMaxCluster * NR + et) * 2;
                        for (uint32_t c = 0; c < csize; ++c)
                            gm = fmaxf(gm, got[c * NR * 2]);
                        if (gm != -INFINITY)
                            for (uint32_t c = 0; c < csize; ++c)
                                gl += got[c * NR * 2 + 1] * ex2_approx(got[c * NR * 2] - gm);
                    }
                    // p_rj / rows = 2^(s_rj - shift_r); padding rows get +inf (p = 0)
                    shift[et] =
                        (et < g.rows && gl > 0.f) ? gm + lg2_approx(gl * static_cast<float>(g.rows)) : INFINITY;
                }
                if (kClosed) {
                    // S, summed over the cluster in rank order
                    float S = 0.f;
                    if (landed) {
                        const float *got = sslots + sb * kMaxCluster * 128 + et;
                        for (uint32_t c = 0; c < csize; ++c)
                            S += got[c * 128];
                    }
                    sfin[et] = S;
                }
            }
            ok = !named_sync_or(1, kEpi, *abort != 0);
            ++hk;
            // ---- pass C: I_j from the logits still in TMEM, every kEW-th tile
            if (ok) {
                for (int i = wg; i < mt; i += kEW) {
                    const int j = (t0 + i) * kTileKeys + key_in_tile;
                    // kClosed: this key's row, read again below for k_j . S, on its way
                    // into L1 while the I_j sum runs
                    const uint8_t *krow = nullptr;
                    if (kClosed && j < n) {
                        if (!g.paged) {
                            krow = a.k + (static_cast<size_t>(e) * g.nmax + j) * 256;
                        } else {
                            const HeadId id = head_id(g, static_cast<int>(e));
                            const int phys = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + j / kBlock];
                            if (phys >= 0 && phys < g.num_blocks) // else recorded by the producer
                                krow = a.k + ((((static_cast<size_t>(id.l) * g.num_blocks + phys) * kBlock + j % kBlock) *
                                                   g.Hkv + id.h) * 256);
                        }
                        if (krow) {
                            asm volatile("prefetch.global.L1 [%0];" ::"l"(krow) : "memory");
                            asm volatile("prefetch.global.L1 [%0];" ::"l"(krow + 128) : "memory");
                        }
                    }
                    float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f; // four short add chains
#pragma unroll
                    for (int c = 0; c < NR / 32; ++c) {
                        float v[32];
                        tmem_ld32(cols + i * NR + c * 32, v);
                        tmem_wait_ld();
                        const float4 *sh4 = reinterpret_cast<const float4 *>(shift + c * 32);
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 sh = sh4[q];
                            acc0 += ex2_approx(fmaf(v[4 * q + 0], c2, -sh.x));
                            acc1 += ex2_approx(fmaf(v[4 * q + 1], c2, -sh.y));
                            acc2 += ex2_approx(fmaf(v[4 * q + 2], c2, -sh.z));
                            acc3 += ex2_approx(fmaf(v[4 * q + 3], c2, -sh.w));
                        }
                    }
                    if (j < n)
                        a.out_imp[obase + j] = (acc0 + acc1) + (acc2 + acc3);
                    if (kClosed && j < n) {
                        // k_j . S from the key row, read again through L2 (this CTA staged it
                        // moments ago), then R_j by the rank-one identity
                        const uint4 *row = reinterpret_cast<const uint4 *>(krow);
                        float d0 = 0.f, d1 = 0.f;
                        if (row) {
                            const float4 *s4 = reinterpret_cast<const float4 *>(sfin);
#pragma unroll
                            for (int c = 0; c < 16; ++c) {
                                const uint4 v = __ldg(row + c);
                                const float4 sa = s4[2 * c], sb4 = s4[2 * c + 1];
                                d0 = fmaf(__uint_as_float(v.x << 16), sa.x, d0);
                                d1 = fmaf(__uint_as_float(v.x & 0xFFFF0000u), sa.y, d1);
                                d0 = fmaf(__uint_as_float(v.y << 16), sa.z, d0);
                                d1 = fmaf(__uint_as_float(v.y & 0xFFFF0000u), sa.w, d1);
                                d0 = fmaf(__uint_as_float(v.z << 16), sb4.x, d0);
                                d1 = fmaf(__uint_as_float(v.z & 0xFFFF0000u), sb4.y, d1);
                                d0 = fmaf(__uint_as_float(v.w << 16), sb4.z, d0);
                                d1 = fmaf(__uint_as_float(v.w & 0xFFFF0000u), sb4.w, d1);
                            }
                        }
                        const float iv = a.out_inv[obase + j]; // written by this thread in pass A
                        const float denom = n > 1 ? 1.f / static_cast<float>(n - 1) : 0.f;
                        a.out_red[obase + j] = (iv * (d0 + d1) - (iv > 0.f ? 1.f : 0.f)) * denom;
                    }
                }
            }
            // this TMEM half may be reused (each warp releases its own reads)
            tc_fence_before();
            if (mt > 0) {
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&tfree[hb]);
                ++qk;
            }
        }
    }
    tc_fence_before();
    cluster_sync(); // no remote store or arrival is still addressed to a CTA that exits
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, a.tmem_cols);
    }
}

} // namespace rkv
