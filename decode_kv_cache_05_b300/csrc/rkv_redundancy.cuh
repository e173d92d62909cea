// rkv_redundancy: mean cosine similarity of each key to the head's other keys.
//
// R-KV flags repeated content by the cosine similarity of key vectors
// (hotdry.top blog, R-KV section, first step); the R-KV review page ("How
// R-KV decides what to drop") credits batched redundancy scoring for keeping
// the cost on the decode path low. Definition used here, for a head with N keys:
//     R_i = (1/(N-1)) * sum_{j != i} (k_i . k_j) * inv_i * inv_j,  inv = 1/|k|.
//
// Design: a dense key Gram G = K K^T on the 5th-generation tensor cores, never
// written to HBM. One CTA per (head, pair of 128-row tiles):
//   warp 0      TMA producer: the two row tiles (A operands) plus the head's
//               inverse norms once, then every 128-key column tile (B operand)
//               through a STAGES-deep 128B-swizzled ring.
//   warp 1      TMEM owner / MMA issuer: per column tile, two 128x128x128
//               tcgen05 MMAs (one per row tile) into a double-buffered fp32
//               accumulator (2 buffers x 2 row tiles x 128 columns = 512).
//   warps 2..9  epilogue (one warpgroup per row tile, one row per thread):
//               tcgen05.ld the 128 accumulator columns, fused row mean
//               sum_j G_ij * inv_j with the diagonal and the ragged tail
//               masked, then R_i = sum * inv_i / (N-1).
// The inverse norms come from rkv_importance, which computes them from the
// same staged K tiles.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

constexpr int kRedThreads = 320;
constexpr int kRedStages = 4;

struct RedArgs {
    Geom g;
    const float *inv;
    float *out_red;
    int pairs; // CTAs per head: ceil(ceil(max_seq_len / 128) / 2)
};

struct RedSmem {
    static constexpr int kA = 0;                                   // 2 row tiles
    static constexpr int kB = 2 * kTileBytes;                      // ring
    static constexpr int kInv = kB + kRedStages * kTileBytes;      // float[npad]
    // barriers follow the inverse norms (offset depends on npad)
    static constexpr int kNumBars = 2 * kRedStages + 1 + 2 + 2;
    static int bytes(int npad) { return kInv + npad * 4 + 8 * kNumBars + 16 + 1024; }
};

__global__ void __launch_bounds__(kRedThreads, 1)
    rkv_redundancy_kernel(const __grid_constant__ CUtensorMap kmap, const RedArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x / a.pairs;
    const HeadId id = head_id(g, e);

    int n = g.seq_lens[id.b];
    if (n < 0 || n > g.nmax)
        n = 0; // rkv_importance records the error
    const int tiles = (n + kTileKeys - 1) / kTileKeys;
    const int rt0 = 2 * (blockIdx.x % a.pairs);
    if (rt0 >= tiles)
        return;
    const int nrt = min(2, tiles - rt0);

    uint8_t *a_s = smem + RedSmem::kA;
    uint8_t *b_s = smem + RedSmem::kB;
    float *inv_s = reinterpret_cast<float *>(smem + RedSmem::kInv);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + RedSmem::kInv + g.npad * 4);
    uint64_t *full = bars;
    uint64_t *empty = bars + kRedStages;
    uint64_t *afull = bars + 2 * kRedStages;
    uint64_t *acc_full = afull + 1;
    uint64_t *acc_empty = acc_full + 2;
    uint32_t *misc = reinterpret_cast<uint32_t *>(acc_empty + 2);
    volatile uint32_t *abort = misc + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRedStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(afull, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 8);
        }
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(&misc[0], 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    const int nblk_seq = (n + kBlock - 1) / kBlock;

    // Issue the TMA loads of key tile `tile` into `dst` (one warp; lanes split boxes).
    auto load_tile = [&](uint8_t *dst, int tile, uint64_t *bar) {
        if (!g.paged) {
            if (lane < 2)
                tma_load_2d(dst + lane * kHalfBytes, &kmap, lane * 64, e * g.nmax + tile * kTileKeys, bar);
        } else if (lane < 16) {
            const int blk8 = lane >> 1, half = lane & 1;
            const int lb = min(tile * 8 + blk8, nblk_seq - 1);
            int phys = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + lb];
            if (phys < 0 || phys >= g.num_blocks)
                phys = 0; // rkv_importance records the error
            tma_load_4d(dst + half * kHalfBytes + blk8 * (kBlock * 128), &kmap, half * 64, id.h, 0,
                        id.l * g.num_blocks + phys, bar);
        }
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0) {
            prefetch_tmap(&kmap);
            mbar_expect_tx(afull, nrt * kTileBytes + tiles * kTileKeys * 4);
            bulk_load(inv_s, a.inv + static_cast<size_t>(e) * g.npad, tiles * kTileKeys * 4, afull);
        }
        __syncwarp();
        for (int r = 0; r < nrt; ++r)
            load_tile(a_s + r * kTileBytes, rt0 + r, afull);
        __syncwarp();
        for (int ct = 0; ct < tiles; ++ct) {
            const int s = ct % kRedStages;
            if (ct >= kRedStages && !mbar_wait(&empty[s], ((ct / kRedStages) - 1) & 1, abort))
                break;
            if (lane == 0)
                mbar_expect_tx(&full[s], kTileBytes);
            __syncwarp();
            load_tile(b_s + s * kTileBytes, ct, &full[s]);
            __syncwarp();
        }
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            bool ok = mbar_wait(afull, 0, abort);
            for (int ct = 0; ok && ct < tiles; ++ct) {
                const int s = ct % kRedStages, buf = ct & 1;
                if (!mbar_wait(&full[s], (ct / kRedStages) & 1, abort))
                    break;
                if (ct >= 2 && !mbar_wait(&acc_empty[buf], ((ct >> 1) - 1) & 1, abort))
                    break;
                tc_fence_after();
                const uint32_t bbase = smem_u32(b_s + s * kTileBytes);
                for (int r = 0; r < nrt; ++r) {
                    const uint32_t abase = smem_u32(a_s + r * kTileBytes);
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t koff = (k >> 2) * kHalfBytes + (k & 3) * 32;
                        umma_bf16(tmem + (buf * 2 + r) * 128, sdesc_sw128(abase + koff), sdesc_sw128(bbase + koff),
                                  idesc, k > 0 ? 1u : 0u);
                    }
                }
                umma_commit(&empty[s]);
                umma_commit(&acc_full[buf]);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - 2;             // 0..7
        const int r = ew >> 2;               // row tile of this warpgroup
        const int q4 = warp & 3;             // TMEM lane quarter
        const int i = (rt0 + r) * kTileKeys + q4 * 32 + lane;
        const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
        float sum = 0.f;
        bool ok = mbar_wait(afull, 0, abort);
        for (int ct = 0; ok && ct < tiles; ++ct) {
            const int buf = ct & 1;
            if (!mbar_wait(&acc_full[buf], (ct >> 1) & 1, abort))
                break;
            tc_fence_after();
            if (r < nrt) {
                const bool edge = (ct == tiles - 1) || (ct == rt0 + r);
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float v[32];
                    tmem_ld32(tmem + lane_addr + (buf * 2 + r) * 128 + cc * 32, v);
                    tmem_wait_ld();
                    const int jb = ct * kTileKeys + cc * 32;
                    const float4 *iv = reinterpret_cast<const float4 *>(inv_s + jb);
                    if (!edge) {
#pragma unroll
                        for (int q = 0; q < 8; ++q) {
                            const float4 w = iv[q];
                            sum = fmaf(v[4 * q + 0], w.x, sum);
                            sum = fmaf(v[4 * q + 1], w.y, sum);
                            sum = fmaf(v[4 * q + 2], w.z, sum);
                            sum = fmaf(v[4 * q + 3], w.w, sum);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < 32; ++c) {
                            const int j = jb + c;
                            const float t = v[c] * inv_s[j];
                            sum += (j < n && j != i) ? t : 0.f;
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0)
                mbar_arrive(&acc_empty[buf]);
        }
        if (r < nrt && i < n && !*abort)
            a.out_red[static_cast<size_t>(e) * g.npad + i] = n > 1 ? sum * inv_s[i] / static_cast<float>(n - 1) : 0.f;
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

} // namespace rkv
