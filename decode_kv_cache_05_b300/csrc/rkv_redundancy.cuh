// rkv_redundancy: mean cosine similarity of each key to the head's other keys.
//
// R-KV flags repeated content by the cosine similarity of key vectors
// (hotdry.top blog, R-KV section, first step); the R-KV review page ("How
// R-KV decides what to drop") credits batched redundancy scoring for keeping
// the cost on the decode path low. Definition used here, for a head with N keys:
//     R_i = (1/(N-1)) * sum_{j != i} (k_i . k_j) * inv_i * inv_j,  inv = 1/|k|.
//
// Design: a dense key Gram G = K K^T on the 5th-generation tensor cores, never
// written to HBM. The kernel is persistent (one CTA per SM); a work item is a
// (head, pair of 128-row tiles) and items are dealt round-robin to the CTAs.
//   warp 0      TMA producer: the item's two row tiles (A operands) into one
//               of two A buffers, so the next item's rows load while the
//               current item multiplies; then every other 128-key column
//               tile (B operand) through a STAGES-deep 128B-swizzled ring.
//               The item's own row tiles are also two of its column tiles:
//               those are multiplied from the A buffer, not loaded again.
//   warp 1      TMEM owner / MMA issuer: per column tile, two 128x128x128
//               tcgen05 MMAs (one per row tile) into a double-buffered fp32
//               accumulator (2 buffers x 2 row tiles x 128 columns = 512).
//   warps 2..9  epilogue (one warpgroup per row tile, four lanes per row):
//               tcgen05.ld the 128 accumulator columns, fused row sum
//               sum_j G_ij * inv_j over all j < N (only a ragged last tile is
//               masked), then R_i = (inv_i * sum - [k_i != 0]) / (N-1): the
//               diagonal term inv_i^2 G_ii equals 1 up to fp32 rounding and is
//               removed after the sum instead of being masked in it. The
//               column tile's inverse norms inv_j come through a small
//               shared-memory ring.
//   warp 10     fills that ring (bulk copies), so that the producer never
//               waits for the epilogue to free an inverse-norm slot.
// The inverse norms come from rkv_importance, which computes them from the
// same staged K tiles.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

constexpr int kRedThreads = 352;
constexpr int kRedStages = 3;

struct RedArgs {
    Geom g;
    const float *inv;
    float *out_red;
    int pairs; // items per head: ceil(ceil(max_seq_len / 128) / 2)
    int item0; // this launch's items: [item0, items) in the order of red_item_map
    int items; // end of this launch's items (heads * pairs for all of them)
    int heads;
    int interleave; // 1: a head's items consecutive (its half block right after its full ones)
};

// Item order: first every head's full 256-row blocks, then the half blocks
// (one 128-row tile) that an odd tile count leaves, so that the cheap items
// fill in at the end of each CTA's round-robin share instead of being spread
// unevenly (on 1152-token heads this cuts the longest share from ~17.5 to
// 16 half-block units, against 15.6 on average).
//
// With `interleave` (problems with many items per CTA, where the balance above
// no longer matters), a head's blocks are consecutive instead: the CTAs that
// work on a head at the same time then share its key tiles through L2, where
// a half block dealt at the very end would fetch all of them from HBM again.
__host__ __device__ inline void red_item_map(const RedArgs &a, int item, int tiles_max, int &e, int &pair)
{
    if (a.interleave) {
        e = item / a.pairs;
        pair = item % a.pairs;
        return;
    }
    const int full = tiles_max / 2;
    const int fitems = a.heads * full;
    if (item < fitems) {
        e = item / full;
        pair = item % full;
    } else {
        e = item - fitems;
        pair = full;
    }
}

struct RedSmem {
    static constexpr int kInvSlots = 4;                            // inverse-norm ring (one column tile each)
    static constexpr int kA = 0;                                   // 2 buffers x 2 row tiles
    static constexpr int kB = 4 * kTileBytes;                      // ring
    static constexpr int kInv = kB + kRedStages * kTileBytes;      // float[kInvSlots][128]
    static constexpr int kBars = kInv + kInvSlots * kTileKeys * 4;
    static constexpr int kNumBars = 2 * kRedStages + 2 + 2 + 2 + 2 + 2 * kInvSlots;
    static constexpr int kMisc = kBars + 8 * kNumBars;
    static constexpr int kBytes = kMisc + 16;
    // Requested dynamic shared memory: everything above plus whatever is
    // left of the 227 KB limit, which absorbs a base address that is not
    // 1024-byte aligned (the kernel checks that it fits).
    static constexpr int kAlloc = 232448;
};
static_assert(RedSmem::kBytes <= RedSmem::kAlloc, "redundancy kernel exceeds 227 KB of shared memory");

// Geometry of one work item, computed identically by every role.
struct RedItem {
    int e, n, tiles, rt0, nrt;
    HeadId id;
};

__device__ __forceinline__ bool red_item(const RedArgs &a, int item, RedItem &it)
{
    const Geom &g = a.g;
    int pair;
    red_item_map(a, item, (g.nmax + kTileKeys - 1) / kTileKeys, it.e, pair);
    it.id = head_id(g, it.e);
    int n = __ldg(g.seq_lens + it.id.b); // L1-cached: every role reads it at every item
    if (n < 0 || n > g.nmax)
        n = 0; // rkv_importance records the error
    if (!triggered(g, n))
        n = 0; // left for a later call
    it.n = n;
    it.tiles = (n + kTileKeys - 1) / kTileKeys;
    it.rt0 = 2 * pair;
    it.nrt = min(2, it.tiles - it.rt0);
    return it.rt0 < it.tiles;
}

__global__ void __launch_bounds__(kRedThreads, 1)
    rkv_redundancy_kernel(const __grid_constant__ CUtensorMap kmap, const RedArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (smem - smem_raw + RedSmem::kBytes > RedSmem::kAlloc) {
        if (threadIdx.x == 0)
            record_error(kErrDevice); // the layout does not fit: launch nothing further
        return;
    }

    uint8_t *a_s = smem + RedSmem::kA;
    uint8_t *b_s = smem + RedSmem::kB;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + RedSmem::kBars);
    uint64_t *full = bars;
    uint64_t *empty = bars + kRedStages;
    uint64_t *afull = bars + 2 * kRedStages;
    uint64_t *aempty = afull + 2;
    uint64_t *acc_full = aempty + 2;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *ifull = acc_empty + 2;
    uint64_t *iempty = ifull + RedSmem::kInvSlots;
    float *inv_s = reinterpret_cast<float *>(smem + RedSmem::kInv);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + RedSmem::kMisc);
    volatile uint32_t *abort = misc + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kRedStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&afull[b], 1);
            mbar_init(&aempty[b], 1);
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 8);
        }
        for (int b = 0; b < RedSmem::kInvSlots; ++b) {
            mbar_init(&ifull[b], 1);
            mbar_init(&iempty[b], 8);
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
    pdl_wait();
    pdl_trigger();

    // This lane's pool block for key tile `tile` of head `it` (paged layout;
    // lanes 0..15 each own one 16-row block half), looked up ahead of the
    // TMA issue so that the table load overlaps the ring wait.
    auto tile_phys = [&](const RedItem &it, int tile) -> int {
        if (!g.paged || lane >= 16)
            return 0;
        const int nblk_seq = (it.n + kBlock - 1) / kBlock;
        const int lb = min(tile * 8 + (lane >> 1), nblk_seq - 1);
        const int phys = g.block_table[static_cast<size_t>(it.id.b) * g.max_blocks + lb];
        return (phys < 0 || phys >= g.num_blocks) ? 0 : phys; // rkv_importance records the error
    };
    // Issue the TMA loads of key tile `tile` of head `it` into `dst` (one warp;
    // lanes split the boxes).
    auto load_tile = [&](const RedItem &it, uint8_t *dst, int tile, int phys, uint64_t *bar) {
        if (!g.paged) {
            if (lane < 2)
                tma_load_2d(dst + lane * kHalfBytes, &kmap, lane * 64, it.e * g.nmax + tile * kTileKeys, bar);
        } else if (lane < 16) {
            const int blk8 = lane >> 1, half = lane & 1;
            tma_load_4d(dst + half * kHalfBytes + blk8 * (kBlock * 128), &kmap, half * 64, it.id.h, 0,
                        it.id.l * g.num_blocks + phys, bar);
        }
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0)
            prefetch_tmap(&kmap);
        int kk = 0;   // A loads issued (items, in processing order)
        int ctg = 0;  // B tiles issued
        bool ok = true;
        // the item's row tiles into A buffer kk & 1, once the MMA is done with
        // that buffer's previous item
        auto load_a = [&](const RedItem &it) -> bool {
            const int ab = kk & 1;
            if (kk >= 2 && !mbar_wait(&aempty[ab], ((kk >> 1) - 1) & 1, abort))
                return false;
            ++kk;
            if (lane == 0)
                mbar_expect_tx(&afull[ab], it.nrt * kTileBytes);
            __syncwarp();
            for (int r = 0; r < it.nrt; ++r)
                load_tile(it, a_s + (ab * 2 + r) * kTileBytes, it.rt0 + r, tile_phys(it, it.rt0 + r), &afull[ab]);
            __syncwarp();
            return true;
        };
        auto next_item = [&](int from, RedItem &it) -> int {
            for (int item = from; item < a.items; item += gridDim.x)
                if (red_item(a, item, it))
                    return item;
            return a.items;
        };
        RedItem cur, nxt;
        int item = next_item(a.item0 + static_cast<int>(blockIdx.x), cur);
        if (item < a.items)
            ok = load_a(cur);
        while (ok && item < a.items) {
            const int nitem = next_item(item + gridDim.x, nxt);
            // the next item's rows go out once a few of this item's column
            // tiles are queued: early enough to land before its first MMA,
            // late enough that the MMA has left the buffer's previous item
            const int a_at = min(kRedStages, cur.tiles - 1);
            for (int ct = 0; ct < cur.tiles; ++ct) {
                // the item's own row tiles are multiplied from the A buffer:
                // no second copy of them goes through the ring
                if (ct < cur.rt0 || ct >= cur.rt0 + cur.nrt) {
                    const int s = ctg % kRedStages;
                    const int phys = tile_phys(cur, ct);
                    if (ctg >= kRedStages && !mbar_wait(&empty[s], ((ctg / kRedStages) - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    if (lane == 0)
                        mbar_expect_tx(&full[s], kTileBytes);
                    __syncwarp();
                    load_tile(cur, b_s + s * kTileBytes, ct, phys, &full[s]);
                    __syncwarp();
                    ++ctg;
                }
                if (ct == a_at && nitem < a.items && !load_a(nxt)) {
                    ok = false;
                    break;
                }
            }
            item = nitem;
            cur = nxt;
        }
        if (*abort && lane == 0) {
            for (int c = max(0, ctg - kRedStages); c < ctg; ++c)
                mbar_drain(&full[c % kRedStages], (c / kRedStages) & 1);
            for (int c = max(0, kk - 2); c < kk; ++c)
                mbar_drain(&afull[c & 1], (c >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
            int kk = 0, ctg = 0, bcnt = 0; // items, column tiles, ring tiles consumed
            bool ok = true;
            for (int item = a.item0 + static_cast<int>(blockIdx.x); ok && item < a.items; item += gridDim.x) {
                RedItem it;
                if (!red_item(a, item, it))
                    continue;
                const int ab = kk & 1;
                if (!mbar_wait(&afull[ab], (kk >> 1) & 1, abort))
                    break;
                for (int ct = 0; ct < it.tiles; ++ct, ++ctg) {
                    const int buf = ctg & 1, s = bcnt % kRedStages;
                    const bool own = ct >= it.rt0 && ct < it.rt0 + it.nrt; // B operand = an A tile
                    if ((!own && !mbar_wait(&full[s], (bcnt / kRedStages) & 1, abort)) ||
                        (ctg >= 2 && !mbar_wait(&acc_empty[buf], ((ctg >> 1) - 1) & 1, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t bbase = own ? smem_u32(a_s + (ab * 2 + (ct - it.rt0)) * kTileBytes)
                                               : smem_u32(b_s + s * kTileBytes);
                    for (int r = 0; r < it.nrt; ++r) {
                        const uint32_t abase = smem_u32(a_s + (ab * 2 + r) * kTileBytes);
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const uint32_t koff = (k >> 2) * kHalfBytes + (k & 3) * 32;
                            umma_bf16(tmem + (buf * 2 + r) * 128, sdesc_sw128(abase + koff),
                                      sdesc_sw128(bbase + koff), idesc, k > 0 ? 1u : 0u);
                        }
                    }
                    if (!own) {
                        umma_commit(&empty[s]);
                        ++bcnt;
                    }
                    umma_commit(&acc_full[buf]);
                }
                if (ok)
                    umma_commit(&aempty[ab]);
                ++kk;
            }
            if (*abort && ctg > 0)
                mbar_drain(&acc_full[(ctg - 1) & 1], ((ctg - 1) >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == kRedThreads / 32 - 1) {
        // --------------------------------------------- inverse-norm loader
        // Each column tile's 128 inverse norms into a small ring for the
        // epilogue, in a warp of its own: a slot is free only once the
        // epilogue has finished that tile's sums, and waiting for that in the
        // producer would hold back the key tiles the MMAs need.
        if (lane == 0) {
            int ictg = 0;
            bool ok = true;
            for (int item = a.item0 + static_cast<int>(blockIdx.x); ok && item < a.items; item += gridDim.x) {
                RedItem it;
                if (!red_item(a, item, it))
                    continue;
                for (int ct = 0; ct < it.tiles; ++ct, ++ictg) {
                    const int is = ictg % RedSmem::kInvSlots;
                    if (ictg >= RedSmem::kInvSlots &&
                        !mbar_wait(&iempty[is], ((ictg / RedSmem::kInvSlots) - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    mbar_expect_tx(&ifull[is], kTileKeys * 4);
                    bulk_load(inv_s + is * kTileKeys, a.inv + static_cast<size_t>(it.e) * g.npad + ct * kTileKeys,
                              kTileKeys * 4, &ifull[is]);
                }
            }
            if (*abort) {
                for (int c = max(0, ictg - RedSmem::kInvSlots); c < ictg; ++c)
                    mbar_drain(&ifull[c % RedSmem::kInvSlots], (c / RedSmem::kInvSlots) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        // One warpgroup per row tile; the accumulator is read in the 16x256b
        // TMEM layout (lane t: rows t/4, t/4 + 8 of each 16-row block, columns
        // 2(t%4), 2(t%4)+1 of every 8), so that each lane needs a quarter of
        // the column inverse norms; the four lanes of a row add their sums by
        // shuffles at the end of the item. (One row per lane with the 32x32b
        // layout took 4.79 ms on a paged Qwen2-7B cache on B300, this 4.60.)
        const int ew = warp - 2;             // 0..7
        const int r = ew >> 2;               // row tile of this warpgroup
        const int q4 = warp & 3;             // TMEM lane quarter
        const int g8 = lane >> 2, kq = lane & 3;
        const int row = q4 * 32 + (kq >> 1) * 16 + (kq & 1) * 8 + g8; // the row whose sum this lane writes
        int ctg = 0;
        bool ok = true;
        for (int item = a.item0 + static_cast<int>(blockIdx.x); ok && item < a.items; item += gridDim.x) {
            RedItem it;
            if (!red_item(a, item, it))
                continue;
            const int i = (it.rt0 + r) * kTileKeys + row;
            const bool mine = r < it.nrt;
            // this row's inverse norm, fetched now so that its latency is hidden
            const float inv_i = (mine && i < it.n) ? __ldg(a.inv + static_cast<size_t>(it.e) * g.npad + i) : 0.f;
            float part[4][2]; // rows g8, g8 + 8, 16 + g8, 24 + g8 of the quarter; two chains each
#pragma unroll
            for (int q = 0; q < 4; ++q)
                part[q][0] = part[q][1] = 0.f;
            for (int ct = 0; ct < it.tiles; ++ct, ++ctg) {
                const int buf = ctg & 1, is = ctg % RedSmem::kInvSlots;
                if (!mbar_wait(&acc_full[buf], (ctg >> 1) & 1, abort) ||
                    !mbar_wait(&ifull[is], (ctg / RedSmem::kInvSlots) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // the whole 128-column accumulator slice into registers with one
                // wait, then the TMEM buffer goes back to the MMA warp at once
                float v[2][64];
                if (mine) {
#pragma unroll
                    for (int blk = 0; blk < 2; ++blk)
                        tmem_ld_16x256b_x16(tmem + (static_cast<uint32_t>(q4 * 32 + blk * 16) << 16) +
                                                (buf * 2 + r) * 128,
                                            v[blk]);
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&acc_empty[buf]);
                if (mine) {
                    const int jb = ct * kTileKeys;
                    const float2 *iv = reinterpret_cast<const float2 *>(inv_s + is * kTileKeys) + kq;
                    if (jb + kTileKeys <= it.n) {
#pragma unroll
                        for (int rep = 0; rep < 16; ++rep) {
                            const float2 w = iv[4 * rep];
#pragma unroll
                            for (int q = 0; q < 4; ++q)
                                fma2(part[q][0], part[q][1], v[q >> 1][4 * rep + 2 * (q & 1)],
                                     v[q >> 1][4 * rep + 2 * (q & 1) + 1], w.x, w.y);
                        }
                    } else {
                        // ragged last tile: columns j >= N are left out of the sums
#pragma unroll
                        for (int rep = 0; rep < 16; ++rep) {
                            const float2 w = iv[4 * rep];
                            const int j = jb + 8 * rep + 2 * kq;
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                const float t0 = v[q >> 1][4 * rep + 2 * (q & 1)] * w.x;
                                const float t1 = v[q >> 1][4 * rep + 2 * (q & 1) + 1] * w.y;
                                part[q][0] += j < it.n ? t0 : 0.f;
                                part[q][1] += j + 1 < it.n ? t1 : 0.f;
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&iempty[is]);
            }
            float rs[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                rs[q] = part[q][0] + part[q][1];
                rs[q] += __shfl_xor_sync(0xffffffffu, rs[q], 1);
                rs[q] += __shfl_xor_sync(0xffffffffu, rs[q], 2);
            }
            const float sum = kq == 0 ? rs[0] : kq == 1 ? rs[1] : kq == 2 ? rs[2] : rs[3];
            if (ok && mine && i < it.n && !*abort)
                a.out_red[static_cast<size_t>(it.e) * g.npad + i] =
                    it.n > 1 ? (inv_i * sum - (inv_i > 0.f ? 1.f : 0.f)) / static_cast<float>(it.n - 1) : 0.f;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// Wide form of the single-CTA Gram: 128 x 256 MMAs (two key tiles per MMA)
// instead of 128 x 128, half as many MMA instructions per flop. Same items
// (a head's pair of 128-row tiles), same fused row-mean epilogue.
//   shared memory (the same 226 KB as above, laid out differently):
//     A  two buffers of the item's two row tiles, half-major: [rt0 dims 0-63]
//        [rt1 dims 0-63][rt0 dims 64-127][rt1 dims 64-127] (16 KB each), so
//        that a row tile is a 128-row operand and the pair a 256-row one;
//     B  a ring of three 32 KB entries, each two key tiles' halves of the same
//        64 dims: one 256-row B operand for four K = 16 steps (a column pair
//        takes two entries; the item's own pair is multiplied from A);
//   TMEM  two 256-column accumulators: with two row tiles, one per row tile,
//        drained by its epilogue warpgroup while the other row tile's MMAs
//        run; with one row tile, the two alternate by column pair.
constexpr int kWideThreads = 352;

struct WideSmem {
    static constexpr int kEntries = 3;                          // B ring entries
    static constexpr int kInvSlots = 2;                         // float[2][256]
    static constexpr int kA = 0;                                // 2 buffers x 64 KB
    static constexpr int kB = 2 * 2 * kTileBytes;               // ring
    static constexpr int kInv = kB + kEntries * kTileBytes;
    static constexpr int kXs = kInv + kInvSlots * 256 * 4;      // float[128]: one-row-tile items' partials
    static constexpr int kBars = kXs + 128 * 4;
    // entry full/empty; A full/empty; accumulator full/empty; inverse-norm full/empty
    static constexpr int kNumBars = 2 * kEntries + 2 + 2 + 2 + 2 + 2 * kInvSlots;
    static constexpr int kMisc = kBars + 8 * kNumBars;
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = 232448;
};
static_assert(WideSmem::kBytes <= WideSmem::kAlloc, "wide Gram kernel exceeds 227 KB of shared memory");

__global__ void __launch_bounds__(kWideThreads, 1)
    rkv_redundancy_wide_kernel(const __grid_constant__ CUtensorMap kmap, const RedArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (smem - smem_raw + WideSmem::kBytes > WideSmem::kAlloc) {
        if (threadIdx.x == 0)
            record_error(kErrDevice); // the layout does not fit: launch nothing further
        return;
    }
    uint8_t *a_s = smem + WideSmem::kA;
    uint8_t *b_s = smem + WideSmem::kB;
    float *inv_s = reinterpret_cast<float *>(smem + WideSmem::kInv);
    float *xs = reinterpret_cast<float *>(smem + WideSmem::kXs);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + WideSmem::kBars);
    uint64_t *efull = bars;
    uint64_t *eempty = efull + WideSmem::kEntries;
    uint64_t *afull = eempty + WideSmem::kEntries;
    uint64_t *aempty = afull + 2;
    uint64_t *acc_full = aempty + 2;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *ifull = acc_empty + 2;
    uint64_t *iempty = ifull + WideSmem::kInvSlots;
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + WideSmem::kMisc);
    volatile uint32_t *abort = misc + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < WideSmem::kEntries; ++s) {
            mbar_init(&efull[s], 1);
            mbar_init(&eempty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&afull[b], 1);
            mbar_init(&aempty[b], 1);
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 4); // the four warps of the draining warpgroup
        }
        for (int b = 0; b < WideSmem::kInvSlots; ++b) {
            mbar_init(&ifull[b], 1);
            mbar_init(&iempty[b], 8); // every epilogue warp, for every column pair
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
    pdl_wait();
    pdl_trigger();

    // Tile loads, one warp, one round: `parts` 16 KB halves (128 rows x 64 dims,
    // swizzled) go to dst_of(part); part p is half h_of(p) of key tile
    // tile_of(p). Contiguous layout: lane p issues part p; paged layout: lanes
    // 8p .. 8p+7 issue part p's eight 16-row blocks (pool block ids looked up
    // by the same lanes beforehand, so that the table loads overlap a wait).
    auto part_phys = [&](const RedItem &it, int tile) -> int { // this lane's block of `tile` (paged)
        if (!g.paged)
            return 0;
        const int nblk_seq = (it.n + kBlock - 1) / kBlock;
        const int lb = min(tile * 8 + (lane & 7), nblk_seq - 1);
        const int phys = g.block_table[static_cast<size_t>(it.id.b) * g.max_blocks + lb];
        return (phys < 0 || phys >= g.num_blocks) ? 0 : phys; // rkv_importance records the error
    };
    auto load_parts = [&](const RedItem &it, int parts, int phys, uint64_t *bar, auto tile_of, auto h_of,
                          auto dst_of) {
        if (!g.paged) {
            if (lane < parts)
                tma_load_2d(dst_of(lane), &kmap, h_of(lane) * 64, it.e * g.nmax + tile_of(lane) * kTileKeys, bar);
        } else if (lane < 8 * parts) {
            const int p = lane >> 3;
            tma_load_4d(dst_of(p) + (lane & 7) * (kBlock * 128), &kmap, h_of(p) * 64, it.id.h, 0,
                        it.id.l * g.num_blocks + phys, bar);
        }
    };

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0)
            prefetch_tmap(&kmap);
        int kk = 0, ec = 0; // items' A loads issued; ring entries issued
        bool ok = true;
        auto load_a = [&](const RedItem &it) -> bool {
            const int ab = kk & 1;
            if (kk >= 2 && !mbar_wait(&aempty[ab], ((kk >> 1) - 1) & 1, abort))
                return false;
            ++kk;
            if (lane == 0)
                mbar_expect_tx(&afull[ab], it.nrt * kTileBytes);
            __syncwarp();
            uint8_t *abuf = a_s + ab * 2 * kTileBytes;
            for (int r = 0; r < it.nrt; ++r) {
                // both halves of row tile r in one round (part = half)
                const int tile = it.rt0 + r;
                const int phys = part_phys(it, tile);
                load_parts(it, 2, phys, &afull[ab], [&](int) { return tile; }, [&](int p) { return p; },
                           [&](int p) { return abuf + p * kTileBytes + r * kHalfBytes; });
            }
            __syncwarp();
            return true;
        };
        auto next_item = [&](int from, RedItem &it) -> int {
            for (int item = from; item < a.items; item += gridDim.x)
                if (red_item(a, item, it))
                    return item;
            return a.items;
        };
        RedItem cur, nxt;
        int item = next_item(a.item0 + static_cast<int>(blockIdx.x), cur);
        if (item < a.items)
            ok = load_a(cur);
        while (ok && item < a.items) {
            const int nitem = next_item(item + gridDim.x, nxt);
            const int cps = (cur.tiles + 1) / 2;     // column pairs
            const int own = cur.rt0 / 2;             // the pair multiplied from A
            const int a_at = min(1, cps - 1);        // the next item's rows go out after this pair
            for (int cp = 0; cp < cps; ++cp) {
                if (cp != own) {
                    const int ntl = min(2, cur.tiles - 2 * cp);
                    // this lane's pool block of its tile (part = tile of the pair)
                    const int phys = part_phys(cur, 2 * cp + ((lane >> 3) & 1));
                    for (int h = 0; h < 2; ++h, ++ec) {
                        const int s = ec % WideSmem::kEntries;
                        if (ec >= WideSmem::kEntries &&
                            !mbar_wait(&eempty[s], ((ec / WideSmem::kEntries) - 1) & 1, abort)) {
                            ok = false;
                            break;
                        }
                        if (lane == 0)
                            mbar_expect_tx(&efull[s], ntl * kHalfBytes);
                        __syncwarp();
                        uint8_t *entry = b_s + s * kTileBytes;
                        load_parts(cur, ntl, phys, &efull[s], [&](int p) { return 2 * cp + p; }, [&](int) { return h; },
                                   [&](int p) { return entry + p * kHalfBytes; });
                        __syncwarp();
                    }
                    if (!ok)
                        break;
                }
                if (cp == a_at && nitem < a.items && !load_a(nxt)) {
                    ok = false;
                    break;
                }
            }
            item = nitem;
            cur = nxt;
        }
        if (*abort && lane == 0) {
            for (int c = max(0, ec - WideSmem::kEntries); c < ec; ++c)
                mbar_drain(&efull[c % WideSmem::kEntries], (c / WideSmem::kEntries) & 1);
            for (int c = max(0, kk - 2); c < kk; ++c)
                mbar_drain(&afull[c & 1], (c >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            int kk = 0, ec = 0;          // items; ring entries consumed
            int use[2] = {0, 0};         // uses of each accumulator
            bool ok = true;
            for (int item = a.item0 + static_cast<int>(blockIdx.x); ok && item < a.items; item += gridDim.x) {
                RedItem it;
                if (!red_item(a, item, it))
                    continue;
                const int ab = kk & 1;
                if (!mbar_wait(&afull[ab], (kk >> 1) & 1, abort))
                    break;
                const uint32_t abase = smem_u32(a_s + ab * 2 * kTileBytes);
                const int cps = (it.tiles + 1) / 2, own = it.rt0 / 2;
                for (int cp = 0; ok && cp < cps; ++cp) {
                    const int ntl = min(2, it.tiles - 2 * cp);
                    const uint32_t idesc = idesc_bf16_f32(128, ntl * 128);
                    // accumulator of each row tile for this pair
                    int acc_of[2];
                    for (int r = 0; r < it.nrt; ++r)
                        acc_of[r] = it.nrt == 2 ? r : (cp & 1);
                    // Row tile by row tile: row tile 0's accumulator is complete after
                    // its eight MMAs, so that its drain overlaps all eight of row tile
                    // 1's (interleaving the two by 64-dim half would leave it four; on
                    // B300 that order took 80.0 us on a Llama-3-8B cache, this 76.3).
                    // Both halves' ring entries stay held until row tile 1 has used them.
                    uint32_t bbase[2] = {0u, 0u};
                    int es[2] = {0, 0};
                    for (int r = 0; ok && r < it.nrt; ++r) {
                        const int b = acc_of[r];
                        if (use[b] >= 1 && !mbar_wait(&acc_empty[b], (use[b] - 1) & 1, abort)) {
                            ok = false;
                            break;
                        }
                        for (int h = 0; h < 2; ++h) {
                            if (r == 0) {
                                if (cp == own) {
                                    bbase[h] = abase + h * kTileBytes; // the item's own row tiles, [rt0 | rt1] of half h
                                } else {
                                    es[h] = (ec + h) % WideSmem::kEntries;
                                    if (!mbar_wait(&efull[es[h]], ((ec + h) / WideSmem::kEntries) & 1, abort)) {
                                        ok = false;
                                        break;
                                    }
                                    bbase[h] = smem_u32(b_s + es[h] * kTileBytes);
                                }
                            }
                            tc_fence_after();
                            const uint32_t arow = abase + h * kTileBytes + r * kHalfBytes;
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                umma_bf16(tmem + b * 256, sdesc_sw128(arow + k * 32), sdesc_sw128(bbase[h] + k * 32),
                                          idesc, (h > 0 || k > 0) ? 1u : 0u);
                            if (r == it.nrt - 1 && cp != own)
                                umma_commit(&eempty[es[h]]);
                        }
                        if (!ok)
                            break;
                        umma_commit(&acc_full[b]);
                    }
                    if (!ok)
                        break;
                    if (cp != own)
                        ec += 2;
                    if (!ok)
                        break;
                    for (int r = 0; r < it.nrt; ++r)
                        ++use[acc_of[r]];
                }
                if (ok)
                    umma_commit(&aempty[ab]);
                ++kk;
            }
            if (*abort) {
                for (int b = 0; b < 2; ++b)
                    if (use[b] > 0)
                        mbar_drain(&acc_full[b], (use[b] - 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == kWideThreads / 32 - 1) {
        // --------------------------------------------- inverse-norm loader
        if (lane == 0) {
            int ic = 0;
            bool ok = true;
            for (int item = a.item0 + static_cast<int>(blockIdx.x); ok && item < a.items; item += gridDim.x) {
                RedItem it;
                if (!red_item(a, item, it))
                    continue;
                const int cps = (it.tiles + 1) / 2;
                for (int cp = 0; cp < cps; ++cp, ++ic) {
                    const int is = ic % WideSmem::kInvSlots;
                    if (ic >= WideSmem::kInvSlots &&
                        !mbar_wait(&iempty[is], ((ic / WideSmem::kInvSlots) - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    const int nf = min(256, g.npad - cp * 256); // floats of this pair inside the head's row
                    mbar_expect_tx(&ifull[is], nf * 4);
                    bulk_load(inv_s + is * 256, a.inv + static_cast<size_t>(it.e) * g.npad + cp * 256, nf * 4,
                              &ifull[is]);
                }
            }
            if (*abort) {
                for (int c = max(0, ic - WideSmem::kInvSlots); c < ic; ++c)
                    mbar_drain(&ifull[c % WideSmem::kInvSlots], (c / WideSmem::kInvSlots) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        // One warpgroup per accumulator. The accumulator is read with the
        // 16x256b TMEM shape: lane t of a warp holds rows t/4 and t/4 + 8 of
        // each 16-row block and columns 2(t%4), 2(t%4)+1 of every 8-column
        // group, so it needs a quarter of the column inverse norms (one 8-byte
        // shared load per 8 columns, against one 16-byte load per 4 columns
        // with one row per thread; on B300 the Llama-3-8B cache took 76.0 us
        // that way, 73.5 us this way). A row's sum is spread over four lanes
        // and added by shuffles at the end of the item.
        const int ew = warp - 2;          // 0..7
        const int wg = ew >> 2;           // accumulator this warpgroup drains
        const int q4 = warp & 3;          // TMEM lane quarter
        const int g8 = lane >> 2, kq = lane & 3;
        int ic = 0, duse = 0;             // column pairs seen; drains of accumulator wg
        bool ok = true;
        for (int item = a.item0 + static_cast<int>(blockIdx.x); ok && item < a.items; item += gridDim.x) {
            RedItem it;
            if (!red_item(a, item, it))
                continue;
            float part[4][2]; // rows g8, g8 + 8, 16 + g8, 24 + g8 of the quarter; two chains each
#pragma unroll
            for (int q = 0; q < 4; ++q)
                part[q][0] = part[q][1] = 0.f;
            const int cps = (it.tiles + 1) / 2;
            for (int cp = 0; cp < cps; ++cp, ++ic) {
                const int is = ic % WideSmem::kInvSlots;
                if (!mbar_wait(&ifull[is], (ic / WideSmem::kInvSlots) & 1, abort)) {
                    ok = false;
                    break;
                }
                const bool mine = it.nrt == 2 || (cp & 1) == wg;
                if (mine) {
                    if (!mbar_wait(&acc_full[wg], duse & 1, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const int ncols = min(2, it.tiles - 2 * cp) * 128;
                    const float *inv_t = inv_s + is * 256;
                    for (int half = 0; half < ncols / 128; ++half) {
                        float v[2][64];
#pragma unroll
                        for (int blk = 0; blk < 2; ++blk)
                            tmem_ld_16x256b_x16(tmem + (static_cast<uint32_t>(q4 * 32 + blk * 16) << 16) + wg * 256 +
                                                    half * 128,
                                                v[blk]);
                        tmem_wait_ld();
                        if (half == ncols / 128 - 1) {
                            // the accumulator goes back to the MMA warp as soon as it is read
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                mbar_arrive(&acc_empty[wg]);
                        }
                        const int jb0 = cp * 256 + half * 128;
                        const float2 *iv = reinterpret_cast<const float2 *>(inv_t + half * 128) + kq;
                        if (jb0 + 128 <= it.n) {
#pragma unroll
                            for (int rep = 0; rep < 16; ++rep) {
                                const float2 w = iv[4 * rep];
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    fma2(part[q][0], part[q][1], v[q >> 1][4 * rep + 2 * (q & 1)],
                                         v[q >> 1][4 * rep + 2 * (q & 1) + 1], w.x, w.y);
                            }
                        } else {
                            // ragged last tile: columns j >= N are left out (their
                            // products are not formed into the sums at all)
#pragma unroll
                            for (int rep = 0; rep < 16; ++rep) {
                                const float2 w = iv[4 * rep];
                                const int j = jb0 + 8 * rep + 2 * kq;
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    const float t0 = v[q >> 1][4 * rep + 2 * (q & 1)] * w.x;
                                    const float t1 = v[q >> 1][4 * rep + 2 * (q & 1) + 1] * w.y;
                                    part[q][0] += j < it.n ? t0 : 0.f;
                                    part[q][1] += j + 1 < it.n ? t1 : 0.f;
                                }
                            }
                        }
                    }
                    ++duse;
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&iempty[is]);
            }
            // every epilogue warp takes the same decision to go on
            ok = !named_sync_or(1, 256, !ok || *abort);
            if (!ok)
                break;
            // each row's four lanes add their sums; lane kq then owns row q = kq
            float rs[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                rs[q] = part[q][0] + part[q][1];
                rs[q] += __shfl_xor_sync(0xffffffffu, rs[q], 1);
                rs[q] += __shfl_xor_sync(0xffffffffu, rs[q], 2);
            }
            float sum = kq == 0 ? rs[0] : kq == 1 ? rs[1] : kq == 2 ? rs[2] : rs[3];
            const int row = q4 * 32 + (kq >> 1) * 16 + (kq & 1) * 8 + g8;
            const int rtile = it.nrt == 2 ? wg : 0;
            const int i = (it.rt0 + rtile) * kTileKeys + row;
            if (it.nrt == 1) {
                // the two warpgroups summed alternate column pairs of the one row tile
                if (wg == 1)
                    xs[row] = sum;
                named_sync(1, 256);
                if (wg == 0)
                    sum += xs[row];
                named_sync(1, 256); // xs free again for the next item
            }
            if ((it.nrt == 2 || wg == 0) && i < it.n) {
                const float inv_i = __ldg(a.inv + static_cast<size_t>(it.e) * g.npad + i);
                a.out_red[static_cast<size_t>(it.e) * g.npad + i] =
                    it.n > 1 ? (inv_i * sum - (inv_i > 0.f ? 1.f : 0.f)) / static_cast<float>(it.n - 1) : 0.f;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

} // namespace rkv

namespace rkv {

// ---------------------------------------------------------------------------
// The same redundancy score on CTA pairs (cta_group::2). A cluster of two CTAs
// owns a 256-row block of one head: the even CTA holds rows [0,128) of the
// block, the odd CTA rows [128,256). Column tiles are 256 keys, each CTA
// staging its half (keys [0,128) of the tile in the even CTA, [128,256) in the
// odd one); a last tile with at most 128 valid keys is a 128-key tile, 64 in
// each CTA. One thread of the even CTA issues 256x256x16 MMAs that read both
// CTAs' halves, so each SM reads only its own A and B halves from shared
// memory per MMA: half the operand traffic per flop of a single-CTA 128x128
// tile, which is what limits the single-CTA kernel above.
//   warp 0      producer (both CTAs): own A half per item into one of two A
//               buffers, own B half per column tile through a STAGES ring;
//               completion is counted on the even CTA's barriers. The
//               diagonal column tile (the item's own 256 keys) is multiplied
//               from the A buffers instead.
//   warp 1      even CTA: MMA issuer; commits are multicast to both CTAs.
//   warps 2..9  epilogue (both CTAs): one warpgroup per 128-column half of
//               the 256 accumulator columns, one row per thread; the two
//               partial row sums are added through shared memory.
//   warp 10     each column tile's 256 inverse norms into a local ring.
constexpr int kPairThreads = 352;
constexpr int kPairStages = 4;

struct PairSmem {
    static constexpr int kInvSlots = 8;
    static constexpr int kA = 0;                                        // 2 A buffers (own 128 rows)
    static constexpr int kB = 2 * kTileBytes;                           // ring of own B halves
    static constexpr int kInv = kB + kPairStages * kTileBytes;          // float[kInvSlots][256]
    static constexpr int kPart = kInv + kInvSlots * 256 * 4;            // float[128]
    static constexpr int kBars = kPart + 128 * 4;
    static constexpr int kNumBars = 2 * kPairStages + 2 + 2 + 2 + 2 + 2 * kInvSlots;
    static constexpr int kMisc = kBars + 8 * kNumBars;
    static constexpr int kBytes = kMisc + 16;
    static constexpr int kAlloc = kBytes + 1024; // + alignment slack
};
static_assert(PairSmem::kAlloc <= 232448, "pair redundancy kernel exceeds 227 KB of shared memory");

struct PairItem {
    int e, n, ctiles, row0;
    HeadId id;
};

// Work item = (head, 256-row block); rows [row0, row0 + 256), column tiles of 256 keys.
__device__ __forceinline__ bool pair_item(const RedArgs &a, int item, PairItem &it)
{
    const Geom &g = a.g;
    int pair;
    red_item_map(a, item, (g.nmax + kTileKeys - 1) / kTileKeys, it.e, pair);
    it.id = head_id(g, it.e);
    int n = __ldg(g.seq_lens + it.id.b);
    if (n < 0 || n > g.nmax)
        n = 0; // rkv_importance records the error
    if (!triggered(g, n))
        n = 0; // left for a later call
    it.n = n;
    it.ctiles = (n + 255) / 256;
    it.row0 = 256 * pair;
    return it.row0 < n;
}

// Column tile ct of item `it` is the item's own 256-row block at full width:
// each CTA's 128-key half of it is exactly that CTA's A rows.
__device__ __forceinline__ bool pair_own_tile(const PairItem &it, int ct)
{
    return 256 * ct == it.row0 && it.n - 256 * ct > 128;
}

__global__ void __launch_bounds__(kPairThreads, 1)
    rkv_redundancy_pair_kernel(const __grid_constant__ CUtensorMap kmap, const RedArgs a)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = align1024(smem_raw);
    const Geom &g = a.g;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank(); // 0: even CTA (MMA issuer), 1: odd CTA
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;

    uint8_t *a_s = smem + PairSmem::kA;
    uint8_t *b_s = smem + PairSmem::kB;
    float *inv_s = reinterpret_cast<float *>(smem + PairSmem::kInv);
    float *part = reinterpret_cast<float *>(smem + PairSmem::kPart);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + PairSmem::kBars);
    uint64_t *full = bars;                              // even CTA: both B halves landed
    uint64_t *empty = full + kPairStages;               // both CTAs: MMA done with the stage
    uint64_t *afull = empty + kPairStages;              // even CTA: both A halves landed
    uint64_t *aempty = afull + 2;                       // both CTAs: MMA done with the A buffer
    uint64_t *acc_full = aempty + 2;                    // both CTAs: accumulator ready
    uint64_t *acc_empty = acc_full + 2;                 // even CTA: 16 epilogue warps done
    uint64_t *ifull = acc_empty + 2;                    // local
    uint64_t *iempty = ifull + PairSmem::kInvSlots;     // local
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + PairSmem::kMisc);
    volatile uint32_t *abort = misc + 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&afull[b], 1);
            mbar_init(&aempty[b], 1);
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 16);
        }
        for (int b = 0; b < PairSmem::kInvSlots; ++b) {
            mbar_init(&ifull[b], 1);
            mbar_init(&iempty[b], 8);
        }
        misc[1] = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc_pair(&misc[0], 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync(); // barriers of both CTAs initialised; TMEM allocated
    tc_fence_after();
    const uint32_t tmem = misc[0];
    pdl_wait();
    pdl_trigger();

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0)
            prefetch_tmap(&kmap);
        int kk = 0, ctg = 0;
        bool ok = true;
        // Own 128-row half of a 256-row block starting at row `r0`.
        auto load_half = [&](const PairItem &it, uint8_t *dst, int r0, uint32_t bar) {
            if (!g.paged) {
                if (lane < 2)
                    tma_load_2d_pair(dst + lane * kHalfBytes, &kmap, lane * 64, it.e * g.nmax + r0, bar);
            } else if (lane < 16) {
                const int nblk_seq = (it.n + kBlock - 1) / kBlock;
                const int blk8 = lane >> 1, half = lane & 1;
                const int lb = min(r0 / kBlock + blk8, nblk_seq - 1);
                int phys = g.block_table[static_cast<size_t>(it.id.b) * g.max_blocks + lb];
                if (phys < 0 || phys >= g.num_blocks)
                    phys = 0; // rkv_importance records the error
                tma_load_4d_pair(dst + half * kHalfBytes + blk8 * (kBlock * 128), &kmap, half * 64, it.id.h, 0,
                                 it.id.l * g.num_blocks + phys, bar);
            }
        };
        for (int item = a.item0 + pair; ok && item < a.items; item += npairs) {
            PairItem it;
            if (!pair_item(a, item, it))
                continue;
            const int ab = kk & 1;
            if (kk >= 2 && !mbar_wait(&aempty[ab], ((kk >> 1) - 1) & 1, abort))
                break;
            ++kk;
            if (rank == 0 && lane == 0)
                mbar_expect_tx(&afull[ab], 2 * kTileBytes);
            __syncwarp();
            load_half(it, a_s + ab * kTileBytes, it.row0 + 128 * static_cast<int>(rank), cluster_addr(&afull[ab], 0));
            __syncwarp();
            for (int ct = 0; ct < it.ctiles; ++ct) {
                // the diagonal 256-key tile holds exactly each CTA's own A
                // rows: multiplied from the A buffer, not loaded again
                if (pair_own_tile(it, ct))
                    continue;
                const int s = ctg % kPairStages;
                if (ctg >= kPairStages && !mbar_wait(&empty[s], ((ctg / kPairStages) - 1) & 1, abort)) {
                    ok = false;
                    break;
                }
                if (rank == 0 && lane == 0)
                    mbar_expect_tx(&full[s], 2 * kTileBytes);
                __syncwarp();
                // a last tile with at most 128 valid keys is multiplied as a
                // 128-wide tile: 64 keys in each CTA (a full box is still loaded)
                const int wh = it.n - 256 * ct > 128 ? 128 : 64;
                load_half(it, b_s + s * kTileBytes, 256 * ct + wh * static_cast<int>(rank),
                          cluster_addr(&full[s], 0));
                __syncwarp();
                ++ctg;
            }
        }
        if (*abort && lane == 0) {
            if (rank == 0) {
                for (int c = max(0, ctg - kPairStages); c < ctg; ++c)
                    mbar_drain(&full[c % kPairStages], (c / kPairStages) & 1);
                for (int c = max(0, kk - 2); c < kk; ++c)
                    mbar_drain(&afull[c & 1], (c >> 1) & 1);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------- MMA (even CTA only)
        if (rank == 0 && lane == 0) {
            constexpr uint32_t idesc_full = idesc_bf16_f32(256, 256);
            constexpr uint32_t idesc_half = idesc_bf16_f32(256, 128);
            int kk = 0, ctg = 0, bcnt = 0; // items, column tiles, ring tiles consumed
            bool ok = true;
            for (int item = a.item0 + pair; ok && item < a.items; item += npairs) {
                PairItem it;
                if (!pair_item(a, item, it))
                    continue;
                const int ab = kk & 1;
                if (!mbar_wait(&afull[ab], (kk >> 1) & 1, abort))
                    break;
                const uint32_t abase = smem_u32(a_s + ab * kTileBytes);
                for (int ct = 0; ct < it.ctiles; ++ct, ++ctg) {
                    const int s = bcnt % kPairStages, buf = ctg & 1;
                    const bool own = pair_own_tile(it, ct); // B operand = the A buffer
                    if ((!own && !mbar_wait(&full[s], (bcnt / kPairStages) & 1, abort)) ||
                        (ctg >= 2 && !mbar_wait(&acc_empty[buf], ((ctg >> 1) - 1) & 1, abort))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t bbase = own ? abase : smem_u32(b_s + s * kTileBytes);
                    const uint32_t idesc = it.n - 256 * ct > 128 ? idesc_full : idesc_half;
#pragma unroll
                    for (int k = 0; k < 8; ++k) {
                        const uint32_t koff = (k >> 2) * kHalfBytes + (k & 3) * 32;
                        umma_bf16_pair(tmem + buf * 256, sdesc_sw128(abase + koff), sdesc_sw128(bbase + koff), idesc,
                                       k > 0 ? 1u : 0u);
                    }
                    if (!own) {
                        umma_commit_pair(&empty[s], 0x3);
                        ++bcnt;
                    }
                    umma_commit_pair(&acc_full[buf], 0x3);
                }
                if (ok)
                    umma_commit_pair(&aempty[ab], 0x3);
                ++kk;
            }
            if (*abort && ctg > 0)
                mbar_drain(&acc_full[(ctg - 1) & 1], ((ctg - 1) >> 1) & 1);
        }
        __syncwarp();
    } else if (warp == kPairThreads / 32 - 1) {
        // --------------------------------------------- inverse-norm loader
        // Each 256-key column tile's inverse norms into a local ring, in a
        // warp of its own so that the producer never waits for the epilogue.
        if (lane == 0) {
            int ictg = 0;
            bool ok = true;
            for (int item = a.item0 + pair; ok && item < a.items; item += npairs) {
                PairItem it;
                if (!pair_item(a, item, it))
                    continue;
                for (int ct = 0; ct < it.ctiles; ++ct, ++ictg) {
                    const int is = ictg % PairSmem::kInvSlots;
                    if (ictg >= PairSmem::kInvSlots &&
                        !mbar_wait(&iempty[is], ((ictg / PairSmem::kInvSlots) - 1) & 1, abort)) {
                        ok = false;
                        break;
                    }
                    const int cnt = min(256, g.npad - 256 * ct); // 128 or 256: stays inside the head's plane
                    mbar_expect_tx(&ifull[is], cnt * 4);
                    bulk_load(inv_s + is * 256, a.inv + static_cast<size_t>(it.e) * g.npad + 256 * ct, cnt * 4,
                              &ifull[is]);
                }
            }
            if (*abort) {
                for (int c = max(0, ictg - PairSmem::kInvSlots); c < ictg; ++c)
                    mbar_drain(&ifull[c % PairSmem::kInvSlots], (c / PairSmem::kInvSlots) & 1);
            }
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- epilogue
        const int ew = warp - 2;             // 0..7
        const int wg = ew >> 2;              // column half of the accumulator
        const int q4 = warp & 3;             // TMEM lane quarter
        const uint32_t lane_addr = static_cast<uint32_t>(q4 * 32) << 16;
        const int rloc = q4 * 32 + lane;     // row within this CTA's 128
        int ctg = 0;
        bool ok = true;
        for (int item = a.item0 + pair; ok && item < a.items; item += npairs) {
            PairItem it;
            if (!pair_item(a, item, it))
                continue;
            const int i = it.row0 + 128 * static_cast<int>(rank) + rloc;
            const float inv_i = i < it.n ? __ldg(a.inv + static_cast<size_t>(it.e) * g.npad + i) : 0.f;
            float part4[4] = {0.f, 0.f, 0.f, 0.f}; // four chains: the FMA latency is not serialised
            for (int ct = 0; ct < it.ctiles; ++ct, ++ctg) {
                const int buf = ctg & 1, is = ctg % PairSmem::kInvSlots;
                if (!mbar_wait(&acc_full[buf], (ctg >> 1) & 1, abort) ||
                    !mbar_wait(&ifull[is], (ctg / PairSmem::kInvSlots) & 1, abort)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // tile width: 256 keys, or 128 for a last tile with at most 128
                // valid keys; this warpgroup takes the second half of its columns
                const int wh = it.n - 256 * ct > 128 ? 128 : 64;
                const int j0 = 256 * ct + wh * wg; // first key of this warpgroup's columns
                const bool edge = j0 + wh > it.n;  // ragged last tile
                const float *inv_t = inv_s + is * 256 + wh * wg;
                // the warpgroup's accumulator columns into registers with one
                // wait, then the TMEM buffer goes back to the MMA warp at once
                float v[4][32];
                const bool live = j0 < it.n;
                if (live) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc)
                        if (cc * 32 < wh)
                            tmem_ld32(tmem + lane_addr + buf * 256 + wg * wh + cc * 32, v[cc]);
                    tmem_wait_ld();
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    mbar_arrive_cluster_relaxed(cluster_addr(&acc_empty[buf], 0));
                if (live) {
#pragma unroll
                    for (int cc = 0; cc < 4; ++cc) {
                        if (cc * 32 >= wh)
                            break;
                        const float4 *iv = reinterpret_cast<const float4 *>(inv_t + cc * 32);
                        if (!edge) {
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                const float4 w = iv[q];
                                fma2(part4[0], part4[1], v[cc][4 * q + 0], v[cc][4 * q + 1], w.x, w.y);
                                fma2(part4[2], part4[3], v[cc][4 * q + 2], v[cc][4 * q + 3], w.z, w.w);
                            }
                        } else {
#pragma unroll
                            for (int c = 0; c < 32; ++c) {
                                const int j = j0 + cc * 32 + c;
                                const float t = v[cc][c] * inv_t[cc * 32 + c];
                                part4[c & 3] += j < it.n ? t : 0.f;
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(&iempty[is]);
            }
            const float sum = (part4[0] + part4[1]) + (part4[2] + part4[3]);
            // add the two column halves' partial sums of each row
            if (wg == 1)
                part[rloc] = sum;
            // every epilogue warp takes the same decision to go on, so that
            // none is left waiting alone at a named barrier
            ok = !named_sync_or(1, 256, !ok || *abort);
            if (ok && wg == 0 && i < it.n) {
                // the diagonal term inv_i^2 G_ii is 1 up to fp32 rounding (0 for a zero key)
                a.out_red[static_cast<size_t>(it.e) * g.npad + i] =
                    it.n > 1 ? (inv_i * (sum + part[rloc]) - (inv_i > 0.f ? 1.f : 0.f)) /
                                   static_cast<float>(it.n - 1)
                             : 0.f;
            }
            named_sync(1, 256);
        }
    }
    tc_fence_before();
    cluster_sync(); // both CTAs done: no MMA, commit or remote arrival in flight
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

} // namespace rkv
