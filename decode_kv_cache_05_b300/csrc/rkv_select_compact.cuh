// rkv_select_compact: steps 3-5 of the compression event in one launch --
// normalise, blend and select (rkv_select's computation) followed by the
// in-place compaction of K and V and the freed-block emission (rkv_compact's
// computation), for per-KV-head selection.
//
// The R-KV review page ("How R-KV decides what to drop") keeps kv_budget tokens
// with a protected window and blends the two scores with mix_lambda, then
// compacts the cache and hands evicted blocks back (FREE_BLOCKS); the
// hotdry.top blog (Ada-KV section) gives the paged block size of 16.
//
// One cluster of C CTAs per (layer, sequence, KV head), as in rkv_compact:
//   1. the CTA of rank 0 runs the selection of the head in its shared memory
//      (score rows bulk-copied in, min-max, blend, radix select, ascending
//      emission) and writes the kept indices to keep_idx and to a shared
//      array keep_s;
//   2. one cluster barrier; every other CTA copies the kept indices of its own
//      slots out of rank 0's keep_s (distributed shared memory) into its
//      unused selection scratch;
//   3. all C CTAs move the kept rows in rounds, exactly as rkv_compact does.
// Compared with two launches, the kept indices never travel through global
// memory before the moves, and the selection's latency is paid once inside a
// kernel that is already resident instead of in a launch of its own.
#pragma once

#include "rkv_compact.cuh"
#include "rkv_select.cuh"

namespace rkv {

static_assert(kSelThreads == kCpThreads, "the fused kernel runs the selection on the compaction CTA's threads");

struct SelCompactArgs {
    CompactArgs c; // compaction outputs (c.keep unused: the kept indices come from the selection)
    SelArgs s;     // selection inputs and outputs (s.keep: keep_idx, s.scores: optional scores)
};

// Dynamic shared memory: the selection scratch, then keep_s[budget].
__host__ __device__ constexpr size_t selcp_keep_offset(int npad) { return (sel_smem_bytes(npad, false) + 15) & ~size_t(15); }
__host__ __device__ constexpr size_t selcp_smem_bytes(int npad, int budget)
{
    return selcp_keep_offset(npad) + static_cast<size_t>(budget) * 4;
}

__global__ void __launch_bounds__(kCpThreads) rkv_select_compact_kernel(const SelCompactArgs a)
{
    extern __shared__ __align__(16) uint32_t scp_smem[];
    __shared__ int32_t table_s[kMaxSeq / kBlock];
    __shared__ int sh_sum;
    __shared__ uint32_t sh_sel_ok;
    const Geom &g = a.c.g;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int e = blockIdx.x / csize; // one cluster per head
    const HeadId id = head_id(g, e);
    int32_t *keep_s = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(scp_smem) + selcp_keep_offset(g.npad));

    pdl_wait();
    pdl_trigger();
    int n = g.seq_lens[id.b];
    bool ok = n >= 0 && n <= g.nmax;
    if (!ok)
        n = 0;
    const bool trig = triggered(g, n);
    const int kb = min(n, g.budget);
    const int new_len = trig ? kb : n; // a sequence left for a later call keeps its length
    const int nblk = (n + kBlock - 1) / kBlock;

    // ---- freed blocks and new length: one CTA per sequence
    if (id.l == 0 && id.h == 0 && crank == 0)
        emit_freed(a.c, id, n, ok, new_len, nblk, &sh_sum);

    // ---- steps 3-4 in rank 0 (keep_idx, the optional scores and keep_s)
    if (crank == 0) {
        const bool sel_ok = select_unit<false>(a.s, e, scp_smem, keep_s);
        if (threadIdx.x == 0)
            sh_sel_ok = sel_ok ? 1u : 0u;
    }

    // ---- block table row (paged), validated; every CTA loads the same row
    if (g.paged && trig) {
        for (int i = threadIdx.x; i < nblk; i += kCpThreads) {
            const int p = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + i];
            ok = ok && p >= 0 && p < g.num_blocks;
            table_s[i] = p;
        }
    }
    ok = __syncthreads_and(ok);
    cluster_sync(); // (A) rank 0's keep_s and selection flag are complete
    uint32_t sel_ok;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(sel_ok) : "r"(cluster_addr(&sh_sel_ok, 0)) : "memory");
    // the same decision in every CTA of the cluster (n, the table and the flag are the same)
    const bool moves = ok && trig && n > g.budget && sel_ok != 0;
    if (!ok && n > 0 && threadIdx.x == 0 && crank == 0)
        record_error(kErrDevice); // a block id outside the pool: the head is left as it was
    if (!moves) {
        cluster_sync(); // (B) rank 0 stays resident until every peer has read its flag
        return;
    }

    const int per_round = static_cast<int>(csize) * kCpRows;
    const int rounds = (kb + per_round - 1) / per_round;
    // a peer's kept sources, round by round, in its (unused) selection scratch
    int32_t *keep_l = reinterpret_cast<int32_t *>(scp_smem);
    if (crank != 0) {
        const uint32_t remote = cluster_addr(keep_s, 0);
        for (int t = threadIdx.x; t < rounds * kCpRows; t += kCpThreads) {
            const int j = (t / kCpRows) * per_round + static_cast<int>(crank) * kCpRows + t % kCpRows;
            int32_t v = -1;
            if (j < kb)
                asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(remote + 4u * j) : "memory");
            keep_l[t] = v;
        }
        __syncthreads();
    }
    // rank 0 is still resident: it leaves only after the first round's cluster
    // barrier, which every peer reaches after its copy above
    const int32_t *src = crank == 0 ? keep_s : keep_l;
    const int stride = crank == 0 ? per_round : kCpRows;
    move_kept_rows(a.c, e, id, table_s, kb, crank, csize, [&](int r, int i) { return src[r * stride + i]; });
}

// ---------------------------------------------------------------------------
// One CTA per head, no cluster: kScpSoloThreads threads run the selection,
// then move the kept rows in rounds of kScpSoloRows slots, each round's loads
// and stores separated by __syncthreads (a barrier of the CTA alone, where the
// cluster form needs a cluster barrier per round and leaves its other CTAs
// waiting while the first one selects). Two CTAs fit an SM.
constexpr int kScpSoloThreads = 512;
constexpr int kScpSoloRows = kScpSoloThreads / 4;             // 16 threads x 16 bytes per row, 4 rows per thread
constexpr int kScpSoloItems = kScpSoloRows * 16 / kScpSoloThreads;

__host__ __device__ constexpr size_t selcp_solo_keep_offset(int npad)
{
    return (sel_smem_bytes(npad, false, kScpSoloThreads) + 15) & ~size_t(15);
}
__host__ __device__ constexpr size_t selcp_solo_smem_bytes(int npad, int budget)
{
    return selcp_solo_keep_offset(npad) + static_cast<size_t>(budget) * 4;
}

__global__ void __launch_bounds__(kScpSoloThreads, 2) rkv_select_compact_solo_kernel(const SelCompactArgs a)
{
    extern __shared__ __align__(16) uint32_t scp_smem[];
    __shared__ int32_t table_s[kMaxSeq / kBlock];
    __shared__ int sh_sum;
    const Geom &g = a.c.g;
    const int e = blockIdx.x;
    const HeadId id = head_id(g, e);
    int32_t *keep_s = reinterpret_cast<int32_t *>(reinterpret_cast<uint8_t *>(scp_smem) + selcp_solo_keep_offset(g.npad));

    pdl_wait();
    pdl_trigger();
    int n = g.seq_lens[id.b];
    bool ok = n >= 0 && n <= g.nmax;
    if (!ok)
        n = 0;
    const bool trig = triggered(g, n);
    const int kb = min(n, g.budget);
    const int new_len = trig ? kb : n; // a sequence left for a later call keeps its length
    const int nblk = (n + kBlock - 1) / kBlock;

    if (id.l == 0 && id.h == 0)
        emit_freed(a.c, id, n, ok, new_len, nblk, &sh_sum);

    // ---- steps 3-4 (keep_idx, the optional scores and keep_s)
    const bool sel_ok = select_unit<false, kScpSoloThreads>(a.s, e, scp_smem, keep_s);

    // ---- block table row (paged), validated
    if (g.paged && trig) {
        for (int i = threadIdx.x; i < nblk; i += kScpSoloThreads) {
            const int p = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + i];
            ok = ok && p >= 0 && p < g.num_blocks;
            table_s[i] = p;
        }
    }
    ok = __syncthreads_and(ok); // also: keep_s complete
    if (!ok && n > 0 && threadIdx.x == 0)
        record_error(kErrDevice); // a block id outside the pool: the head is left as it was
    if (!(ok && trig && n > g.budget && sel_ok))
        return;

    // ---- step 5: in-place rounds (sources of a later round lie past this round's slots)
    const size_t row_bytes = kHeadDim * 2;
    auto row_ptr = [&](uint8_t *base, int t) -> uint8_t * {
        if (!g.paged)
            return base + (static_cast<size_t>(e) * g.nmax + t) * row_bytes;
        const int blk = table_s[t / kBlock];
        return base + ((((static_cast<size_t>(id.l) * g.num_blocks + blk) * kBlock + (t % kBlock)) * g.Hkv + id.h) *
                       row_bytes);
    };
    const int rounds = (kb + kScpSoloRows - 1) / kScpSoloRows;
    for (int r = 0; r < rounds; ++r) {
        uint4 kx[kScpSoloItems], vx[kScpSoloItems];
        int dx[kScpSoloItems];
#pragma unroll
        for (int q = 0; q < kScpSoloItems; ++q) {
            const int flat = threadIdx.x + q * kScpSoloThreads;
            const int j = r * kScpSoloRows + (flat >> 4);
            const int col = flat & 15;
            dx[q] = -1;
            if (j < kb) {
                const int src = keep_s[j];
                if (src != j) {
                    dx[q] = j;
                    kx[q] = cp_ld(reinterpret_cast<const uint4 *>(row_ptr(a.c.k, src)) + col);
                    vx[q] = cp_ld(reinterpret_cast<const uint4 *>(row_ptr(a.c.v, src)) + col);
                }
            }
        }
        __syncthreads(); // every load of this round has read its row
#pragma unroll
        for (int q = 0; q < kScpSoloItems; ++q) {
            if (dx[q] >= 0) {
                const int col = (threadIdx.x + q * kScpSoloThreads) & 15;
                cp_st(reinterpret_cast<uint4 *>(row_ptr(a.c.k, dx[q])) + col, kx[q]);
                cp_st(reinterpret_cast<uint4 *>(row_ptr(a.c.v, dx[q])) + col, vx[q]);
            }
        }
    }
}

} // namespace rkv
