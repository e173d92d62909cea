// rkv_compact: move kept K/V rows into the kept slots, in place, and emit the
// freed paged blocks and the new lengths.
//
// The R-KV review page ("How R-KV decides what to drop") describes two-phase
// compaction in the SGLang port and FREE_BLOCKS, which hands evicted blocks
// back to the allocator instead of stranding them; the hotdry.top blog
// (Ada-KV section) gives the paged block size of 16.
//
// In-place safety: keep[] is ascending with keep[j] >= j, so slot j is never a
// source for a later slot. A cluster of C CTAs per head sweeps the slots in
// rounds of C x 128 rows; in each round every CTA first loads its 128 source
// rows (K and V) into registers, the cluster synchronises, then every CTA
// stores. Sources of round r+1 lie at or past the end of round r's
// destinations, so one cluster barrier per round is enough.
// Paged: slot j and token t both address block_table[b][. / 16], row . % 16;
// freed = table entries ceil(k_b/16) .. ceil(N_b/16)-1.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

constexpr int kCpThreads = 256;
constexpr int kCpRows = 128;                          // rows per CTA per round
constexpr int kCpItems = kCpRows * 16 / kCpThreads;   // uint4 per thread per tensor

struct CompactArgs {
    Geom g;
    uint8_t *k;
    uint8_t *v;
    const int32_t *keep;
    int32_t *freed_off;
    int32_t *freed_ids;
    int32_t *new_lens;
};

__global__ void __launch_bounds__(kCpThreads) rkv_compact_kernel(const CompactArgs a)
{
    __shared__ int32_t table_s[kMaxSeq / kBlock];
    __shared__ int sh_sum;
    const Geom &g = a.g;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int e = blockIdx.x / csize; // one cluster per head
    const HeadId id = head_id(g, e);

    int n = g.seq_lens[id.b];
    bool ok = n >= 0 && n <= g.nmax;
    if (!ok)
        n = 0;
    const int kb = min(n, g.budget);
    const int nblk = (n + kBlock - 1) / kBlock;

    // ---- freed blocks and new length: one CTA per sequence
    if (id.l == 0 && id.h == 0 && crank == 0) {
        if (threadIdx.x == 0)
            sh_sum = 0;
        __syncthreads();
        int part = 0;
        if (g.paged) {
            for (int b2 = threadIdx.x; b2 < id.b; b2 += kCpThreads) {
                const int n2 = g.seq_lens[b2];
                if (n2 >= 0 && n2 <= g.nmax)
                    part += (n2 + kBlock - 1) / kBlock - (min(n2, g.budget) + kBlock - 1) / kBlock;
            }
        }
        atomicAdd(&sh_sum, part);
        __syncthreads();
        const int off = sh_sum;
        const int first = (kb + kBlock - 1) / kBlock;
        const int cnt = g.paged ? nblk - first : 0;
        if (threadIdx.x == 0) {
            a.new_lens[id.b] = kb;
            a.freed_off[id.b] = off;
            if (id.b == g.B - 1)
                a.freed_off[g.B] = off + cnt;
            if (!ok)
                record_error(kErrDevice);
        }
        for (int i = threadIdx.x; i < cnt; i += kCpThreads)
            a.freed_ids[off + i] = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + first + i];
    }

    // ---- block table row (paged) and validation of keep[]
    const int32_t *keep = a.keep + static_cast<size_t>(e) * g.budget;
    if (g.paged) {
        for (int i = threadIdx.x; i < nblk; i += kCpThreads) {
            const int p = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + i];
            ok = ok && p >= 0 && p < g.num_blocks;
            table_s[i] = p;
        }
    }
    for (int j = threadIdx.x; j < kb; j += kCpThreads) {
        const int s = keep[j];
        ok = ok && s >= j && s < n && (j == 0 || s > keep[j - 1]);
    }
    ok = __syncthreads_and(ok);
    if (!ok) {
        if (threadIdx.x == 0)
            record_error(kErrDevice);
        // every CTA of the cluster reaches the same decision: no round runs
        return;
    }

    const size_t row_bytes = kHeadDim * 2;
    auto row_ptr = [&](uint8_t *base, int t) -> uint8_t * {
        if (!g.paged)
            return base + (static_cast<size_t>(e) * g.nmax + t) * row_bytes;
        const int blk = table_s[t / kBlock];
        return base + ((((static_cast<size_t>(id.l) * g.num_blocks + blk) * kBlock + (t % kBlock)) * g.Hkv + id.h) *
                       row_bytes);
    };

    const int per_round = static_cast<int>(csize) * kCpRows;
    const int rounds = (kb + per_round - 1) / per_round;
    for (int r = 0; r < rounds; ++r) {
        const int base = r * per_round + static_cast<int>(crank) * kCpRows;
        uint4 kr[kCpItems], vr[kCpItems];
        int dst[kCpItems];
#pragma unroll
        for (int q = 0; q < kCpItems; ++q) {
            const int flat = threadIdx.x + q * kCpThreads;
            const int j = base + (flat >> 4);
            const int col = flat & 15;
            dst[q] = -1;
            if (j < kb) {
                const int s = keep[j];
                if (s != j) {
                    dst[q] = j;
                    kr[q] = __ldcg(reinterpret_cast<const uint4 *>(row_ptr(a.k, s)) + col);
                    vr[q] = __ldcg(reinterpret_cast<const uint4 *>(row_ptr(a.v, s)) + col);
                }
            }
        }
        cluster_sync();
#pragma unroll
        for (int q = 0; q < kCpItems; ++q) {
            if (dst[q] >= 0) {
                const int col = (threadIdx.x + q * kCpThreads) & 15;
                __stcg(reinterpret_cast<uint4 *>(row_ptr(a.k, dst[q])) + col, kr[q]);
                __stcg(reinterpret_cast<uint4 *>(row_ptr(a.v, dst[q])) + col, vr[q]);
            }
        }
    }
}

} // namespace rkv
