// rkv_compact: move kept K/V rows into the kept slots, in place, and emit the
// freed paged blocks and the new lengths.
//
// The R-KV review page ("How R-KV decides what to drop") describes two-phase
// compaction in the SGLang port and FREE_BLOCKS, which hands evicted blocks
// back to the allocator instead of stranding them; the hotdry.top blog
// (Ada-KV section) gives the paged block size of 16.
//
// In-place safety: keep[] is ascending with keep[j] >= j, so a row is only
// ever read by a slot at or before its own position. A cluster of C CTAs per
// head sweeps the slots in rounds of C x 64 rows. A round's stores may begin
// once every CTA's loads of that round (and of all earlier rounds) have
// completed, which one cluster barrier per round provides; the loads of the
// next round read rows at or past the next round's first slot, beyond this
// round's destinations, so they are issued before the barrier and overlap it
// and the stores (register double buffer).
// Paged: slot j and token t both address block_table[b][. / 16], row . % 16;
// freed = table entries ceil(k_b/16) .. ceil(N_b/16)-1.
#pragma once

#include "rkv_device.cuh"
#include "rkv_geom.cuh"

namespace rkv {

#ifndef RKV_CP_ROWS
#define RKV_CP_ROWS 64
#endif
#ifndef RKV_CP_PIPE
#define RKV_CP_PIPE 0
#endif
#ifndef RKV_CP_HINT
#define RKV_CP_HINT 1
#endif

constexpr int kCpThreads = 256;
constexpr int kCpRows = RKV_CP_ROWS;                  // rows per CTA per round
constexpr int kCpItems = kCpRows * 16 / kCpThreads;   // uint4 per thread per tensor

__device__ __forceinline__ uint4 cp_ld(const uint4 *p)
{
#if RKV_CP_HINT == 1
    return __ldcs(p);
#elif RKV_CP_HINT == 0
    return __ldcg(p);
#else
    return *p;
#endif
}

__device__ __forceinline__ void cp_st(uint4 *p, const uint4 &v)
{
#if RKV_CP_HINT == 1
    __stcs(p, v);
#elif RKV_CP_HINT == 0
    __stcg(p, v);
#else
    *p = v;
#endif
}

struct CompactArgs {
    Geom g;
    uint8_t *k;
    uint8_t *v;
    const int32_t *keep;
    int32_t *freed_off;
    int32_t *freed_ids;
    int32_t *new_lens;
};

// Freed-block CSR slice and new length of sequence id.b, written by one CTA
// per sequence (all its threads call this).
__device__ __forceinline__ void emit_freed(const CompactArgs &a, const HeadId &id, int n, bool ok, int new_len,
                                           int nblk, int *sh_sum)
{
    const Geom &g = a.g;
    const int nthreads = static_cast<int>(blockDim.x);
    if (threadIdx.x == 0)
        *sh_sum = 0;
    __syncthreads();
    int part = 0;
    if (g.paged) {
        for (int b2 = threadIdx.x; b2 < id.b; b2 += nthreads) {
            const int n2 = g.seq_lens[b2];
            if (n2 >= 0 && n2 <= g.nmax && triggered(g, n2))
                part += (n2 + kBlock - 1) / kBlock - (min(n2, g.budget) + kBlock - 1) / kBlock;
        }
    }
    atomicAdd(sh_sum, part);
    __syncthreads();
    const int off = *sh_sum;
    const int first = (new_len + kBlock - 1) / kBlock;
    const int cnt = g.paged ? nblk - first : 0;
    if (threadIdx.x == 0) {
        a.new_lens[id.b] = new_len;
        a.freed_off[id.b] = off;
        if (id.b == g.B - 1)
            a.freed_off[g.B] = off + cnt;
        if (!ok)
            record_error(kErrDevice);
    }
    for (int i = threadIdx.x; i < cnt; i += nthreads)
        a.freed_ids[off + i] = g.block_table[static_cast<size_t>(id.b) * g.max_blocks + first + i];
}

// The in-place move of one head's kept rows by a cluster of csize CTAs, in
// rounds of csize x kCpRows slots (see the file comment for why it is safe).
// src_of(r, i) is the kept token of this CTA's slot i of round r, i.e. of
// slot j = r * csize * kCpRows + crank * kCpRows + i. Every CTA of the cluster
// must call this with the same kb (the cluster barrier of each round).
template <typename SrcOf>
__device__ __forceinline__ void move_kept_rows(const CompactArgs &a, int e, const HeadId &id, const int32_t *table_s,
                                               int kb, uint32_t crank, uint32_t csize, SrcOf src_of)
{
    const Geom &g = a.g;
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
    // rows whose slot already holds them (keep[j] == j) need no move
    uint4 kr[2][kCpItems], vr[2][kCpItems];
    int dst[2][kCpItems];
    auto load_round = [&](int r, uint4 (&kx)[kCpItems], uint4 (&vx)[kCpItems], int (&dx)[kCpItems]) {
        const int base = r * per_round + static_cast<int>(crank) * kCpRows;
#pragma unroll
        for (int q = 0; q < kCpItems; ++q) {
            const int flat = threadIdx.x + q * kCpThreads;
            const int i = flat >> 4;
            const int j = base + i;
            const int col = flat & 15;
            dx[q] = -1;
            if (j < kb) {
                const int src = src_of(r, i);
                if (src != j) {
                    dx[q] = j;
                    kx[q] = cp_ld(reinterpret_cast<const uint4 *>(row_ptr(a.k, src)) + col);
                    vx[q] = cp_ld(reinterpret_cast<const uint4 *>(row_ptr(a.v, src)) + col);
                }
            }
        }
    };
    auto store_round = [&](const uint4 (&kx)[kCpItems], const uint4 (&vx)[kCpItems], const int (&dx)[kCpItems]) {
#pragma unroll
        for (int q = 0; q < kCpItems; ++q) {
            if (dx[q] >= 0) {
                const int col = (threadIdx.x + q * kCpThreads) & 15;
                cp_st(reinterpret_cast<uint4 *>(row_ptr(a.k, dx[q])) + col, kx[q]);
                cp_st(reinterpret_cast<uint4 *>(row_ptr(a.v, dx[q])) + col, vx[q]);
            }
        }
    };
#if RKV_CP_PIPE == 0
    for (int r = 0; r < rounds; ++r) {
        load_round(r, kr[0], vr[0], dst[0]);
        cluster_sync();
        store_round(kr[0], vr[0], dst[0]);
    }
    return;
#endif
    if (rounds > 0)
        load_round(0, kr[0], vr[0], dst[0]);
    for (int r = 0; r < rounds; r += 2) {
        if (r + 1 < rounds)
            load_round(r + 1, kr[1], vr[1], dst[1]);
        cluster_sync(); // loads of rounds <= r complete in every CTA
        store_round(kr[0], vr[0], dst[0]);
        if (r + 1 >= rounds)
            break;
        if (r + 2 < rounds)
            load_round(r + 2, kr[0], vr[0], dst[0]);
        cluster_sync(); // loads of rounds <= r + 1 complete in every CTA
        store_round(kr[1], vr[1], dst[1]);
    }
}

__global__ void __launch_bounds__(kCpThreads) rkv_compact_kernel(const CompactArgs a)
{
    __shared__ int32_t table_s[kMaxSeq / kBlock];
    __shared__ int sh_sum;
    const Geom &g = a.g;
    const uint32_t crank = cluster_rank(), csize = cluster_size();
    const int e = blockIdx.x / csize; // one cluster per head
    const HeadId id = head_id(g, e);

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
        emit_freed(a, id, n, ok, new_len, nblk, &sh_sum);

    if (!trig)
        return; // every CTA of the cluster decides alike; nothing moves

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
    const int per_round = static_cast<int>(csize) * kCpRows;
    move_kept_rows(a, e, id, table_s, kb, crank, csize,
                   [&](int r, int i) { return keep[r * per_round + static_cast<int>(crank) * kCpRows + i]; });
}

} // namespace rkv
