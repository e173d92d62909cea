// librkv: rkv_compress_host -- the compression event for a KV cache that
// lives in host memory. Host-side runtime code only: it cuts the layers into
// chunks and runs, per chunk,
//     host->device copy (stream h2d)  ->  rkv_compress (caller's stream)
//                                     ->  device->host copy (stream d2h)
// over three device slots, so that the chunk c+1 upload, the chunk c kernels
// and the chunk c-1 download are in flight together. The two directions use
// separate copy engines and PCIe is full duplex, so the downloads overlap the
// uploads instead of following them; the kernels hide behind the copies.
//
// Every dependency is an event: a slot is refilled only after its previous
// download has been read out (ev_out), the kernels of a chunk wait for its
// upload (ev_in), its download waits for its kernels (ev_comp), and the
// caller's stream waits for the last download (ev_done).
#include "rkv.h"

#include <algorithm>
#include <cstdint>
#include <mutex>

namespace {

constexpr int kSlots = 3;
constexpr size_t kAutoChunkBytes = size_t(20) << 20; // K+V bytes per chunk when chunk_layers == 0
constexpr int kMaxDevices = 64;

inline size_t up256(size_t x) { return (x + 255) & ~size_t(255); }

// Bytes of one layer of each per-layer array.
struct LayerBytes {
    size_t kv;    // K (or V)
    size_t q;     // q_window
    size_t keep;  // out_keep_idx
    size_t score; // one of the three score planes
};

LayerBytes layer_bytes(const rkv_problem *p)
{
    LayerBytes s;
    const size_t row = static_cast<size_t>(p->head_dim) * 2;
    if (p->layout == RKV_LAYOUT_PAGED)
        s.kv = static_cast<size_t>(p->num_blocks) * p->block_size * p->num_kv_heads * row;
    else
        s.kv = static_cast<size_t>(p->batch) * p->num_kv_heads * p->max_seq_len * row;
    s.q = static_cast<size_t>(p->batch) * p->num_q_heads * p->window * row;
    s.keep = static_cast<size_t>(p->batch) * p->num_kv_heads * p->budget * 4;
    s.score = static_cast<size_t>(p->batch) * p->num_kv_heads * p->max_seq_len * 4;
    return s;
}

int chunk_of(const rkv_problem *p, int32_t chunk_layers)
{
    if (p->num_layers == 0)
        return 0;
    if (chunk_layers > 0)
        return std::min<int>(chunk_layers, p->num_layers);
    const size_t per = 2 * layer_bytes(p).kv;
    const size_t c = per ? std::max<size_t>(1, kAutoChunkBytes / per) : size_t(p->num_layers);
    return static_cast<int>(std::min<size_t>(c, static_cast<size_t>(p->num_layers)));
}

// Byte offsets of everything in the device workspace.
struct Plan {
    int chunk = 0;
    LayerBytes lb{};
    size_t lens = 0, table = 0, off = 0, ids = 0, newl = 0; // per-call arrays
    size_t slot0 = 0, slot = 0;                             // first slot, bytes per slot
    size_t s_k = 0, s_v = 0, s_q = 0, s_keep = 0, s_scores = 0; // offsets inside a slot
    size_t comp = 0, comp_bytes = 0;                        // rkv_compress workspace
    size_t total = 0;
};

rkv_status make_plan(const rkv_problem *p, int32_t chunk_layers, Plan *pl)
{
    if (chunk_layers < 0)
        return RKV_ERR_INVALID_ARG;
    size_t ws = 0;
    const rkv_status st = rkv_workspace_size(p, &ws); // validates the problem
    if (st != RKV_OK)
        return st;
    pl->chunk = chunk_of(p, chunk_layers);
    pl->lb = layer_bytes(p);
    const size_t B = static_cast<size_t>(p->batch);
    const size_t table_n = p->layout == RKV_LAYOUT_PAGED ? B * p->max_blocks_per_seq : 0;
    size_t at = 0;
    pl->lens = at;
    at += up256(B * 4);
    pl->table = at;
    at += up256(table_n * 4);
    pl->off = at;
    at += up256((B + 1) * 4);
    pl->ids = at;
    at += up256(std::max<size_t>(table_n, 1) * 4);
    pl->newl = at;
    at += up256(B * 4);
    const size_t c = static_cast<size_t>(pl->chunk);
    size_t in_slot = 0;
    pl->s_k = in_slot;
    in_slot += up256(c * pl->lb.kv);
    pl->s_v = in_slot;
    in_slot += up256(c * pl->lb.kv);
    pl->s_q = in_slot;
    in_slot += up256(c * pl->lb.q);
    pl->s_keep = in_slot;
    in_slot += up256(c * pl->lb.keep);
    pl->s_scores = in_slot;
    in_slot += up256(3 * c * pl->lb.score);
    pl->slot0 = at;
    pl->slot = in_slot;
    at += kSlots * in_slot;
    rkv_problem pc = *p;
    pc.num_layers = pl->chunk;
    size_t comp = 0;
    if (rkv_workspace_size(&pc, &comp) != RKV_OK)
        return RKV_ERR_INVALID_ARG;
    pl->comp = at;
    pl->comp_bytes = std::max<size_t>(comp, 256);
    at += pl->comp_bytes;
    pl->total = at;
    return RKV_OK;
}

// The copy streams and events of one device, created on first use and kept
// for the life of the process.
struct CopyEngine {
    std::mutex mu;
    bool ready = false;
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t start = nullptr, meta = nullptr, done = nullptr;
    cudaEvent_t in[kSlots] = {}, comp[kSlots] = {}, out[kSlots] = {};
};

CopyEngine g_engine[kMaxDevices];

bool create(CopyEngine &e)
{
    const unsigned ev = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&e.h2d, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&e.d2h, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.start, ev) != cudaSuccess || cudaEventCreateWithFlags(&e.meta, ev) != cudaSuccess ||
        cudaEventCreateWithFlags(&e.done, ev) != cudaSuccess)
        return false;
    for (int s = 0; s < kSlots; ++s)
        if (cudaEventCreateWithFlags(&e.in[s], ev) != cudaSuccess ||
            cudaEventCreateWithFlags(&e.comp[s], ev) != cudaSuccess ||
            cudaEventCreateWithFlags(&e.out[s], ev) != cudaSuccess)
            return false;
    return true;
}

#define RKV_TRY(x)                                                                                                     \
    do {                                                                                                               \
        if ((x) != cudaSuccess)                                                                                        \
            return RKV_ERR_CUDA;                                                                                       \
    } while (0)

// After a failure part-way through a call: the caller's stream waits for
// every copy already queued on the library's streams, so that the caller's
// host buffers are not read or written after it has synchronised the stream
// (best effort: a CUDA error here leaves nothing better to do).
void join_after_error(CopyEngine &e, cudaStream_t stream)
{
    if (cudaEventRecord(e.done, e.h2d) == cudaSuccess)
        (void)cudaStreamWaitEvent(stream, e.done, 0);
    if (cudaEventRecord(e.done, e.d2h) == cudaSuccess)
        (void)cudaStreamWaitEvent(stream, e.done, 0);
}

inline const uint8_t *cbytes(const void *p) { return static_cast<const uint8_t *>(p); }
inline uint8_t *bytes(void *p) { return static_cast<uint8_t *>(p); }

rkv_status enqueue(CopyEngine &e, const rkv_problem *p, const Plan &pl, const void *k_in, const void *v_in,
                   void *k_out, void *v_out, const void *q_window, const int32_t *seq_lens,
                   const int32_t *block_table, int32_t *out_keep_idx, int32_t *out_freed_off,
                   int32_t *out_freed_ids, int32_t *out_new_seq_lens, float *out_scores, uint8_t *ws,
                   cudaStream_t stream)
{
    const bool paged = p->layout == RKV_LAYOUT_PAGED;
    const size_t B = static_cast<size_t>(p->batch);
    const size_t table_bytes = paged ? B * p->max_blocks_per_seq * 4 : 0;
    int32_t *d_lens = reinterpret_cast<int32_t *>(ws + pl.lens);
    int32_t *d_table = paged ? reinterpret_cast<int32_t *>(ws + pl.table) : nullptr;
    int32_t *d_off = reinterpret_cast<int32_t *>(ws + pl.off);
    int32_t *d_ids = paged ? reinterpret_cast<int32_t *>(ws + pl.ids) : nullptr;
    int32_t *d_newl = reinterpret_cast<int32_t *>(ws + pl.newl);

    // everything starts after the work already queued on the caller's stream
    RKV_TRY(cudaEventRecord(e.start, stream));
    RKV_TRY(cudaStreamWaitEvent(e.h2d, e.start, 0));
    RKV_TRY(cudaStreamWaitEvent(e.d2h, e.start, 0));
    if (B > 0)
        RKV_TRY(cudaMemcpyAsync(d_lens, seq_lens, B * 4, cudaMemcpyHostToDevice, e.h2d));
    if (table_bytes > 0)
        RKV_TRY(cudaMemcpyAsync(d_table, block_table, table_bytes, cudaMemcpyHostToDevice, e.h2d));
    RKV_TRY(cudaEventRecord(e.meta, e.h2d));
    RKV_TRY(cudaStreamWaitEvent(stream, e.meta, 0));

    const long long heads = static_cast<long long>(p->num_layers) * p->batch * p->num_kv_heads;
    if (heads == 0) {
        // nothing to copy per layer; rkv_compress writes what it writes for
        // an empty problem (freed_off[0] = 0 when there is no sequence)
        uint8_t *slot = ws + pl.slot0;
        rkv_status st = rkv_compress(p, slot + pl.s_k, slot + pl.s_v, slot + pl.s_q, d_lens, d_table,
                                     reinterpret_cast<int32_t *>(slot + pl.s_keep), d_off, d_ids, d_newl, nullptr,
                                     ws + pl.comp, pl.comp_bytes, stream);
        if (st != RKV_OK)
            return st;
        if (B == 0)
            RKV_TRY(cudaMemcpyAsync(out_freed_off, d_off, 4, cudaMemcpyDeviceToHost, stream));
        return RKV_OK;
    }

    const LayerBytes &lb = pl.lb;
    const int L = p->num_layers;
    const int nchunks = (L + pl.chunk - 1) / pl.chunk;
    for (int i = 0; i < nchunks; ++i) {
        const int s = i % kSlots;
        const int l0 = i * pl.chunk;
        const int nl = std::min(pl.chunk, L - l0);
        uint8_t *slot = ws + pl.slot0 + static_cast<size_t>(s) * pl.slot;
        uint8_t *dk = slot + pl.s_k, *dv = slot + pl.s_v, *dq = slot + pl.s_q;
        int32_t *dkeep = reinterpret_cast<int32_t *>(slot + pl.s_keep);
        float *dscores = out_scores ? reinterpret_cast<float *>(slot + pl.s_scores) : nullptr;

        // upload, once the slot's previous download has read it out
        if (i >= kSlots)
            RKV_TRY(cudaStreamWaitEvent(e.h2d, e.out[s], 0));
        RKV_TRY(cudaMemcpyAsync(dk, cbytes(k_in) + l0 * lb.kv, nl * lb.kv, cudaMemcpyHostToDevice, e.h2d));
        RKV_TRY(cudaMemcpyAsync(dv, cbytes(v_in) + l0 * lb.kv, nl * lb.kv, cudaMemcpyHostToDevice, e.h2d));
        RKV_TRY(cudaMemcpyAsync(dq, cbytes(q_window) + l0 * lb.q, nl * lb.q, cudaMemcpyHostToDevice, e.h2d));
        RKV_TRY(cudaEventRecord(e.in[s], e.h2d));

        // compress the chunk on the caller's stream
        RKV_TRY(cudaStreamWaitEvent(stream, e.in[s], 0));
        if (dscores)
            RKV_TRY(cudaMemsetAsync(dscores, 0, 3 * nl * lb.score, stream));
        rkv_problem pc = *p;
        pc.num_layers = nl;
        const rkv_status st = rkv_compress(&pc, dk, dv, dq, d_lens, d_table, dkeep, d_off, d_ids, d_newl, dscores,
                                           ws + pl.comp, pl.comp_bytes, stream);
        if (st != RKV_OK)
            return st;
        RKV_TRY(cudaEventRecord(e.comp[s], stream));

        // download
        RKV_TRY(cudaStreamWaitEvent(e.d2h, e.comp[s], 0));
        RKV_TRY(cudaMemcpyAsync(bytes(k_out) + l0 * lb.kv, dk, nl * lb.kv, cudaMemcpyDeviceToHost, e.d2h));
        RKV_TRY(cudaMemcpyAsync(bytes(v_out) + l0 * lb.kv, dv, nl * lb.kv, cudaMemcpyDeviceToHost, e.d2h));
        RKV_TRY(cudaMemcpyAsync(bytes(out_keep_idx) + l0 * lb.keep, dkeep, nl * lb.keep, cudaMemcpyDeviceToHost,
                                e.d2h));
        if (dscores)
            for (int t = 0; t < 3; ++t)
                RKV_TRY(cudaMemcpyAsync(bytes(out_scores) + (static_cast<size_t>(t) * L + l0) * lb.score,
                                        bytes(dscores) + static_cast<size_t>(t) * nl * lb.score, nl * lb.score,
                                        cudaMemcpyDeviceToHost, e.d2h));
        RKV_TRY(cudaEventRecord(e.out[s], e.d2h));
    }

    // the per-sequence outputs (every chunk writes the same values; the d2h
    // stream has already waited for the last chunk's kernels)
    RKV_TRY(cudaMemcpyAsync(out_freed_off, d_off, (B + 1) * 4, cudaMemcpyDeviceToHost, e.d2h));
    RKV_TRY(cudaMemcpyAsync(out_new_seq_lens, d_newl, B * 4, cudaMemcpyDeviceToHost, e.d2h));
    if (paged && table_bytes > 0)
        RKV_TRY(cudaMemcpyAsync(out_freed_ids, d_ids, table_bytes, cudaMemcpyDeviceToHost, e.d2h));
    RKV_TRY(cudaEventRecord(e.done, e.d2h));
    RKV_TRY(cudaStreamWaitEvent(stream, e.done, 0));
    return RKV_OK;
}

} // namespace

extern "C" {

rkv_status rkv_compress_host_workspace_size(const rkv_problem *p, int32_t chunk_layers, size_t *bytes)
{
    if (!bytes)
        return RKV_ERR_INVALID_ARG;
    Plan pl;
    const rkv_status st = make_plan(p, chunk_layers, &pl);
    if (st != RKV_OK)
        return st;
    *bytes = pl.total;
    return RKV_OK;
}

rkv_status rkv_compress_host(const rkv_problem *p, int32_t chunk_layers, const void *k_in, const void *v_in,
                             void *k_out, void *v_out, const void *q_window, const int32_t *seq_lens,
                             const int32_t *block_table, int32_t *out_keep_idx, int32_t *out_freed_off,
                             int32_t *out_freed_ids, int32_t *out_new_seq_lens, float *out_scores, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream)
{
    Plan pl;
    rkv_status st = make_plan(p, chunk_layers, &pl);
    if (st != RKV_OK)
        return st;
    const bool paged = p->layout == RKV_LAYOUT_PAGED;
    if (!k_in || !v_in || !k_out || !v_out || !q_window || !seq_lens || !out_keep_idx || !out_freed_off ||
        !out_new_seq_lens || (paged && (!block_table || !out_freed_ids)))
        return RKV_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < pl.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return RKV_ERR_WORKSPACE;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return RKV_ERR_CUDA;
    CopyEngine &e = g_engine[dev];
    std::lock_guard<std::mutex> lock(e.mu);
    if (!e.ready) {
        if (!create(e))
            return RKV_ERR_CUDA;
        e.ready = true;
    }
    st = enqueue(e, p, pl, k_in, v_in, k_out, v_out, q_window, seq_lens, block_table, out_keep_idx, out_freed_off,
                 out_freed_ids, out_new_seq_lens, out_scores, static_cast<uint8_t *>(workspace), stream);
    if (st != RKV_OK)
        join_after_error(e, stream);
    return st;
}

} // extern "C"
