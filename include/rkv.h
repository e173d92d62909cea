/*
 * rkv.h -- C ABI of librkv, the B300 (sm_103a) implementation of the R-KV
 * decode-time KV-cache compression event.
 *
 * The method (sources by page title and section):
 *   - "R-KV: Redundancy-Aware KV Cache Compression for Reasoning Models"
 *     (hysenlabs project review), section "How R-KV decides what to drop:
 *     budget, buffer and cross-layer scoring": compression runs at decode time
 *     once a sequence holds budget + buffer tokens; kv_budget tokens are kept;
 *     a local window (window_size) is protected; mix_lambda blends two scores;
 *     FREE_BLOCKS hands evicted blocks back to the allocator. Flag values in
 *     "Installing R-KV and running a first math evaluation".
 *   - hotdry.top blog "KV缓存压缩三剑客：R-KV、EvolKV与Ada-KV的工程实践",
 *     R-KV section: redundancy from the cosine similarity of key vectors,
 *     importance from multi-head attention, eviction by high importance and
 *     low redundancy, lambda about 0.1. Ada-KV section: paged blocks of 16.
 *
 * What one call computes, for every (layer l, sequence b, KV head h) with
 * N = seq_lens[b] cached tokens, G = Hq / Hkv and w = window:
 *   I_j  = mean over the w*G rows r (window position x query head of the
 *          group) of softmax_j(q_r . k_j / sqrt(d)), over all N keys;
 *   R_i  = mean over j != i of cos(k_i, k_j)  (divisor N-1; a zero key has
 *          cosine 0);
 *   I^, R^ = min-max normalised over the N tokens (a constant vector -> 0);
 *   S_j  = lambda * I^_j - (1 - lambda) * R^_j;
 *   keep = the last w tokens plus the (budget - w) largest S among the first
 *          N - w (equal S -> lower index), ascending; N <= budget keeps all
 *          (with RKV_SELECT_SHARED_HEADS, S summed over the KV heads);
 *   slot j of the head receives token keep[j] (K and V, in place);
 *   paged: blocks ceil(min(N,budget)/16) .. ceil(N/16)-1 of the sequence's
 *          block table are returned as freed (table order, batch order).
 *
 * Conventions for every entry point:
 *   - All data pointers are DEVICE pointers owned by the caller, except the
 *     cache, query and output pointers of rkv_compress_host, which are HOST
 *     pointers. No call allocates device memory; every call is asynchronous
 *     on `stream` and does not synchronise the host (except
 *     rkv_device_status).
 *   - bf16 tensors are raw 16-bit storage (e.g. torch.bfloat16), row-major.
 *   - Errors found on the host (shapes, alignment, sizes) return a status and
 *     launch nothing. Errors found on the device (a seq_len above max_seq_len,
 *     a block id outside the pool, invalid kept indices, a bounded in-kernel
 *     wait that gave up) set a per-device error word that rkv_device_status
 *     reports (one word shared by all calls on the device; see there); the
 *     affected heads are skipped and the cache contents for that sequence are
 *     then unspecified.
 *   - Entry points may be called from several host threads at once: the
 *     library's host-side caches (device attributes, kernel attributes,
 *     occupancy) are thread-safe.
 *   - Supported: head_dim == 128, 1 <= window <= budget, window * Hq/Hkv <= 64,
 *     max_seq_len <= 8192, paged block_size == 16, pointers 16-byte aligned.
 */
#ifndef RKV_H
#define RKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define RKV_API __attribute__((visibility("default")))
#else
#define RKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rkv_status {
    RKV_OK = 0,
    RKV_ERR_INVALID_ARG = 1,   /* bad shape/parameter/pointer, detected on the host */
    RKV_ERR_WORKSPACE = 2,     /* workspace missing or too small */
    RKV_ERR_UNSUPPORTED = 3,   /* valid but outside the supported envelope above */
    RKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    RKV_ERR_DEVICE = 5,        /* a kernel found invalid device-side input */
    RKV_ERR_TIMEOUT = 6        /* a bounded in-kernel wait gave up */
} rkv_status;

typedef enum rkv_layout {
    RKV_LAYOUT_CONTIGUOUS = 0, /* K/V: [L][B][Hkv][max_seq_len][d] */
    RKV_LAYOUT_PAGED = 1       /* K/V: [L][num_blocks][block_size][Hkv][d] + block_table */
} rkv_layout;

/*
 * How step 2 computes R_i (all give the mean pairwise key cosine above):
 *   RKV_REDUNDANCY_GRAM         a dense N x N key Gram per head on the tensor
 *                               cores, row-mean fused into the epilogue (the
 *                               default; 2*N^2*d flops per head);
 *   RKV_REDUNDANCY_CLOSED_FORM  the exact rank-one identity
 *                               sum_{j!=i} cos(k_i,k_j) = k^_i.(sum_j k^_j) - |k^_i|^2,
 *                               in a kernel of its own after importance: two
 *                               passes over each key row, the second from
 *                               shared memory for heads of up to 1280 keys
 *                               (HBM-bound; the fastest closed form on B300);
 *   RKV_REDUNDANCY_CLOSED_FORM_FUSED  the same identity inside the importance
 *                               kernel's pass over K (one launch for steps
 *                               1-2; HBM reads the keys once for both). It
 *                               spends more SM time than the two-kernel form
 *                               (the extra per-key work lands on the
 *                               importance kernel's epilogue): choose it when
 *                               HBM bandwidth, not SM time, is what the rest
 *                               of the workload competes for.
 * They agree to fp32 rounding (about 1e-6 on normalised scores).
 */
typedef enum rkv_redundancy_method {
    RKV_REDUNDANCY_GRAM = 0,
    RKV_REDUNDANCY_CLOSED_FORM = 1,
    RKV_REDUNDANCY_CLOSED_FORM_FUSED = 2
} rkv_redundancy_method;

/*
 * Which tokens step 4 keeps:
 *   RKV_SELECT_PER_HEAD      each (layer, sequence, KV head) keeps its own top
 *                            tokens by its own S (the default);
 *   RKV_SELECT_SHARED_HEADS  one keep set per (layer, sequence): the KV heads'
 *                            S (each normalised and blended per head) are
 *                            summed over the heads and the top tokens of the
 *                            sum are kept by every head -- the eviction that
 *                            tensor-parallel serving needs, where all ranks
 *                            must evict the same tokens (R-KV review page:
 *                            identical eviction on every rank, eviction-score
 *                            all-reduce; on one GPU the all-reduce is this
 *                            local sum over heads). A paged block then holds
 *                            the same tokens for every head.
 */
typedef enum rkv_selection {
    RKV_SELECT_PER_HEAD = 0,
    RKV_SELECT_SHARED_HEADS = 1
} rkv_selection;

/*
 * Which sequences one call compresses:
 *   RKV_TRIGGER_ANY                 every sequence holding more than budget
 *                                   tokens (the default; the caller decides
 *                                   when to call);
 *   RKV_TRIGGER_BUDGET_PLUS_BUFFER  only sequences holding at least
 *                                   budget + buffer tokens, decided on the
 *                                   device from seq_lens (R-KV review page:
 *                                   compression starts when the cache reaches
 *                                   budget + buffer). The other sequences are
 *                                   left as they are: no row moves, no block
 *                                   is freed, out_new_seq_lens = N_b and
 *                                   out_keep_idx holds the identity prefix.
 *                                   With this trigger the same call can run
 *                                   at every decode step, e.g. replayed from a
 *                                   captured CUDA graph.
 */
typedef enum rkv_trigger {
    RKV_TRIGGER_ANY = 0,
    RKV_TRIGGER_BUDGET_PLUS_BUFFER = 1
} rkv_trigger;

typedef struct rkv_problem {
    int32_t num_layers;         /* L */
    int32_t batch;              /* B */
    int32_t num_kv_heads;       /* Hkv */
    int32_t num_q_heads;        /* Hq, a multiple of Hkv (GQA: q head g -> KV head g / (Hq/Hkv)) */
    int32_t head_dim;           /* d, must be 128 */
    int32_t max_seq_len;        /* Nmax: upper bound of seq_lens; contiguous row capacity per head */
    int32_t layout;             /* rkv_layout */
    int32_t block_size;         /* paged: tokens per block, must be 16 */
    int32_t num_blocks;         /* paged: blocks in the pool (per layer plane) */
    int32_t max_blocks_per_seq; /* paged: row length of block_table, >= ceil(max_seq_len/16) */
    int32_t budget;             /* tokens kept per head (kv_budget) */
    int32_t buffer;             /* trigger slack: compression is due at budget+buffer tokens */
    int32_t window;             /* window_size: recent tokens always kept, and the query window */
    float mix_lambda;           /* lambda in S = lambda*I^ - (1-lambda)*R^ */
    int32_t redundancy;         /* rkv_redundancy_method (0: dense Gram) */
    int32_t selection;          /* rkv_selection (0: per KV head) */
    int32_t trigger;            /* rkv_trigger (0: compress whatever exceeds the budget) */
} rkv_problem;

/* Human-readable name of a status. Never NULL. */
RKV_API const char *rkv_status_string(rkv_status status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
RKV_API int rkv_version(void);

/* Per-head stride (in floats) of the score buffers used by the stage calls:
 * round_up(max_seq_len, 128). Score buffers are [L][B][Hkv][stride] fp32. */
RKV_API int32_t rkv_score_stride(const rkv_problem *p);

/* Bytes of device workspace rkv_compress needs (a multiple of 256). */
RKV_API rkv_status rkv_workspace_size(const rkv_problem *p, size_t *bytes);

/*
 * The whole compression event (all five steps) for every (layer, sequence,
 * KV head), launched on `stream`.
 *   k_cache, v_cache  bf16, in/out, layout per p->layout. Compacted in place:
 *                     slots [0, min(N_b, budget)) of each head receive the
 *                     kept tokens in ascending token order; the rest of the
 *                     head's rows are left as they were.
 *   q_window          bf16 [L][B][Hq][window][d]: the last `window` queries,
 *                     in any order along the window axis (importance is a
 *                     mean over the window rows), so a ring buffer that the
 *                     decode loop overwrites one position per step serves
 *                     as is.
 *   seq_lens          int32 [B]: N_b, 0 <= N_b <= max_seq_len.
 *   block_table       int32 [B][max_blocks_per_seq] (paged) or NULL
 *                     (contiguous). Read only. Entries below ceil(N_b/16)
 *                     must be distinct pool block ids, disjoint between
 *                     sequences.
 *   out_keep_idx      int32 [L][B][Hkv][budget]: kept token indices,
 *                     ascending, -1 past min(N_b, budget).
 *   out_freed_off     int32 [B+1]: CSR offsets of freed blocks per sequence
 *                     (all zero for the contiguous layout).
 *   out_freed_ids     int32 [B * max_blocks_per_seq] (paged) or NULL
 *                     (contiguous): freed block ids, sequence-major, table order.
 *   out_new_seq_lens  int32 [B]: min(N_b, budget).
 *   out_scores        NULL, or fp32 [3][L][B][Hkv][max_seq_len]: I^, R^, S
 *                     (entries at and past N_b are left untouched).
 *   workspace         device scratch of rkv_workspace_size bytes, 256-byte
 *                     aligned; its contents need no initialisation.
 * Returns RKV_OK once all kernels are queued.
 */
RKV_API rkv_status rkv_compress(const rkv_problem *p, void *k_cache, void *v_cache, const void *q_window,
                        const int32_t *seq_lens, const int32_t *block_table,
                        int32_t *out_keep_idx, int32_t *out_freed_off, int32_t *out_freed_ids,
                        int32_t *out_new_seq_lens, float *out_scores,
                        void *workspace, size_t workspace_bytes, cudaStream_t stream);

/*
 * rkv_compress without a caller-provided workspace. There is no counterpart
 * on the method's pages: this entry point exists for callers that cannot
 * allocate device memory at the point where they compress -- for example an
 * engine that has handed all free HBM to its KV block pool and runs its
 * decode step without access to an allocator, or a plugin host that gives
 * its extensions device pointers but no way to obtain more memory.
 *
 * Same arguments, computation and results as rkv_compress, minus `workspace`
 * and `workspace_bytes`. The scratch lives in one static device array of
 * RKV_NOALLOC_SCRATCH_BYTES per GPU (16 MiB), reserved on every GPU that
 * loads the library and held until the process exits. A problem whose
 * rkv_workspace_size exceeds it is rejected with RKV_ERR_WORKSPACE before
 * anything is launched (for instance, 32 layers x 8 KV heads x 1152 tokens
 * needs 3.4 MiB and fits; 28 layers x 128 sequences x 4 KV heads does not).
 * No cudaMalloc, cudaFree or other allocating call is made.
 *
 * The first call on each device looks up the array's device address (with
 * that device current) and caches it together with the id of the device's
 * current CUDA context. A call made in another context (for instance after
 * cudaDeviceReset, which tears the context down and loads the module again,
 * possibly at another address) looks the address up afresh. Make the first
 * call in each context before any stream capture. Every call on a device shares the one array, and calls whose
 * kernels overlap on the GPU (different streams, or different host threads)
 * race on it: serialise them. Each call writes every scratch value before
 * reading it, so nothing in the array needs to start at zero.
 */
#define RKV_NOALLOC_SCRATCH_BYTES (16u << 20)
RKV_API rkv_status rkv_compress_noalloc(const rkv_problem *p, void *k_cache, void *v_cache,
                                        const void *q_window, const int32_t *seq_lens,
                                        const int32_t *block_table, int32_t *out_keep_idx,
                                        int32_t *out_freed_off, int32_t *out_freed_ids,
                                        int32_t *out_new_seq_lens, float *out_scores, cudaStream_t stream);

/*
 * The compression event for a KV cache held in HOST memory: the offload tier
 * of a serving engine that parks long sequences' caches in CPU memory and
 * compresses them on the GPU. There is no counterpart on the method's pages;
 * the computation is rkv_compress's, on the same kernels.
 *
 * The layers are taken in chunks of `chunk_layers` (0: the library picks
 * about 20 MiB of K+V per chunk). Each chunk's K, V and q_window rows are
 * copied host->device into one of three device slots of the workspace,
 * rkv_compress runs on the slot (on `stream`), and the compacted K/V and kept
 * indices (and scores) are copied device->host. The copies run on two
 * library-owned streams of the current device, one per direction, so the
 * copies of successive chunks overlap each other and the kernels, and the
 * call takes about the longer of the two directions instead of their sum.
 *
 *   chunk_layers      layers per chunk, >= 0 (0: automatic).
 *   k_in, v_in        host, bf16, the cache as rkv_compress takes it
 *                     (contiguous or paged layout); read only.
 *   k_out, v_out      host, bf16, same shape: receive the whole compacted
 *                     cache; rows that rkv_compress leaves alone carry the
 *                     k_in / v_in values. May be the same buffers as k_in /
 *                     v_in.
 *   q_window, seq_lens, block_table, out_keep_idx, out_freed_off,
 *   out_freed_ids, out_new_seq_lens
 *                     host, shapes and meaning as for rkv_compress.
 *   out_scores        host fp32 [3][L][B][Hkv][max_seq_len], or NULL; entries
 *                     at and past N_b are written as 0.
 *   workspace         DEVICE scratch of rkv_compress_host_workspace_size
 *                     bytes (for the same problem and chunk_layers), 256-byte
 *                     aligned; its contents need no initialisation.
 *   stream            the kernels run on it. The copies are ordered after the
 *                     work already queued on `stream`, and `stream` waits for
 *                     all of them: once `stream` has been synchronised, every
 *                     host output is written.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister) for
 * the copies to overlap; pageable memory gives the same results with the
 * copies serialised. They must stay valid until `stream` has been
 * synchronised. Calls on one device share the library's copy streams and are
 * queued under a per-device lock, so they may come from several host
 * threads. Device-side errors are reported by rkv_device_status as for
 * rkv_compress. Argument checks (problem, pointers, workspace) happen before
 * anything is queued. If a later step fails (a CUDA error while queuing a
 * chunk), the call returns that status after making `stream` wait for every
 * copy it had already queued: keep the host buffers valid until `stream` has
 * been synchronised, whatever the status.
 */
RKV_API rkv_status rkv_compress_host_workspace_size(const rkv_problem *p, int32_t chunk_layers, size_t *bytes);
RKV_API rkv_status rkv_compress_host(const rkv_problem *p, int32_t chunk_layers, const void *k_in,
                                     const void *v_in, void *k_out, void *v_out, const void *q_window,
                                     const int32_t *seq_lens, const int32_t *block_table,
                                     int32_t *out_keep_idx, int32_t *out_freed_off, int32_t *out_freed_ids,
                                     int32_t *out_new_seq_lens, float *out_scores, void *workspace,
                                     size_t workspace_bytes, cudaStream_t stream);

/*
 * Step 1 alone (kernel rkv_importance): importance I (un-normalised) and the
 * fp32 inverse key norms 1/|k_j| (0 for a zero key) that step 2 consumes.
 *   out_importance, out_inv_norm  fp32 [L][B][Hkv][rkv_score_stride(p)];
 *                                 written for j < N_b only.
 */
RKV_API rkv_status rkv_importance(const rkv_problem *p, const void *k_cache, const void *q_window,
                          const int32_t *seq_lens, const int32_t *block_table,
                          float *out_importance, float *out_inv_norm, cudaStream_t stream);

/*
 * Steps 1-2 (importance, inverse key norms and redundancy). With
 * p->redundancy == RKV_REDUNDANCY_CLOSED_FORM_FUSED this is ONE launch of the
 * importance kernel that also forms R from the same pass over the keys (the
 * R-KV review page credits a fused redundancy kernel; the method's redundancy
 * is the mean pairwise key cosine, reached here through the exact rank-one
 * identity): while a CTA's key tiles stream through shared memory for the
 * attention scores, it also sums inv_j * k_j into S; the CTAs of a head
 * exchange their partial S with the softmax statistics; each key's k_j . S is
 * then taken from its row read a second time through L2 (the same CTA read it
 * microseconds earlier), so HBM sees the keys once. With the other methods
 * it is rkv_importance followed by rkv_redundancy (two launches).
 *   out_importance, out_inv_norm, out_redundancy  fp32 [L][B][Hkv][stride];
 *                                 written for j < N_b only.
 */
RKV_API rkv_status rkv_importance_redundancy(const rkv_problem *p, const void *k_cache, const void *q_window,
                                             const int32_t *seq_lens, const int32_t *block_table,
                                             float *out_importance, float *out_inv_norm, float *out_redundancy,
                                             cudaStream_t stream);

/*
 * Step 2 alone (kernel rkv_redundancy): redundancy R (un-normalised) from a
 * dense key Gram on the tensor cores, with the row mean fused in the epilogue,
 * or, with either closed-form method, from the rank-one identity (kernel
 * rkv_redundancy_closed).
 *   inv_norm        fp32 [L][B][Hkv][stride], as written by rkv_importance.
 *   out_redundancy  fp32 [L][B][Hkv][stride]; written for j < N_b only.
 */
RKV_API rkv_status rkv_redundancy(const rkv_problem *p, const void *k_cache, const int32_t *seq_lens,
                          const int32_t *block_table, const float *inv_norm,
                          float *out_redundancy, cudaStream_t stream);

/*
 * Steps 3-4 (kernel rkv_select): normalise, blend and select.
 *   importance, redundancy  fp32 [L][B][Hkv][stride], 16-byte aligned (each
 *                           head's row is copied to shared memory whole).
 *   out_keep_idx, out_scores as for rkv_compress (out_scores may be NULL).
 */
RKV_API rkv_status rkv_select(const rkv_problem *p, const float *importance, const float *redundancy,
                      const int32_t *seq_lens, int32_t *out_keep_idx, float *out_scores,
                      cudaStream_t stream);

/*
 * Step 5 (kernel rkv_compact): in-place ordered gather of K and V to the kept
 * slots, freed-block CSR and new lengths. keep_idx as written by rkv_select
 * (ascending, -1 padded); it is validated on the device before any row moves.
 */
RKV_API rkv_status rkv_compact(const rkv_problem *p, void *k_cache, void *v_cache, const int32_t *seq_lens,
                       const int32_t *block_table, const int32_t *keep_idx,
                       int32_t *out_freed_off, int32_t *out_freed_ids, int32_t *out_new_seq_lens,
                       cudaStream_t stream);

/*
 * Steps 3-5 in one launch (kernel rkv_select_compact): normalise, blend and
 * select as rkv_select does, then compact K and V and emit the freed blocks
 * and new lengths as rkv_compact does, with the kept indices handed from the
 * selection to the moves inside the kernel (shared memory of the head's CTA,
 * or of its cluster when there are fewer heads than SMs) instead of through a
 * second launch. rkv_compress uses it for
 * per-KV-head selection. Arguments as for rkv_select and rkv_compact:
 *   importance, redundancy  fp32 [L][B][Hkv][stride], 16-byte aligned;
 *   k_cache, v_cache        compacted in place;
 *   out_keep_idx            int32 [L][B][Hkv][budget], written as rkv_select
 *                           writes it (it is an output here, not an input);
 *   out_freed_off, out_freed_ids, out_new_seq_lens, out_scores  as for
 *                           rkv_compress (out_scores may be NULL).
 * With RKV_SELECT_SHARED_HEADS, or if a head's selection scratch does not
 * fit a CTA's shared memory, the call runs the rkv_select and rkv_compact
 * kernels one after the other instead (same results).
 */
RKV_API rkv_status rkv_select_compact(const rkv_problem *p, const float *importance, const float *redundancy,
                                      const int32_t *seq_lens, const int32_t *block_table, void *k_cache,
                                      void *v_cache, int32_t *out_keep_idx, int32_t *out_freed_off,
                                      int32_t *out_freed_ids, int32_t *out_new_seq_lens, float *out_scores,
                                      cudaStream_t stream);

/*
 * FREE_BLOCKS on the device (R-KV review page: evicted blocks go back to the
 * allocator instead of being stranded). Appends the blocks one rkv_compress
 * call freed -- its CSR output, total = freed_off[batch] ids -- to a
 * caller-owned device stack of free pool blocks:
 *   free_stack[*free_top .. *free_top + total) = freed_ids[0 .. total);
 *   *free_top += total.
 *   freed_off   int32 [batch + 1], freed_ids int32 [>= total] (device; as
 *               written by rkv_compress / rkv_compact on the same stream);
 *               freed_ids may be NULL for the contiguous layout, which never
 *               frees a block.
 *   free_stack  int32 [capacity], free_top int32 [1] (device).
 * One small kernel on `stream`; no host synchronisation, so it can follow
 * rkv_compress inside a captured CUDA graph. If the stack would overflow,
 * nothing is written and the device error word is set (RKV_ERR_DEVICE from
 * rkv_device_status).
 */
RKV_API rkv_status rkv_free_blocks_push(const int32_t *freed_off, const int32_t *freed_ids, int32_t batch,
                                        int32_t *free_stack, int32_t *free_top, int32_t capacity,
                                        cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the calling thread's current
 * device's error word: RKV_OK, RKV_ERR_DEVICE or RKV_ERR_TIMEOUT (or
 * RKV_ERR_CUDA if the synchronisation itself failed).
 * There is ONE error word per device, shared by every call on every stream
 * and host thread of the process: it holds the first device-side error since
 * it was last cleared, with no record of which call raised it, and a read
 * clears it for everyone. A caller that needs to attribute an error to one
 * call should check the status after that call alone, with no other call on
 * the device in flight.
 */
RKV_API rkv_status rkv_device_status(cudaStream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* RKV_H */
