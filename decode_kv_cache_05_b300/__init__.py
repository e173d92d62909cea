"""R-KV decode-time KV-cache compression on one B300 (sm_103a).

The product is the C-ABI library librkv.so (include/rkv.h); this package is its
Python binding: argument marshalling with torch tensors for device memory and
streams. See `rkv_compress` for the whole event and the stage calls
(`rkv_importance`, `rkv_redundancy`, `rkv_select_compact`, or `rkv_select` and
`rkv_compact` separately) for its kernels one at a time; `rkv_compress_host`
runs the event on a cache held in host memory, with the copies overlapped.
"""

from ._binding import (  # noqa: F401
    EXPORTS,
    LAYOUT_CONTIGUOUS,
    LAYOUT_PAGED,
    LIB_PATH,
    RKV_ERR_CUDA,
    RKV_ERR_DEVICE,
    RKV_ERR_INVALID_ARG,
    RKV_ERR_TIMEOUT,
    RKV_ERR_UNSUPPORTED,
    RKV_ERR_WORKSPACE,
    NOALLOC_SCRATCH_BYTES,
    REDUNDANCY_CLOSED_FORM,
    REDUNDANCY_CLOSED_FORM_FUSED,
    REDUNDANCY_GRAM,
    SELECT_PER_HEAD,
    SELECT_SHARED_HEADS,
    TRIGGER_ANY,
    TRIGGER_BUDGET_PLUS_BUFFER,
    RKV_OK,
    Problem,
    RKVError,
    allocate_outputs,
    library,
    make_problem,
    rkv_compact,
    rkv_compress,
    rkv_compress_host,
    rkv_compress_noalloc,
    rkv_device_status,
    rkv_free_blocks_push,
    rkv_importance,
    rkv_importance_redundancy,
    rkv_redundancy,
    rkv_select,
    rkv_select_compact,
    host_workspace_size,
    score_stride,
    status_string,
    workspace_size,
)


def problem_for(shape, num_blocks: int = 0, redundancy: int = REDUNDANCY_GRAM,
                selection: int = SELECT_PER_HEAD, trigger: int = TRIGGER_ANY) -> Problem:
    """rkv_problem for a workload shape (any object with the attributes
    layers, batch, kv_heads, q_heads, head_dim, max_seq_len, budget, buffer,
    window, mix_lambda, paged, block_size, blocks_per_seq)."""
    return make_problem(num_layers=shape.layers, batch=shape.batch, num_kv_heads=shape.kv_heads,
                        num_q_heads=shape.q_heads, head_dim=shape.head_dim, max_seq_len=shape.max_seq_len,
                        budget=shape.budget, buffer=shape.buffer, window=shape.window,
                        mix_lambda=shape.mix_lambda, paged=shape.paged, block_size=shape.block_size,
                        num_blocks=num_blocks, max_blocks_per_seq=shape.blocks_per_seq if shape.paged else 0,
                        redundancy=redundancy, selection=selection, trigger=trigger)
