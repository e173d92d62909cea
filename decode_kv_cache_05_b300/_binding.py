"""ctypes binding of librkv (include/rkv.h). Argument marshalling only: every
step of the compression event runs in the library's CUDA kernels. Torch is
used for device memory and streams.

The library is built in-tree (decode_kv_cache_05_b300/librkv.so). If it is
missing, every call raises; there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "librkv.so")

RKV_OK = 0
RKV_ERR_INVALID_ARG = 1
RKV_ERR_WORKSPACE = 2
RKV_ERR_UNSUPPORTED = 3
RKV_ERR_CUDA = 4
RKV_ERR_DEVICE = 5
RKV_ERR_TIMEOUT = 6

LAYOUT_CONTIGUOUS = 0
LAYOUT_PAGED = 1

REDUNDANCY_GRAM = 0                # dense key Gram on the tensor cores
REDUNDANCY_CLOSED_FORM = 1         # exact rank-one identity, a kernel of its own after importance
REDUNDANCY_CLOSED_FORM_FUSED = 2   # the same identity inside importance's pass over the keys

SELECT_PER_HEAD = 0          # each KV head keeps its own tokens
SELECT_SHARED_HEADS = 1      # one keep set per (layer, sequence) from S summed over the KV heads

TRIGGER_ANY = 0                     # compress every sequence above the budget
TRIGGER_BUDGET_PLUS_BUFFER = 1      # only sequences holding budget + buffer tokens (decided on the device)

EXPORTS = ("rkv_status_string", "rkv_version", "rkv_score_stride", "rkv_workspace_size", "rkv_compress",
           "rkv_importance", "rkv_redundancy", "rkv_select", "rkv_compact", "rkv_device_status",
           "rkv_compress_noalloc", "rkv_free_blocks_push", "rkv_compress_host",
           "rkv_compress_host_workspace_size", "rkv_select_compact", "rkv_importance_redundancy")

# Size of the static device scratch behind rkv_compress_noalloc (include/rkv.h).
NOALLOC_SCRATCH_BYTES = 16 << 20


class RKVError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Problem(ctypes.Structure):
    """Mirror of struct rkv_problem."""
    _fields_ = [(n, ctypes.c_int32) for n in (
        "num_layers", "batch", "num_kv_heads", "num_q_heads", "head_dim", "max_seq_len", "layout",
        "block_size", "num_blocks", "max_blocks_per_seq", "budget", "buffer", "window")] + [
        ("mix_lambda", ctypes.c_float), ("redundancy", ctypes.c_int32), ("selection", ctypes.c_int32),
        ("trigger", ctypes.c_int32)]

    @property
    def paged(self) -> bool:
        return self.layout == LAYOUT_PAGED

    @property
    def heads(self) -> int:
        return self.num_layers * self.batch * self.num_kv_heads


def make_problem(*, num_layers, batch, num_kv_heads, num_q_heads, max_seq_len, budget, window, mix_lambda,
                 buffer=0, head_dim=128, paged=False, block_size=16, num_blocks=0,
                 max_blocks_per_seq=0, redundancy=REDUNDANCY_GRAM, selection=SELECT_PER_HEAD,
                 trigger=TRIGGER_ANY) -> Problem:
    return Problem(num_layers, batch, num_kv_heads, num_q_heads, head_dim, max_seq_len,
                   LAYOUT_PAGED if paged else LAYOUT_CONTIGUOUS, block_size, num_blocks, max_blocks_per_seq,
                   budget, buffer, window, float(mix_lambda), int(redundancy), int(selection), int(trigger))


_lib = None


def library() -> ctypes.CDLL:
    """Loads librkv.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"librkv.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                               "or python -m decode_kv_cache_05_b300.build")
        lib = ctypes.CDLL(LIB_PATH)
        P = ctypes.POINTER(Problem)
        vp, i32p, f32p = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p
        lib.rkv_status_string.argtypes = [ctypes.c_int]
        lib.rkv_status_string.restype = ctypes.c_char_p
        lib.rkv_version.restype = ctypes.c_int
        lib.rkv_score_stride.argtypes = [P]
        lib.rkv_score_stride.restype = ctypes.c_int32
        lib.rkv_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
        lib.rkv_compress.argtypes = [P, vp, vp, vp, i32p, i32p, i32p, i32p, i32p, i32p, f32p, vp, ctypes.c_size_t, vp]
        lib.rkv_importance.argtypes = [P, vp, vp, i32p, i32p, f32p, f32p, vp]
        lib.rkv_importance_redundancy.argtypes = [P, vp, vp, i32p, i32p, f32p, f32p, f32p, vp]
        lib.rkv_redundancy.argtypes = [P, vp, i32p, i32p, f32p, f32p, vp]
        lib.rkv_select.argtypes = [P, f32p, f32p, i32p, i32p, f32p, vp]
        lib.rkv_compact.argtypes = [P, vp, vp, i32p, i32p, i32p, i32p, i32p, i32p, vp]
        lib.rkv_select_compact.argtypes = [P, f32p, f32p, i32p, i32p, vp, vp, i32p, i32p, i32p, i32p, f32p, vp]
        lib.rkv_device_status.argtypes = [vp]
        lib.rkv_compress_noalloc.argtypes = [P, vp, vp, vp, i32p, i32p, i32p, i32p, i32p, i32p, f32p, vp]
        lib.rkv_free_blocks_push.argtypes = [i32p, i32p, ctypes.c_int32, i32p, i32p, ctypes.c_int32, vp]
        lib.rkv_compress_host_workspace_size.argtypes = [P, ctypes.c_int32, ctypes.POINTER(ctypes.c_size_t)]
        lib.rkv_compress_host.argtypes = [P, ctypes.c_int32, vp, vp, vp, vp, vp, i32p, i32p, i32p, i32p, i32p, i32p,
                                          f32p, vp, ctypes.c_size_t, vp]
        for name in ("rkv_workspace_size", "rkv_compress", "rkv_importance", "rkv_redundancy", "rkv_select",
                     "rkv_compact", "rkv_device_status", "rkv_compress_noalloc", "rkv_free_blocks_push",
                     "rkv_compress_host", "rkv_compress_host_workspace_size", "rkv_select_compact",
                     "rkv_importance_redundancy"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return library().rkv_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != RKV_OK:
        raise RKVError(status, where)


def _ptr(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None, name: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _hptr(t: Optional[torch.Tensor], dtype: Optional[torch.dtype] = None, name: str = "tensor") -> Optional[int]:
    """Host pointer of a CPU tensor (page-locked for the copies to overlap)."""
    if t is None:
        return None
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a CPU tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def score_stride(p: Problem) -> int:
    return int(library().rkv_score_stride(ctypes.byref(p)))


def workspace_size(p: Problem) -> int:
    n = ctypes.c_size_t(0)
    _check(library().rkv_workspace_size(ctypes.byref(p), ctypes.byref(n)), "rkv_workspace_size")
    return int(n.value)


def allocate_outputs(p: Problem, device, scores: bool = False) -> dict:
    """Caller-owned output and workspace buffers for rkv_compress (torch allocations)."""
    out = {
        "keep_idx": torch.empty((p.num_layers, p.batch, p.num_kv_heads, p.budget), dtype=torch.int32, device=device),
        "freed_off": torch.empty(p.batch + 1, dtype=torch.int32, device=device),
        "freed_ids": torch.empty(max(1, p.batch * max(p.max_blocks_per_seq, 1)), dtype=torch.int32, device=device),
        "new_seq_lens": torch.empty(p.batch, dtype=torch.int32, device=device),
        "scores": (torch.zeros((3, p.num_layers, p.batch, p.num_kv_heads, p.max_seq_len), dtype=torch.float32,
                               device=device) if scores else None),
        "workspace": torch.empty(max(256, workspace_size(p)), dtype=torch.uint8, device=device),
    }
    return out


def rkv_compress(p: Problem, k_cache: torch.Tensor, v_cache: torch.Tensor, q_window: torch.Tensor,
                 seq_lens: torch.Tensor, block_table: Optional[torch.Tensor], keep_idx: torch.Tensor,
                 freed_off: torch.Tensor, freed_ids: Optional[torch.Tensor], new_seq_lens: torch.Tensor,
                 scores: Optional[torch.Tensor], workspace: torch.Tensor,
                 stream: Optional[torch.cuda.Stream] = None) -> None:
    st = library().rkv_compress(
        ctypes.byref(p), _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
        _ptr(q_window, torch.bfloat16, "q_window"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(block_table, torch.int32, "block_table"), _ptr(keep_idx, torch.int32, "keep_idx"),
        _ptr(freed_off, torch.int32, "freed_off"), _ptr(freed_ids, torch.int32, "freed_ids"),
        _ptr(new_seq_lens, torch.int32, "new_seq_lens"), _ptr(scores, torch.float32, "scores"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "rkv_compress")


def rkv_compress_noalloc(p: Problem, k_cache: torch.Tensor, v_cache: torch.Tensor, q_window: torch.Tensor,
                         seq_lens: torch.Tensor, block_table: Optional[torch.Tensor], keep_idx: torch.Tensor,
                         freed_off: torch.Tensor, freed_ids: Optional[torch.Tensor], new_seq_lens: torch.Tensor,
                         scores: Optional[torch.Tensor], stream: Optional[torch.cuda.Stream] = None) -> None:
    """rkv_compress for callers that cannot provide a device workspace: the
    library's static per-GPU scratch (NOALLOC_SCRATCH_BYTES) is used instead.
    Calls that overlap on one GPU race on that scratch; serialise them."""
    st = library().rkv_compress_noalloc(
        ctypes.byref(p), _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
        _ptr(q_window, torch.bfloat16, "q_window"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(block_table, torch.int32, "block_table"), _ptr(keep_idx, torch.int32, "keep_idx"),
        _ptr(freed_off, torch.int32, "freed_off"), _ptr(freed_ids, torch.int32, "freed_ids"),
        _ptr(new_seq_lens, torch.int32, "new_seq_lens"), _ptr(scores, torch.float32, "scores"), _stream(stream))
    _check(st, "rkv_compress_noalloc")


def host_workspace_size(p: Problem, chunk_layers: int = 0) -> int:
    """Device workspace bytes of rkv_compress_host for this problem and chunking."""
    n = ctypes.c_size_t(0)
    _check(library().rkv_compress_host_workspace_size(ctypes.byref(p), int(chunk_layers), ctypes.byref(n)),
           "rkv_compress_host_workspace_size")
    return int(n.value)


def rkv_compress_host(p: Problem, k_in: torch.Tensor, v_in: torch.Tensor, k_out: torch.Tensor,
                      v_out: torch.Tensor, q_window: torch.Tensor, seq_lens: torch.Tensor,
                      block_table: Optional[torch.Tensor], keep_idx: torch.Tensor, freed_off: torch.Tensor,
                      freed_ids: Optional[torch.Tensor], new_seq_lens: torch.Tensor, scores: Optional[torch.Tensor],
                      workspace: torch.Tensor, chunk_layers: int = 0,
                      stream: Optional[torch.cuda.Stream] = None) -> None:
    """The compression event on a KV cache in host memory: every tensor but
    `workspace` (a CUDA tensor of host_workspace_size bytes) is a CPU tensor,
    best page-locked. Chunks of layers are uploaded, compressed and downloaded
    with the copies overlapped; the host outputs are complete once `stream`
    has been synchronised."""
    st = library().rkv_compress_host(
        ctypes.byref(p), int(chunk_layers), _hptr(k_in, torch.bfloat16, "k_in"), _hptr(v_in, torch.bfloat16, "v_in"),
        _hptr(k_out, torch.bfloat16, "k_out"), _hptr(v_out, torch.bfloat16, "v_out"),
        _hptr(q_window, torch.bfloat16, "q_window"), _hptr(seq_lens, torch.int32, "seq_lens"),
        _hptr(block_table, torch.int32, "block_table"), _hptr(keep_idx, torch.int32, "keep_idx"),
        _hptr(freed_off, torch.int32, "freed_off"), _hptr(freed_ids, torch.int32, "freed_ids"),
        _hptr(new_seq_lens, torch.int32, "new_seq_lens"), _hptr(scores, torch.float32, "scores"),
        _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(), _stream(stream))
    _check(st, "rkv_compress_host")


def rkv_importance(p: Problem, k_cache, q_window, seq_lens, block_table, out_importance, out_inv_norm,
                   stream=None) -> None:
    st = library().rkv_importance(
        ctypes.byref(p), _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(q_window, torch.bfloat16, "q_window"),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(out_importance, torch.float32, "out_importance"), _ptr(out_inv_norm, torch.float32, "out_inv_norm"),
        _stream(stream))
    _check(st, "rkv_importance")


def rkv_importance_redundancy(p: Problem, k_cache, q_window, seq_lens, block_table, out_importance, out_inv_norm,
                              out_redundancy, stream=None) -> None:
    st = library().rkv_importance_redundancy(
        ctypes.byref(p), _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(q_window, torch.bfloat16, "q_window"),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(out_importance, torch.float32, "out_importance"), _ptr(out_inv_norm, torch.float32, "out_inv_norm"),
        _ptr(out_redundancy, torch.float32, "out_redundancy"), _stream(stream))
    _check(st, "rkv_importance_redundancy")


def rkv_redundancy(p: Problem, k_cache, seq_lens, block_table, inv_norm, out_redundancy, stream=None) -> None:
    st = library().rkv_redundancy(
        ctypes.byref(p), _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(block_table, torch.int32, "block_table"), _ptr(inv_norm, torch.float32, "inv_norm"),
        _ptr(out_redundancy, torch.float32, "out_redundancy"), _stream(stream))
    _check(st, "rkv_redundancy")


def rkv_select(p: Problem, importance, redundancy, seq_lens, out_keep_idx, out_scores=None, stream=None) -> None:
    st = library().rkv_select(
        ctypes.byref(p), _ptr(importance, torch.float32, "importance"),
        _ptr(redundancy, torch.float32, "redundancy"), _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(out_keep_idx, torch.int32, "out_keep_idx"), _ptr(out_scores, torch.float32, "out_scores"),
        _stream(stream))
    _check(st, "rkv_select")


def rkv_compact(p: Problem, k_cache, v_cache, seq_lens, block_table, keep_idx, out_freed_off, out_freed_ids,
                out_new_seq_lens, stream=None) -> None:
    st = library().rkv_compact(
        ctypes.byref(p), _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(keep_idx, torch.int32, "keep_idx"), _ptr(out_freed_off, torch.int32, "out_freed_off"),
        _ptr(out_freed_ids, torch.int32, "out_freed_ids"), _ptr(out_new_seq_lens, torch.int32, "out_new_seq_lens"),
        _stream(stream))
    _check(st, "rkv_compact")


def rkv_select_compact(p: Problem, importance, redundancy, seq_lens, block_table, k_cache, v_cache, out_keep_idx,
                       out_freed_off, out_freed_ids, out_new_seq_lens, out_scores=None, stream=None) -> None:
    st = library().rkv_select_compact(
        ctypes.byref(p), _ptr(importance, torch.float32, "importance"), _ptr(redundancy, torch.float32, "redundancy"),
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(block_table, torch.int32, "block_table"),
        _ptr(k_cache, torch.bfloat16, "k_cache"), _ptr(v_cache, torch.bfloat16, "v_cache"),
        _ptr(out_keep_idx, torch.int32, "out_keep_idx"), _ptr(out_freed_off, torch.int32, "out_freed_off"),
        _ptr(out_freed_ids, torch.int32, "out_freed_ids"), _ptr(out_new_seq_lens, torch.int32, "out_new_seq_lens"),
        _ptr(out_scores, torch.float32, "out_scores"), _stream(stream))
    _check(st, "rkv_select_compact")


def rkv_free_blocks_push(freed_off, freed_ids, batch: int, free_stack, free_top, stream=None) -> None:
    """Appends the freed block ids of a compression call to a device stack of
    free blocks (free_stack int32 [capacity], free_top int32 [1])."""
    st = library().rkv_free_blocks_push(
        _ptr(freed_off, torch.int32, "freed_off"), _ptr(freed_ids, torch.int32, "freed_ids"), int(batch),
        _ptr(free_stack, torch.int32, "free_stack"), _ptr(free_top, torch.int32, "free_top"),
        int(free_stack.numel()), _stream(stream))
    _check(st, "rkv_free_blocks_push")


def rkv_device_status(stream=None) -> int:
    """Synchronises the stream; returns and clears the device error word."""
    return int(library().rkv_device_status(_stream(stream)))
