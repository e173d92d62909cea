"""CPU oracle for the R-KV compression event -- TEST INFRASTRUCTURE ONLY.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import
this package. It is a plain fp64 C restatement of the method (rkv_oracle.c;
the readings taken where the pages are silent are listed in rkv_oracle.h) with
numpy marshalling here. It shares no code with the CUDA library.

Parity pins (tests/test_oracle_pins.py): hand-derived tiny examples
(tests/golden/), the rank-1 closed form of the mean cosine, softmax sums,
orthonormal/duplicate key invariants, scale invariance, the lambda = 0 / 1
limits, brute-force subset enumeration for the selection, and a naive gather
for compaction. No function here is "parity unpinned".
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rkv_oracle.c")
_HDR = os.path.join(_HERE, "rkv_oracle.h")
_LIB = os.path.join(_HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP over heads). Returns the .so path."""
    stale = (not os.path.exists(_LIB) or
             os.path.getmtime(_LIB) < max(os.path.getmtime(_SRC), os.path.getmtime(_HDR)))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


class _Problem(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "layers", "batch", "kv_heads", "q_heads", "head_dim", "max_seq_len",
        "paged", "block_size", "num_blocks", "max_blocks", "budget", "window")] + [
        ("mix_lambda", ctypes.c_double)]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.POINTER
        u16, i32, f64 = P(ctypes.c_uint16), P(ctypes.c_int32), P(ctypes.c_double)
        lib.orc_importance.argtypes = [u16, ctypes.c_int, u16, ctypes.c_int, ctypes.c_int, f64]
        lib.orc_redundancy.argtypes = [u16, ctypes.c_int, ctypes.c_int, f64]
        lib.orc_minmax.argtypes = [f64, ctypes.c_int, f64]
        lib.orc_mix.argtypes = [f64, f64, ctypes.c_int, ctypes.c_double, f64]
        lib.orc_select.argtypes = [f64, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32]
        lib.orc_select.restype = ctypes.c_int
        lib.orc_redundancy_closed.argtypes = [u16, ctypes.c_int, ctypes.c_int, f64]
        for name in ("orc_compress", "orc_compress_closed"):
            getattr(lib, name).argtypes = [P(_Problem), u16, u16, u16, i32, i32, i32, i32, i32, i32, f64]
            getattr(lib, name).restype = ctypes.c_int
        lib.orc_compact.argtypes = [P(_Problem), u16, u16, i32, i32, i32]
        lib.orc_compact.restype = ctypes.c_int
        lib.orc_freed_blocks.argtypes = [P(_Problem), i32, i32, i32, i32, i32]
        lib.orc_freed_blocks.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray], ctype):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, "bf16 data is passed as raw uint16 bit patterns"
    return a


def bf16_bits_from_float(x: np.ndarray) -> np.ndarray:
    """Round float values to bf16 (nearest even) and return the bit patterns.
    Used by the pins to build exact small inputs."""
    f = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)


def bf16_to_float(bits: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


# ---- per-head definitions -------------------------------------------------

def importance(q: np.ndarray, k: np.ndarray) -> np.ndarray:
    """q: [rows][d] bf16 bits, k: [n][d] bf16 bits -> I [n] (fp64)."""
    q, k = _u16(q), _u16(k)
    n, d = k.shape
    out = np.zeros(n, dtype=np.float64)
    _load().orc_importance(_ptr(q, ctypes.c_uint16), q.shape[0], _ptr(k, ctypes.c_uint16), n, d,
                           _ptr(out, ctypes.c_double))
    return out


def redundancy(k: np.ndarray) -> np.ndarray:
    """k: [n][d] bf16 bits -> R [n] (fp64), mean pairwise cosine, self excluded."""
    k = _u16(k)
    n, d = k.shape
    out = np.zeros(n, dtype=np.float64)
    _load().orc_redundancy(_ptr(k, ctypes.c_uint16), n, d, _ptr(out, ctypes.c_double))
    return out


def redundancy_closed(k: np.ndarray) -> np.ndarray:
    """The same R from the rank-one identity of the cosine sum (two passes
    over the keys); equal to redundancy() up to fp64 rounding."""
    k = _u16(k)
    n, d = k.shape
    out = np.zeros(n, dtype=np.float64)
    _load().orc_redundancy_closed(_ptr(k, ctypes.c_uint16), n, d, _ptr(out, ctypes.c_double))
    return out


def minmax(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    _load().orc_minmax(_ptr(x, ctypes.c_double), x.size, _ptr(out, ctypes.c_double))
    return out


def mix(imp_hat: np.ndarray, red_hat: np.ndarray, lam: float) -> np.ndarray:
    a = np.ascontiguousarray(imp_hat, dtype=np.float64)
    b = np.ascontiguousarray(red_hat, dtype=np.float64)
    out = np.zeros_like(a)
    _load().orc_mix(_ptr(a, ctypes.c_double), _ptr(b, ctypes.c_double), a.size, lam,
                    _ptr(out, ctypes.c_double))
    return out


def select(s: np.ndarray, budget: int, window: int) -> np.ndarray:
    """Kept indices (ascending, -1 padded to `budget`)."""
    s = np.ascontiguousarray(s, dtype=np.float64)
    keep = np.full(budget, -1, dtype=np.int32)
    _load().orc_select(_ptr(s, ctypes.c_double), s.size, budget, window, _ptr(keep, ctypes.c_int32))
    return keep


def select_shared(S: np.ndarray, n: int, budget: int, window: int) -> np.ndarray:
    """Eviction shared by the KV heads of one (layer, sequence): S[h][j] are
    the heads' blended scores; the per-token score is their sum over the heads
    (R-KV review page: every tensor-parallel rank evicts the same tokens, the
    SGLang port all-reduces the eviction scores; on one device that reduction
    is this sum), and the ordinary windowed top-budget rule is applied to it.
    Returns the kept indices (ascending, -1 padded), the same for every head."""
    total = np.zeros(n, dtype=np.float64)
    for h in range(S.shape[0]):
        total += np.asarray(S[h, :n], dtype=np.float64)
    return select(total, budget, window), total


def compress_head(q: np.ndarray, k: np.ndarray, budget: int, window: int, lam: float) -> dict:
    """All scores and the kept list of one (layer, sequence, KV head)."""
    I = importance(q, k)
    R = redundancy(k)
    Ih, Rh = minmax(I), minmax(R)
    S = mix(Ih, Rh, lam)
    return dict(I=I, R=R, I_hat=Ih, R_hat=Rh, S=S, keep=select(S, budget, window))


# ---- whole event ----------------------------------------------------------

def problem(*, layers, batch, kv_heads, q_heads, head_dim, max_seq_len, budget, window, mix_lambda,
            paged=False, block_size=16, num_blocks=0, max_blocks=0) -> _Problem:
    return _Problem(layers, batch, kv_heads, q_heads, head_dim, max_seq_len, int(paged), block_size,
                    num_blocks, max_blocks, budget, window, float(mix_lambda))


def compress(p: _Problem, k_cache: np.ndarray, v_cache: np.ndarray, q_window: np.ndarray,
             seq_lens: np.ndarray, block_table: Optional[np.ndarray] = None,
             closed_form: bool = False) -> dict:
    """Run the event on host copies. k_cache/v_cache are modified in place
    (pass copies). Returns keep_idx, freed_off, freed_ids, new_seq_lens and
    the score planes I, R, I_hat, R_hat, S ([L][B][Hkv][Nmax], zero past N_b).
    closed_form: redundancy by the rank-one identity instead of the pairwise sum."""
    k_cache, v_cache, q_window = _u16(k_cache), _u16(v_cache), _u16(q_window)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    L, B, H, N = p.layers, p.batch, p.kv_heads, p.max_seq_len
    keep = np.full((L, B, H, p.budget), -1, dtype=np.int32)
    freed_off = np.zeros(B + 1, dtype=np.int32)
    freed_ids = np.zeros(max(1, B * max(p.max_blocks, 1)), dtype=np.int32)
    new_lens = np.zeros(B, dtype=np.int32)
    scores = np.zeros((5, L, B, H, N), dtype=np.float64)
    fn = _load().orc_compress_closed if closed_form else _load().orc_compress
    rc = fn(ctypes.byref(p), _ptr(k_cache, ctypes.c_uint16), _ptr(v_cache, ctypes.c_uint16),
            _ptr(q_window, ctypes.c_uint16), _ptr(seq_lens, ctypes.c_int32),
            _ptr(bt, ctypes.c_int32), _ptr(keep, ctypes.c_int32),
            _ptr(freed_off, ctypes.c_int32), _ptr(freed_ids, ctypes.c_int32),
            _ptr(new_lens, ctypes.c_int32), _ptr(scores, ctypes.c_double))
    if rc:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return dict(keep_idx=keep, freed_off=freed_off, freed_ids=freed_ids[:freed_off[-1]].copy(),
                new_seq_lens=new_lens, I=scores[0], R=scores[1], I_hat=scores[2], R_hat=scores[3],
                S=scores[4])


def compact(p: _Problem, k_cache: np.ndarray, v_cache: np.ndarray, seq_lens: np.ndarray,
            block_table: Optional[np.ndarray], keep_idx: np.ndarray) -> None:
    """In-place gather of K/V with given kept indices (host copies)."""
    k_cache, v_cache = _u16(k_cache), _u16(v_cache)
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    keep_idx = np.ascontiguousarray(keep_idx, dtype=np.int32)
    rc = _load().orc_compact(ctypes.byref(p), _ptr(k_cache, ctypes.c_uint16), _ptr(v_cache, ctypes.c_uint16),
                             _ptr(seq_lens, ctypes.c_int32), _ptr(bt, ctypes.c_int32),
                             _ptr(keep_idx, ctypes.c_int32))
    if rc:
        raise ValueError(f"oracle rejected the compaction (code {rc})")


def freed_blocks(p: _Problem, seq_lens: np.ndarray, block_table: Optional[np.ndarray]):
    seq_lens = np.ascontiguousarray(seq_lens, dtype=np.int32)
    bt = None if block_table is None else np.ascontiguousarray(block_table, dtype=np.int32)
    B = p.batch
    freed_off = np.zeros(B + 1, dtype=np.int32)
    freed_ids = np.zeros(max(1, B * max(p.max_blocks, 1)), dtype=np.int32)
    new_lens = np.zeros(B, dtype=np.int32)
    rc = _load().orc_freed_blocks(ctypes.byref(p), _ptr(seq_lens, ctypes.c_int32), _ptr(bt, ctypes.c_int32),
                                  _ptr(freed_off, ctypes.c_int32), _ptr(freed_ids, ctypes.c_int32),
                                  _ptr(new_lens, ctypes.c_int32))
    if rc:
        raise ValueError(f"oracle rejected the problem (code {rc})")
    return freed_off, freed_ids[:freed_off[-1]].copy(), new_lens
