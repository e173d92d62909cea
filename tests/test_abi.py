"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point declared in include/rkv.h, and rejects invalid problems
before touching the device."""

import ctypes
import os
import re

import pytest

import decode_kv_cache_05_b300 as rkv
from decode_kv_cache_05_b300 import build as rkv_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    rkv_build.build()
    return rkv.library()


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "rkv.h")).read()
    return sorted(set(re.findall(r"RKV_API\s+[\w\s\*]*?\b(rkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    assert {"rkv_compress", "rkv_workspace_size", "rkv_status_string", "rkv_importance", "rkv_redundancy",
            "rkv_select", "rkv_compact", "rkv_device_status"} <= set(names)
    assert set(names) == set(rkv.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name
    assert lib.rkv_version() >= 100


def test_noalloc_scratch_size_matches_header():
    """The binding's copy of RKV_NOALLOC_SCRATCH_BYTES is the header's."""
    text = open(os.path.join(ROOT, "include", "rkv.h")).read()
    m = re.search(r"#define\s+RKV_NOALLOC_SCRATCH_BYTES\s+\((\d+)u\s*<<\s*(\d+)\)", text)
    assert m, "RKV_NOALLOC_SCRATCH_BYTES not found in include/rkv.h"
    assert rkv.NOALLOC_SCRATCH_BYTES == int(m.group(1)) << int(m.group(2))


def test_host_queries_are_thread_safe(lib):
    """Several host threads asking for workspace sizes at once get the same
    answers as one thread (the library's host-side caches are thread-safe)."""
    import threading
    problems = [_p(), _p(num_layers=2, batch=3), _p(paged=True, num_blocks=500, max_blocks_per_seq=72)]
    want = [(rkv.workspace_size(q), rkv.host_workspace_size(q)) for q in problems]
    errors = []

    def worker():
        try:
            for _ in range(200):
                for q, w in zip(problems, want):
                    assert (rkv.workspace_size(q), rkv.host_workspace_size(q)) == w
        except Exception as exc:  # noqa: BLE001 - reported below
            errors.append(exc)

    threads = [threading.Thread(target=worker) for _ in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors[0]


def test_status_strings(lib):
    for code in range(7):
        assert rkv.status_string(code)
    assert rkv.status_string(99) == "unknown status"


def _p(**kw):
    base = dict(num_layers=32, batch=1, num_kv_heads=8, num_q_heads=32, max_seq_len=1152, budget=1024,
                window=8, mix_lambda=0.1, buffer=128)
    base.update(kw)
    return rkv.make_problem(**base)


def test_workspace_size_and_stride(lib):
    p = _p()
    assert rkv.score_stride(p) == 1152
    # three fp32 planes [L][B][Hkv][stride], each rounded up to 256 bytes
    assert rkv.workspace_size(p) == 3 * (32 * 8 * 1152 * 4)
    p2 = _p(max_seq_len=1100)
    assert rkv.score_stride(p2) == 1152


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=64), rkv.RKV_ERR_UNSUPPORTED),
    (dict(window=0), rkv.RKV_ERR_INVALID_ARG),
    (dict(window=2000), rkv.RKV_ERR_INVALID_ARG),
    (dict(num_q_heads=30), rkv.RKV_ERR_INVALID_ARG),
    (dict(max_seq_len=9000), rkv.RKV_ERR_UNSUPPORTED),
    (dict(window=32), rkv.RKV_ERR_UNSUPPORTED),           # 32 * 4 = 128 query rows > 64
    (dict(paged=True, block_size=32, num_blocks=100, max_blocks_per_seq=72), rkv.RKV_ERR_UNSUPPORTED),
    (dict(paged=True, num_blocks=100, max_blocks_per_seq=10), rkv.RKV_ERR_INVALID_ARG),
    (dict(mix_lambda=float("nan")), rkv.RKV_ERR_INVALID_ARG),
    (dict(redundancy=7), rkv.RKV_ERR_INVALID_ARG),
    (dict(selection=-1), rkv.RKV_ERR_INVALID_ARG),
    (dict(trigger=2), rkv.RKV_ERR_INVALID_ARG),
    (dict(buffer=-1), rkv.RKV_ERR_INVALID_ARG),
])
def test_invalid_problems_rejected_on_host(lib, kw, code):
    n = ctypes.c_size_t(0)
    assert lib.rkv_workspace_size(ctypes.byref(_p(**kw)), ctypes.byref(n)) == code


def test_null_pointers_rejected_without_launch(lib):
    p = _p()
    st = lib.rkv_compress(ctypes.byref(p), None, None, None, None, None, None, None, None, None, None, None, 0, None)
    assert st == rkv.RKV_ERR_INVALID_ARG


def test_misaligned_pointers_rejected(lib):
    p = _p()
    fake = 0x10000  # never dereferenced: validation fails first
    st = lib.rkv_compress(ctypes.byref(p), fake + 2, fake, fake, fake, None, fake, fake, None, fake, None,
                          fake, 1 << 30, None)
    assert st == rkv.RKV_ERR_INVALID_ARG


def test_workspace_too_small_rejected(lib):
    p = _p()
    fake = 0x10000
    st = lib.rkv_compress(ctypes.byref(p), fake, fake, fake, fake, None, fake, fake, None, fake, None,
                          fake, 1024, None)
    assert st == rkv.RKV_ERR_WORKSPACE


def test_problem_struct_matches_header():
    """The ctypes mirror has the header's fields, in order (13 int32, the
    float lambda, the int32 redundancy method, selection and trigger)."""
    text = open(os.path.join(ROOT, "include", "rkv.h")).read()
    body = text[text.index("typedef struct rkv_problem {"):text.index("} rkv_problem;")]
    fields = re.findall(r"^\s+(int32_t|float)\s+(\w+);", body, flags=re.M)
    assert [name for _, name in fields] == [name for name, _ in rkv.Problem._fields_]
    assert ctypes.sizeof(rkv.Problem) == 4 * len(fields)


def test_host_path_workspace_size(lib):
    # contiguous: one layer of K+V is 8 x 1152 x 256 B x 2 = 4.7 MB, so the automatic chunk
    # (about 20 MiB of K+V) is four layers
    p = _p()
    kv = 8 * 1152 * 256
    slot = 2 * kv + 32 * 8 * 256 + 8 * 1024 * 4 + 3 * 8 * 1152 * 4  # K, V, queries, kept indices, scores
    meta = 4 * 256  # seq_lens, freed_off, freed_ids (one entry), new lengths; no block table
    assert rkv.host_workspace_size(p, 1) == meta + 3 * slot + rkv.workspace_size(_p(num_layers=1))
    assert rkv.host_workspace_size(p, 4) == meta + 3 * 4 * slot + rkv.workspace_size(_p(num_layers=4))
    assert rkv.host_workspace_size(p) == rkv.host_workspace_size(p, 4)
    assert rkv.host_workspace_size(p, 1000) == rkv.host_workspace_size(p, 32)


def test_host_path_rejects_bad_arguments_before_any_device_work(lib):
    p = _p(num_layers=2)
    n = ctypes.c_size_t(0)
    assert lib.rkv_compress_host_workspace_size(ctypes.byref(p), -1, ctypes.byref(n)) == rkv.RKV_ERR_INVALID_ARG
    assert lib.rkv_compress_host_workspace_size(ctypes.byref(_p(head_dim=64)), 0, ctypes.byref(n)) == \
        rkv.RKV_ERR_UNSUPPORTED
    need = rkv.host_workspace_size(p)
    buf = ctypes.create_string_buffer(64)
    h = ctypes.addressof(buf)
    fake_ws = 1 << 20  # never dereferenced: every case below fails its host-side checks first

    def call(**kw):
        a = dict(k_in=h, v_in=h, k_out=h, v_out=h, q=h, lens=h, table=None, keep=h, off=h, ids=None, newl=h,
                 scores=None, ws=fake_ws, nbytes=need, chunk=0)
        a.update(kw)
        return lib.rkv_compress_host(ctypes.byref(p), a["chunk"], a["k_in"], a["v_in"], a["k_out"], a["v_out"],
                                     a["q"], a["lens"], a["table"], a["keep"], a["off"], a["ids"], a["newl"],
                                     a["scores"], a["ws"], a["nbytes"], None)

    assert call(k_in=None) == rkv.RKV_ERR_INVALID_ARG
    assert call(v_out=None) == rkv.RKV_ERR_INVALID_ARG
    assert call(newl=None) == rkv.RKV_ERR_INVALID_ARG
    assert call(chunk=-2) == rkv.RKV_ERR_INVALID_ARG
    assert call(ws=None) == rkv.RKV_ERR_WORKSPACE
    assert call(nbytes=need - 1) == rkv.RKV_ERR_WORKSPACE
    assert call(ws=fake_ws + 16) == rkv.RKV_ERR_WORKSPACE  # not 256-byte aligned
