"""rkv_compress_noalloc: the compression event for callers that cannot
allocate device memory when they compress (an engine whose free HBM all
belongs to its KV block pool, a plugin host that hands out device pointers
but no allocator). It must give the same results as rkv_compress, call after
call, while using only the library's static per-GPU scratch.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test."""

import ctypes

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import synthetic

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _call(fn, p, wl, k, v, out, with_workspace):
    args = [ctypes.byref(p), k.data_ptr(), v.data_ptr(), wl.q_window.data_ptr(), wl.seq_lens.data_ptr(),
            None if wl.block_table is None else wl.block_table.data_ptr(), out["keep_idx"].data_ptr(),
            out["freed_off"].data_ptr(), out["freed_ids"].data_ptr() if wl.shape.paged else None,
            out["new_seq_lens"].data_ptr(), out["scores"].data_ptr()]
    if with_workspace:
        args += [out["workspace"].data_ptr(), out["workspace"].numel()]
    args.append(torch.cuda.current_stream().cuda_stream)
    return fn(*args)


def _run(fn, p, wl, k0, v0, with_workspace):
    k, v = k0.clone(), v0.clone()
    out = rkv.allocate_outputs(p, "cuda", scores=True)
    st = _call(fn, p, wl, k, v, out, with_workspace)
    assert st == rkv.RKV_OK, rkv.status_string(st)
    assert rkv.rkv_device_status() == rkv.RKV_OK
    res = {key: out[key].cpu().numpy() for key in ("keep_idx", "freed_off", "freed_ids", "new_seq_lens", "scores")}
    res["k"], res["v"] = synthetic.bf16_bits(k), synthetic.bf16_bits(v)
    return res


def _assert_identical(ref, got, shape, where):
    """Same kernels, same inputs, same launch configuration: the results must
    be bit-identical to rkv_compress's (which the parity tests hold to the
    oracle), so a stale value picked up from the shared static scratch cannot
    hide inside a tolerance."""
    for key in ("scores", "keep_idx", "k", "v", "freed_off", "new_seq_lens"):
        assert np.array_equal(ref[key], got[key]), f"{where}: {key} differs"
    if shape.paged:
        n = int(ref["freed_off"][-1])
        assert np.array_equal(ref["freed_ids"][:n], got["freed_ids"][:n]), f"{where}: freed_ids differ"


def test_noalloc_matches_workspace_entry_on_two_calls():
    """The largest problem first (the whole 32-layer Llama-3-8B cache: 3.4 MiB
    of scratch), then a smaller paged one, each called twice in a row: the
    later calls find the array holding an earlier call's values, which they
    must overwrite before reading."""
    lib = rkv.library()
    cases = [(1, {}), (4, dict(layers=2, batch=6))]
    sizes = []
    for wid, kw in cases:
        wl = synthetic.generate(wid, device="cuda", **kw)
        p = rkv.problem_for(wl.shape, wl.num_blocks)
        sizes.append(rkv.workspace_size(p))
        assert sizes[-1] <= rkv.NOALLOC_SCRATCH_BYTES
        k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()
        ref = _run(lib.rkv_compress, p, wl, k0, v0, True)
        for call in range(2):  # two calls in a row share (and reuse) the static scratch
            got = _run(lib.rkv_compress_noalloc, p, wl, k0, v0, False)
            _assert_identical(ref, got, wl.shape, f"workload {wid}, call {call}")
    assert sizes[0] > sizes[1]


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = rkv.library()
    p = rkv.problem_for(synthetic.WORKLOADS[4], num_blocks=128 * 72)
    assert rkv.workspace_size(p) > rkv.NOALLOC_SCRATCH_BYTES
    fake = 0x10000  # never dereferenced: the size check comes first
    st = lib.rkv_compress_noalloc(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake, fake, None,
                                  None)
    assert st == rkv.RKV_ERR_WORKSPACE
