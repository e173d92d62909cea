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
from helpers import BAND, SCORE_TOL

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


def _same_within_tolerance(ref, got, shape, lens):
    """The tolerance the parity tests use: scores within 1e-3, kept sets equal
    outside the 1e-3 band around the threshold, K/V and free lists exact."""
    s_ref = ref["scores"]
    assert np.max(np.abs(got["scores"] - s_ref)) <= SCORE_TOL
    L, B, H = shape.layers, shape.batch, shape.kv_heads
    for l in range(L):
        for b in range(B):
            n = int(lens[b])
            for h in range(H):
                a, c = ref["keep_idx"][l, b, h], got["keep_idx"][l, b, h]
                if n <= shape.budget:
                    assert np.array_equal(a, c)
                    continue
                cand, take = n - shape.window, shape.budget - shape.window
                S = s_ref[2, l, b, h, :cand]
                thr = np.sort(S)[::-1][take - 1]
                unsure = set(np.nonzero(np.abs(S - thr) <= BAND)[0].tolist())
                assert set(a.tolist()) - unsure == set(c.tolist()) - unsure
    for key in ("k", "v", "freed_off", "new_seq_lens"):
        assert np.array_equal(ref[key], got[key]), key
    if shape.paged:
        assert np.array_equal(ref["freed_ids"][:ref["freed_off"][-1]], got["freed_ids"][:got["freed_off"][-1]])


@pytest.mark.parametrize("wid,kw", [(1, dict(layers=4)), (4, dict(layers=2, batch=6))])
def test_noalloc_matches_workspace_entry_on_two_calls(wid, kw):
    lib = rkv.library()
    wl = synthetic.generate(wid, device="cuda", **kw)
    p = rkv.problem_for(wl.shape, wl.num_blocks)
    assert rkv.workspace_size(p) <= rkv.NOALLOC_SCRATCH_BYTES
    lens = wl.seq_lens.cpu().numpy()
    k0, v0 = wl.k_cache.clone(), wl.v_cache.clone()

    def run(fn, with_workspace):
        k, v = k0.clone(), v0.clone()
        out = rkv.allocate_outputs(p, "cuda", scores=True)
        st = _call(fn, p, wl, k, v, out, with_workspace)
        assert st == rkv.RKV_OK, rkv.status_string(st)
        assert rkv.rkv_device_status() == rkv.RKV_OK
        res = {key: out[key].cpu().numpy() for key in ("keep_idx", "freed_off", "freed_ids", "new_seq_lens",
                                                       "scores")}
        res["k"], res["v"] = synthetic.bf16_bits(k), synthetic.bf16_bits(v)
        return res

    ref = run(lib.rkv_compress, True)
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        got = run(lib.rkv_compress_noalloc, False)
        _same_within_tolerance(ref, got, wl.shape, lens)


def test_noalloc_rejects_problems_larger_than_its_scratch():
    lib = rkv.library()
    p = rkv.problem_for(synthetic.WORKLOADS[4], num_blocks=128 * 72)
    assert rkv.workspace_size(p) > rkv.NOALLOC_SCRATCH_BYTES
    fake = 0x10000  # never dereferenced: the size check comes first
    st = lib.rkv_compress_noalloc(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, fake, fake, None,
                                  None)
    assert st == rkv.RKV_ERR_WORKSPACE
