"""rkv_compress_host: the compression event on a KV cache held in host memory,
uploaded, compressed and downloaded chunk by chunk with the copies of both
directions overlapped. Its results must pass the same oracle parity as
rkv_compress (scores within 1e-3, kept sets outside the 1e-3 band, K/V and
freed lists bit-exact), for every chunking, for page-locked and pageable host
memory and for outputs written over the inputs."""

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import synthetic
from helpers import check_full

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _host(t: torch.Tensor, pinned: bool) -> torch.Tensor:
    h = t.detach().cpu().contiguous()
    return h.pin_memory() if pinned else h.clone()


def run_host(wl: synthetic.Workload, chunk_layers: int, pinned: bool = True, alias: bool = False,
             scores: bool = True, trigger: int = rkv.TRIGGER_ANY) -> dict:
    s = wl.shape
    p = rkv.problem_for(s, wl.num_blocks, trigger=trigger)
    hk, hv = _host(wl.k_cache, pinned), _host(wl.v_cache, pinned)
    k0, v0 = synthetic.bf16_bits(hk), synthetic.bf16_bits(hv)
    hq, hl = _host(wl.q_window, pinned), _host(wl.seq_lens, pinned)
    ht = _host(wl.block_table, pinned) if s.paged else None
    ko = hk if alias else _host(torch.zeros_like(wl.k_cache), pinned)
    vo = hv if alias else _host(torch.zeros_like(wl.v_cache), pinned)

    def out(shape, dtype, fill):
        t = torch.full(shape, fill, dtype=dtype)
        return t.pin_memory() if pinned else t

    keep = out((s.layers, s.batch, s.kv_heads, s.budget), torch.int32, -7)
    off = out((s.batch + 1,), torch.int32, -7)
    ids = out((max(1, s.batch * s.blocks_per_seq),), torch.int32, -7) if s.paged else None
    newl = out((s.batch,), torch.int32, -7)
    sc = out((3, s.layers, s.batch, s.kv_heads, s.max_seq_len), torch.float32, float("nan")) if scores else None
    ws = torch.empty(rkv.host_workspace_size(p, chunk_layers), dtype=torch.uint8, device=DEV)
    rkv.rkv_compress_host(p, hk, hv, ko, vo, hq, hl, ht, keep, off, ids, newl, sc, ws, chunk_layers=chunk_layers)
    st = rkv.rkv_device_status()
    assert st == rkv.RKV_OK, rkv.status_string(st)
    return {"keep_idx": keep.numpy(), "freed_off": off.numpy(), "freed_ids": None if ids is None else ids.numpy(),
            "new_seq_lens": newl.numpy(), "scores": None if sc is None else sc.numpy(),
            "k0": k0, "v0": v0, "k": synthetic.bf16_bits(ko), "v": synthetic.bf16_bits(vo)}


def _scores_past_n_are_zero(res: dict, lens: np.ndarray):
    for b, n in enumerate(lens):
        assert np.all(res["scores"][:, :, b, :, int(n):] == 0.0)


@pytest.mark.parametrize("chunk", [0, 1, 2, 5])
def test_host_path_contiguous_matches_oracle(chunk):
    # 5 layers: chunks of 2 leave a ragged last chunk, 5 is one chunk, 1 cycles the three slots
    wl = synthetic.generate(1, device=DEV, layers=5)
    res = run_host(wl, chunk)
    check_full(wl, res)
    _scores_past_n_are_zero(res, wl.seq_lens.cpu().numpy())


@pytest.mark.parametrize("chunk", [0, 1, 3])
def test_host_path_paged_matches_oracle(chunk):
    wl = synthetic.generate(4, device=DEV, layers=4, batch=3)
    res = run_host(wl, chunk)
    check_full(wl, res)


def test_host_path_ragged_lengths_pageable_memory():
    shape = synthetic.custom_shape(layers=3, batch=8, kv_heads=2, q_heads=8, budget=256, buffer=64, window=8,
                                   paged=True)
    wl = synthetic.generate(shape, device=DEV, seed=321, seq_lens=np.array([1, 1, 127, 129, 256, 257, 300, 320]))
    res = run_host(wl, 2, pinned=False)
    check_full(wl, res)
    _scores_past_n_are_zero(res, wl.seq_lens.cpu().numpy())


def test_host_path_in_place_without_scores():
    wl = synthetic.generate(1, device=DEV, layers=4)
    ref = run_host(wl, 1)
    got = run_host(wl, 1, alias=True, scores=False)
    for key in ("keep_idx", "k", "v", "freed_off", "new_seq_lens"):
        assert np.array_equal(ref[key], got[key]), key


@pytest.mark.parametrize("trigger", [rkv.TRIGGER_ANY, rkv.TRIGGER_BUDGET_PLUS_BUFFER])
def test_host_path_in_place_ragged_and_triggered(trigger):
    # outputs over the inputs with ragged lengths (and, with the device trigger,
    # sequences it leaves alone): the host cache must equal what separate
    # output buffers receive
    shape = synthetic.custom_shape(layers=3, batch=6, kv_heads=2, q_heads=8, budget=256, buffer=64, window=8)
    lens = np.array([1, 200, 256, 257, 300, 320])
    wl = synthetic.generate(shape, device=DEV, seed=55, seq_lens=lens)
    ref = run_host(wl, 1, trigger=trigger)
    got = run_host(wl, 2, alias=True, scores=False, trigger=trigger)
    for key in ("keep_idx", "k", "v", "freed_off", "new_seq_lens"):
        assert np.array_equal(ref[key], got[key]), key
    if trigger == rkv.TRIGGER_BUDGET_PLUS_BUFFER:
        assert got["new_seq_lens"].tolist() == [1, 200, 256, 257, 300, 256]
    else:
        check_full(wl, ref)


def test_host_path_equals_device_path():
    wl = synthetic.generate(4, device=DEV, layers=2, batch=4)
    host = run_host(wl, 1)
    p = rkv.problem_for(wl.shape, wl.num_blocks)
    out = rkv.allocate_outputs(p, DEV, scores=True)
    rkv.rkv_compress(p, wl.k_cache, wl.v_cache, wl.q_window, wl.seq_lens, wl.block_table, out["keep_idx"],
                     out["freed_off"], out["freed_ids"], out["new_seq_lens"], out["scores"], out["workspace"])
    assert rkv.rkv_device_status() == rkv.RKV_OK
    assert np.array_equal(host["keep_idx"], out["keep_idx"].cpu().numpy())
    assert np.array_equal(host["k"], synthetic.bf16_bits(wl.k_cache))
    assert np.array_equal(host["v"], synthetic.bf16_bits(wl.v_cache))
    assert np.array_equal(host["freed_off"], out["freed_off"].cpu().numpy())
    n = int(host["freed_off"][-1])
    assert np.array_equal(host["freed_ids"][:n], out["freed_ids"].cpu().numpy()[:n])
    lens = wl.seq_lens.cpu().numpy()
    dev_scores = out["scores"].cpu().numpy()
    for b, nb in enumerate(lens):
        assert np.max(np.abs(host["scores"][:, :, b, :, :nb] - dev_scores[:, :, b, :, :nb])) <= 1e-6


def test_host_path_empty_batch():
    p = rkv.make_problem(num_layers=3, batch=0, num_kv_heads=2, num_q_heads=4, max_seq_len=256, budget=64,
                         window=8, mix_lambda=0.1)
    # nothing is read or written per layer; one-element stand-ins carry the pointers
    k = torch.zeros(8, dtype=torch.bfloat16).pin_memory()
    i32 = torch.zeros(8, dtype=torch.int32).pin_memory()
    off = torch.full((1,), 5, dtype=torch.int32).pin_memory()
    ws = torch.empty(rkv.host_workspace_size(p), dtype=torch.uint8, device=DEV)
    rkv.rkv_compress_host(p, k, k, k, k, k, i32, None, i32, off, None, i32, None, ws)
    assert rkv.rkv_device_status() == rkv.RKV_OK
    assert off.tolist() == [0]
