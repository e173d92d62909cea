"""GPU parity of head-shared eviction (RKV_SELECT_SHARED_HEADS): one keep set
per (layer, sequence) from the blended scores summed over the KV heads, kept
by every head. Oracle: the per-head scores of the whole-event oracle, summed
over the heads in fp64, and its windowed top-budget rule (oracle.select_shared).
Acceptance as for per-head eviction: per-head normalised scores within 1e-3,
the kept set identical outside the 1e-3 band of the summed score, every head's
row identical, compaction and freed lists bit-exact."""

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import oracle
import synthetic
from helpers import check_keep_row, check_scores_row, oracle_problem

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_shared(wl, redundancy=rkv.REDUNDANCY_GRAM):
    p = rkv.problem_for(wl.shape, wl.num_blocks, redundancy=redundancy, selection=rkv.SELECT_SHARED_HEADS)
    k0, v0 = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    out = rkv.allocate_outputs(p, wl.k_cache.device, scores=True)
    rkv.rkv_compress(p, wl.k_cache, wl.v_cache, wl.q_window, wl.seq_lens, wl.block_table, out["keep_idx"],
                     out["freed_off"], out["freed_ids"] if wl.shape.paged else None, out["new_seq_lens"],
                     out["scores"], out["workspace"])
    st = rkv.rkv_device_status()
    assert st == rkv.RKV_OK, rkv.status_string(st)
    res = {k: v.cpu().numpy() for k, v in out.items() if v is not None and k != "workspace"}
    res["k0"], res["v0"] = k0, v0
    res["k"], res["v"] = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    return res


def check_shared(wl, res):
    s = wl.shape
    p = oracle_problem(wl)
    lens = wl.seq_lens.cpu().numpy()
    bt = None if wl.block_table is None else wl.block_table.cpu().numpy()
    orc = oracle.compress(p, res["k0"].copy(), res["v0"].copy(), synthetic.bf16_bits(wl.q_window), lens, bt)
    for l in range(s.layers):
        for b in range(s.batch):
            n = int(lens[b])
            for h in range(s.kv_heads):
                row = {name: orc[name][l, b, h] for name in ("I_hat", "R_hat", "S")}
                check_scores_row(res["scores"][:, l, b, h], row, n, f"l={l} b={b} h={h}")
            _, total = oracle.select_shared(orc["S"][l, b], n, s.budget, s.window)
            first = res["keep_idx"][l, b, 0]
            check_keep_row(first, total, n, s.budget, s.window, f"l={l} b={b} shared")
            for h in range(1, s.kv_heads):
                assert np.array_equal(res["keep_idx"][l, b, h], first), f"l={l} b={b}: head {h} differs"
    k_ref, v_ref = res["k0"].copy(), res["v0"].copy()
    oracle.compact(p, k_ref, v_ref, lens, bt, res["keep_idx"])
    assert np.array_equal(res["k"], k_ref) and np.array_equal(res["v"], v_ref)
    off, ids, new_lens = oracle.freed_blocks(p, lens, bt)
    assert np.array_equal(res["freed_off"], off) and np.array_equal(res["new_seq_lens"], new_lens)
    if s.paged:
        assert np.array_equal(res["freed_ids"][:off[-1]], ids)


REDUCED = {0: dict(), 1: dict(layers=2), 2: dict(layers=1, batch=2), 4: dict(layers=2, batch=4)}


@pytest.mark.parametrize("wid", sorted(REDUCED))
def test_shared_selection_reduced(wid):
    wl = synthetic.generate(wid, device=DEV, **REDUCED[wid])
    check_shared(wl, run_shared(wl))


def test_shared_selection_closed_form_ragged_paged():
    shape = synthetic.custom_shape(layers=2, batch=6, kv_heads=4, q_heads=16, budget=256, buffer=64, window=8,
                                   paged=True)
    wl = synthetic.generate(shape, device=DEV, seed=21, seq_lens=np.array([1, 100, 256, 257, 300, 320]))
    check_shared(wl, run_shared(wl, redundancy=rkv.REDUNDANCY_CLOSED_FORM))


def test_shared_selection_one_kv_head_equals_per_head():
    shape = synthetic.custom_shape(layers=2, batch=2, kv_heads=1, q_heads=4, budget=96, buffer=40, window=4)
    wl_a = synthetic.generate(shape, device=DEV, seed=5)
    wl_b = synthetic.generate(shape, device=DEV, seed=5)
    res = run_shared(wl_a)
    p = rkv.problem_for(shape)
    out = rkv.allocate_outputs(p, DEV)
    rkv.rkv_compress(p, wl_b.k_cache, wl_b.v_cache, wl_b.q_window, wl_b.seq_lens, None, out["keep_idx"],
                     out["freed_off"], None, out["new_seq_lens"], None, out["workspace"])
    assert rkv.rkv_device_status() == rkv.RKV_OK
    assert np.array_equal(res["keep_idx"], out["keep_idx"].cpu().numpy())
