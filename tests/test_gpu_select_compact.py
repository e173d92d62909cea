"""rkv_select_compact (steps 3-5 in one launch) against the two separate
stage calls rkv_select + rkv_compact on the same importance and redundancy
rows: kept indices, scores, compacted K/V, freed blocks and new lengths must
be bit-identical (the same arithmetic, one launch instead of two). The whole
event through rkv_compress, which uses the fused kernel, is held to the oracle
by the parity tests. Problems with fewer heads than SMs take the cluster
kernel (a cluster of CTAs per head), larger ones the one-CTA-per-head kernel:
the cases cover both."""

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def _scores_rows(wl, p):
    stride = rkv.score_stride(p)
    imp = torch.zeros(p.heads * stride, dtype=torch.float32, device=DEV)
    inv = torch.zeros_like(imp)
    red = torch.zeros_like(imp)
    rkv.rkv_importance(p, wl.k_cache, wl.q_window, wl.seq_lens, wl.block_table, imp, inv)
    rkv.rkv_redundancy(p, wl.k_cache, wl.seq_lens, wl.block_table, inv, red)
    return imp, red


def _run(wl, p, imp, red, fused):
    k, v = wl.k_cache.clone(), wl.v_cache.clone()
    out = rkv.allocate_outputs(p, DEV, scores=True)
    out["keep_idx"].fill_(-9)
    if fused:
        rkv.rkv_select_compact(p, imp, red, wl.seq_lens, wl.block_table, k, v, out["keep_idx"], out["freed_off"],
                               out["freed_ids"] if p.paged else None, out["new_seq_lens"], out["scores"])
    else:
        rkv.rkv_select(p, imp, red, wl.seq_lens, out["keep_idx"], out["scores"])
        rkv.rkv_compact(p, k, v, wl.seq_lens, wl.block_table, out["keep_idx"], out["freed_off"],
                        out["freed_ids"] if p.paged else None, out["new_seq_lens"])
    assert rkv.rkv_device_status() == rkv.RKV_OK
    res = {key: out[key].cpu().numpy() for key in ("keep_idx", "scores", "freed_off", "new_seq_lens", "freed_ids")}
    res["k"], res["v"] = synthetic.bf16_bits(k), synthetic.bf16_bits(v)
    return res


CASES = [
    dict(wid=1, kw=dict(layers=2)),
    dict(wid=4, kw=dict(layers=1, batch=8)),
    dict(wid=2, kw=dict(layers=1, batch=2)),
    dict(wid=3, kw=dict(layers=1, batch=1)),
    # ragged lengths around the budget and the 16-row blocks, some empty
    dict(shape=dict(layers=1, batch=8, kv_heads=2, q_heads=8, budget=256, buffer=64, window=8, paged=True),
         lens=[0, 1, 127, 129, 256, 257, 300, 320]),
    dict(shape=dict(layers=2, batch=3, kv_heads=2, q_heads=8, budget=2000, buffer=100, window=8),
         lens=[100, 700, 2100]),
    # at least as many heads as SMs: one CTA per head instead of a cluster
    dict(wid=1, kw=dict(layers=20)),
    dict(wid=4, kw=dict(layers=2, batch=20)),
    dict(shape=dict(layers=10, batch=8, kv_heads=2, q_heads=8, budget=256, buffer=64, window=8, paged=True),
         lens=[0, 1, 127, 129, 256, 257, 300, 320]),
    dict(shape=dict(layers=25, batch=3, kv_heads=2, q_heads=8, budget=2000, buffer=100, window=8),
         lens=[100, 700, 2100]),
]


@pytest.mark.parametrize("case", range(len(CASES)))
@pytest.mark.parametrize("trigger", [rkv.TRIGGER_ANY, rkv.TRIGGER_BUDGET_PLUS_BUFFER])
def test_fused_select_compact_equals_separate_calls(case, trigger):
    c = CASES[case]
    if "wid" in c:
        wl = synthetic.generate(c["wid"], device=DEV, **c["kw"])
    else:
        shape = synthetic.custom_shape(**c["shape"])
        wl = synthetic.generate(shape, device=DEV, seed=300 + case, seq_lens=np.maximum(c["lens"], 1))
        if 0 in c["lens"]:
            wl.seq_lens.copy_(torch.tensor(c["lens"], dtype=torch.int32))
    p = rkv.problem_for(wl.shape, wl.num_blocks, trigger=trigger)
    imp, red = _scores_rows(wl, p)
    a = _run(wl, p, imp, red, fused=True)
    b = _run(wl, p, imp, red, fused=False)
    for key in ("keep_idx", "scores", "k", "v", "freed_off", "new_seq_lens"):
        assert np.array_equal(a[key], b[key]), key
    if p.paged:
        n = int(b["freed_off"][-1])
        assert np.array_equal(a["freed_ids"][:n], b["freed_ids"][:n])
