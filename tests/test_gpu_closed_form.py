"""GPU parity of the closed-form redundancy (RKV_REDUNDANCY_CLOSED_FORM, a
kernel of its own, and RKV_REDUNDANCY_CLOSED_FORM_FUSED, inside the
importance kernel's pass over K) against the CPU oracle, which computes the
pairwise definition: the rank-one identity is exact, so the same acceptance
applies as for the dense Gram (normalised scores within 1e-3, kept sets equal
outside the 1e-3 band, compaction bit-exact)."""

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import synthetic
from helpers import check_full, check_sampled_run, run_gpu, run_gpu_sampled, sample_heads

pytestmark = pytest.mark.gpu

DEV = "cuda"
CF = rkv.REDUNDANCY_CLOSED_FORM
CFF = rkv.REDUNDANCY_CLOSED_FORM_FUSED
BOTH = pytest.mark.parametrize("method", [CF, CFF], ids=["separate", "fused"])


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


REDUCED = {0: dict(), 1: dict(layers=2), 2: dict(layers=1, batch=2), 3: dict(layers=1, batch=1),
           4: dict(layers=2, batch=4)}


@BOTH
@pytest.mark.parametrize("wid", sorted(REDUCED))
def test_closed_form_event_parity_reduced(wid, method):
    wl = synthetic.generate(wid, device=DEV, **REDUCED[wid])
    worst = check_full(wl, run_gpu(wl, redundancy=method))
    print(f"closed form ({method}), workload {wid} reduced: worst abs error {worst}")


EDGE = [
    dict(shape=dict(layers=1, batch=8, kv_heads=2, q_heads=8, budget=256, buffer=64, window=8, paged=True),
         lens=[0, 1, 127, 129, 256, 257, 300, 320]),
    dict(shape=dict(layers=1, batch=1, kv_heads=1, q_heads=4, budget=8000, buffer=192, window=16, keys="clusters"),
         lens=[8192]),
    dict(shape=dict(layers=1, batch=2, kv_heads=2, q_heads=4, budget=100, buffer=60, window=4, mix_lambda=0.0),
         lens=[160, 130]),
]


@BOTH
@pytest.mark.parametrize("case", range(len(EDGE)))
def test_closed_form_edge_cases(case, method):
    c = EDGE[case]
    shape = synthetic.custom_shape(**c["shape"])
    wl = synthetic.generate(shape, device=DEV, seed=300 + case, seq_lens=np.maximum(c["lens"], 1))
    if 0 in c["lens"]:
        wl.seq_lens.copy_(torch.tensor(c["lens"], dtype=torch.int32))
    check_full(wl, run_gpu(wl, redundancy=method))


def test_zero_keys_both_methods():
    """Zero key rows have cosine 0 with everything (R = 0 before
    normalisation) under both methods."""
    for method in (rkv.REDUNDANCY_GRAM, CF, CFF):
        wl = synthetic.generate(0, device=DEV, seed=77)
        wl.k_cache[0, 0, :, 5:9] = 0
        wl.k_cache[0, 0, 2, 100] = 0
        check_full(wl, run_gpu(wl, redundancy=method))


def test_closed_form_matches_gram():
    """The two methods agree on every normalised score to well inside the
    tolerance (they differ only by fp32 rounding)."""
    wl_a = synthetic.generate(1, device=DEV, layers=4)
    wl_b = synthetic.generate(1, device=DEV, layers=4)
    a = run_gpu(wl_a, redundancy=rkv.REDUNDANCY_GRAM)
    b = run_gpu(wl_b, redundancy=CF)
    n = wl_a.shape.max_seq_len
    err = np.max(np.abs(a["scores"][..., :n] - b["scores"][..., :n]))
    assert err < 1e-4, err


@pytest.mark.parametrize("wid,count,method", [(1, 24, CF), (4, 16, CF), (1, 24, CFF), (4, 16, CFF)])
def test_closed_form_full_size_sampled(wid, count, method):
    wl = synthetic.generate(wid, device=DEV)
    heads = sample_heads(wl, count, seed=50 + wid)
    worst = check_sampled_run(wl, run_gpu_sampled(wl, heads, redundancy=method))
    print(f"closed form ({method}), workload {wid} full size: worst abs error {worst}")
    del wl
    torch.cuda.empty_cache()


def _stage_rows(wl, p):
    stride = rkv.score_stride(p)
    z = lambda: torch.zeros(p.heads * stride, dtype=torch.float32, device=DEV)  # noqa: E731
    return z(), z(), z(), stride


@BOTH
@pytest.mark.parametrize("wid,kw", [(0, {}), (1, dict(layers=3)), (2, dict(layers=1, batch=2)),
                                    (3, dict(layers=1, batch=1)), (4, dict(layers=1, batch=6))])
def test_importance_redundancy_stage(wid, kw, method):
    """rkv_importance_redundancy (steps 1-2; with the fused method one launch:
    importance and R from one pass over K) against the oracle's pairwise
    redundancy and importance, per head, and against rkv_redundancy's closed-
    form kernel on the same inverse norms (same identity, other summation
    order: agreement to fp32 rounding)."""
    import oracle
    wl = synthetic.generate(wid, device=DEV, **kw)
    p = rkv.problem_for(wl.shape, wl.num_blocks, redundancy=method)
    imp, inv, red, stride = _stage_rows(wl, p)
    rkv.rkv_importance_redundancy(p, wl.k_cache, wl.q_window, wl.seq_lens, wl.block_table, imp, inv, red)
    assert rkv.rkv_device_status() == rkv.RKV_OK
    red2 = torch.zeros_like(red)
    rkv.rkv_redundancy(p, wl.k_cache, wl.seq_lens, wl.block_table, inv, red2)  # the separate closed-form kernel
    assert rkv.rkv_device_status() == rkv.RKV_OK
    s = wl.shape
    lens = wl.seq_lens.cpu().numpy()
    R, R2 = red.view(s.layers, s.batch, s.kv_heads, stride).cpu().numpy(), \
        red2.view(s.layers, s.batch, s.kv_heads, stride).cpu().numpy()
    I = imp.view(s.layers, s.batch, s.kv_heads, stride).cpu().numpy()
    G = s.group
    for l in range(s.layers):
        for b in range(s.batch):
            n = int(lens[b])
            for h in range(s.kv_heads):
                k = synthetic.bf16_bits(synthetic.logical_rows(wl, wl.k_cache, l, b, h, n))
                q = synthetic.bf16_bits(wl.q_window[l, b, h * G:(h + 1) * G]).reshape(G * s.window, -1)
                ref = oracle.redundancy(k)
                rng = max(ref.max() - ref.min(), 1e-12)
                assert np.max(np.abs(R[l, b, h, :n] - ref)) <= 1e-4 * rng, (l, b, h)
                assert np.max(np.abs(R[l, b, h, :n] - R2[l, b, h, :n])) <= 1e-4 * rng, (l, b, h)
                iref = oracle.importance(q, k)
                assert np.max(np.abs(I[l, b, h, :n] - iref)) <= 1e-4 * (iref.max() - iref.min()), (l, b, h)


@pytest.mark.parametrize("q_heads", [8, 16])
def test_closed_form_large_logits(q_heads):
    """The fused kernel's exact two-pass softmax statistics (logits 8x the
    usual scale) together with the closed-form redundancy it forms."""
    shape = synthetic.custom_shape(layers=2, batch=2, kv_heads=2, q_heads=q_heads, budget=300, buffer=200, window=8)
    wl = synthetic.generate(shape, device=DEV, seed=78, seq_lens=np.array([500, 333]))
    wl.k_cache.mul_(8.0)
    wl.q_window.mul_(8.0)
    check_full(wl, run_gpu(wl, redundancy=CFF))
