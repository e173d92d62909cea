"""GPU parity of the closed-form redundancy (RKV_REDUNDANCY_CLOSED_FORM)
against the CPU oracle, which computes the pairwise definition: the rank-one
identity is exact, so the same acceptance applies as for the dense Gram
(normalised scores within 1e-3, kept sets equal outside the 1e-3 band,
compaction bit-exact)."""

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import synthetic
from helpers import check_full, check_sampled_run, run_gpu, run_gpu_sampled, sample_heads

pytestmark = pytest.mark.gpu

DEV = "cuda"
CF = rkv.REDUNDANCY_CLOSED_FORM


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


REDUCED = {0: dict(), 1: dict(layers=2), 2: dict(layers=1, batch=2), 3: dict(layers=1, batch=1),
           4: dict(layers=2, batch=4)}


@pytest.mark.parametrize("wid", sorted(REDUCED))
def test_closed_form_event_parity_reduced(wid):
    wl = synthetic.generate(wid, device=DEV, **REDUCED[wid])
    worst = check_full(wl, run_gpu(wl, redundancy=CF))
    print(f"closed form, workload {wid} reduced: worst abs error {worst}")


EDGE = [
    dict(shape=dict(layers=1, batch=8, kv_heads=2, q_heads=8, budget=256, buffer=64, window=8, paged=True),
         lens=[0, 1, 127, 129, 256, 257, 300, 320]),
    dict(shape=dict(layers=1, batch=1, kv_heads=1, q_heads=4, budget=8000, buffer=192, window=16, keys="clusters"),
         lens=[8192]),
    dict(shape=dict(layers=1, batch=2, kv_heads=2, q_heads=4, budget=100, buffer=60, window=4, mix_lambda=0.0),
         lens=[160, 130]),
]


@pytest.mark.parametrize("case", range(len(EDGE)))
def test_closed_form_edge_cases(case):
    c = EDGE[case]
    shape = synthetic.custom_shape(**c["shape"])
    wl = synthetic.generate(shape, device=DEV, seed=300 + case, seq_lens=np.maximum(c["lens"], 1))
    if 0 in c["lens"]:
        wl.seq_lens.copy_(torch.tensor(c["lens"], dtype=torch.int32))
    check_full(wl, run_gpu(wl, redundancy=CF))


def test_zero_keys_both_methods():
    """Zero key rows have cosine 0 with everything (R = 0 before
    normalisation) under both methods."""
    for method in (rkv.REDUNDANCY_GRAM, CF):
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


@pytest.mark.parametrize("wid,count", [(1, 24), (4, 16)])
def test_closed_form_full_size_sampled(wid, count):
    wl = synthetic.generate(wid, device=DEV)
    heads = sample_heads(wl, count, seed=50 + wid)
    worst = check_sampled_run(wl, run_gpu_sampled(wl, heads, redundancy=CF))
    print(f"closed form, workload {wid} full size: worst abs error {worst}")
    del wl
    torch.cuda.empty_cache()
