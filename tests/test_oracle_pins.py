"""Pins for the CPU oracle: each test checks it against something other than
itself -- a hand-derived closed form, an identity, an invariant, brute force,
or an independent library routine -- so that a dropped term, a wrong sign or
index, or a transposed operand fails at least one of them."""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
bf = oracle.bf16_bits_from_float


def f32(x):
    return np.asarray(x, dtype=np.float32)


# ---------------------------------------------------------------- importance

def test_importance_hand_case_single_query():
    # d = 4 -> scale 1/2. q = (2,0,0,0); keys e1, e2, -e1 -> logits 1, 0, -1.
    q = bf(f32([[2, 0, 0, 0]]))
    k = bf(f32([[1, 0, 0, 0], [0, 1, 0, 0], [-1, 0, 0, 0]]))
    z = math.e + 1 + 1 / math.e
    want = np.array([math.e / z, 1 / z, 1 / math.e / z])
    np.testing.assert_allclose(oracle.importance(q, k), want, rtol=0, atol=1e-15)


def test_importance_hand_case_mean_over_rows():
    # Second row (0,2,0,0) -> logits 0, 1, 0 -> probabilities (1, e, 1)/(e+2).
    q = bf(f32([[2, 0, 0, 0], [0, 2, 0, 0]]))
    k = bf(f32([[1, 0, 0, 0], [0, 1, 0, 0], [-1, 0, 0, 0]]))
    z1 = math.e + 1 + 1 / math.e
    p1 = np.array([math.e, 1, 1 / math.e]) / z1
    p2 = np.array([1, math.e, 1]) / (math.e + 2)
    np.testing.assert_allclose(oracle.importance(q, k), (p1 + p2) / 2, rtol=0, atol=1e-15)


def test_importance_scale_is_inverse_sqrt_d():
    # d = 16 -> scale 1/4. q = 4*e1, keys e1 and 0 -> logits 1 and 0.
    d = 16
    q = np.zeros((1, d), np.float32); q[0, 0] = 4
    k = np.zeros((2, d), np.float32); k[0, 0] = 1
    want = np.array([math.e, 1]) / (math.e + 1)
    np.testing.assert_allclose(oracle.importance(bf(q), bf(k)), want, rtol=0, atol=1e-15)


def test_importance_sums_to_one_and_matches_torch_softmax():
    rng = np.random.default_rng(1)
    q = bf(rng.standard_normal((12, 128)).astype(np.float32))
    k = bf(rng.standard_normal((300, 128)).astype(np.float32))
    imp = oracle.importance(q, k)
    assert abs(imp.sum() - 1.0) < 1e-12
    qt = torch.from_numpy(oracle.bf16_to_float(q).astype(np.float64))
    kt = torch.from_numpy(oracle.bf16_to_float(k).astype(np.float64))
    ref = torch.softmax(qt @ kt.T / math.sqrt(128), dim=-1).mean(0).numpy()
    np.testing.assert_allclose(imp, ref, rtol=1e-12, atol=1e-16)


def test_importance_zero_queries_uniform():
    k = bf(np.random.default_rng(2).standard_normal((37, 128)).astype(np.float32))
    q = np.zeros((8, 128), np.uint16)
    imp = oracle.importance(q, k)
    np.testing.assert_allclose(imp, np.full(37, 1 / 37), rtol=0, atol=1e-15)
    # uniform -> constant -> normalises to zero
    assert np.all(oracle.minmax(imp) == 0)


def test_importance_key_permutation_equivariant():
    rng = np.random.default_rng(3)
    q = bf(rng.standard_normal((4, 128)).astype(np.float32))
    k = bf(rng.standard_normal((50, 128)).astype(np.float32))
    perm = rng.permutation(50)
    np.testing.assert_allclose(oracle.importance(q, k)[perm], oracle.importance(q, k[perm]), atol=1e-15)


# ---------------------------------------------------------------- redundancy

def test_redundancy_hand_case():
    # keys (1,0), (0,1), (1,1): cos = 0, 1/sqrt2, 1/sqrt2.
    k = bf(f32([[1, 0], [0, 1], [1, 1]]))
    s = 1 / math.sqrt(2)
    np.testing.assert_allclose(oracle.redundancy(k), [s / 2, s / 2, s], rtol=0, atol=1e-15)


def test_redundancy_rank1_closed_form():
    # mean_{j != i} cos(k_i, k_j) = (khat_i . sum_j khat_j - |khat_i|^2) / (N - 1)
    rng = np.random.default_rng(4)
    kb = bf(rng.standard_normal((257, 128)).astype(np.float32))
    kf = oracle.bf16_to_float(kb).astype(np.float64)
    kh = kf / np.linalg.norm(kf, axis=1, keepdims=True)
    closed = (kh @ kh.sum(0) - (kh * kh).sum(1)) / (kf.shape[0] - 1)
    np.testing.assert_allclose(oracle.redundancy(kb), closed, rtol=0, atol=1e-13)


def test_redundancy_orthonormal_zero_and_duplicate_maximal():
    n, d = 10, 16
    k = np.zeros((n, d), np.float32)
    k[np.arange(n), np.arange(n)] = 1.0
    assert np.all(np.abs(oracle.redundancy(bf(k))) < 1e-15)
    k[7] = k[2]  # one exact duplicate pair
    r = oracle.redundancy(bf(k))
    want = np.zeros(n); want[[2, 7]] = 1 / (n - 1)
    np.testing.assert_allclose(r, want, atol=1e-15)
    assert set(np.argsort(-r)[:2]) == {2, 7}


def test_redundancy_scale_invariant_and_zero_key():
    rng = np.random.default_rng(5)
    k = rng.standard_normal((20, 128)).astype(np.float32)
    k = oracle.bf16_to_float(bf(k))
    k2 = k.copy(); k2[3] *= 4.0  # exact in bf16
    np.testing.assert_allclose(oracle.redundancy(bf(k)), oracle.redundancy(bf(k2)), atol=1e-15)
    k3 = k.copy(); k3[5] = 0.0
    r3 = oracle.redundancy(bf(k3))
    assert r3[5] == 0.0
    kf = k.astype(np.float64); kh = kf / np.linalg.norm(kf, axis=1, keepdims=True)
    kh[5] = 0
    closed = (kh @ kh.sum(0) - (kh * kh).sum(1)) / 19
    np.testing.assert_allclose(r3, closed, atol=1e-13)


def test_redundancy_single_key_zero():
    assert oracle.redundancy(bf(f32([[1, 2, 3, 4]]))).tolist() == [0.0]


def test_closed_form_redundancy_hand_case_and_degenerate_heads():
    s = 1 / math.sqrt(2)
    k = bf(f32([[1, 0], [0, 1], [1, 1]]))
    np.testing.assert_allclose(oracle.redundancy_closed(k), [s / 2, s / 2, s], rtol=0, atol=1e-15)
    assert oracle.redundancy_closed(bf(f32([[1, 2, 3, 4]]))).tolist() == [0.0]
    # orthonormal keys with one exact duplicate pair and one zero key
    n, d = 10, 16
    kk = np.zeros((n, d), np.float32)
    kk[np.arange(n), np.arange(n)] = 1.0
    kk[7] = kk[2]
    kk[4] = 0.0
    want = np.zeros(n); want[[2, 7]] = 1 / (n - 1)
    np.testing.assert_allclose(oracle.redundancy_closed(bf(kk)), want, atol=1e-15)


@pytest.mark.parametrize("seed", range(4))
def test_closed_form_redundancy_equals_pairwise_definition(seed):
    # the rank-one identity against the n^2 pairwise sum: two independent formulas
    rng = np.random.default_rng(40 + seed)
    n = int(rng.integers(2, 300))
    k = rng.standard_normal((n, 128)).astype(np.float32)
    k[rng.integers(0, n)] = 0.0                         # a zero key
    k[rng.integers(0, n)] = k[rng.integers(0, n)] * 2   # a scaled duplicate
    kb = bf(k)
    np.testing.assert_allclose(oracle.redundancy_closed(kb), oracle.redundancy(kb), rtol=0, atol=1e-13)


def test_closed_form_event_equals_pairwise_event():
    shape = synthetic.custom_shape(layers=2, batch=3, kv_heads=2, q_heads=6, budget=40, buffer=24,
                                   window=4, ragged=True)
    wl = synthetic.generate(shape, seed=22, seq_lens=np.array([30, 41, 64]))
    p = oracle.problem(layers=2, batch=3, kv_heads=2, q_heads=6, head_dim=128, max_seq_len=64,
                       budget=40, window=4, mix_lambda=0.1)
    k0, v0 = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    q, lens = synthetic.bf16_bits(wl.q_window), wl.seq_lens.numpy()
    a = oracle.compress(p, k0.copy(), v0.copy(), q, lens)
    b = oracle.compress(p, k0.copy(), v0.copy(), q, lens, closed_form=True)
    for name in ("I", "R", "I_hat", "R_hat", "S"):
        np.testing.assert_allclose(b[name], a[name], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(b["keep_idx"], a["keep_idx"])


# ---------------------------------------------------------- normalise / mix

def test_minmax_and_mix_limits():
    x = np.array([3.0, 1.0, 2.0, 5.0])
    np.testing.assert_allclose(oracle.minmax(x), [0.5, 0.0, 0.25, 1.0])
    assert np.all(oracle.minmax(np.full(5, 2.5)) == 0.0)
    a, b = np.array([0.0, 0.5, 1.0]), np.array([1.0, 0.25, 0.0])
    np.testing.assert_allclose(oracle.mix(a, b, 1.0), a)
    np.testing.assert_allclose(oracle.mix(a, b, 0.0), -b)
    np.testing.assert_allclose(oracle.mix(a, b, 0.1), 0.1 * a - 0.9 * b)


# ---------------------------------------------------------------- selection

def _brute_force_keep(s, budget, window):
    n = len(s)
    if n <= budget:
        return list(range(n))
    win = list(range(n - window, n))
    best = None
    for comb in itertools.combinations(range(n - window), budget - window):
        total = sum(s[i] for i in comb)
        key = (-total, comb)  # larger sum first; ties -> lexicographically smallest
        if best is None or key < best[0]:
            best = (key, comb)
    return sorted(list(best[1]) + win)


@pytest.mark.parametrize("seed", range(12))
def test_select_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 13))
    budget = int(rng.integers(1, 9))
    window = int(rng.integers(1, budget + 1))
    # small integers make exact ties common; the sums are then exact too
    s = rng.integers(-3, 4, size=n).astype(np.float64)
    keep = oracle.select(s, budget, window)
    kept = [int(i) for i in keep if i >= 0]
    assert kept == _brute_force_keep(list(s), budget, window)
    assert len(kept) == min(n, budget)
    assert np.all(keep[len(kept):] == -1)
    if n > budget:
        assert set(range(n - window, n)) <= set(kept)
    assert kept == sorted(kept)


@pytest.mark.parametrize("seed", range(8))
def test_shared_selection_brute_force(seed):
    """Head-shared eviction keeps the subset with the largest score summed
    over the heads (brute force over all subsets of a tiny head group)."""
    rng = np.random.default_rng(100 + seed)
    heads, n = int(rng.integers(1, 5)), int(rng.integers(2, 12))
    budget = int(rng.integers(1, n + 1))
    window = int(rng.integers(1, budget + 1))
    S = rng.integers(-3, 4, size=(heads, n)).astype(np.float64)
    keep, total = oracle.select_shared(S, n, budget, window)
    kept = [int(i) for i in keep if i >= 0]
    per_token = [sum(S[h, j] for h in range(heads)) for j in range(n)]  # summed by hand, not by the oracle
    assert np.array_equal(total, per_token)
    assert kept == _brute_force_keep(per_token, budget, window)


def test_shared_selection_special_cases():
    rng = np.random.default_rng(7)
    S1 = rng.standard_normal((1, 40))
    # one head: identical to the per-head rule
    assert np.array_equal(oracle.select_shared(S1, 40, 24, 4)[0], oracle.select(S1[0], 24, 4))
    # identical heads: the sum ranks exactly like any one head
    S4 = np.repeat(S1, 4, axis=0)
    assert np.array_equal(oracle.select_shared(S4, 40, 24, 4)[0], oracle.select(S1[0], 24, 4))
    # a head that is constant contributes no preference
    S2 = np.vstack([S1, np.full((1, 40), 0.25)])
    assert np.array_equal(oracle.select_shared(S2, 40, 24, 4)[0], oracle.select(S1[0], 24, 4))


def test_lambda_one_is_attention_topk_and_lambda_zero_is_least_redundant():
    wl = synthetic.generate(synthetic.custom_shape(kv_heads=1, q_heads=4, budget=48, buffer=16, window=4),
                            seed=11)
    q = synthetic.bf16_bits(wl.q_window[0, 0])  # [4][4][128]
    k = synthetic.bf16_bits(wl.k_cache[0, 0, 0])
    n, budget, w = k.shape[0], 48, 4
    qt = torch.from_numpy(oracle.bf16_to_float(q).reshape(-1, 128).astype(np.float64))
    kt = torch.from_numpy(oracle.bf16_to_float(k).astype(np.float64))
    attn = torch.softmax(qt @ kt.T / math.sqrt(128), dim=-1).mean(0).numpy()
    kh = kt.numpy() / np.linalg.norm(kt.numpy(), axis=1, keepdims=True)
    red = (kh @ kh.sum(0) - 1.0) / (n - 1)

    got1 = oracle.compress_head(q.reshape(-1, 128), k, budget, w, 1.0)["keep"]
    want1 = sorted(list(np.argsort(-attn[: n - w], kind="stable")[: budget - w]) + list(range(n - w, n)))
    assert got1.tolist() == want1

    got0 = oracle.compress_head(q.reshape(-1, 128), k, budget, w, 0.0)["keep"]
    want0 = sorted(list(np.argsort(red[: n - w], kind="stable")[: budget - w]) + list(range(n - w, n)))
    assert got0.tolist() == want0


# -------------------------------------------------------------- compaction

def _naive_gather_contig(cache, seq_lens, keep, budget):
    out = cache.copy()
    L, B, H = cache.shape[:3]
    for l in range(L):
        for b in range(B):
            kb = min(int(seq_lens[b]), budget)
            for h in range(H):
                idx = keep[l, b, h, :kb]
                out[l, b, h, :kb] = cache[l, b, h, idx]
    return out


@pytest.mark.parametrize("paged", [False, True])
def test_compress_invariants_and_naive_gather(paged):
    shape = synthetic.custom_shape(layers=2, batch=3, kv_heads=2, q_heads=6, budget=40, buffer=24,
                                   window=4, paged=paged, ragged=True)
    wl = synthetic.generate(shape, seed=21, seq_lens=np.array([30, 41, 64]))
    p = oracle.problem(layers=2, batch=3, kv_heads=2, q_heads=6, head_dim=128, max_seq_len=64,
                       budget=40, window=4, mix_lambda=0.1, paged=paged, block_size=16,
                       num_blocks=wl.num_blocks, max_blocks=4 if paged else 0)
    k0, v0 = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    q = synthetic.bf16_bits(wl.q_window)
    lens = wl.seq_lens.numpy()
    bt = None if wl.block_table is None else wl.block_table.numpy()
    k, v = k0.copy(), v0.copy()
    out = oracle.compress(p, k, v, q, lens, bt)
    keep = out["keep_idx"]
    for l in range(2):
        for b in range(3):
            n = int(lens[b]); kb = min(n, 40)
            assert out["new_seq_lens"][b] == kb
            for h in range(2):
                kept = keep[l, b, h]
                assert np.all(kept[kb:] == -1)
                assert np.all(np.diff(kept[:kb]) > 0) and kept[0] >= 0 and kept[kb - 1] < n
                if n > 40:
                    assert set(range(n - 4, n)) <= set(kept[:kb].tolist())
                # scores: importance sums to one; normalised scores in [0, 1]
                assert abs(out["I"][l, b, h, :n].sum() - 1) < 1e-12
                assert out["I_hat"][l, b, h, :n].min() >= 0 and out["I_hat"][l, b, h, :n].max() <= 1
    if not paged:
        np.testing.assert_array_equal(k, _naive_gather_contig(k0, lens, keep, 40))
        np.testing.assert_array_equal(v, _naive_gather_contig(v0, lens, keep, 40))
        assert out["freed_off"].tolist() == [0, 0, 0, 0]
    else:
        # logical view through the block table, then the same naive gather
        def logical(pool):
            L = pool.shape[0]
            outl = np.zeros((L, 3, 2, 64, 128), np.uint16)
            for b in range(3):
                blocks = bt[b]
                outl[:, b] = pool[:, blocks].reshape(L, 64, 2, 128).transpose(0, 2, 1, 3)
            return outl
        np.testing.assert_array_equal(logical(k), _naive_gather_contig(logical(k0), lens, keep, 40))
        np.testing.assert_array_equal(logical(v), _naive_gather_contig(logical(v0), lens, keep, 40))
        # freed blocks: ceil(N/16) - ceil(k/16) per sequence, in table order
        off, ids = out["freed_off"], out["freed_ids"]
        for b in range(3):
            n = int(lens[b]); kb = min(n, 40)
            first, last = -(-kb // 16), -(-n // 16)
            assert off[b + 1] - off[b] == last - first
            assert ids[off[b]:off[b + 1]].tolist() == bt[b, first:last].tolist()
            assert sorted(ids[off[b]:off[b + 1]].tolist() + bt[b, :first].tolist()) == sorted(bt[b, :last].tolist())


def test_compact_with_given_indices_matches_naive():
    rng = np.random.default_rng(7)
    L, B, H, N, d, budget = 1, 2, 2, 24, 128, 16
    k0 = rng.integers(0, 65535, size=(L, B, H, N, d)).astype(np.uint16)
    v0 = rng.integers(0, 65535, size=(L, B, H, N, d)).astype(np.uint16)
    lens = np.array([24, 10], np.int32)
    keep = np.full((L, B, H, budget), -1, np.int32)
    for b in range(B):
        for h in range(H):
            n = int(lens[b]); kb = min(n, budget)
            keep[0, b, h, :kb] = np.sort(rng.choice(n, kb, replace=False))
    p = oracle.problem(layers=L, batch=B, kv_heads=H, q_heads=H, head_dim=d, max_seq_len=N,
                       budget=budget, window=1, mix_lambda=0.1)
    k, v = k0.copy(), v0.copy()
    oracle.compact(p, k, v, lens, None, keep)
    np.testing.assert_array_equal(k, _naive_gather_contig(k0, lens, keep, budget))
    np.testing.assert_array_equal(v, _naive_gather_contig(v0, lens, keep, budget))


# ------------------------------------------------------------ page figures

def test_page_figures_and_workload_flags():
    g = json.load(open(os.path.join(GOLDEN, "pages_figures.json")))
    for wid in (0, 1, 4):
        s = synthetic.WORKLOADS[wid]
        assert s.budget == g["kv_budget"]["value"] and s.window == g["window_size"]["value"]
        assert s.buffer == g["divide_length"]["value"]
    for s in synthetic.WORKLOADS.values():
        lo, hi = g["mix_lambda_range"]["value"]
        assert s.mix_lambda == g["mix_lambda"]["value"] and lo <= s.mix_lambda <= hi
        assert s.block_size in g["paged_block_sizes"]["value"]
    m = g["kv_gb_per_32k_tokens_r1_llama8b"]
    per_token = m["model"]["layers"] * m["model"]["kv_heads"] * m["model"]["head_dim"] * 2 * m["model"]["bytes_per_value"]
    assert per_token == 128 * 1024
    assert abs(per_token * m["tokens"] / 1e9 - m["value"]) < 0.1
