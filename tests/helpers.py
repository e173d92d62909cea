"""Shared test helpers: run the CUDA path through the C ABI on a synthetic
workload, run the oracle on the same bf16 bytes, and compare them with the
acceptance rules of the method:
  - normalised scores (I^, R^, S) within 1e-3 absolute;
  - kept sets identical except tokens whose oracle S lies within 1e-3 of the
    oracle's (budget - window)-th candidate score;
  - compacted K/V and freed-block lists bit-exact given the GPU's kept indices.
"""

from __future__ import annotations

import numpy as np
import torch

import decode_kv_cache_05_b300 as rkv
import oracle
import synthetic

SCORE_TOL = 1e-3
BAND = 1e-3


def oracle_problem(wl: synthetic.Workload):
    s = wl.shape
    return oracle.problem(layers=s.layers, batch=s.batch, kv_heads=s.kv_heads, q_heads=s.q_heads,
                          head_dim=s.head_dim, max_seq_len=s.max_seq_len, budget=s.budget, window=s.window,
                          mix_lambda=s.mix_lambda, paged=s.paged, block_size=s.block_size,
                          num_blocks=wl.num_blocks, max_blocks=s.blocks_per_seq if s.paged else 0)


def run_gpu(wl: synthetic.Workload, scores: bool = True, redundancy: int = rkv.REDUNDANCY_GRAM) -> dict:
    """rkv_compress on the workload's (device) tensors. K/V are compacted in
    place; the originals are returned as host copies."""
    p = rkv.problem_for(wl.shape, wl.num_blocks, redundancy=redundancy)
    dev = wl.k_cache.device
    k0, v0 = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    out = rkv.allocate_outputs(p, dev, scores=scores)
    rkv.rkv_compress(p, wl.k_cache, wl.v_cache, wl.q_window, wl.seq_lens, wl.block_table, out["keep_idx"],
                     out["freed_off"], out["freed_ids"] if wl.shape.paged else None, out["new_seq_lens"],
                     out["scores"], out["workspace"])
    st = rkv.rkv_device_status()
    assert st == rkv.RKV_OK, rkv.status_string(st)
    res = {k: (v.cpu().numpy() if isinstance(v, torch.Tensor) and k != "workspace" else None)
           for k, v in out.items()}
    res["k0"], res["v0"] = k0, v0
    res["k"], res["v"] = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    res["problem"] = p
    return res


def check_keep_row(keep_gpu: np.ndarray, s_oracle: np.ndarray, n: int, budget: int, w: int, where: str = ""):
    kb = min(n, budget)
    assert np.all(keep_gpu[kb:] == -1), where
    kept = keep_gpu[:kb]
    assert np.all(np.diff(kept) > 0), f"{where}: not ascending"
    if n <= budget:
        assert kept.tolist() == list(range(n)), where
        return
    assert kept[0] >= 0 and kept[-1] < n, where
    cand, take = n - w, budget - w
    assert set(range(cand, n)) <= set(kept.tolist()), f"{where}: window not kept"
    if take == 0:
        return
    thr = np.sort(s_oracle[:cand])[::-1][take - 1]
    sure_keep = np.nonzero(s_oracle[:cand] > thr + BAND)[0]
    sure_drop = np.nonzero(s_oracle[:cand] < thr - BAND)[0]
    ks = set(kept.tolist())
    missing = [int(j) for j in sure_keep if j not in ks]
    extra = [int(j) for j in sure_drop if j in ks]
    assert not missing and not extra, f"{where}: missing {missing[:8]} extra {extra[:8]}"


def check_scores_row(gpu_scores: np.ndarray, orc: dict, n: int, where: str = ""):
    """gpu_scores: [3][n] (I^, R^, S)."""
    for plane, name in enumerate(("I_hat", "R_hat", "S")):
        err = np.max(np.abs(gpu_scores[plane, :n].astype(np.float64) - orc[name][:n]), initial=0.0)
        assert err <= SCORE_TOL, f"{where}: {name} max abs error {err:.3g}"


def check_full(wl: synthetic.Workload, res: dict, closed_form: bool = False) -> dict:
    """Element-wise comparison of every head against the whole-event oracle
    (closed_form: the oracle's rank-one redundancy routine, which the oracle
    pins hold to the pairwise definition within 1e-13)."""
    s = wl.shape
    p = oracle_problem(wl)
    lens = wl.seq_lens.cpu().numpy()
    bt = None if wl.block_table is None else wl.block_table.cpu().numpy()
    q = synthetic.bf16_bits(wl.q_window)
    k_or, v_or = res["k0"].copy(), res["v0"].copy()
    orc = oracle.compress(p, k_or, v_or, q, lens, bt, closed_form=closed_form)
    del k_or, v_or
    worst = {"I_hat": 0.0, "R_hat": 0.0, "S": 0.0}
    for l in range(s.layers):
        for b in range(s.batch):
            n = int(lens[b])
            for h in range(s.kv_heads):
                where = f"l={l} b={b} h={h} n={n}"
                row = {name: orc[name][l, b, h] for name in ("I_hat", "R_hat", "S")}
                g = res["scores"][:, l, b, h]
                for plane, name in enumerate(("I_hat", "R_hat", "S")):
                    worst[name] = max(worst[name], float(np.max(np.abs(g[plane, :n] - row[name][:n]), initial=0)))
                check_scores_row(g, row, n, where)
                check_keep_row(res["keep_idx"][l, b, h], row["S"], n, s.budget, s.window, where)
    # compaction and freed lists, bit-exact, given the GPU's kept indices
    k_ref, v_ref = res["k0"].copy(), res["v0"].copy()
    oracle.compact(p, k_ref, v_ref, lens, bt, res["keep_idx"])
    assert np.array_equal(res["k"], k_ref), "K compaction differs"
    assert np.array_equal(res["v"], v_ref), "V compaction differs"
    off, ids, new_lens = oracle.freed_blocks(p, lens, bt)
    assert np.array_equal(res["freed_off"], off)
    assert np.array_equal(res["new_seq_lens"], new_lens)
    if s.paged:
        assert np.array_equal(res["freed_ids"][:off[-1]], ids)
    return worst


def logical_head(arr: np.ndarray, wl: synthetic.Workload, l: int, b: int, h: int, n: int) -> np.ndarray:
    """First n logical rows [n][d] of a head from a host copy of a cache."""
    if wl.block_table is None:
        return arr[l, b, h, :n]
    bs = wl.shape.block_size
    nb = -(-n // bs)
    blocks = wl.block_table[b, :nb].cpu().numpy()
    return arr[l][blocks][:, :, h].reshape(nb * bs, -1)[:n]


def check_sampled(wl: synthetic.Workload, res: dict, heads: list) -> dict:
    """Per-head oracle on a sample of (l, b, h) of a full-size run."""
    s = wl.shape
    lens = wl.seq_lens.cpu().numpy()
    worst = {"I_hat": 0.0, "R_hat": 0.0, "S": 0.0}
    G, w = s.group, s.window
    for (l, b, h) in heads:
        n = int(lens[b])
        where = f"l={l} b={b} h={h} n={n}"
        k = logical_head(res["k0"], wl, l, b, h, n)
        v = logical_head(res["v0"], wl, l, b, h, n)
        q = synthetic.bf16_bits(wl.q_window[l, b, h * G:(h + 1) * G]).reshape(G * w, -1)
        orc = oracle.compress_head(q, np.ascontiguousarray(k), s.budget, w, s.mix_lambda)
        g = res["scores"][:, l, b, h]
        for plane, name in enumerate(("I_hat", "R_hat", "S")):
            worst[name] = max(worst[name], float(np.max(np.abs(g[plane, :n] - orc[name][:n]), initial=0.0)))
        check_scores_row(g, orc, n, where)
        keep = res["keep_idx"][l, b, h]
        check_keep_row(keep, orc["S"], n, s.budget, w, where)
        kb = min(n, s.budget)
        kc = logical_head(res["k"], wl, l, b, h, n)
        vc = logical_head(res["v"], wl, l, b, h, n)
        assert np.array_equal(kc[:kb], k[keep[:kb]]), f"{where}: K rows"
        assert np.array_equal(vc[:kb], v[keep[:kb]]), f"{where}: V rows"
        assert np.array_equal(kc[kb:], k[kb:]) and np.array_equal(vc[kb:], v[kb:]), f"{where}: tail rows touched"
    return worst


def _head_rows(wl: synthetic.Workload, cache: torch.Tensor, l: int, b: int, h: int, n: int) -> np.ndarray:
    return synthetic.bf16_bits(synthetic.logical_rows(wl, cache, l, b, h, n))


def run_gpu_sampled(wl: synthetic.Workload, heads: list, redundancy: int = rkv.REDUNDANCY_GRAM) -> dict:
    """rkv_compress on a full-size workload (every head computed, exactly the
    launch a benchmark makes), with host copies of only the sampled heads."""
    s = wl.shape
    lens = wl.seq_lens.cpu().numpy()
    G, w = s.group, s.window
    before = {}
    for (l, b, h) in heads:
        n = int(lens[b])
        before[(l, b, h)] = (_head_rows(wl, wl.k_cache, l, b, h, n), _head_rows(wl, wl.v_cache, l, b, h, n),
                             synthetic.bf16_bits(wl.q_window[l, b, h * G:(h + 1) * G]).reshape(G * w, -1))
    p = rkv.problem_for(s, wl.num_blocks, redundancy=redundancy)
    out = rkv.allocate_outputs(p, wl.k_cache.device, scores=True)
    rkv.rkv_compress(p, wl.k_cache, wl.v_cache, wl.q_window, wl.seq_lens, wl.block_table, out["keep_idx"],
                     out["freed_off"], out["freed_ids"] if s.paged else None, out["new_seq_lens"],
                     out["scores"], out["workspace"])
    st = rkv.rkv_device_status()
    assert st == rkv.RKV_OK, rkv.status_string(st)
    after = {}
    for (l, b, h) in heads:
        n = int(lens[b])
        after[(l, b, h)] = (_head_rows(wl, wl.k_cache, l, b, h, n), _head_rows(wl, wl.v_cache, l, b, h, n),
                            out["scores"][:, l, b, h].cpu().numpy(), out["keep_idx"][l, b, h].cpu().numpy())
    return dict(before=before, after=after, freed_off=out["freed_off"].cpu().numpy(),
                freed_ids=out["freed_ids"].cpu().numpy(), new_seq_lens=out["new_seq_lens"].cpu().numpy())


def check_sampled_run(wl: synthetic.Workload, run: dict) -> dict:
    s = wl.shape
    lens = wl.seq_lens.cpu().numpy()
    worst = {"I_hat": 0.0, "R_hat": 0.0, "S": 0.0}
    for (l, b, h), (k, v, q) in run["before"].items():
        n = int(lens[b])
        where = f"l={l} b={b} h={h} n={n}"
        kc, vc, g, keep = run["after"][(l, b, h)]
        orc = oracle.compress_head(q, k, s.budget, s.window, s.mix_lambda)
        for plane, name in enumerate(("I_hat", "R_hat", "S")):
            worst[name] = max(worst[name], float(np.max(np.abs(g[plane, :n] - orc[name][:n]), initial=0.0)))
        check_scores_row(g, orc, n, where)
        check_keep_row(keep, orc["S"], n, s.budget, s.window, where)
        kb = min(n, s.budget)
        assert np.array_equal(kc[:kb], k[keep[:kb]]), f"{where}: K rows"
        assert np.array_equal(vc[:kb], v[keep[:kb]]), f"{where}: V rows"
        assert np.array_equal(kc[kb:], k[kb:]) and np.array_equal(vc[kb:], v[kb:]), f"{where}: tail rows touched"
    # freed lists and lengths for every sequence (host arithmetic on the table)
    p = oracle_problem(wl)
    bt = None if wl.block_table is None else wl.block_table.cpu().numpy()
    off, ids, new_lens = oracle.freed_blocks(p, lens, bt)
    assert np.array_equal(run["freed_off"], off)
    assert np.array_equal(run["new_seq_lens"], new_lens)
    if s.paged:
        assert np.array_equal(run["freed_ids"][:off[-1]], ids)
    return worst


def sample_heads(wl: synthetic.Workload, count: int, seed: int = 0) -> list:
    """A seeded sample of (l, b, h), always including the first and last head."""
    s = wl.shape
    rng = np.random.default_rng(seed)
    heads = {(0, 0, 0), (s.layers - 1, s.batch - 1, s.kv_heads - 1)}
    while len(heads) < min(count, s.events * s.kv_heads):
        heads.add((int(rng.integers(s.layers)), int(rng.integers(s.batch)), int(rng.integers(s.kv_heads))))
    return sorted(heads)
