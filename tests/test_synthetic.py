"""Host-side checks of the seeded input generator (structure only)."""
import numpy as np
import torch

import synthetic
from synthetic import _chain_depth, _dup_sources, _run_sources


def test_dup_sources_count_and_order():
    rng = np.random.default_rng(0)
    src = _dup_sources(rng, 1152, 0.25)
    pos = np.nonzero(src >= 0)[0]
    assert pos.size == 288 and pos.min() >= 1
    assert np.all(src[pos] < pos)


def test_run_sources_cover_and_lengths():
    rng = np.random.default_rng(1)
    src = _run_sources(rng, 2176)
    covered = int((src >= 0).sum())
    assert covered == int(np.ceil(0.3 * 2176))
    pos = np.nonzero(src >= 0)[0]
    assert np.all(src[pos] < pos)
    # runs: maximal stretches with one source; all but the truncated last are 8..32 long
    lengths = []
    i = 0
    while i < src.size:
        if src[i] < 0:
            i += 1
            continue
        j = i
        while j < src.size and src[j] == src[i] and src[j] >= 0:
            j += 1
        lengths.append(j - i)
        i = j
    assert max(lengths) <= 64  # two adjacent runs may share a source by chance


def test_chain_depth():
    src = np.array([-1, 0, 1, -1, 2, 0])
    assert _chain_depth(src).tolist() == [0, 1, 2, 0, 3, 1]


def test_duplicates_are_near_copies():
    wl = synthetic.generate(0)
    k = wl.k_cache[0, 0].float()  # [H][N][d]
    kn = k / k.norm(dim=-1, keepdim=True)
    cos = torch.einsum("hnd,hmd->hnm", kn, kn)
    cos.diagonal(dim1=1, dim2=2).fill_(0)
    best = cos.max(dim=-1).values  # [H][N]
    # 288 near-duplicate positions per head have a partner with cosine > 0.99
    high = (best > 0.99).sum(dim=-1)
    assert torch.all(high >= 288)


def test_paged_table_is_a_permutation_and_lengths_ragged():
    wl = synthetic.generate(4, layers=1, batch=6)
    bt = wl.block_table.numpy()
    assert sorted(bt.reshape(-1).tolist()) == list(range(wl.num_blocks))
    lens = wl.seq_lens.numpy()
    assert lens.min() >= 1025 and lens.max() <= 1152


def test_logical_rows_paged_roundtrip():
    wl = synthetic.generate(4, layers=1, batch=2)
    n = int(wl.seq_lens[1])
    rows = synthetic.logical_rows(wl, wl.k_cache, 0, 1, 3, n)
    blk = int(wl.block_table[1, 5])
    assert torch.equal(rows[5 * 16 + 7], wl.k_cache[0, blk, 7, 3])
