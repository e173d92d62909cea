"""Decode-loop integration on the GPU: the device-side trigger (compress only
sequences holding budget + buffer tokens), FREE_BLOCKS into a device stack of
free blocks, a window of queries kept as a ring buffer, and the whole call
captured once in a CUDA graph and replayed with new data. Expected results come
from the oracle: triggered sequences are compressed exactly as the oracle
compresses them; the others are left as they were."""

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import oracle
import synthetic
from helpers import check_keep_row, check_scores_row, oracle_problem

pytestmark = pytest.mark.gpu

DEV = "cuda"
TRIG = rkv.TRIGGER_BUDGET_PLUS_BUFFER


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


SHAPE = synthetic.custom_shape(layers=2, batch=8, kv_heads=2, q_heads=8, budget=256, buffer=64, window=8,
                               paged=True)
# below the budget, between budget and budget + buffer, at and above the trigger
LENS_A = np.array([100, 256, 257, 300, 319, 320, 320, 200])
LENS_B = np.array([320, 320, 50, 320, 310, 257, 320, 320])


def expected(wl, k0, v0, lens, stack0, top0):
    """Oracle result of one triggered call plus the free-stack push."""
    s = wl.shape
    p = oracle_problem(wl)
    bt = wl.block_table.cpu().numpy()
    orc = oracle.compress(p, k0.copy(), v0.copy(), synthetic.bf16_bits(wl.q_window), lens, bt)
    trig = lens >= s.budget + s.buffer
    keep = orc["keep_idx"].copy()
    for b in np.nonzero(~trig)[0]:
        kb = min(int(lens[b]), s.budget)
        keep[:, b] = -1
        keep[:, b, :, :kb] = np.arange(kb)
    # freed lists of the triggered sequences only: an untriggered one frees
    # what a sequence of min(N, budget) tokens frees, i.e. nothing
    lens_f = np.where(trig, lens, np.minimum(lens, s.budget)).astype(np.int32)
    off, ids, _ = oracle.freed_blocks(p, lens_f, bt)
    new_lens = np.where(trig, np.minimum(lens, s.budget), lens)
    stack = np.concatenate([stack0[:top0], ids])
    return dict(orc=orc, trig=trig, keep=keep, k0=k0, v0=v0, p=p, bt=bt, off=off, ids=ids, new_lens=new_lens,
                stack=stack, top=top0 + len(ids))


def check(wl, exp, out, k, v, stack, top, lens):
    s = wl.shape
    for l in range(s.layers):
        for b in range(s.batch):
            n = int(lens[b])
            for h in range(s.kv_heads):
                got = out["keep_idx"][l, b, h].cpu().numpy()
                if exp["trig"][b]:
                    check_keep_row(got, exp["orc"]["S"][l, b, h], n, s.budget, s.window, f"l={l} b={b} h={h}")
                    row = {nm: exp["orc"][nm][l, b, h] for nm in ("I_hat", "R_hat", "S")}
                    check_scores_row(out["scores"][:, l, b, h].cpu().numpy(), row, n, f"l={l} b={b} h={h}")
                else:
                    assert np.array_equal(got, exp["keep"][l, b, h]), f"l={l} b={b} h={h}: not identity"
    # compaction, bit-exact against the oracle's gather with the GPU's kept
    # indices (identity rows leave a sequence untouched)
    k_ref, v_ref = exp["k0"].copy(), exp["v0"].copy()
    oracle.compact(exp["p"], k_ref, v_ref, lens, exp["bt"], out["keep_idx"].cpu().numpy())
    assert np.array_equal(synthetic.bf16_bits(k), k_ref), "K cache"
    assert np.array_equal(synthetic.bf16_bits(v), v_ref), "V cache"
    assert np.array_equal(out["freed_off"].cpu().numpy(), exp["off"])
    assert np.array_equal(out["new_seq_lens"].cpu().numpy(), exp["new_lens"])
    nf = exp["off"][-1]
    assert np.array_equal(out["freed_ids"].cpu().numpy()[:nf], exp["ids"])
    assert int(top.item()) == exp["top"]
    assert np.array_equal(stack.cpu().numpy()[:exp["top"]], exp["stack"])


def test_trigger_and_free_stack_eager():
    wl = synthetic.generate(SHAPE, device=DEV, seed=31, seq_lens=LENS_A)
    p = rkv.problem_for(SHAPE, wl.num_blocks, trigger=TRIG)
    out = rkv.allocate_outputs(p, DEV, scores=True)
    k0, v0 = synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache)
    stack = torch.full((4096,), -7, dtype=torch.int32, device=DEV)
    stack[:5] = torch.arange(900, 905, dtype=torch.int32)
    top = torch.tensor([5], dtype=torch.int32, device=DEV)
    exp = expected(wl, k0, v0, LENS_A, stack.cpu().numpy(), 5)
    rkv.rkv_compress(p, wl.k_cache, wl.v_cache, wl.q_window, wl.seq_lens, wl.block_table, out["keep_idx"],
                     out["freed_off"], out["freed_ids"], out["new_seq_lens"], out["scores"], out["workspace"])
    rkv.rkv_free_blocks_push(out["freed_off"], out["freed_ids"], SHAPE.batch, stack, top)
    assert rkv.rkv_device_status() == rkv.RKV_OK
    check(wl, exp, out, wl.k_cache, wl.v_cache, stack, top, LENS_A)


def test_free_stack_overflow_is_reported_and_writes_nothing():
    off = torch.tensor([0, 3, 5], dtype=torch.int32, device=DEV)
    ids = torch.tensor([11, 12, 13, 14, 15], dtype=torch.int32, device=DEV)
    stack = torch.zeros(6, dtype=torch.int32, device=DEV)
    top = torch.tensor([2], dtype=torch.int32, device=DEV)
    rkv.rkv_free_blocks_push(off, ids, 2, stack, top)
    assert rkv.rkv_device_status() == rkv.RKV_ERR_DEVICE
    assert int(top.item()) == 2 and torch.count_nonzero(stack).item() == 0
    top.fill_(1)
    rkv.rkv_free_blocks_push(off, ids, 2, stack, top)
    assert rkv.rkv_device_status() == rkv.RKV_OK
    assert stack.cpu().tolist() == [0, 11, 12, 13, 14, 15] and int(top.item()) == 6


def test_window_ring_buffer_order_does_not_matter():
    """Rotating the window axis of q_window (a ring buffer written one
    position per step) leaves scores equal to fp32 rounding and the kept
    sets identical."""
    shape = synthetic.custom_shape(layers=2, batch=2, kv_heads=2, q_heads=8, budget=200, buffer=56, window=8)
    res = []
    for shift in (0, 3):
        wl = synthetic.generate(shape, device=DEV, seed=41)
        q = torch.roll(wl.q_window, shifts=shift, dims=3).contiguous()
        p = rkv.problem_for(shape)
        out = rkv.allocate_outputs(p, DEV, scores=True)
        rkv.rkv_compress(p, wl.k_cache, wl.v_cache, q, wl.seq_lens, None, out["keep_idx"], out["freed_off"],
                         None, out["new_seq_lens"], out["scores"], out["workspace"])
        assert rkv.rkv_device_status() == rkv.RKV_OK
        res.append((out["scores"].cpu().numpy(), out["keep_idx"].cpu().numpy()))
    assert np.max(np.abs(res[0][0] - res[1][0])) < 1e-5
    assert np.array_equal(res[0][1], res[1][1])


def test_captured_graph_replays_with_new_data():
    """rkv_compress (device trigger) + rkv_free_blocks_push captured once in a
    CUDA graph, replayed on two different batches copied into the same
    buffers, each checked against the oracle."""
    wl_a = synthetic.generate(SHAPE, device=DEV, seed=51, seq_lens=LENS_A)
    wl_b = synthetic.generate(SHAPE, device=DEV, seed=52, seq_lens=LENS_B)
    p = rkv.problem_for(SHAPE, wl_a.num_blocks, trigger=TRIG)
    out = rkv.allocate_outputs(p, DEV, scores=True)
    # static buffers of the graph
    k, v, q = wl_a.k_cache.clone(), wl_a.v_cache.clone(), wl_a.q_window.clone()
    lens, table = wl_a.seq_lens.clone(), wl_a.block_table.clone()
    stack = torch.zeros(4096, dtype=torch.int32, device=DEV)
    top = torch.zeros(1, dtype=torch.int32, device=DEV)

    def step():
        rkv.rkv_compress(p, k, v, q, lens, table, out["keep_idx"], out["freed_off"], out["freed_ids"],
                         out["new_seq_lens"], out["scores"], out["workspace"])
        rkv.rkv_free_blocks_push(out["freed_off"], out["freed_ids"], SHAPE.batch, stack, top)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager first call: one-time set-up happens outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    assert rkv.rkv_device_status() == rkv.RKV_OK
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for wl, lens_np in ((wl_a, LENS_A), (wl_b, LENS_B)):
        k.copy_(wl.k_cache)
        v.copy_(wl.v_cache)
        q.copy_(wl.q_window)
        lens.copy_(wl.seq_lens)
        table.copy_(wl.block_table)
        stack.zero_()
        top.zero_()
        out["scores"].zero_()
        exp = expected(wl, synthetic.bf16_bits(wl.k_cache), synthetic.bf16_bits(wl.v_cache), lens_np,
                       np.zeros(4096, dtype=np.int32), 0)
        graph.replay()
        torch.cuda.synchronize()
        assert rkv.rkv_device_status() == rkv.RKV_OK
        check(wl, exp, out, k, v, stack, top, lens_np)
