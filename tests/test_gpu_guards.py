"""Out-of-bounds writes show up without a sanitizer: every output and the
workspace are views into larger buffers whose guard regions hold a pattern
that must survive the call; the caches are views with guard rows around them."""

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda"
GUARD = 4096  # elements on each side


@pytest.fixture(scope="module", autouse=True)
def _built():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def guarded(shape, dtype, fill):
    """(base, view): the view starts 256-byte aligned, at least GUARD elements
    from either end of the base buffer; everything else in base holds `fill`."""
    n = int(np.prod(shape))
    esz = torch.empty(0, dtype=dtype).element_size()
    slack = 256 // esz
    base = torch.full((n + 2 * GUARD + slack,), fill, dtype=dtype, device=DEV)
    start = GUARD + ((-(base.data_ptr() // esz + GUARD)) % slack)
    view = base[start:start + n].view(*shape)
    base.guard_ranges = ((0, start), (start + n, base.numel()))
    return base, view


def guards_intact(base, fill):
    return all(bool(torch.all(base[a:b] == fill).item()) for a, b in base.guard_ranges)


@pytest.mark.parametrize("wid,kw,redundancy,selection", [
    (0, dict(), rkv.REDUNDANCY_GRAM, rkv.SELECT_PER_HEAD),
    (4, dict(layers=2, batch=4), rkv.REDUNDANCY_GRAM, rkv.SELECT_PER_HEAD),
    (3, dict(layers=1, batch=1), rkv.REDUNDANCY_GRAM, rkv.SELECT_PER_HEAD),
    (4, dict(layers=2, batch=4), rkv.REDUNDANCY_CLOSED_FORM, rkv.SELECT_SHARED_HEADS),
])
def test_no_write_outside_outputs(wid, kw, redundancy, selection):
    wl = synthetic.generate(wid, device=DEV, **kw)
    s = wl.shape
    p = rkv.problem_for(s, wl.num_blocks, redundancy=redundancy, selection=selection)
    # caches inside guard rows
    kb, k = guarded(wl.k_cache.shape, torch.bfloat16, 0.0)
    vb, v = guarded(wl.v_cache.shape, torch.bfloat16, 0.0)
    k.copy_(wl.k_cache)
    v.copy_(wl.v_cache)
    for (a0, a1) in kb.guard_ranges:
        kb[a0:a1] = 7.0
    for (a0, a1) in vb.guard_ranges:
        vb[a0:a1] = -7.0
    L, B, H = s.layers, s.batch, s.kv_heads
    keep_b, keep = guarded((L, B, H, s.budget), torch.int32, -12345)
    off_b, off = guarded((B + 1,), torch.int32, -12345)
    ids_b, ids = guarded((max(1, B * max(s.blocks_per_seq if s.paged else 1, 1)),), torch.int32, -12345)
    len_b, lens = guarded((B,), torch.int32, -12345)
    sc_b, scores = guarded((3, L, B, H, s.max_seq_len), torch.float32, 1234.5)
    ws_bytes = rkv.workspace_size(p)
    ws_b, ws = guarded(((ws_bytes + 255) // 256 * 256 // 4,), torch.float32, 4321.0)
    assert ws.data_ptr() % 256 == 0
    rkv.rkv_compress(p, k, v, wl.q_window, wl.seq_lens, wl.block_table, keep, off, ids if s.paged else None, lens,
                     scores, ws.view(torch.uint8))
    assert rkv.rkv_device_status() == rkv.RKV_OK
    assert guards_intact(kb, 7.0), "K guard rows"
    assert guards_intact(vb, -7.0), "V guard rows"
    for name, base, fill in (("keep_idx", keep_b, -12345), ("freed_off", off_b, -12345),
                             ("freed_ids", ids_b, -12345), ("new_seq_lens", len_b, -12345),
                             ("scores", sc_b, 1234.5), ("workspace", ws_b, 4321.0)):
        assert guards_intact(base, fill), name
    # entries past each sequence's length in the score planes are left untouched
    n = wl.seq_lens.cpu().numpy()
    sc = scores.cpu().numpy()
    for b in range(B):
        assert np.all(sc[:, :, b, :, n[b]:] == 1234.5)
