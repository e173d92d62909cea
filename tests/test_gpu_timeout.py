"""The bounded-wait timeout path, exercised on the GPU without a fault or a hang.

Every in-kernel wait of the library gives up after a limit, records
RKV_ERR_TIMEOUT in the device error word, waits (bounded) for the copies it
issued and returns. Here a test build of the library (librkv_waittest.so, the
same sources compiled with RKV_SELECT_WAIT_TEST) makes rkv_select also wait on
an mbarrier that nothing ever arrives on, with a 2 ms limit. rkv_select is a
single-CTA kernel without clusters, so no peer CTA is left waiting on it. The
test checks that the wait runs out, that the status reads RKV_ERR_TIMEOUT,
that no kept index was written, and that the context stays usable: the
shipped library's rkv_select then gives the oracle's selection on the same
inputs."""

import ctypes

import numpy as np
import pytest
import torch

import decode_kv_cache_05_b300 as rkv
import oracle
import synthetic

pytestmark = pytest.mark.gpu

DEV = "cuda"
SENTINEL = -7


@pytest.fixture(scope="module")
def waittest_lib():
    from decode_kv_cache_05_b300 import build
    build.build()
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    path = build.build_variant("waittest", {"RKV_SELECT_WAIT_TEST": 1, "RKV_SELECT_WAIT_TEST_NS": "2000000ull"})
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.rkv_select.argtypes = [ctypes.POINTER(rkv.Problem), vp, vp, vp, vp, vp, vp]
    lib.rkv_select.restype = ctypes.c_int
    lib.rkv_device_status.argtypes = [vp]
    lib.rkv_device_status.restype = ctypes.c_int
    return lib


def _scores(shape, stride, seed=3):
    rng = np.random.default_rng(seed)
    I = (rng.integers(0, 64, size=(shape.kv_heads, stride)) / 64.0).astype(np.float32)
    R = (rng.integers(0, 64, size=(shape.kv_heads, stride)) / 64.0).astype(np.float32)
    return I, R


def test_select_wait_runs_out_and_reports_timeout(waittest_lib):
    shape = synthetic.custom_shape(kv_heads=2, q_heads=4, budget=96, buffer=64, window=8)
    p = rkv.problem_for(shape)
    stride = rkv.score_stride(p)
    n = shape.max_seq_len
    I, R = _scores(shape, stride)
    imp = torch.from_numpy(I).to(DEV)
    red = torch.from_numpy(R).to(DEV)
    seq = torch.tensor([n], dtype=torch.int32, device=DEV)
    keep = torch.full((1, 1, shape.kv_heads, shape.budget), SENTINEL, dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    assert rkv.rkv_device_status() == rkv.RKV_OK  # no error left over from earlier tests

    st = waittest_lib.rkv_select(ctypes.byref(p), imp.data_ptr(), red.data_ptr(), seq.data_ptr(), keep.data_ptr(),
                                 None, stream)
    assert st == rkv.RKV_OK  # queued; the timeout is found on the device
    assert waittest_lib.rkv_device_status(stream) == rkv.RKV_ERR_TIMEOUT
    assert waittest_lib.rkv_device_status(stream) == rkv.RKV_OK  # reading the word cleared it
    assert torch.all(keep == SENTINEL).item(), "a kernel that gave up must not write kept indices"

    # the context is still usable: the shipped library scores and selects as
    # the oracle does (ties settled on the GPU's own fp32 S, as in the stage
    # test of rkv_select)
    scores = torch.zeros((3, 1, 1, shape.kv_heads, n), dtype=torch.float32, device=DEV)
    rkv.rkv_select(p, imp, red, seq, keep, scores)
    assert rkv.rkv_device_status() == rkv.RKV_OK
    got = keep.cpu().numpy()[0, 0]
    for h in range(shape.kv_heads):
        ih = oracle.minmax(I[h, :n].astype(np.float64))
        rh = oracle.minmax(R[h, :n].astype(np.float64))
        got_s = scores[2, 0, 0, h].cpu().numpy()
        assert np.max(np.abs(got_s - oracle.mix(ih, rh, shape.mix_lambda))) < 1e-6
        want = oracle.select(got_s.astype(np.float64), shape.budget, shape.window)
        assert got[h].tolist() == want.tolist()
