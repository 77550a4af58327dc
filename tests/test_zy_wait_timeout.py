"""Failure detection on the GPU without a fault: a bounded mbarrier wait that
nothing completes runs out, the kernel records it in the device error word
and returns, the host reads the bit through ws_device_error, and the context
stays usable.  (Named to run after the tests that expect a clean word.)"""
import numpy as np
import pytest
import torch

import synth
from cudart import memcpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def test_bounded_wait_runs_out_and_reports(B, oracle):
    import time
    st, _ = B.ws_device_error(True)                           # start clean
    assert st == B.WS_OK
    assert B.ws_selftest_wait_timeout(0) == B.WS_ERR_INVALID_ARGUMENT
    t0 = time.perf_counter()
    B.check(B.ws_selftest_wait_timeout(2000))                 # a 2 ms limit
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    st, flags = B.ws_device_error(True)
    assert st == B.WS_OK and flags & 1, flags                 # the timeout bit, then cleared
    assert 0.0015 < elapsed < 5.0
    st, flags = B.ws_device_error(False)
    assert st == B.WS_OK and flags == 0
    # the context still works
    frames = synth.frames_uniform(3, 1, 48, 64)
    desc = B.preprocess_desc(64, 48, 32, 32)
    src = torch.from_numpy(frames).cuda()
    out = torch.empty((1, 3, 32, 32), dtype=torch.float32, device="cuda")
    B.check(B.ws_preprocess(desc, src.data_ptr(), 1, out.data_ptr(), 0))
    torch.cuda.synchronize()
    assert np.max(np.abs(out.cpu().numpy() - oracle.preprocess(frames, 64, 48, 32, 32))) <= 1e-5


def test_lane_wait_reports_a_kernel_that_gave_up(B, oracle):
    """A bounded wait that runs out on a lane's stream is reported by that
    lane's wait as WS_ERR_DEVICE (its own error word, not the device-wide
    one); the word is cleared, so the next submit is clean and correct."""
    from post_processing_gb300 import Lane
    frames = synth.frames_uniform(21, 2, 108, 192)
    logits = synth.logits_with_ties(22, 2, 20000)
    src = torch.from_numpy(frames).cuda()
    lg = torch.from_numpy(logits).cuda()
    d = B.lane_desc(B.preprocess_desc(192, 108, 64, 64), 2, 2, 20000, 32, input=src.data_ptr(),
                    logits=lg.data_ptr())
    st, _ = B.ws_device_error(True)
    assert st == B.WS_OK
    with Lane(d) as lane:
        lane.acquire()
        assert B.ws_lane_selftest_wait_timeout(lane.handle, 0) == B.WS_ERR_INVALID_ARGUMENT
        B.check(B.ws_lane_selftest_wait_timeout(lane.handle, 2000))
        lane.submit()
        assert B.ws_lane_selftest_wait_timeout(lane.handle, 2000) == B.WS_ERR_LANE_BUSY
        st, _ = B.ws_lane_wait(lane.handle, -1)
        assert st == B.WS_ERR_DEVICE, B.ws_status_string(st)
        assert "0x1" in B.ws_last_error()
        assert lane.state == B.WS_LANE_FREE
        st, flags = B.ws_device_error(False)
        assert st == B.WS_OK and flags == 0          # the device-wide word is untouched
        for _ in range(2):                           # clean again, and correct
            lane.acquire()
            lane.submit()
            lane.wait()
            v, i = np.empty((2, 32), np.float32), np.empty((2, 32), np.int32)
            b = lane.buffers
            memcpy(v.ctypes.data, b.result_val_device, v.nbytes)
            memcpy(i.ctypes.data, b.result_idx_device, i.nbytes)
            wv, wi = oracle.topk(logits, 32)
            assert np.array_equal(i, wi) and np.array_equal(v.view(np.uint32), wv.view(np.uint32))


def test_pool_complete_reports_a_kernel_that_gave_up(B):
    """The same error through the lane pool: complete returns WS_ERR_DEVICE
    with the lane held, and the lane's next job completes cleanly."""
    d = B.lane_desc(B.preprocess_desc(64, 48, 32, 32), 1, 1, 1000, 5)
    st, P = B.ws_pool_create(d, 2)
    B.check(st)
    try:
        st, L = B.ws_pool_acquire(P, -1)
        B.check(st)
        B.check(B.ws_lane_selftest_wait_timeout(L, 2000))
        B.check(B.ws_pool_submit(P, L, 1))
        st, L2, _ = B.ws_pool_complete(P, -1)
        assert st == B.WS_ERR_DEVICE and L2 == L
        B.check(B.ws_pool_recycle(P, L))
        for _ in range(3):
            st, L = B.ws_pool_acquire(P, -1)
            B.check(st)
            B.check(B.ws_pool_submit(P, L, 1))
            st, L, _ = B.ws_pool_complete(P, -1)
            B.check(st)
            B.check(B.ws_pool_recycle(P, L))
    finally:
        B.check(B.ws_pool_destroy(P))
