"""Failure detection on the GPU without a fault: a bounded mbarrier wait that
nothing completes runs out, the kernel records it in the device error word
and returns, the host reads the bit through ws_device_error, and the context
stays usable.  (Named to run after the tests that expect a clean word.)"""
import numpy as np
import pytest
import torch

import synth

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
