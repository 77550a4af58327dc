"""Host-side fault injection into the cleanup paths of ws_lane_create,
ws_lane_rebind and ws_pool_create ("Inside WarpStream TRT", lane section:
failures are explicit; no half-built lane and no silent leak).

Every internal call of those paths that can fail passes a fault point; the
test makes each one fail in turn, before the CUDA call it guards, and checks
the documented status, that every CUDA resource made so far was released
(the library's own counters), and that the next call succeeds.  Nothing
faults, traps or hangs the GPU: the failures are host-side returns."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from cudart import memcpy

pytestmark = pytest.mark.gpu

FIELDS = ("device_allocs", "host_allocs", "graphs", "graph_execs", "events", "streams")


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def live(B):
    st, c = B.ws_debug_get_counters()
    B.check(st)
    return {f: getattr(c, f) for f in FIELDS}


def points(B):
    st, c = B.ws_debug_get_counters()
    B.check(st)
    return c.fault_points


def expected_status(B, message):
    """The status a real failure of the named call gives."""
    if "cudaMalloc" in message or "cudaHostAlloc" in message:
        return B.WS_ERR_OUT_OF_MEMORY
    if any(w in message for w in ("capture", "instantiate", "upload")):
        return B.WS_ERR_CAPTURE
    return B.WS_ERR_CUDA


def lane_descs(B):
    """Lanes that pass many fault points: copy-in input and copy-out result
    (pinned and device slots), stage timing (five events), batch buckets with
    long rows (a Top-K workspace per bucket), a detection lane."""
    pre = B.preprocess_desc(200, 120, 64, 48)
    yield "topk_copy_buckets", B.lane_desc(pre, 3, 3, 20000, 32, input_mode=B.WS_INPUT_COPY,
                                           result_mode=B.WS_RESULT_COPY,
                                           flags=B.WS_LANE_FLAG_BUCKETS | B.WS_LANE_FLAG_STAGE_TIMING)
    yield "topk_mapped", B.lane_desc(pre, 2, 2, 1000, 5, input_mode=B.WS_INPUT_MAPPED,
                                     result_mode=B.WS_RESULT_MAPPED)
    ddesc = B.detect_desc(in_w=320, in_h=192, reg_max=8, num_classes=3, conf=0.3)
    yield "detect", B.lane_desc(B.preprocess_desc(200, 120, 320, 192, letterbox=True, norm="scale"), 2, 0, 0, 0,
                                detect=ddesc, flags=B.WS_LANE_FLAG_NO_TIMING)


@pytest.mark.parametrize("which", ["topk_copy_buckets", "topk_mapped", "detect"])
def test_lane_create_fails_cleanly_at_every_point(B, which):
    desc = dict(lane_descs(B))[which]
    torch.cuda.synchronize()
    base = live(B)
    B.check(B.ws_debug_inject_failure(0, 0))
    st, h = B.ws_lane_create(desc)
    B.check(st)
    n_points = points(B)
    assert n_points >= 10, n_points
    B.check(B.ws_lane_destroy(h))
    assert live(B) == base
    seen = set()
    for n in range(1, n_points + 1):
        B.check(B.ws_debug_inject_failure(n, 1))
        st, h = B.ws_lane_create(desc)
        msg = B.ws_last_error()
        B.check(B.ws_debug_inject_failure(0, 0))
        assert st != B.WS_OK and h is None, (n, msg)
        assert "injected failure" in msg, (n, msg)
        assert st == expected_status(B, msg), (n, B.ws_status_string(st), msg)
        seen.add(st)
        assert live(B) == base, (n, msg, live(B), base)
    assert {B.WS_ERR_OUT_OF_MEMORY, B.WS_ERR_CAPTURE, B.WS_ERR_CUDA} <= seen
    # the next create succeeds and the lane works
    st, h = B.ws_lane_create(desc)
    B.check(st)
    B.check(B.ws_lane_acquire(h))
    B.check(B.ws_lane_submit(h))
    st, _ = B.ws_lane_wait(h, -1)
    B.check(st)
    B.check(B.ws_lane_destroy(h))
    assert live(B) == base


def test_pool_create_fails_cleanly(B):
    pre = B.preprocess_desc(200, 120, 64, 48)
    desc = B.lane_desc(pre, 2, 2, 20000, 32, flags=B.WS_LANE_FLAG_NO_TIMING)
    torch.cuda.synchronize()
    base = live(B)
    B.check(B.ws_debug_inject_failure(0, 0))
    st, P = B.ws_pool_create(desc, 3)
    B.check(st)
    n_points = points(B)
    B.check(B.ws_pool_destroy(P))
    assert live(B) == base
    for n in range(1, n_points + 1):
        B.check(B.ws_debug_inject_failure(n, 1))
        st, P = B.ws_pool_create(desc, 3)
        msg = B.ws_last_error()
        B.check(B.ws_debug_inject_failure(0, 0))
        assert st == expected_status(B, msg) and P is None, (n, B.ws_status_string(st), msg)
        assert live(B) == base, (n, msg)
    st, P = B.ws_pool_create(desc, 3)
    B.check(st)
    B.check(B.ws_pool_destroy(P))
    assert live(B) == base


def run_and_check(B, lane, frames, logits, oracle):
    lane.acquire()
    lane.submit()
    lane.wait()
    b = lane.buffers
    t = np.empty((3, 3, 48, 64), np.float32)
    memcpy(t.ctypes.data, b.tensor, t.nbytes)
    assert np.max(np.abs(t - oracle.preprocess(frames, 200, 120, 64, 48))) <= 1e-5
    v, i = np.empty((3, 32), np.float32), np.empty((3, 32), np.int32)
    memcpy(v.ctypes.data, b.result_val_device, v.nbytes)
    memcpy(i.ctypes.data, b.result_idx_device, i.nbytes)
    wv, wi = oracle.topk(logits, 32)
    assert np.array_equal(i, wi) and np.array_equal(v.view(np.uint32), wv.view(np.uint32))


@pytest.mark.parametrize("count", [1, 2])
def test_rebind_is_all_or_nothing(B, oracle, count):
    """A bucketed lane (buckets 1, 2, 3) re-bound to new input and logits
    slots while `count` consecutive fault points fail, at every position.  A
    refused in-place update falls back to a new executable graph (WS_OK,
    re-instantiated); any other failure returns WS_ERR_CAPTURE and leaves the
    lane on its previous slots, with the graphs already updated put back --
    the next replay still reads the old frames and logits."""
    from post_processing_gb300 import Lane
    old_f = synth.frames_uniform(31, 3, 120, 200)
    old_l = synth.logits_with_ties(32, 3, 20000)
    new_f = synth.frames_uniform(33, 3, 120, 200)
    new_l = synth.logits_with_ties(34, 3, 20000)
    src_old, lg_old = torch.from_numpy(old_f).cuda(), torch.from_numpy(old_l).cuda()
    src_new, lg_new = torch.from_numpy(new_f).cuda(), torch.from_numpy(new_l).cuda()
    pre = B.preprocess_desc(200, 120, 64, 48)
    d = B.lane_desc(pre, 3, 3, 20000, 32, input=src_old.data_ptr(), logits=lg_old.data_ptr(),
                    flags=B.WS_LANE_FLAG_BUCKETS)
    torch.cuda.synchronize()
    with Lane(d) as lane:
        run_and_check(B, lane, old_f, old_l, oracle)
        base = live(B)
        B.check(B.ws_debug_inject_failure(0, 0))
        st, re = B.ws_lane_rebind(lane.handle, src_new.data_ptr(), lg_new.data_ptr())
        B.check(st)
        n_points = points(B)
        assert n_points >= 6 and re == 0
        assert live(B) == base
        run_and_check(B, lane, new_f, new_l, oracle)
        B.check(B.ws_lane_rebind(lane.handle, src_old.data_ptr(), lg_old.data_ptr())[0])
        outcomes = set()
        for n in range(1, n_points + 1):
            B.check(B.ws_debug_inject_failure(n, count))
            st, re = B.ws_lane_rebind(lane.handle, src_new.data_ptr(), lg_new.data_ptr())
            msg = B.ws_last_error()
            B.check(B.ws_debug_inject_failure(0, 0))
            lane.buffers = B.ws_lane_get_buffers(lane.handle)[1]
            if st == B.WS_OK:
                outcomes.add("reinstantiated" if re else "ok")
                assert lane.buffers.input_device == src_new.data_ptr()
                assert lane.buffers.logits == lg_new.data_ptr()
                run_and_check(B, lane, new_f, new_l, oracle)
                B.check(B.ws_lane_rebind(lane.handle, src_old.data_ptr(), lg_old.data_ptr())[0])
            else:
                outcomes.add("refused")
                assert st == B.WS_ERR_CAPTURE, (n, B.ws_status_string(st), msg)
                assert "injected failure" in msg, msg
                assert lane.buffers.input_device == src_old.data_ptr()
                assert lane.buffers.logits == lg_old.data_ptr()
            assert live(B) == base, (n, msg)
            run_and_check(B, lane, old_f, old_l, oracle)
        # one failing point: a refused update falls back to a new executable
        # graph; two in a row: the update and the fallback both fail
        assert "refused" in outcomes
        assert ("reinstantiated" in outcomes) == (count == 1)
