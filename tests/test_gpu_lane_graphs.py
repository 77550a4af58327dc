"""Graph variants of a lane on the GPU: batch buckets (ws_lane_submit_n),
re-binding the producer / network slots with cudaGraphExecUpdate
(ws_lane_rebind), NVTX-instrumented lanes, and the lane pool -- each result
against the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from cudart import _cudart, memcpy

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def host_array(ptr, nbytes, dtype):
    return np.frombuffer((ctypes.c_char * nbytes).from_address(ptr), dtype=dtype)


def mapped_alloc(nbytes):
    """cudaHostAlloc(..., cudaHostAllocMapped); freed by the returned closer."""
    lib = _cudart()
    lib.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
    lib.cudaFreeHost.argtypes = [ctypes.c_void_p]
    p = ctypes.c_void_p()
    assert lib.cudaHostAlloc(ctypes.byref(p), nbytes, 2) == 0
    return p.value, (lambda: lib.cudaFreeHost(p))


def write_input(lane, frames):
    b = lane.buffers
    fb = np.ascontiguousarray(frames).reshape(-1)
    torch.cuda.synchronize()
    if b.input_host:
        host_array(b.input_host, fb.nbytes, np.uint8)[:] = fb
    else:
        memcpy(b.input_device, fb.ctypes.data, fb.nbytes)


def read_topk(lane, rows, k):
    b = lane.buffers
    if b.result_val_host:
        v = host_array(b.result_val_host, rows * k * 4, np.float32).reshape(rows, k).copy()
        i = host_array(b.result_idx_host, rows * k * 4, np.int32).reshape(rows, k).copy()
    else:
        v, i = np.empty((rows, k), np.float32), np.empty((rows, k), np.int32)
        memcpy(v.ctypes.data, b.result_val_device, v.nbytes)
        memcpy(i.ctypes.data, b.result_idx_device, i.nbytes)
    return v, i


def read_tensor(lane, n, dh, dw):
    t = np.empty((n, 3, dh, dw), np.float32)
    memcpy(t.ctypes.data, lane.buffers.tensor, t.nbytes)
    return t


@pytest.mark.parametrize("input_mode,result_mode", [(0, 0), (2, 2), (1, 1)])
def test_bucketed_topk_lane(B, oracle, input_mode, result_mode):
    """Batch 6 -> buckets 1, 2, 4, 6; long rows so each bucket has its own
    Top-K workspace; every n from 1 to 6 in a mixed order."""
    from post_processing_gb300 import Lane
    batch, cols, k = 6, 20000, 32
    pre = B.preprocess_desc(200, 120, 64, 48)
    d = B.lane_desc(pre, batch, batch, cols, k, input_mode=input_mode, result_mode=result_mode,
                    flags=B.WS_LANE_FLAG_BUCKETS | B.WS_LANE_FLAG_STAGE_TIMING)
    with Lane(d) as lane:
        for rep, n in enumerate([3, 1, 6, 5, 2, 4, 1, 6]):
            frames = synth.frames_uniform(100 + rep, batch, 120, 200)
            logits = synth.logits_with_ties(200 + rep, batch, cols)
            write_input(lane, frames)
            lg = np.ascontiguousarray(logits)
            memcpy(lane.buffers.logits, lg.ctypes.data, lg.nbytes)
            lane.acquire()
            lane.submit(n)
            t = lane.wait()
            assert t.preprocess_us > 0 and t.post_us > 0
            tensor = read_tensor(lane, n, 48, 64)
            assert np.max(np.abs(tensor - oracle.preprocess(frames[:n], 200, 120, 64, 48))) <= 1e-5
            v, i = read_topk(lane, batch, k)
            wv, wi = oracle.topk(logits[:n], k)
            assert np.array_equal(i[:n], wi) and np.array_equal(v[:n].view(np.uint32), wv.view(np.uint32)), n


def test_bucketed_detection_lane(B, oracle):
    from post_processing_gb300 import Lane
    from test_gpu_detect import gpu_decode, unpack
    desc = B.detect_desc()
    pre = B.preprocess_desc(1280, 720, 640, 640, letterbox=True, norm="scale")
    d = B.lane_desc(pre, 4, 0, 0, 0, detect=desc, flags=B.WS_LANE_FLAG_BUCKETS)
    with Lane(d) as lane:
        for n in (3, 1, 4):
            head = synth.yolo_head(300 + n, 4)
            hd = torch.from_numpy(head).cuda()
            memcpy(lane.buffers.logits, hd.data_ptr(), head.nbytes)
            lane.acquire()
            lane.submit(n)
            lane.wait()
            o = torch.empty((4, desc.max_det, 8), dtype=torch.int32, device="cuda")
            c = torch.empty(4, dtype=torch.int32, device="cuda")
            memcpy(o.data_ptr(), lane.buffers.detections_device, o.numel() * 4)
            memcpy(c.data_ptr(), lane.buffers.det_count_device, 16)
            o, c = o.cpu().numpy(), c.cpu().numpy()
            dec = gpu_decode(B, desc, head[:n])
            for b in range(n):
                keep = oracle.nms(dec[b]["boxes"], dec[b]["f4"], dec[b]["cls"], dec[b]["anchor"], desc.iou_thr,
                                  desc.max_det, desc.max_cand)
                assert list(unpack(o[b, :c[b]])["anchor"]) == [int(dec[b]["anchor"][j]) for j in keep]


@pytest.mark.parametrize("input_mode", [0, 1, 2], ids=["device", "mapped", "copy"])
def test_rebind_updates_graph_in_place(B, oracle, input_mode):
    """Two producer slots and two logits slots; the lane follows each rebind
    and its executable graph is updated, not re-instantiated."""
    from post_processing_gb300 import Lane
    batch, cols, k = 2, 1000, 5
    pre = B.preprocess_desc(160, 90, 64, 64)
    fb = 160 * 90 * 3 * batch
    frames = [synth.frames_uniform(10 + j, batch, 90, 160) for j in range(2)]
    logits = [synth.logits_normal(20 + j, batch, cols) for j in range(2)]
    lgs = [torch.from_numpy(x).cuda() for x in logits]
    closers = []
    if input_mode == 0:
        srcs = [torch.from_numpy(f).cuda() for f in frames]
        ptrs = [s.data_ptr() for s in srcs]
    elif input_mode == 1:
        ptrs = []
        for f in frames:
            p, close = mapped_alloc(fb)
            host_array(p, fb, np.uint8)[:] = f.reshape(-1)
            ptrs.append(p)
            closers.append(close)
    else:
        srcs = [torch.from_numpy(f.copy()).pin_memory() for f in frames]
        ptrs = [s.data_ptr() for s in srcs]
    d = B.lane_desc(pre, batch, batch, cols, k, input_mode=input_mode, flags=B.WS_LANE_FLAG_NVTX)
    try:
        with Lane(d) as lane:
            for j in (0, 1, 0, 1):
                assert lane.rebind(input=ptrs[j], logits=lgs[j].data_ptr()) is False   # updated in place
                lane.acquire()
                lane.submit()
                lane.wait()
                tensor = read_tensor(lane, batch, 64, 64)
                assert np.max(np.abs(tensor - oracle.preprocess(frames[j], 160, 90, 64, 64))) <= 1e-5
                v, i = read_topk(lane, batch, k)
                assert np.array_equal(i, oracle.topk(logits[j], k)[1])
            # a rebind while in flight is refused and changes nothing
            lane.acquire()
            lane.submit()
            assert B.ws_lane_rebind(lane.handle, ptrs[0], None)[0] == B.WS_ERR_LANE_BUSY
            lane.wait()
        # destroying the lane frees only what it allocated: the caller's slots
        # are intact and the library has no stale error
        assert np.array_equal(lgs[1].cpu().numpy(), logits[1])
        if input_mode == 0:
            assert np.array_equal(srcs[1].cpu().numpy(), frames[1])
        frame = torch.from_numpy(frames[0][:1].copy()).cuda()       # one 160x90 frame
        out = torch.empty((1, 3, 64, 64), dtype=torch.float32, device="cuda")
        B.check(B.ws_preprocess(pre, frame.data_ptr(), 1, out.data_ptr(), 0))
        torch.cuda.synchronize()
        assert np.max(np.abs(out.cpu().numpy() - oracle.preprocess(frames[0][:1], 160, 90, 64, 64))) <= 1e-5
    finally:
        torch.cuda.synchronize()
        for c in closers:
            c()


def test_pool_on_the_gpu(B, oracle):
    """Three lanes, 24 jobs with distinct frames and logits; each completed
    lane holds its own job's result."""
    batch, cols, k = 1, 1000, 5
    pre = B.preprocess_desc(320, 180, 96, 96)
    d = B.lane_desc(pre, batch, batch, cols, k, flags=B.WS_LANE_FLAG_NO_TIMING | B.WS_LANE_FLAG_NVTX)
    st, P = B.ws_pool_create(d, 3)
    B.check(st)
    try:
        pending = {}
        jobs = [(synth.frames_uniform(500 + j, 1, 180, 320), synth.logits_normal(600 + j, 1, cols)) for j in range(24)]
        done = 0
        j = 0
        while done < len(jobs):
            while j < len(jobs):
                st, L = B.ws_pool_acquire(P, 0)
                if st == B.WS_ERR_TIMEOUT:
                    break
                B.check(st)
                st, buf = B.ws_lane_get_buffers(L)
                B.check(st)
                fr, lg = jobs[j]
                memcpy(buf.input_device, fr.ctypes.data, fr.nbytes)
                memcpy(buf.logits, lg.ctypes.data, lg.nbytes)
                B.check(B.ws_pool_submit(P, L, 1))
                pending[L] = j
                j += 1
            st, L, _ = B.ws_pool_complete(P, -1)
            B.check(st)
            jj = pending.pop(L)
            st, buf = B.ws_lane_get_buffers(L)
            idx = np.empty((1, k), np.int32)
            memcpy(idx.ctypes.data, buf.result_idx_device, idx.nbytes)
            assert np.array_equal(idx, oracle.topk(jobs[jj][1], k)[1]), jj
            t = np.empty((1, 3, 96, 96), np.float32)
            memcpy(t.ctypes.data, buf.tensor, t.nbytes)
            assert np.max(np.abs(t - oracle.preprocess(jobs[jj][0], 320, 180, 96, 96))) <= 1e-5
            B.check(B.ws_pool_recycle(P, L))
            done += 1
    finally:
        assert B.ws_pool_destroy(P) == B.WS_OK


def test_pool_threads_on_the_gpu(B, oracle):
    """Two producer threads and one consumer thread share a pool of four lanes
    on the GPU: 40 jobs with distinct frames and logits, every completed lane
    holds its own job's result.  The lane-to-job record is written before the
    submit, so the consumer always finds it."""
    import threading
    batch, cols, k = 1, 100, 5
    pre = B.preprocess_desc(64, 48, 32, 32)
    d = B.lane_desc(pre, batch, batch, cols, k, flags=B.WS_LANE_FLAG_NO_TIMING)
    st, P = B.ws_pool_create(d, 4)
    B.check(st)
    jobs = [(synth.frames_uniform(700 + j, 1, 48, 64), synth.logits_with_ties(800 + j, 1, cols)) for j in range(40)]
    want = [(oracle.preprocess(fr, 64, 48, 32, 32), oracle.topk(lg, k)) for fr, lg in jobs]
    pending, lock, errors = {}, threading.Lock(), []

    def producer(js):
        try:
            for j in js:
                st, L = B.ws_pool_acquire(P, 5_000_000)
                B.check(st)
                st, buf = B.ws_lane_get_buffers(L)
                B.check(st)
                fr, lg = jobs[j]
                memcpy(buf.input_device, fr.ctypes.data, fr.nbytes)
                memcpy(buf.logits, lg.ctypes.data, lg.nbytes)
                with lock:
                    pending[L] = j
                B.check(B.ws_pool_submit(P, L, 1))
        except Exception as e:   # reported by the main thread
            errors.append(e)

    def consumer(n):
        try:
            for _ in range(n):
                st, L, _ = B.ws_pool_complete(P, 5_000_000)
                B.check(st)
                with lock:
                    j = pending.pop(L)
                st, buf = B.ws_lane_get_buffers(L)
                B.check(st)
                t = np.empty((1, 3, 32, 32), np.float32)
                memcpy(t.ctypes.data, buf.tensor, t.nbytes)
                v = np.empty((1, k), np.float32)
                idx = np.empty((1, k), np.int32)
                memcpy(v.ctypes.data, buf.result_val_device, v.nbytes)
                memcpy(idx.ctypes.data, buf.result_idx_device, idx.nbytes)
                assert np.max(np.abs(t - want[j][0])) <= 1e-5, j
                assert np.array_equal(idx, want[j][1][1]), j
                assert np.array_equal(v.view(np.uint32), want[j][1][0].view(np.uint32)), j
                B.check(B.ws_pool_recycle(P, L))
        except Exception as e:
            errors.append(e)

    try:
        threads = [threading.Thread(target=producer, args=(range(0, 40, 2),)),
                   threading.Thread(target=producer, args=(range(1, 40, 2),)),
                   threading.Thread(target=consumer, args=(40,))]
        for t in threads:
            t.start()
        for t in threads:
            t.join(timeout=120)
        assert not any(t.is_alive() for t in threads), "a pool thread did not finish"
        assert not errors, errors
        assert not pending
    finally:
        assert B.ws_pool_destroy(P) == B.WS_OK
