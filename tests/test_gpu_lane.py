"""Lanes on the GPU: graph replay equals direct launches equals the oracle,
in every input and result mode; per-stage timing; wait with a deadline;
state machine with real work in flight; new inputs in the same buffers."""
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
    buf = (ctypes.c_char * nbytes).from_address(ptr)
    return np.frombuffer(buf, dtype=dtype)


def fill_lane(B, lane, frames, logits):
    """Write frames and logits into the lane's producer / network slots."""
    b = lane.buffers
    fb = frames.reshape(-1)
    torch.cuda.synchronize()
    if b.input_host:
        host_array(b.input_host, fb.nbytes, np.uint8)[:] = fb
    else:
        memcpy(b.input_device, fb.ctypes.data, fb.nbytes)
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    memcpy(b.logits, lg.ctypes.data, lg.nbytes)


def read_lane(B, lane, batch, dh, dw, rows, k):
    b = lane.buffers
    t = np.empty((batch, 3, dh, dw), dtype=np.float32)
    memcpy(t.ctypes.data, b.tensor, t.nbytes)
    if b.result_val_host:
        v = host_array(b.result_val_host, rows * k * 4, np.float32).reshape(rows, k).copy()
        i = host_array(b.result_idx_host, rows * k * 4, np.int32).reshape(rows, k).copy()
    else:
        v = np.empty((rows, k), np.float32)
        i = np.empty((rows, k), np.int32)
        memcpy(v.ctypes.data, b.result_val_device, v.nbytes)
        memcpy(i.ctypes.data, b.result_idx_device, i.nbytes)
    return t, v, i


MODES = [(0, 0, 0), (0, 0, 1), (1, 1, 0), (2, 2, 0), (2, 1, 2), (1, 2, 1), (0, 2, 64)]   # input, result, flags


@pytest.mark.parametrize("name", ["b1_1080p_to_224", "b1_720p_letterbox_640", "b8_4k_to_512"])
@pytest.mark.parametrize("mode", MODES, ids=[f"in{m[0]}-res{m[1]}-f{m[2]}" for m in MODES])
def test_lane_parity(B, oracle, name, mode):
    from post_processing_gb300 import Lane
    w = synth.WORKLOADS[name]
    frames = synth.make_frames(name)
    logits = synth.make_logits(name)
    pre = B.preprocess_desc(w["src_w"], w["src_h"], w["dst_w"], w["dst_h"],
                            letterbox=w["resize"] == "letterbox", norm=w["norm"])
    d = B.lane_desc(pre, w["batch"], w["rows"], w["cols"], w["k"], input_mode=mode[0], result_mode=mode[1],
                    flags=mode[2] | B.WS_LANE_FLAG_STAGE_TIMING)
    with Lane(d) as lane:
        fill_lane(B, lane, frames, logits)
        for _ in range(2):                         # replaying twice gives the same answer
            lane.acquire()
            lane.submit()
            t = lane.wait()
            assert t.gpu_us > 0 and t.preprocess_us > 0 and t.post_us > 0 and t.host_us > 0
            tensor, v, i = read_lane(B, lane, w["batch"], w["dst_h"], w["dst_w"], w["rows"], w["k"])
            want = oracle.preprocess(frames, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"],
                                     letterbox=w["resize"] == "letterbox", norm=w["norm"])
            assert np.max(np.abs(tensor - want)) <= 1e-5
            wv, wi = oracle.topk(logits, w["k"])
            assert np.array_equal(i, wi) and np.array_equal(v.view(np.uint32), wv.view(np.uint32))


def test_new_inputs_in_fixed_buffers(B, oracle):
    from post_processing_gb300 import Lane
    pre = B.preprocess_desc(320, 200, 96, 64)
    d = B.lane_desc(pre, 3, 3, 20000, 32)
    with Lane(d) as lane:
        for seed in range(3):
            frames = synth.frames_uniform(seed, 3, 200, 320)
            logits = synth.logits_with_ties(seed, 3, 20000)
            fill_lane(B, lane, frames, logits)
            lane.acquire()
            lane.submit()
            lane.wait()
            tensor, v, i = read_lane(B, lane, 3, 64, 96, 3, 32)
            assert np.max(np.abs(tensor - oracle.preprocess(frames, 320, 200, 96, 64))) <= 1e-5
            wv, wi = oracle.topk(logits, 32)
            assert np.array_equal(i, wi) and np.array_equal(v.view(np.uint32), wv.view(np.uint32))


def test_wait_deadline_and_state(B):
    """A lane whose stream is held busy times out, stays in flight, then completes."""
    from post_processing_gb300 import Lane
    s = torch.cuda.Stream()
    pre = B.preprocess_desc(64, 48, 32, 32)
    d = B.lane_desc(pre, 1, 1, 100, 5, stream=s.cuda_stream)
    with Lane(d) as lane:
        with torch.cuda.stream(s):
            torch.cuda._sleep(200_000_000)         # ~0.1 s of GPU clock cycles, then done
        lane.acquire()
        lane.submit()
        st, _ = B.ws_lane_wait(lane.handle, 0)
        assert st == B.WS_ERR_TIMEOUT and lane.state == B.WS_LANE_IN_FLIGHT
        assert B.ws_lane_acquire(lane.handle) == B.WS_ERR_LANE_BUSY
        assert B.ws_lane_destroy(lane.handle) == B.WS_ERR_LANE_BUSY
        t = lane.wait(10_000_000)
        assert lane.state == B.WS_LANE_FREE and t.gpu_us > 0


def test_borrowed_buffers(B, oracle):
    from post_processing_gb300 import Lane
    frames = synth.frames_uniform(3, 2, 90, 160)
    logits = synth.logits_normal(4, 2, 1000)
    src = torch.from_numpy(frames).cuda()
    tensor = torch.empty((2, 3, 64, 64), dtype=torch.float32, device="cuda")
    lg = torch.from_numpy(logits).cuda()
    val = torch.empty((2, 5), dtype=torch.float32, device="cuda")
    idx = torch.empty((2, 5), dtype=torch.int32, device="cuda")
    pre = B.preprocess_desc(160, 90, 64, 64, letterbox=True, norm="scale")
    d = B.lane_desc(pre, 2, 2, 1000, 5, input=src.data_ptr(), tensor=tensor.data_ptr(),
                    logits=lg.data_ptr(), result_val=val.data_ptr(), result_idx=idx.data_ptr())
    with Lane(d) as lane:
        assert lane.buffers.tensor == tensor.data_ptr()
        lane.acquire()
        lane.submit()
        lane.wait()
        want = oracle.preprocess(frames, 160, 90, 64, 64, letterbox=True, norm="scale")
        assert np.max(np.abs(tensor.cpu().numpy() - want)) <= 1e-5
        wv, wi = oracle.topk(logits, 5)
        assert np.array_equal(idx.cpu().numpy(), wi)


def test_bench_throughput_configuration(B, oracle):
    """The benchmark's throughput setup: three 64-frame 1080p lanes without
    timing events sharing one stream, replayed in rotation; every replay's
    tensor and Top-K equal the oracle's."""
    from post_processing_gb300 import Lane
    name = "b64_1080p_to_224"
    w = synth.WORKLOADS[name]
    frames = synth.make_frames(name)
    logits = synth.make_logits(name)
    want_t = oracle.preprocess(frames, 1920, 1080, 224, 224)
    want_v, want_i = oracle.topk(logits, 32)
    s = torch.cuda.Stream()
    pre = B.preprocess_desc(1920, 1080, 224, 224)
    lanes = [Lane(B.lane_desc(pre, 64, 64, 1000, 32, stream=s.cuda_stream, flags=B.WS_LANE_FLAG_NO_TIMING))
             for _ in range(3)]
    try:
        for ln in lanes:
            fill_lane(B, ln, frames, logits)
        for step in range(9):
            ln = lanes[step % 3]
            if ln.state == B.WS_LANE_IN_FLIGHT:
                ln.wait()
            ln.acquire()
            ln.submit()
        for ln in lanes:
            if ln.state == B.WS_LANE_IN_FLIGHT:
                t = ln.wait()
                assert t.gpu_us == -1.0
            tensor, v, i = read_lane(B, ln, 64, 224, 224, 64, 32)
            assert np.max(np.abs(tensor - want_t)) <= 1e-5
            assert np.array_equal(i, want_i) and np.array_equal(v.view(np.uint32), want_v.view(np.uint32))
    finally:
        for ln in lanes:
            ln.close()


def test_bf16_bgr_lane(B, oracle):
    """A lane with a BGR producer and a bfloat16 network input."""
    from post_processing_gb300 import Lane
    rgb = synth.frames_uniform(12, 4, 240, 320)
    bgr = rgb.reshape(4, 240, 320, 3)[..., ::-1].copy().reshape(rgb.shape)
    logits = synth.logits_normal(13, 4, 1000)
    pre = B.preprocess_desc(320, 240, 128, 96, channel_order=B.WS_ORDER_BGR, dst_type=B.WS_DTYPE_BF16)
    with Lane(B.lane_desc(pre, 4, 4, 1000, 5)) as lane:
        assert lane.buffers.tensor_bytes == 4 * 3 * 96 * 128 * 2
        fill_lane(B, lane, bgr, logits)
        lane.acquire()
        lane.submit()
        lane.wait()
        raw = np.empty(4 * 3 * 96 * 128, np.uint16)
        memcpy(raw.ctypes.data, lane.buffers.tensor, raw.nbytes)
        got = torch.from_numpy(raw.view(np.int16)).view(torch.bfloat16).float().reshape(4, 3, 96, 128)
        want = torch.from_numpy(oracle.preprocess(rgb, 320, 240, 128, 96)).to(torch.bfloat16).float()
        assert float((got - want).abs().max()) <= 2.0 ** -6 * 4    # at most one bf16 ulp at |x| < 4


def staged_kernel_taken(B, w, batch):
    """ws_preprocess takes the staged bulk-copy kernel above 460,000 output
    pixels (destinations up to 8192 wide)."""
    return batch * w["dst_w"] * w["dst_h"] > 460_000 and w["dst_w"] <= 8192


@pytest.mark.parametrize("name,batch", [("b64_1080p_to_224", 10), ("b64_1080p_to_224", 64), ("b8_4k_to_512", 2),
                                        ("b8_4k_to_512", 8)])
def test_mapped_input_staged_kernel(B, oracle, name, batch):
    """Mapped pinned input read in place by the staged kernel: its bulk copies
    pull the needed source rows straight from host memory across the host
    link (the end-to-end path: "Inside WarpStream TRT", mapped pinned memory).
    The tensor is within 1e-5 of the oracle and the Top-K bit-exact, for two
    replays."""
    from post_processing_gb300 import Lane
    w = synth.WORKLOADS[name]
    assert staged_kernel_taken(B, w, batch)
    frames = synth.make_frames(name, batch=batch)
    rows = w["rows"] * batch // w["batch"] if w["rows"] >= w["batch"] else w["rows"]
    logits = synth.make_logits(name, rows=rows)
    pre = B.preprocess_desc(w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], norm=w["norm"])
    d = B.lane_desc(pre, batch, rows, w["cols"], w["k"], input_mode=B.WS_INPUT_MAPPED,
                    result_mode=B.WS_RESULT_MAPPED)
    with Lane(d) as lane:
        fill_lane(B, lane, frames, logits)
        want = oracle.preprocess(frames, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], norm=w["norm"])
        wv, wi = oracle.topk(logits, w["k"])
        for _ in range(2):
            lane.acquire()
            lane.submit()
            lane.wait()
            tensor, v, i = read_lane(B, lane, batch, w["dst_h"], w["dst_w"], rows, w["k"])
            assert np.max(np.abs(tensor - want)) <= 1e-5
            assert np.array_equal(i, wi) and np.array_equal(v.view(np.uint32), wv.view(np.uint32))


def test_mapped_input_unaligned_borrowed(B, oracle):
    """A borrowed mapped slot whose base, row stride and frame stride are not
    multiples of 16 (a producer's own pinned buffer need not be aligned): the
    staged kernel copies each row's 16-byte window from host memory."""
    from post_processing_gb300 import Lane
    batch, sw, sh, dw, dh = 10, 1920, 1080, 224, 224
    stride, fstride, base_off = 3 * sw + 1, (3 * sw + 1) * sh + 3, 5
    frames = synth.frames_uniform(0x5EED, batch, sh, sw)
    logits = synth.logits_normal(0x5EEE, batch, 1000)
    lib = _cudart()
    lib.cudaHostAlloc.argtypes = [ctypes.POINTER(ctypes.c_void_p), ctypes.c_size_t, ctypes.c_uint]
    lib.cudaFreeHost.argtypes = [ctypes.c_void_p]
    nbytes = base_off + batch * fstride
    ptr = ctypes.c_void_p()
    assert lib.cudaHostAlloc(ctypes.byref(ptr), nbytes, 2) == 0      # cudaHostAllocMapped
    try:
        host = np.frombuffer((ctypes.c_char * nbytes).from_address(ptr.value), dtype=np.uint8)
        host[:] = 0x5A
        fr = frames.reshape(batch, sh, 3 * sw)
        for b in range(batch):
            rows = host[base_off + b * fstride: base_off + b * fstride + sh * stride].reshape(sh, stride)
            rows[:, :3 * sw] = fr[b]
        pre = B.preprocess_desc(sw, sh, dw, dh, row_stride=stride, frame_stride=fstride)
        d = B.lane_desc(pre, batch, batch, 1000, 32, input_mode=B.WS_INPUT_MAPPED, input=ptr.value + base_off)
        with Lane(d) as lane:
            lg = np.ascontiguousarray(logits)
            memcpy(lane.buffers.logits, lg.ctypes.data, lg.nbytes)
            lane.acquire()
            lane.submit()
            lane.wait()
            tensor, v, i = read_lane(B, lane, batch, dh, dw, batch, 32)
            assert np.max(np.abs(tensor - oracle.preprocess(frames, sw, sh, dw, dh))) <= 1e-5
            wv, wi = oracle.topk(logits, 32)
            assert np.array_equal(i, wi) and np.array_equal(v.view(np.uint32), wv.view(np.uint32))
    finally:
        lib.cudaFreeHost(ptr)


@pytest.mark.parametrize("name", ["b64_1080p_to_224", "b8_4k_to_512"])
def test_bench_throughput_lanes_on_own_streams(B, oracle, name):
    """The benchmark's headline configuration: four lanes without timing
    events, each on its own stream, replayed in rotation so that one lane's
    preprocess overlaps the previous lane's Top-K.  Each lane holds different
    frames and logits; after three rotations every lane's tensor and Top-K
    equal the oracle's for its own inputs."""
    from post_processing_gb300 import Lane
    w = synth.WORKLOADS[name]
    pre = B.preprocess_desc(w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], norm=w["norm"])
    lanes, wants = [], []
    try:
        for j in range(4):
            frames = synth.frames_uniform(0x4A00 + j, w["batch"], w["src_h"], w["src_w"])
            logits = synth.logits_with_ties(0x4B00 + j, w["rows"], w["cols"])
            ln = Lane(B.lane_desc(pre, w["batch"], w["rows"], w["cols"], w["k"], flags=B.WS_LANE_FLAG_NO_TIMING))
            lanes.append(ln)
            fill_lane(B, ln, frames, logits)
            wants.append((oracle.preprocess(frames, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], norm=w["norm"]),
                          oracle.topk(logits, w["k"])))
        streams = {ln.buffers.stream for ln in lanes}
        assert len(streams) == 4
        for step in range(12):
            ln = lanes[step % 4]
            if ln.state == B.WS_LANE_IN_FLIGHT:
                ln.wait()
            ln.acquire()
            ln.submit()
        for ln, (want_t, (want_v, want_i)) in zip(lanes, wants):
            if ln.state == B.WS_LANE_IN_FLIGHT:
                ln.wait()
            tensor, v, i = read_lane(B, ln, w["batch"], w["dst_h"], w["dst_w"], w["rows"], w["k"])
            assert np.max(np.abs(tensor - want_t)) <= 1e-5
            assert np.array_equal(i, want_i) and np.array_equal(v.view(np.uint32), want_v.view(np.uint32))
    finally:
        for ln in lanes:
            ln.close()
