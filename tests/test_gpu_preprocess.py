"""GPU preprocess against the oracle: every element within 1e-5 absolute.

Inputs are the seeded synthetic workloads (the five inference
configurations at full size) and small odd shapes that span several blocks
and ragged tails: widths that are not multiples of 4 or 16, padded row and
frame strides, misaligned base pointers (per-pixel kernel), upscales,
letterbox in both orientations, 1x1 frames.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu
TOL = 1e-5


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def run_gpu(B, frames, sw, sh, dw, dh, *, letterbox=False, norm="mean_std", row_stride=None,
            frame_stride=None, offset=0, pad_value=114):
    """frames: uint8 [B, H, stride] laid out with the given strides."""
    batch = frames.shape[0]
    rs = 3 * sw if row_stride is None else row_stride
    fs = rs * sh if frame_stride is None else frame_stride
    flat = np.zeros(offset + batch * fs + 64, np.uint8)
    for b in range(batch):
        for j in range(sh):
            flat[offset + b * fs + j * rs: offset + b * fs + j * rs + 3 * sw] = frames[b, j, :3 * sw]
    dev = torch.from_numpy(flat).cuda()
    out = torch.full((batch, 3, dh, dw), float("nan"), dtype=torch.float32, device="cuda")
    d = B.preprocess_desc(sw, sh, dw, dh, letterbox=letterbox, norm=norm, row_stride=rs,
                          frame_stride=fs, pad_value=pad_value)
    B.check(B.ws_preprocess(d, dev.data_ptr() + offset, batch, out.data_ptr(),
                            torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return out.cpu().numpy()


def compare(got, want):
    assert got.shape == want.shape
    assert not np.isnan(got).any(), "unwritten output elements"
    err = float(np.max(np.abs(got.astype(np.float64) - want.astype(np.float64))))
    assert err <= TOL, f"max abs error {err}"
    return err


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_parity(B, oracle, name):
    w = synth.WORKLOADS[name]
    frames = synth.make_frames(name)
    lb = w["resize"] == "letterbox"
    got = run_gpu(B, frames, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], letterbox=lb, norm=w["norm"])
    want = oracle.preprocess(frames, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], letterbox=lb,
                             norm=w["norm"])
    compare(got, want)


ODD = [
    # sw, sh, dw, dh, letterbox, norm, extra row bytes, extra frame bytes, base offset, batch
    (1, 1, 1, 1, False, "mean_std", 0, 0, 0, 1),
    (1, 1, 7, 5, False, "scale", 0, 0, 0, 2),
    (3, 5, 3, 5, False, "mean_std", 0, 0, 0, 3),
    (5, 3, 11, 2, False, "mean_std", 0, 0, 0, 2),
    (37, 29, 80, 61, False, "mean_std", 0, 0, 0, 2),        # upscale, 3*37 = 111 bytes per row
    (640, 1, 7, 3, False, "scale", 0, 0, 0, 1),
    (100, 60, 33, 17, False, "mean_std", 0, 0, 0, 4),       # dst width not a multiple of 4
    (96, 64, 64, 64, True, "scale", 0, 0, 0, 2),             # letterbox, rows padded
    (64, 96, 67, 64, True, "mean_std", 0, 0, 0, 2),          # letterbox, columns padded, odd split
    (1000, 999, 640, 640, True, "scale", 0, 0, 0, 1),
    (200, 120, 64, 48, False, "mean_std", 16, 32, 0, 3),     # padded, aligned strides (staged)
    (200, 120, 64, 48, False, "mean_std", 5, 7, 0, 3),       # unaligned strides (per-pixel)
    (200, 120, 64, 48, False, "mean_std", 0, 0, 3, 2),       # misaligned base (per-pixel)
    (1920, 1080, 224, 224, False, "mean_std", 0, 0, 1, 1),   # config shape, misaligned base
    (4000, 3, 512, 7, False, "mean_std", 0, 0, 0, 1),        # 12000-byte rows, 2 rows
    (21, 700, 8, 300, False, "scale", 0, 0, 0, 2),            # 63-byte rows: bulk part 48 + tail 15
    (2, 50000, 3, 60000, False, "scale", 10, 0, 0, 1),       # tall: 64-bit y taps, tail-only rows
    (40000, 2, 30000, 1, False, "mean_std", 0, 0, 0, 1),     # wide: per-pixel kernel, 64-bit x taps
]


@pytest.mark.parametrize("case", ODD, ids=[f"{c[0]}x{c[1]}-{c[2]}x{c[3]}-lb{int(c[4])}-o{c[8]}" for c in ODD])
def test_odd_shapes(B, oracle, case):
    sw, sh, dw, dh, lb, norm, er, ef, off, batch = case
    rs = 3 * sw + er
    fs = rs * sh + ef
    frames = synth.frames_uniform(sw * 7 + sh, batch, sh, sw, row_stride=rs)
    got = run_gpu(B, frames, sw, sh, dw, dh, letterbox=lb, norm=norm, row_stride=rs, frame_stride=fs,
                  offset=off)
    buf = np.zeros((batch, fs), np.uint8)
    buf[:, :rs * sh] = frames.reshape(batch, -1)
    want = oracle.preprocess(buf, sw, sh, dw, dh, letterbox=lb, norm=norm, row_stride=rs, frame_stride=fs)
    compare(got, want)


def test_extreme_bytes_and_pad_values(B, oracle):
    for val in (0, 255):
        frames = np.full((2, 50, 3 * 70), val, np.uint8)
        for pad in (0, 114, 255):
            got = run_gpu(B, frames, 70, 50, 64, 64, letterbox=True, pad_value=pad)
            want = oracle.preprocess(frames, 70, 50, 64, 64, letterbox=True, pad_value=pad)
            compare(got, want)


def test_repeat_calls_are_identical(B):
    frames = synth.make_frames("b1_1080p_to_224")
    a = run_gpu(B, frames, 1920, 1080, 224, 224)
    b = run_gpu(B, frames, 1920, 1080, 224, 224)
    assert np.array_equal(a, b)


def test_no_device_error_raised(B):
    st, flags = B.ws_device_error(False)
    assert st == B.WS_OK and flags == 0
