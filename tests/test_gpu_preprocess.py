"""GPU preprocess against the oracle: every element within 1e-5 absolute.

Inputs are the seeded synthetic workloads (the five inference
configurations at full size) and small odd shapes that span several blocks
and ragged tails: widths that are not multiples of 4 or 16, padded row and
frame strides, misaligned base pointers and strides that are not multiples
of 16 (the staged kernel copies each row's 16-byte window), upscales,
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


@pytest.fixture(autouse=True)
def no_index_out_of_range(B):
    """Under the checked build (WS_BOUNDS_CHECK=1 loads libws_bounds.so)
    every test must leave the device error word without the bounds bit: no
    index into a stage slot or the column-tap table, and no source tap, was
    out of range."""
    yield
    if B.ws_build_features() & B.WS_FEATURE_BOUNDS_CHECK:
        torch.cuda.synchronize()
        st, flags = B.ws_device_error(True)
        assert st == B.WS_OK and flags & 0x4 == 0, f"a bounds check failed (device error bits {flags:#x})"


def run_gpu(B, frames, sw, sh, dw, dh, *, letterbox=False, norm="mean_std", row_stride=None,
            frame_stride=None, offset=0, pad_value=114, path=0):
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
    B.check(B.ws_preprocess_path(d, dev.data_ptr() + offset, batch, out.data_ptr(), path,
                                 torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return out.cpu().numpy()


PATHS = [0, 1, 2]   # WS_PRE_PATH_AUTO, _STAGED (the bulk-copy ring), _DIRECT


def compare(got, want):
    assert got.shape == want.shape
    assert not np.isnan(got).any(), "unwritten output elements"
    err = float(np.max(np.abs(got.astype(np.float64) - want.astype(np.float64))))
    assert err <= TOL, f"max abs error {err}"
    return err


@pytest.mark.parametrize("path", PATHS, ids=["auto", "staged", "direct"])
@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_parity(B, oracle, name, path):
    w = synth.WORKLOADS[name]
    frames = synth.make_frames(name)
    lb = w["resize"] == "letterbox"
    got = run_gpu(B, frames, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], letterbox=lb, norm=w["norm"],
                  path=path)
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
    (200, 120, 64, 48, False, "mean_std", 16, 32, 0, 3),     # padded, aligned strides
    (200, 120, 64, 48, False, "mean_std", 5, 7, 0, 3),       # unaligned row and frame strides
    (200, 120, 64, 48, False, "mean_std", 0, 0, 3, 2),       # misaligned base
    (1920, 1080, 224, 224, False, "mean_std", 0, 0, 1, 1),   # config shape, misaligned base
    (1920, 1080, 224, 224, False, "mean_std", 1, 0, 3, 3),   # config shape, stride 5761, base + 3
    (1366, 768, 224, 224, False, "mean_std", 0, 0, 0, 3),    # 4098-byte rows: every row start differs mod 16
    (1280, 720, 640, 640, True, "scale", 7, 5, 9, 2),        # letterbox, everything unaligned
    (4000, 3, 512, 7, False, "mean_std", 0, 0, 0, 1),        # 12000-byte rows, 2 rows
    (21, 700, 8, 300, False, "scale", 0, 0, 0, 2),            # 63-byte rows: 64-byte windows
    (2, 50000, 3, 60000, False, "scale", 10, 0, 0, 1),       # tall: 64-bit y taps, 6-byte rows
    (40000, 2, 30000, 1, False, "mean_std", 0, 0, 0, 1),     # wide: per-pixel kernel, 64-bit x taps
    (20000, 6, 4000, 5, False, "mean_std", 0, 0, 0, 2),      # 60 KB rows: a one-stage ring
    (20000, 6, 4000, 5, False, "scale", 7, 3, 5, 2),         # the same, nothing aligned
    (40000, 4, 1000, 3, False, "mean_std", 0, 0, 0, 1),      # 120 KB rows: no ring fits, per-pixel kernel
]


@pytest.mark.parametrize("path", [1, 2], ids=["staged", "direct"])
@pytest.mark.parametrize("case", ODD, ids=[f"{c[0]}x{c[1]}-{c[2]}x{c[3]}-lb{int(c[4])}-o{c[8]}" for c in ODD])
def test_odd_shapes(B, oracle, case, path):
    sw, sh, dw, dh, lb, norm, er, ef, off, batch = case
    rs = 3 * sw + er
    fs = rs * sh + ef
    frames = synth.frames_uniform(sw * 7 + sh, batch, sh, sw, row_stride=rs)
    got = run_gpu(B, frames, sw, sh, dw, dh, letterbox=lb, norm=norm, row_stride=rs, frame_stride=fs,
                  offset=off, path=path)
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


# ---- precision- and format-specialised outputs ------------------------------

def run_gpu_typed(B, frames, sw, sh, dw, dh, dst_type, channel_order=0, letterbox=False, norm="mean_std",
                  offset=0, path=1):
    batch = frames.shape[0]
    flat = np.zeros(offset + frames.size + 64, np.uint8)
    flat[offset:offset + frames.size] = frames.reshape(-1)
    dev = torch.from_numpy(flat).cuda()
    tdt = {B.WS_DTYPE_F32: torch.float32, B.WS_DTYPE_F16: torch.float16, B.WS_DTYPE_BF16: torch.bfloat16}[dst_type]
    out = torch.full((batch, 3, dh, dw), float("nan"), dtype=tdt, device="cuda")
    d = B.preprocess_desc(sw, sh, dw, dh, letterbox=letterbox, norm=norm, channel_order=channel_order,
                          dst_type=dst_type)
    B.check(B.ws_preprocess_path(d, dev.data_ptr() + offset, batch, out.data_ptr(), path,
                                 torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return out.cpu()


def rounded(oracle_f32, dst_type, B):
    """The FP32 oracle rounded to the output format (torch: round to nearest even)."""
    tdt = {B.WS_DTYPE_F16: torch.float16, B.WS_DTYPE_BF16: torch.bfloat16}[dst_type]
    return torch.from_numpy(oracle_f32).to(tdt)


def ulp_of(x, dst_type, B):
    """Spacing of the format at |x| (one unit in the last place)."""
    mant = 10 if dst_type == B.WS_DTYPE_F16 else 7
    # exact binade from the float's exponent (a float log2 of 2.0 may land
    # just below 1); clamped to the smallest normal exponent of the format
    _, e = torch.frexp(x.float())
    e = torch.clamp(e.float() - 1, min=-14.0 if dst_type == B.WS_DTYPE_F16 else -126.0)
    return torch.pow(2.0, e - mant)


SHAPES_TYPED = [("b64_1080p_to_224", 8), ("b1_720p_letterbox_640", 1), ("b8_4k_to_512", 2), (None, 2)]


@pytest.mark.parametrize("path", [1, 2], ids=["staged", "direct"])
@pytest.mark.parametrize("dst", ["f16", "bf16"])
@pytest.mark.parametrize("name,batch", SHAPES_TYPED, ids=[str(s[0]) for s in SHAPES_TYPED])
def test_half_outputs(B, oracle, dst, name, batch, path):
    """Half outputs equal the FP32 oracle rounded to the format, except where
    the two FP32 values (within 1e-5 of each other) straddle a rounding
    boundary: there an element may differ by one unit in the last place, plus
    the FP32 difference itself."""
    dst_type = B.WS_DTYPE_F16 if dst == "f16" else B.WS_DTYPE_BF16
    if name is None:   # ragged shape, per-pixel kernel (misaligned base)
        sw, sh, dw, dh, lb, norm, off = 101, 67, 37, 29, False, "mean_std", 3
        frames = synth.frames_uniform(5, batch, sh, sw)
    else:
        w = synth.WORKLOADS[name]
        sw, sh, dw, dh, lb, norm, off = (w["src_w"], w["src_h"], w["dst_w"], w["dst_h"],
                                          w["resize"] == "letterbox", w["norm"], 0)
        frames = synth.make_frames(name, batch=batch)
    got = run_gpu_typed(B, frames, sw, sh, dw, dh, dst_type, letterbox=lb, norm=norm, offset=off, path=path)
    want32 = oracle.preprocess(frames, sw, sh, dw, dh, letterbox=lb, norm=norm)
    want = rounded(want32, dst_type, B)
    diff = (got.float() - want.float()).abs()
    assert not torch.isnan(got.float()).any()
    # |round(a) - round(b)| <= |a - b| + one ulp, and |a - b| <= 1e-5 for the
    # FP32 values (near zero that 1e-5 spans several half ulps)
    assert torch.all(diff <= ulp_of(want, dst_type, B) + TOL), float(diff.max())
    assert float((diff > 0).float().mean()) < 1e-3          # boundary cases only
    # and the value is the FP32 result within the format's rounding (one ulp
    # covers a rounding that lands on the next binade)
    assert torch.all((got.float() - torch.from_numpy(want32)).abs() <= ulp_of(want, dst_type, B) + 1e-5)


@pytest.mark.parametrize("name", ["b1_1080p_to_224", "b1_720p_letterbox_640"])
def test_bgr_source(B, oracle, name):
    """A BGR frame gives exactly the planes of the same picture stored as RGB."""
    w = synth.WORKLOADS[name]
    rgb = synth.make_frames(name)
    bgr = rgb.reshape(rgb.shape[0], w["src_h"], w["src_w"], 3)[..., ::-1].copy().reshape(rgb.shape)
    lb = w["resize"] == "letterbox"
    got = run_gpu_typed(B, bgr, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], B.WS_DTYPE_F32,
                        channel_order=B.WS_ORDER_BGR, letterbox=lb, norm=w["norm"]).numpy()
    want = oracle.preprocess(rgb, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], letterbox=lb, norm=w["norm"])
    compare(got, want)
    # the per-pixel kernel too (misaligned base)
    got2 = run_gpu_typed(B, bgr, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], B.WS_DTYPE_F32,
                         channel_order=B.WS_ORDER_BGR, letterbox=lb, norm=w["norm"], offset=1).numpy()
    compare(got2, want)
