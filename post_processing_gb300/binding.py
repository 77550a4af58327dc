"""ctypes binding of ``include/ws.h`` (argument marshalling only).

Every function of the header is exposed under its own name and returns the
raw ``ws_status``; ``check()`` turns a non-zero status into ``WsError`` with
the library's message.  All computation happens in ``libws.so`` on the GPU:
this module never computes a result itself, and importing it fails loudly
when the library has not been built.

Pointers are plain integers (``tensor.data_ptr()``, ``stream.cuda_stream``),
so PyTorch only supplies device memory, pinned host memory and streams.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

WS_OK = 0
WS_ERR_INVALID_ARGUMENT = 1
WS_ERR_UNSUPPORTED = 2
WS_ERR_CUDA = 3
WS_ERR_OUT_OF_MEMORY = 4
WS_ERR_LANE_STATE = 5
WS_ERR_LANE_BUSY = 6
WS_ERR_TIMEOUT = 7
WS_ERR_CAPTURE = 8
WS_ERR_DEVICE = 9

WS_RESIZE_STRETCH, WS_RESIZE_LETTERBOX = 0, 1
WS_NORM_MEAN_STD, WS_NORM_SCALE = 0, 1
WS_ORDER_RGB, WS_ORDER_BGR = 0, 1
WS_DTYPE_F32, WS_DTYPE_F16, WS_DTYPE_BF16 = 0, 1, 2
WS_PRE_PATH_AUTO, WS_PRE_PATH_STAGED, WS_PRE_PATH_DIRECT = 0, 1, 2
WS_INPUT_DEVICE, WS_INPUT_MAPPED, WS_INPUT_COPY = 0, 1, 2
WS_RESULT_DEVICE, WS_RESULT_MAPPED, WS_RESULT_COPY = 0, 1, 2
WS_LANE_FLAG_NO_GRAPH = 1
WS_LANE_FLAG_STAGE_TIMING = 2
WS_LANE_FLAG_NO_TIMING = 4
WS_LANE_FLAG_NO_DEVICE = 8
WS_LANE_FLAG_NVTX = 16
WS_LANE_FLAG_BUCKETS = 32
WS_LANE_FLAG_NO_PDL = 64
WS_POST_TOPK, WS_POST_DETECT = 0, 1
WS_LANE_FREE, WS_LANE_ACQUIRED, WS_LANE_IN_FLIGHT = 0, 1, 2

_i32, _i64, _u32, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32, ctypes.c_float
_vp, _sz = ctypes.c_void_p, ctypes.c_size_t


class ws_preprocess_desc(ctypes.Structure):
    _fields_ = [("src_w", _i32), ("src_h", _i32), ("src_row_stride", _i64), ("src_frame_stride", _i64),
                ("dst_w", _i32), ("dst_h", _i32), ("resize", _i32), ("pad_value", _i32), ("norm", _i32),
                ("mean", _f32 * 3), ("std", _f32 * 3), ("scale", _f32), ("channel_order", _i32),
                ("dst_type", _i32)]


class ws_detect_desc(ctypes.Structure):
    _fields_ = [("in_w", _i32), ("in_h", _i32), ("nlevels", _i32), ("strides", _i32 * 4), ("reg_max", _i32),
                ("num_classes", _i32), ("logit_thr", _f32), ("iou_thr", _f32), ("max_cand", _i32),
                ("max_det", _i32)]


class ws_lane_desc(ctypes.Structure):
    _fields_ = [("pre", ws_preprocess_desc), ("batch", _i32), ("rows", _i64), ("cols", _i64), ("k", _i32),
                ("input_mode", _i32), ("result_mode", _i32), ("flags", _u32), ("input", _vp),
                ("tensor", _vp), ("logits", _vp), ("result_val", _vp), ("result_idx", _vp),
                ("stream", _vp), ("fake_polls", _i32), ("post", _i32), ("detect", ws_detect_desc),
                ("detections", _vp), ("det_count", _vp)]


class ws_lane_buffers(ctypes.Structure):
    _fields_ = [("input_host", _vp), ("input_device", _vp), ("tensor", _vp), ("logits", _vp),
                ("result_val_host", _vp), ("result_idx_host", _vp), ("result_val_device", _vp),
                ("result_idx_device", _vp), ("input_bytes", _sz), ("tensor_bytes", _sz),
                ("logits_bytes", _sz), ("result_bytes", _sz), ("stream", _vp),
                ("detections_host", _vp), ("det_count_host", _vp), ("detections_device", _vp),
                ("det_count_device", _vp)]


class ws_debug_counters(ctypes.Structure):
    _fields_ = [("device_allocs", _i64), ("host_allocs", _i64), ("graphs", _i64), ("graph_execs", _i64),
                ("events", _i64), ("streams", _i64), ("fault_points", _i64)]


class ws_lane_timing(ctypes.Structure):
    _fields_ = [("gpu_us", _f32), ("preprocess_us", _f32), ("post_us", _f32), ("host_us", ctypes.c_double)]


class ws_candidate(ctypes.Structure):
    _fields_ = [("x1", _f32), ("y1", _f32), ("x2", _f32), ("y2", _f32), ("logit", _f32), ("cls", _i32),
                ("anchor", _i32), ("pad_", _i32)]


class ws_detection(ctypes.Structure):
    _fields_ = [("x1", _f32), ("y1", _f32), ("x2", _f32), ("y2", _f32), ("score", _f32), ("cls", _i32),
                ("anchor", _i32), ("pad_", _i32)]


# name: (restype, argtypes) -- one entry per declaration in include/ws.h
SIGNATURES = {
    "ws_status_string": (ctypes.c_char_p, [_i32]),
    "ws_last_error": (ctypes.c_char_p, []),
    "ws_version": (_i32, []),
    "ws_build_features": (_i32, []),
    "ws_device_error": (_i32, [ctypes.POINTER(_u32), _i32]),
    "ws_selftest_wait_timeout": (_i32, [_u32, _vp]),
    "ws_debug_inject_failure": (_i32, [_i32, _i32]),
    "ws_debug_get_counters": (_i32, [ctypes.POINTER(ws_debug_counters)]),
    "ws_preprocess_validate": (_i32, [ctypes.POINTER(ws_preprocess_desc), _i32]),
    "ws_preprocess": (_i32, [ctypes.POINTER(ws_preprocess_desc), _vp, _i32, _vp, _vp]),
    "ws_preprocess_path": (_i32, [ctypes.POINTER(ws_preprocess_desc), _vp, _i32, _vp, _i32, _vp]),
    "ws_topk_validate": (_i32, [_i64, _i64, _i32]),
    "ws_topk_workspace_bytes": (_i32, [_i64, _i64, _i32, ctypes.POINTER(_sz)]),
    "ws_topk_workspace_init": (_i32, [_vp, _sz, _vp]),
    "ws_topk": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp, _sz, _vp]),
    "ws_topk_noalloc": (_i32, [_vp, _i64, _i64, _i32, _vp, _vp, _vp]),
    "ws_detect_validate": (_i32, [ctypes.POINTER(ws_detect_desc), _i32, ctypes.POINTER(_i64)]),
    "ws_detect_workspace_bytes": (_i32, [ctypes.POINTER(ws_detect_desc), _i32, ctypes.POINTER(_sz)]),
    "ws_detect_workspace_init": (_i32, [_vp, _sz, _vp]),
    "ws_detect_decode": (_i32, [ctypes.POINTER(ws_detect_desc), _vp, _i32, _vp, _vp, _vp]),
    "ws_detect_nms": (_i32, [ctypes.POINTER(ws_detect_desc), _vp, _vp, _i32, _vp, _vp, _vp]),
    "ws_detect": (_i32, [ctypes.POINTER(ws_detect_desc), _vp, _i32, _vp, _vp, _vp, _sz, _vp]),
    "ws_lane_create": (_i32, [ctypes.POINTER(ws_lane_desc), ctypes.POINTER(_vp)]),
    "ws_lane_get_buffers": (_i32, [_vp, ctypes.POINTER(ws_lane_buffers)]),
    "ws_lane_acquire": (_i32, [_vp]),
    "ws_lane_submit": (_i32, [_vp]),
    "ws_lane_submit_n": (_i32, [_vp, _i32]),
    "ws_lane_rebind": (_i32, [_vp, _vp, _vp, ctypes.POINTER(_i32)]),
    "ws_lane_wait": (_i32, [_vp, _i64, ctypes.POINTER(ws_lane_timing)]),
    "ws_lane_selftest_wait_timeout": (_i32, [_vp, _u32]),
    "ws_lane_release": (_i32, [_vp]),
    "ws_lane_destroy": (_i32, [_vp]),
    "ws_lane_state": (_i32, [_vp]),
    "ws_pool_create": (_i32, [ctypes.POINTER(ws_lane_desc), _i32, ctypes.POINTER(_vp)]),
    "ws_pool_lane": (_i32, [_vp, _i32, ctypes.POINTER(_vp)]),
    "ws_pool_acquire": (_i32, [_vp, _i64, ctypes.POINTER(_vp)]),
    "ws_pool_submit": (_i32, [_vp, _vp, _i32]),
    "ws_pool_complete": (_i32, [_vp, _i64, ctypes.POINTER(_vp), ctypes.POINTER(ws_lane_timing)]),
    "ws_pool_recycle": (_i32, [_vp, _vp]),
    "ws_pool_destroy": (_i32, [_vp]),
}


def _library_path() -> str:
    """libws.so, or the checked build libws_bounds.so when WS_BOUNDS_CHECK=1."""
    return _build.BOUNDS_LIBRARY if os.environ.get("WS_BOUNDS_CHECK") == "1" else _build.LIBRARY


def _load():
    path = _library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -m post_processing_gb300.build or "
            "__graft_entry__.build()); there is no fallback implementation")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()
LIBRARY_PATH = _library_path()


class WsError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{ws_status_string(status)}: {message}")
        self.status = status


def check(status: int) -> int:
    if status != WS_OK:
        raise WsError(status, ws_last_error())
    return status


# ---- one Python function per C entry point, same names ----------------------

def ws_status_string(status: int) -> str:
    return lib.ws_status_string(status).decode()


def ws_last_error() -> str:
    return lib.ws_last_error().decode()


def ws_version() -> int:
    return lib.ws_version()


WS_FEATURE_BOUNDS_CHECK = 1


def ws_build_features() -> int:
    return lib.ws_build_features()


def ws_device_error(clear: bool = False) -> tuple[int, int]:
    flags = _u32(0)
    st = lib.ws_device_error(ctypes.byref(flags), int(clear))
    return st, flags.value


def ws_selftest_wait_timeout(limit_us: int, stream: int = 0) -> int:
    return lib.ws_selftest_wait_timeout(limit_us, stream)


def ws_debug_inject_failure(nth: int, count: int = 1) -> int:
    return lib.ws_debug_inject_failure(nth, count)


def ws_debug_get_counters() -> tuple[int, ws_debug_counters]:
    c = ws_debug_counters()
    st = lib.ws_debug_get_counters(ctypes.byref(c))
    return st, c


def ws_preprocess_validate(desc: ws_preprocess_desc, batch: int) -> int:
    return lib.ws_preprocess_validate(ctypes.byref(desc), batch)


def ws_preprocess(desc: ws_preprocess_desc, src: int, batch: int, dst: int, stream: int = 0) -> int:
    return lib.ws_preprocess(ctypes.byref(desc), src, batch, dst, stream)


def ws_preprocess_path(desc: ws_preprocess_desc, src: int, batch: int, dst: int, path: int, stream: int = 0) -> int:
    return lib.ws_preprocess_path(ctypes.byref(desc), src, batch, dst, path, stream)


def ws_topk_validate(rows: int, cols: int, k: int) -> int:
    return lib.ws_topk_validate(rows, cols, k)


def ws_topk_workspace_bytes(rows: int, cols: int, k: int) -> tuple[int, int]:
    n = _sz(0)
    st = lib.ws_topk_workspace_bytes(rows, cols, k, ctypes.byref(n))
    return st, n.value


def ws_topk_workspace_init(workspace: int, nbytes: int, stream: int = 0) -> int:
    return lib.ws_topk_workspace_init(workspace, nbytes, stream)


def ws_topk(x: int, rows: int, cols: int, k: int, out_val: int, out_idx: int,
            workspace: int | None, workspace_bytes: int, stream: int = 0) -> int:
    return lib.ws_topk(x, rows, cols, k, out_val, out_idx, workspace or None, workspace_bytes, stream)


def ws_topk_noalloc(x: int, rows: int, cols: int, k: int, out_val: int, out_idx: int,
                    stream: int = 0) -> int:
    return lib.ws_topk_noalloc(x, rows, cols, k, out_val, out_idx, stream)


def ws_detect_validate(desc: ws_detect_desc, batch: int) -> tuple[int, int]:
    a = _i64(0)
    st = lib.ws_detect_validate(ctypes.byref(desc), batch, ctypes.byref(a))
    return st, a.value


def ws_detect_workspace_bytes(desc: ws_detect_desc, batch: int) -> tuple[int, int]:
    n = _sz(0)
    st = lib.ws_detect_workspace_bytes(ctypes.byref(desc), batch, ctypes.byref(n))
    return st, n.value


def ws_detect_workspace_init(workspace: int, nbytes: int, stream: int = 0) -> int:
    return lib.ws_detect_workspace_init(workspace, nbytes, stream)


def ws_detect_decode(desc: ws_detect_desc, head: int, batch: int, cand: int, count: int, stream: int = 0) -> int:
    return lib.ws_detect_decode(ctypes.byref(desc), head, batch, cand, count, stream)


def ws_detect_nms(desc: ws_detect_desc, cand: int, count: int, batch: int, out: int, out_count: int,
                  stream: int = 0) -> int:
    return lib.ws_detect_nms(ctypes.byref(desc), cand, count, batch, out, out_count, stream)


def ws_detect(desc: ws_detect_desc, head: int, batch: int, out: int, out_count: int, workspace: int,
              workspace_bytes: int, stream: int = 0) -> int:
    return lib.ws_detect(ctypes.byref(desc), head, batch, out, out_count, workspace, workspace_bytes, stream)


def detect_desc(in_w: int = 640, in_h: int = 640, strides=(8, 16, 32), reg_max: int = 16, num_classes: int = 80,
                conf: float = 0.25, iou_thr: float = 0.45, max_cand: int = 1024, max_det: int = 300) -> ws_detect_desc:
    """Descriptor with the confidence given as a probability (its logit is the threshold)."""
    import math
    d = ws_detect_desc()
    d.in_w, d.in_h = in_w, in_h
    d.nlevels = len(strides)
    d.strides[:] = list(strides) + [0] * (4 - len(strides))
    d.reg_max, d.num_classes = reg_max, num_classes
    d.logit_thr = math.log(conf / (1.0 - conf))
    d.iou_thr = iou_thr
    d.max_cand, d.max_det = max_cand, max_det
    return d


def ws_lane_create(desc: ws_lane_desc) -> tuple[int, int | None]:
    h = _vp()
    st = lib.ws_lane_create(ctypes.byref(desc), ctypes.byref(h))
    return st, h.value


def ws_lane_get_buffers(lane: int) -> tuple[int, ws_lane_buffers]:
    b = ws_lane_buffers()
    st = lib.ws_lane_get_buffers(lane, ctypes.byref(b))
    return st, b


def ws_lane_acquire(lane: int) -> int:
    return lib.ws_lane_acquire(lane)


def ws_lane_submit(lane: int) -> int:
    return lib.ws_lane_submit(lane)


def ws_lane_submit_n(lane: int, n: int) -> int:
    return lib.ws_lane_submit_n(lane, n)


def ws_lane_rebind(lane: int, input: int | None = None, logits: int | None = None) -> tuple[int, int]:
    """(status, 1 if an executable graph had to be re-instantiated else 0)."""
    r = _i32(0)
    st = lib.ws_lane_rebind(lane, input, logits, ctypes.byref(r))
    return st, r.value


def ws_lane_wait(lane: int, timeout_us: int = -1) -> tuple[int, ws_lane_timing]:
    t = ws_lane_timing()
    st = lib.ws_lane_wait(lane, timeout_us, ctypes.byref(t))
    return st, t


def ws_lane_selftest_wait_timeout(lane: int, limit_us: int) -> int:
    return lib.ws_lane_selftest_wait_timeout(lane, limit_us)


def ws_lane_release(lane: int) -> int:
    return lib.ws_lane_release(lane)


def ws_lane_destroy(lane: int) -> int:
    return lib.ws_lane_destroy(lane)


def ws_lane_state(lane: int | None) -> int:
    return lib.ws_lane_state(lane)


# ---- descriptor helpers ------------------------------------------------------

def preprocess_desc(src_w: int, src_h: int, dst_w: int, dst_h: int, *, letterbox: bool = False,
                    pad_value: int = 114, norm: str = "mean_std",
                    mean=(0.485, 0.456, 0.406), std=(0.229, 0.224, 0.225), scale: float = 1.0 / 255.0,
                    row_stride: int | None = None, frame_stride: int | None = None,
                    channel_order: int = WS_ORDER_RGB, dst_type: int = WS_DTYPE_F32) -> ws_preprocess_desc:
    d = ws_preprocess_desc()
    d.src_w, d.src_h, d.dst_w, d.dst_h = src_w, src_h, dst_w, dst_h
    d.src_row_stride = 3 * src_w if row_stride is None else row_stride
    d.src_frame_stride = d.src_row_stride * src_h if frame_stride is None else frame_stride
    d.resize = WS_RESIZE_LETTERBOX if letterbox else WS_RESIZE_STRETCH
    d.pad_value = pad_value
    d.norm = WS_NORM_MEAN_STD if norm == "mean_std" else WS_NORM_SCALE
    d.mean[:] = list(mean)
    d.std[:] = list(std)
    d.scale = scale
    d.channel_order = channel_order
    d.dst_type = dst_type
    return d


def lane_desc(pre: ws_preprocess_desc, batch: int, rows: int, cols: int, k: int, *,
              input_mode: int = WS_INPUT_DEVICE, result_mode: int = WS_RESULT_DEVICE, flags: int = 0,
              input: int | None = None, tensor: int | None = None, logits: int | None = None,
              result_val: int | None = None, result_idx: int | None = None, stream: int | None = None,
              fake_polls: int = 0, detect: ws_detect_desc | None = None, detections: int | None = None,
              det_count: int | None = None) -> ws_lane_desc:
    """A lane descriptor; with `detect` the lane post-processes a detection head
    (rows, cols and k are then ignored)."""
    d = ws_lane_desc()
    d.pre = pre
    d.batch, d.rows, d.cols, d.k = batch, rows, cols, k
    d.input_mode, d.result_mode, d.flags = input_mode, result_mode, flags
    d.input, d.tensor, d.logits = input, tensor, logits
    d.result_val, d.result_idx, d.stream = result_val, result_idx, stream
    d.fake_polls = fake_polls
    if detect is not None:
        d.post, d.detect = WS_POST_DETECT, detect
        d.detections, d.det_count = detections, det_count
    return d


def ws_pool_create(desc: ws_lane_desc, lanes: int) -> tuple[int, int | None]:
    h = _vp()
    st = lib.ws_pool_create(ctypes.byref(desc), lanes, ctypes.byref(h))
    return st, h.value


def ws_pool_lane(pool: int, i: int) -> tuple[int, int | None]:
    h = _vp()
    st = lib.ws_pool_lane(pool, i, ctypes.byref(h))
    return st, h.value


def ws_pool_acquire(pool: int, timeout_us: int = -1) -> tuple[int, int | None]:
    h = _vp()
    st = lib.ws_pool_acquire(pool, timeout_us, ctypes.byref(h))
    return st, h.value


def ws_pool_submit(pool: int, lane: int, n: int) -> int:
    return lib.ws_pool_submit(pool, lane, n)


def ws_pool_complete(pool: int, timeout_us: int = -1) -> tuple[int, int | None, ws_lane_timing]:
    h = _vp()
    t = ws_lane_timing()
    st = lib.ws_pool_complete(pool, timeout_us, ctypes.byref(h), ctypes.byref(t))
    return st, h.value, t


def ws_pool_recycle(pool: int, lane: int) -> int:
    return lib.ws_pool_recycle(pool, lane)


def ws_pool_destroy(pool: int) -> int:
    return lib.ws_pool_destroy(pool)
