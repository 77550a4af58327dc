"""PyTorch-tensor front end of the C ABI (marshalling only).

Tensors supply device memory, pinned host memory and streams; every result
is computed by ``libws.so`` on the GPU.
"""
from __future__ import annotations

import torch

from . import binding as B


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def preprocess(frames: torch.Tensor, desc: B.ws_preprocess_desc, batch: int | None = None,
               out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """ws_preprocess on a uint8 CUDA tensor holding `batch` frames."""
    if frames.dtype != torch.uint8 or not frames.is_cuda:
        raise TypeError("frames must be a uint8 CUDA tensor")
    if batch is None:
        batch = frames.shape[0]
    if out is None:
        dtype = {B.WS_DTYPE_F32: torch.float32, B.WS_DTYPE_F16: torch.float16,
                 B.WS_DTYPE_BF16: torch.bfloat16}[desc.dst_type]
        out = torch.empty((batch, 3, desc.dst_h, desc.dst_w), dtype=dtype, device=frames.device)
    B.check(B.ws_preprocess(desc, frames.data_ptr(), batch, out.data_ptr(), _stream(stream)))
    return out


def topk_workspace(rows: int, cols: int, k: int, device="cuda", stream=None) -> torch.Tensor | None:
    """A zeroed workspace for ws_topk of this shape (None when none is needed)."""
    st, n = B.ws_topk_workspace_bytes(rows, cols, k)
    B.check(st)
    if n == 0:
        return None
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    B.check(B.ws_topk_workspace_init(ws.data_ptr(), n, _stream(stream)))
    return ws


def topk(x: torch.Tensor, k: int, out_val: torch.Tensor | None = None, out_idx: torch.Tensor | None = None,
         workspace: torch.Tensor | None = None, stream=None):
    """ws_topk on a float32 CUDA tensor [rows, cols] (or [cols])."""
    if x.dtype != torch.float32 or not x.is_cuda or not x.is_contiguous():
        raise TypeError("x must be a contiguous float32 CUDA tensor")
    rows, cols = (1, x.shape[0]) if x.dim() == 1 else x.shape
    if out_val is None:
        out_val = torch.empty((rows, k), dtype=torch.float32, device=x.device)
    if out_idx is None:
        out_idx = torch.empty((rows, k), dtype=torch.int32, device=x.device)
    if workspace is None:
        workspace = topk_workspace(rows, cols, k, x.device, stream)
    wptr, wbytes = (workspace.data_ptr(), workspace.numel()) if workspace is not None else (None, 0)
    B.check(B.ws_topk(x.data_ptr(), rows, cols, k, out_val.data_ptr(), out_idx.data_ptr(), wptr, wbytes,
                      _stream(stream)))
    return out_val, out_idx


def detect_workspace(desc: B.ws_detect_desc, batch: int, device="cuda", stream=None) -> torch.Tensor:
    """A zeroed, 256-byte aligned workspace for ws_detect of this geometry and batch."""
    st, n = B.ws_detect_workspace_bytes(desc, batch)
    B.check(st)
    ws = torch.empty(n + 256, dtype=torch.uint8, device=device)
    off = (-ws.data_ptr()) % 256
    ws = ws[off:off + n]
    B.check(B.ws_detect_workspace_init(ws.data_ptr(), n, _stream(stream)))
    return ws


def detect(head: torch.Tensor, desc: B.ws_detect_desc, workspace: torch.Tensor | None = None,
           out: torch.Tensor | None = None, out_count: torch.Tensor | None = None, stream=None):
    """ws_detect on a float32 CUDA head [batch, 4*reg_max + num_classes, A].

    Returns (detections, counts): detections is the raw int32 [batch, max_det,
    8] buffer of ws_detection records and counts the int32 [batch] kept per
    image; detection_fields() gives named views of it."""
    if head.dtype != torch.float32 or not head.is_cuda or not head.is_contiguous() or head.dim() != 3:
        raise TypeError("head must be a contiguous float32 CUDA tensor [batch, channels, anchors]")
    batch = head.shape[0]
    if workspace is None:
        workspace = detect_workspace(desc, batch, head.device, stream)
    if out is None:
        out = torch.empty((batch, desc.max_det, 8), dtype=torch.int32, device=head.device)
    if out_count is None:
        out_count = torch.empty(batch, dtype=torch.int32, device=head.device)
    B.check(B.ws_detect(desc, head.data_ptr(), batch, out.data_ptr(), out_count.data_ptr(), workspace.data_ptr(),
                        workspace.numel(), _stream(stream)))
    return out, out_count


def detection_fields(detections: torch.Tensor) -> dict:
    """Named views of a [..., 8] int32 ws_detection buffer: boxes (x1, y1, x2,
    y2) and score as float32, class and anchor as int32."""
    f = detections.view(torch.float32)
    return {"boxes": f[..., 0:4], "score": f[..., 4], "cls": detections[..., 5], "anchor": detections[..., 6]}


class Pool:
    """ws_pool_*: N identical lanes with a producer / consumer hand-off;
    destroyed by close() or `with`.  Lanes are returned as raw handles."""

    def __init__(self, desc: B.ws_lane_desc, lanes: int):
        st, h = B.ws_pool_create(desc, lanes)
        B.check(st)
        self.handle = h
        self.size = lanes
        self._batch = desc.batch

    def lane(self, i: int) -> int:
        st, h = B.ws_pool_lane(self.handle, i)
        B.check(st)
        return h

    def buffers(self, lane: int) -> B.ws_lane_buffers:
        st, b = B.ws_lane_get_buffers(lane)
        B.check(st)
        return b

    def acquire(self, timeout_us: int = -1) -> int | None:
        """A free lane, or None if none became free in time (back-pressure)."""
        st, h = B.ws_pool_acquire(self.handle, timeout_us)
        if st == B.WS_ERR_TIMEOUT:
            return None
        B.check(st)
        return h

    def submit(self, lane: int, n: int | None = None):
        """Submit the lane's whole batch, or its first n frames."""
        B.check(B.ws_pool_submit(self.handle, lane, self._batch if n is None else n))

    def complete(self, timeout_us: int = -1):
        """(lane, timing) of the oldest submission, or (None, None) on timeout."""
        st, h, t = B.ws_pool_complete(self.handle, timeout_us)
        if st == B.WS_ERR_TIMEOUT:
            return None, None
        B.check(st)
        return h, t

    def recycle(self, lane: int):
        B.check(B.ws_pool_recycle(self.handle, lane))

    def close(self):
        if self.handle is not None:
            B.check(B.ws_pool_destroy(self.handle))
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


class Lane:
    """One fixed-shape lane (ws_lane_*); destroyed by close() or `with`."""

    def __init__(self, desc: B.ws_lane_desc):
        st, h = B.ws_lane_create(desc)
        B.check(st)
        self.handle = h
        st, self.buffers = B.ws_lane_get_buffers(h)
        B.check(st)

    def acquire(self):
        B.check(B.ws_lane_acquire(self.handle))

    def submit(self, n: int | None = None):
        """Submit the whole batch, or the first n frames (ws_lane_submit_n)."""
        B.check(B.ws_lane_submit(self.handle) if n is None else B.ws_lane_submit_n(self.handle, n))

    def rebind(self, input: int | None = None, logits: int | None = None) -> bool:
        """Point the lane at new slots; True if a graph was re-instantiated."""
        st, re = B.ws_lane_rebind(self.handle, input, logits)
        B.check(st)
        st, self.buffers = B.ws_lane_get_buffers(self.handle)
        B.check(st)
        return bool(re)

    def wait(self, timeout_us: int = -1) -> B.ws_lane_timing:
        st, t = B.ws_lane_wait(self.handle, timeout_us)
        B.check(st)
        return t

    def release(self):
        B.check(B.ws_lane_release(self.handle))

    @property
    def state(self) -> int:
        return B.ws_lane_state(self.handle)

    def close(self):
        if self.handle is not None:
            B.check(B.ws_lane_destroy(self.handle))
            self.handle = None

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
