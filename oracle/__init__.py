"""The oracle: a plain CPU definition of the preprocess, the exact Top-K and
the detection decode + NMS.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product (``post_processing_gb300``) never imports it, and it
imports nothing from the product.

The arithmetic lives in ``ws_oracle.cpp`` (plain C++17, compiled with
``-O2 -ffp-contract=off``); this module only builds it with g++ and marshals
numpy arrays through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "ws_oracle.cpp")
LIBRARY = os.path.join(_HERE, "liboracle.so")
CXXFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None


def build(source: str = SOURCE, output: str = LIBRARY, force: bool = False) -> str:
    """Compile the oracle into a shared library (skipped when up to date)."""
    if (not force and os.path.exists(output)
            and os.path.getmtime(output) >= os.path.getmtime(source)):
        return output
    tmp = output + ".tmp%d" % os.getpid()
    subprocess.run(["g++", *CXXFLAGS, source, "-o", tmp], check=True)
    os.replace(tmp, output)
    return output


def load(path: str | None = None):
    """Load (building first if needed) an oracle library; returns a handle."""
    global _lib
    if path is None and _lib is not None:
        return _lib
    lib = ctypes.CDLL(path or build())
    i64, i32, f32p = ctypes.c_int64, ctypes.c_int, ctypes.POINTER(ctypes.c_float)
    lib.oracle_inner_box.argtypes = [i32, i32, i32, i32, i32] + [ctypes.POINTER(i32)] * 4
    lib.oracle_inner_box.restype = i32
    lib.oracle_axis_tap.argtypes = [i64, i64, i64, ctypes.POINTER(i64), ctypes.POINTER(i64), f32p]
    lib.oracle_axis_tap.restype = i32
    lib.oracle_preprocess.argtypes = [ctypes.c_void_p, i64, i64, i32, i32, i32, i32, i32, i32, i32,
                                      i32, f32p, f32p, ctypes.c_float, ctypes.c_void_p]
    lib.oracle_preprocess.restype = i32
    lib.oracle_topk.argtypes = [ctypes.c_void_p, i64, i64, i32, ctypes.c_void_p, ctypes.c_void_p]
    lib.oracle_topk.restype = i32
    vp = ctypes.c_void_p
    lib.oracle_anchor.argtypes = [i64, i32, i32, vp, i32, ctypes.POINTER(ctypes.c_double),
                                  ctypes.POINTER(ctypes.c_double), ctypes.POINTER(i32)]
    lib.oracle_anchor.restype = i32
    lib.oracle_decode.argtypes = [vp, i64, i32, i32, i32, i32, vp, i32, ctypes.c_float, i32,
                                  vp, vp, vp, vp, vp, ctypes.POINTER(i32)]
    lib.oracle_decode.restype = i32
    lib.oracle_nms.argtypes = [vp, vp, vp, vp, i32, ctypes.c_float, i32, i32, vp]
    lib.oracle_nms.restype = i32
    if path is None:
        _lib = lib
    return lib


class Oracle:
    """numpy front end of one oracle library (the built one by default)."""

    def __init__(self, path: str | None = None):
        self.lib = load(path)

    def inner_box(self, src_w, src_h, dst_w, dst_h, letterbox):
        out = [ctypes.c_int() for _ in range(4)]
        rc = self.lib.oracle_inner_box(src_w, src_h, dst_w, dst_h, int(letterbox),
                                       *[ctypes.byref(o) for o in out])
        if rc != 0:
            raise ValueError("invalid box sizes")
        return tuple(o.value for o in out)   # nw, nh, left, top

    def axis_tap(self, x, S, D):
        i0, i1, w = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_float()
        if self.lib.oracle_axis_tap(x, S, D, ctypes.byref(i0), ctypes.byref(i1), ctypes.byref(w)):
            raise ValueError("invalid tap")
        return i0.value, i1.value, w.value

    def preprocess(self, frames: np.ndarray, src_w: int, src_h: int, dst_w: int, dst_h: int,
                   letterbox: bool = False, pad_value: int = 114, norm: str = "mean_std",
                   mean=(0.485, 0.456, 0.406), std=(0.229, 0.224, 0.225),
                   scale: float = 1.0 / 255.0, row_stride: int | None = None,
                   frame_stride: int | None = None) -> np.ndarray:
        """frames: uint8 array of shape [B, H, stride] or [B, H, W, 3]."""
        frames = np.ascontiguousarray(frames, dtype=np.uint8)
        batch = frames.shape[0]
        flat = frames.reshape(batch, -1)
        rs = 3 * src_w if row_stride is None else row_stride
        fs = flat.shape[1] if frame_stride is None else frame_stride
        out = np.empty((batch, 3, dst_h, dst_w), dtype=np.float32)
        m = (ctypes.c_float * 3)(*mean)
        s = (ctypes.c_float * 3)(*std)
        rc = self.lib.oracle_preprocess(
            flat.ctypes.data, rs, fs, src_w, src_h, batch, dst_w, dst_h, int(letterbox),
            int(pad_value), 0 if norm == "mean_std" else 1, m, s, ctypes.c_float(scale),
            out.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_preprocess rejected its arguments")
        return out

    def topk(self, x: np.ndarray, k: int):
        x = np.ascontiguousarray(x, dtype=np.float32)
        if x.ndim == 1:
            x = x[None, :]
        rows, cols = x.shape
        val = np.empty((rows, k), dtype=np.float32)
        idx = np.empty((rows, k), dtype=np.int32)
        rc = self.lib.oracle_topk(x.ctypes.data, rows, cols, k, val.ctypes.data, idx.ctypes.data)
        if rc != 0:
            raise ValueError("oracle_topk rejected its arguments")
        return val, idx

    # ---- detection decode + NMS ------------------------------------------------

    def anchor(self, a, in_w, in_h, strides):
        st = np.ascontiguousarray(strides, dtype=np.int32)
        cx, cy, s = ctypes.c_double(), ctypes.c_double(), ctypes.c_int()
        if self.lib.oracle_anchor(a, in_w, in_h, st.ctypes.data, st.size, ctypes.byref(cx),
                                  ctypes.byref(cy), ctypes.byref(s)):
            raise ValueError("anchor out of range")
        return cx.value, cy.value, s.value

    def decode(self, head: np.ndarray, reg_max: int, num_classes: int, in_w: int, in_h: int, strides,
               logit_thr: float, max_cand: int = 1 << 20):
        """head: float32 [4*reg_max + num_classes, A] of one image."""
        head = np.ascontiguousarray(head, dtype=np.float32)
        A = head.shape[1]
        st = np.ascontiguousarray(strides, dtype=np.int32)
        cap = min(max_cand, A)
        boxes = np.empty((cap, 4), np.float32)
        logits = np.empty(cap, np.float32)
        scores = np.empty(cap, np.float32)
        classes = np.empty(cap, np.int32)
        anchors = np.empty(cap, np.int32)
        total = ctypes.c_int()
        n = self.lib.oracle_decode(head.ctypes.data, A, reg_max, num_classes, in_w, in_h, st.ctypes.data,
                                   st.size, ctypes.c_float(logit_thr), cap, boxes.ctypes.data,
                                   logits.ctypes.data, scores.ctypes.data, classes.ctypes.data,
                                   anchors.ctypes.data, ctypes.byref(total))
        if n < 0:
            raise ValueError("oracle_decode rejected its arguments")
        return dict(boxes=boxes[:n], logits=logits[:n], scores=scores[:n], classes=classes[:n],
                    anchors=anchors[:n], total=total.value)

    def nms(self, boxes, logits, classes, anchors, iou_thr: float, max_det: int, max_cand: int = 1 << 30):
        boxes = np.ascontiguousarray(boxes, dtype=np.float32).reshape(-1, 4)
        logits = np.ascontiguousarray(logits, dtype=np.float32)
        classes = np.ascontiguousarray(classes, dtype=np.int32)
        anchors = np.ascontiguousarray(anchors, dtype=np.int32)
        n = boxes.shape[0]
        keep = np.empty(max(max_det, 1), np.int32)
        k = self.lib.oracle_nms(boxes.ctypes.data, logits.ctypes.data, classes.ctypes.data, anchors.ctypes.data,
                                n, ctypes.c_float(iou_thr), max_cand, max_det, keep.ctypes.data)
        if k < 0:
            raise ValueError("oracle_nms rejected its arguments")
        return keep[:k]
