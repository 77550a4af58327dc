"""GB300-native fused RGB8 -> FP32 NCHW preprocess, exact Top-K and
detection decode + NMS.

The compute lives in ``libws.so`` (hand-written CUDA for sm_103a, C ABI in
``include/ws.h``).  ``binding`` mirrors the C ABI one function per entry
point; ``api`` adds PyTorch-tensor conveniences that only marshal
pointers, shapes and streams.
"""
from . import binding
from .binding import WsError, check
from .api import (Lane, Pool, detect, detect_workspace, detection_fields, preprocess, topk,
                  topk_workspace)

__all__ = ["binding", "WsError", "check", "Lane", "Pool", "preprocess", "topk", "topk_workspace", "detect",
           "detect_workspace", "detection_fields"]
