"""Seeded synthetic inputs for the fused preprocess and the exact Top-K.

This module holds only random-number generation and the shapes of the
workloads; none of the preprocess or Top-K arithmetic lives here.  Both the
CPU oracle (in ``oracle/``) and the CUDA path (in ``post_processing_gb300``)
are fed from these generators, and neither is imported here.

Generators, each from its published definition:

* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014; the 64-bit finaliser constants of Vigna's
  ``splitmix64.c``): output ``i`` of a stream with seed ``s`` is
  ``mix(s + (i + 1) * GOLDEN_GAMMA)`` modulo 2**64.
* Uniform bytes: the eight little-endian bytes of each SplitMix64 output.
* Uniform doubles: the top 53 bits of an output times 2**-53.
* Normal deviates: the Box-Muller transform (Box and Muller, 1958) in double
  precision, rounded once to float32.

The workload recipes (frame sizes, value distributions, the 5 % duplicated
entries of the long-row case) follow the inference configurations that the
WarpStream TRT write-up (problem-statement table: interleaved RGB8 producer,
FP32 NCHW network input, FP32 logits, K <= 32) and the yolo.cu README
(640x640 letterbox input) describe.
"""
from __future__ import annotations

import numpy as np

GOLDEN_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK64 = (1 << 64) - 1


def _mix(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def splitmix64(seed: int, n: int) -> np.ndarray:
    """First ``n`` outputs of the SplitMix64 stream seeded with ``seed``."""
    seed = int(seed) & _MASK64
    with np.errstate(over="ignore"):
        ctr = np.arange(1, n + 1, dtype=np.uint64) * GOLDEN_GAMMA
        ctr += np.uint64(seed)
        return _mix(ctr)


def splitmix64_scalar(seed: int, n: int) -> list[int]:
    """Plain-integer SplitMix64, used to cross-check the vectorised one."""
    out = []
    state = int(seed) & _MASK64
    for _ in range(n):
        state = (state + 0x9E3779B97F4A7C15) & _MASK64
        z = state
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK64
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK64
        out.append(z ^ (z >> 31))
    return out


def derive_seed(seed: int, *ids: int) -> int:
    """A child seed: one SplitMix64 output per id, chained."""
    s = int(seed) & _MASK64
    for i in ids:
        s = int(splitmix64(s ^ (int(i) & _MASK64), 1)[0])
    return s


def uniform_bytes(seed: int, n: int) -> np.ndarray:
    words = splitmix64(seed, (n + 7) // 8)
    return words.view("<u1")[:n].copy()


def uniform_doubles(seed: int, n: int) -> np.ndarray:
    """Uniform in [0, 1): top 53 bits of each output times 2**-53."""
    return (splitmix64(seed, n) >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normal(seed: int, n: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    """N(mu, sigma) deviates by Box-Muller in double, rounded to float32."""
    return normal_f64(seed, n, mu, sigma).astype(np.float32)


def normal_f64(seed: int, n: int, mu: float = 0.0, sigma: float = 1.0) -> np.ndarray:
    pairs = (n + 1) // 2
    w = splitmix64(seed, 2 * pairs)
    u1 = ((w[0::2] >> np.uint64(11)).astype(np.float64) + 1.0) * (2.0 ** -53)  # (0, 1]
    u2 = (w[1::2] >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)          # [0, 1)
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * pairs, dtype=np.float64)
    z[0::2] = r * np.cos(2.0 * np.pi * u2)
    z[1::2] = r * np.sin(2.0 * np.pi * u2)
    return mu + sigma * z[:n]


# --------------------------------------------------------------------------
# Frames (interleaved RGB8, row stride = 3 * width unless stated)
# --------------------------------------------------------------------------

def frames_uniform(seed: int, batch: int, height: int, width: int,
                   row_stride: int | None = None) -> np.ndarray:
    """``batch`` independent uniform RGB8 frames, shape [B, H, stride]."""
    stride = 3 * width if row_stride is None else row_stride
    out = np.empty((batch, height, stride), dtype=np.uint8)
    for b in range(batch):
        out[b] = uniform_bytes(derive_seed(seed, b), height * stride).reshape(height, stride)
    return out


def frames_gradient_noise(seed: int, batch: int, height: int, width: int,
                          noise: int = 32) -> np.ndarray:
    """Smooth gradient plus uniform integer noise in [-noise, noise], clamped.

    R ramps along x, G along y, B along x + y; the noise is drawn per byte.
    Shape [B, H, 3 * W].
    """
    x = np.arange(width, dtype=np.float64)
    y = np.arange(height, dtype=np.float64)[:, None]
    base = np.empty((height, width, 3), dtype=np.float64)
    base[..., 0] = 255.0 * x / max(width - 1, 1)
    base[..., 1] = 255.0 * y / max(height - 1, 1)
    base[..., 2] = 255.0 * (x + y) / max(width + height - 2, 1)
    base = np.floor(base + 0.5).astype(np.int32)
    span = 2 * noise + 1
    out = np.empty((batch, height, 3 * width), dtype=np.uint8)
    for b in range(batch):
        w = splitmix64(derive_seed(seed, b), height * width * 3)
        nz = (w % np.uint64(span)).astype(np.int32) - noise
        img = np.clip(base + nz.reshape(height, width, 3), 0, 255).astype(np.uint8)
        out[b] = img.reshape(height, 3 * width)
    return out


# --------------------------------------------------------------------------
# Logits / scores
# --------------------------------------------------------------------------

def logits_normal(seed: int, rows: int, cols: int) -> np.ndarray:
    return normal(seed, rows * cols).reshape(rows, cols)


def scores_logistic(seed: int, n: int, mu: float = -4.0, sigma: float = 2.0) -> np.ndarray:
    """sigma(z) with z ~ N(mu, sigma), evaluated in double, rounded to float32."""
    z = normal_f64(seed, n, mu, sigma)
    return (1.0 / (1.0 + np.exp(-z))).astype(np.float32)


def logits_with_ties(seed: int, rows: int, cols: int, frac: float = 0.05) -> np.ndarray:
    """N(0, 1) rows where a fraction ``frac`` of positions copy another entry.

    For each row, every position d is picked with probability ``frac`` and
    then set to x[s] with s uniform over the row, so equal values (ties that
    the lower index must win) appear throughout the row.
    """
    x = logits_normal(seed, rows, cols)
    for r in range(rows):
        u = uniform_doubles(derive_seed(seed, 1, r), cols)
        dst = np.nonzero(u < frac)[0]
        src = (splitmix64(derive_seed(seed, 2, r), dst.size) % np.uint64(cols)).astype(np.int64)
        x[r, dst] = x[r, src]
    return x


# --------------------------------------------------------------------------
# The five inference workloads
# --------------------------------------------------------------------------

MEAN = (0.485, 0.456, 0.406)
STD = (0.229, 0.224, 0.225)

WORKLOADS = {
    # name: dict(source frames, geometry, normalisation, logits, K)
    "b1_224_identity": dict(
        batch=1, src_w=224, src_h=224, dst_w=224, dst_h=224, resize="stretch",
        norm="mean_std", rows=1, cols=1000, k=5, frames="uniform", logits="normal"),
    "b1_1080p_to_224": dict(
        batch=1, src_w=1920, src_h=1080, dst_w=224, dst_h=224, resize="stretch",
        norm="mean_std", rows=1, cols=1000, k=5, frames="gradient_noise", logits="normal"),
    "b1_720p_letterbox_640": dict(
        batch=1, src_w=1280, src_h=720, dst_w=640, dst_h=640, resize="letterbox",
        norm="scale", rows=1, cols=8400 * 80, k=32, frames="uniform", logits="logistic"),
    "b64_1080p_to_224": dict(
        batch=64, src_w=1920, src_h=1080, dst_w=224, dst_h=224, resize="stretch",
        norm="mean_std", rows=64, cols=1000, k=32, frames="uniform", logits="normal"),
    "b8_4k_to_512": dict(
        batch=8, src_w=3840, src_h=2160, dst_w=512, dst_h=512, resize="stretch",
        norm="mean_std", rows=32, cols=131072, k=32, frames="uniform", logits="ties"),
}

BASE_SEED = 0x57A70000


def workload_seed(name: str, tensor_id: int) -> int:
    return derive_seed(BASE_SEED, list(WORKLOADS).index(name), tensor_id)


def make_frames(name: str, batch: int | None = None) -> np.ndarray:
    w = WORKLOADS[name]
    b = w["batch"] if batch is None else batch
    seed = workload_seed(name, 0)
    if w["frames"] == "gradient_noise":
        return frames_gradient_noise(seed, b, w["src_h"], w["src_w"])
    return frames_uniform(seed, b, w["src_h"], w["src_w"])


def make_logits(name: str, rows: int | None = None) -> np.ndarray:
    w = WORKLOADS[name]
    r = w["rows"] if rows is None else rows
    seed = workload_seed(name, 1)
    if w["logits"] == "logistic":
        return scores_logistic(seed, r * w["cols"]).reshape(r, w["cols"])
    if w["logits"] == "ties":
        return logits_with_ties(seed, r, w["cols"])
    return logits_normal(seed, r, w["cols"])


# --------------------------------------------------------------------------
# Detection head (YOLO-style, before the DFL decode)
# --------------------------------------------------------------------------

YOLO_STRIDES = (8, 16, 32)


def yolo_anchor_count(in_w: int, in_h: int, strides=YOLO_STRIDES) -> int:
    return sum((in_w // s) * (in_h // s) for s in strides)


def yolo_head(seed: int, batch: int, in_w: int = 640, in_h: int = 640, reg_max: int = 16,
              num_classes: int = 80, dfl_sigma: float = 2.0, cls_mu: float = -8.0,
              cls_sigma: float = 2.0, strides=YOLO_STRIDES) -> np.ndarray:
    """Raw head output [batch, 4*reg_max + num_classes, A]: DFL bin logits
    N(0, dfl_sigma) and class logits N(cls_mu, cls_sigma).  With the defaults
    about 2 % of the anchors of a 640x640 input clear a 0.25 confidence, and
    neighbouring anchors' boxes overlap, so suppression has work to do."""
    A = yolo_anchor_count(in_w, in_h, strides)
    ch = 4 * reg_max + num_classes
    out = np.empty((batch, ch, A), np.float32)
    for b in range(batch):
        out[b, :4 * reg_max] = normal(derive_seed(seed, b, 0), 4 * reg_max * A, 0.0, dfl_sigma).reshape(4 * reg_max, A)
        out[b, 4 * reg_max:] = normal(derive_seed(seed, b, 1), num_classes * A, cls_mu, cls_sigma).reshape(num_classes, A)
    return out


def clustered_candidates(seed: int, objects: int, per_object: int, num_classes: int = 80,
                         in_w: int = 640, in_h: int = 640, jitter: float = 0.08,
                         logit_mu: float = 0.0, logit_sigma: float = 2.0, anchors: int = 8400) -> dict:
    """Detection candidates the way a detector's dense head emits them: around
    each of ``objects`` random boxes, ``per_object`` copies whose corners move
    by N(0, jitter * side), all of the object's class; logits N(mu, sigma);
    distinct anchor ids drawn from [0, anchors).  Returns float32 boxes
    [n, 4] (x1, y1, x2, y2), float32 logits, int32 classes and anchors."""
    n = objects * per_object
    u = uniform_doubles(derive_seed(seed, 0), 4 * objects).reshape(objects, 4)
    w = 16.0 + u[:, 2] * (in_w / 2.0)
    h = 16.0 + u[:, 3] * (in_h / 2.0)
    cx = u[:, 0] * in_w
    cy = u[:, 1] * in_h
    base = np.stack([cx - w / 2, cy - h / 2, cx + w / 2, cy + h / 2], axis=1)
    side = np.stack([w, h, w, h], axis=1)
    z = normal_f64(derive_seed(seed, 1), 4 * n).reshape(n, 4)
    boxes = (np.repeat(base, per_object, axis=0) + jitter * np.repeat(side, per_object, axis=0) * z)
    cls = (splitmix64(derive_seed(seed, 2), objects) % np.uint64(num_classes)).astype(np.int32)
    perm = np.argsort(splitmix64(derive_seed(seed, 3), anchors), kind="stable")[:n].astype(np.int32)
    return dict(boxes=boxes.astype(np.float32), logits=normal(derive_seed(seed, 4), n, logit_mu, logit_sigma),
                classes=np.repeat(cls, per_object), anchors=perm)
