"""Pins of the oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:

* hand-computed values stored under ``tests/golden/`` (each with its source);
* closed forms (identity resize, constant images, letterbox padding);
* exact rational arithmetic of the textbook half-pixel coordinate
  (``fractions.Fraction``), independent of the oracle's integer form;
* a library special case: ``torch.nn.functional.interpolate`` (bilinear,
  ``align_corners=False``, no antialias) in float64, and a stable
  ``torch.sort`` for Top-K;
* brute force on tiny inputs (every permutation of a row with ties, signed
  zeros, NaN and infinities, against selection by repeated arg-max).

The same functions run against deliberately broken copies of the oracle in
``test_oracle_mutations.py`` to show that each plausible mistake is caught.
"""
from __future__ import annotations

import itertools
import math
import os
from fractions import Fraction

import numpy as np

import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
MEAN = np.array(synth.MEAN)
STD = np.array(synth.STD)


# ---------------------------------------------------------------- fixtures

def read_bilinear_cases():
    cases, cur, section, chan = [], None, None, None
    for line in open(os.path.join(GOLDEN, "bilinear_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        if tok[0] == "case":
            sw, sh, dw, dh = map(int, tok[2:6])
            cur = dict(name=tok[1], sw=sw, sh=sh, dw=dw, dh=dh,
                       src=np.zeros((sh, sw, 3), np.uint8), out=np.zeros((3, dh, dw)),
                       rows={"src": [0, 0, 0], "out": [0, 0, 0]})
            cases.append(cur)
        elif tok[0] in ("src", "out"):
            section, chan = tok[0], int(tok[1])
        else:
            vals = [float(t) for t in tok]
            r = cur["rows"][section][chan]
            if section == "src":
                cur["src"][r, :, chan] = np.array(vals, dtype=np.uint8)
            else:
                cur["out"][chan, r, :] = vals
            cur["rows"][section][chan] += 1
    return cases


def read_boxes():
    out = []
    for line in open(os.path.join(GOLDEN, "letterbox_boxes.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            out.append(tuple(int(t) for t in line.split()))
    return out


def _f(tok):
    return {"nan": math.nan, "inf": math.inf, "-inf": -math.inf}.get(tok, None) \
        if tok in ("nan", "inf", "-inf") else float(tok)


def read_topk_rows():
    rows, lines = [], [l.strip() for l in open(os.path.join(GOLDEN, "topk_hand.txt"))]
    lines = [l for l in lines if l and not l.startswith("#")]
    for i in range(0, len(lines), 4):
        k = int(lines[i].split()[1])
        x = np.array([_f(t) for t in lines[i + 1].split()], dtype=np.float32)
        idx = np.array([int(t) for t in lines[i + 2].split()], dtype=np.int32)
        val = np.array([_f(t) for t in lines[i + 3].split()], dtype=np.float32)
        rows.append((k, x, idx, val))
    return rows


def normalise_f64(v, mean=MEAN, std=STD):
    """The page's normalisation in float64: (v/255 - mean) / std."""
    v = np.asarray(v, dtype=np.float64)
    return (v / 255.0 - mean.reshape(-1, 1, 1)) / std.reshape(-1, 1, 1)


# ---------------------------------------------------------------- preprocess

def pin_bilinear_golden(o):
    for c in read_bilinear_cases():
        out = o.preprocess(c["src"][None], c["sw"], c["sh"], c["dw"], c["dh"],
                           norm="scale", scale=1.0)[0]
        assert np.array_equal(out, c["out"].astype(np.float32)), \
            f"{c['name']}: {out} != {c['out']}"


def pin_letterbox_boxes(o):
    for sw, sh, dw, dh, nw, nh, left, top in read_boxes():
        got = o.inner_box(sw, sh, dw, dh, True)
        assert got == (nw, nh, left, top), f"{sw}x{sh}->{dw}x{dh}: {got}"
        assert o.inner_box(sw, sh, dw, dh, False) == (dw, dh, 0, 0)


def pin_axis_taps(o):
    """(i0, i1, w) against exact rational evaluation of the textbook formula."""
    rng = np.random.default_rng(1)
    pairs = [(1920, 224), (1080, 224), (3840, 512), (2160, 512), (1280, 640), (720, 360),
             (224, 224), (2, 4), (4, 2), (3, 2), (1, 5), (5, 1), (7, 640), (640, 7)]
    pairs += [(int(a), int(b)) for a, b in rng.integers(1, 300, size=(24, 2))]
    for S, D in pairs:
        xs = range(D) if D <= 700 else rng.integers(0, D, 200)
        for x in xs:
            x = int(x)
            c = Fraction(2 * x + 1, 2) * Fraction(S, D) - Fraction(1, 2)
            x0 = math.floor(c)
            frac = c - x0
            i0, i1, w = o.axis_tap(x, S, D)
            assert i0 == min(max(x0, 0), S - 1), (S, D, x, i0)
            assert i1 == min(max(x0 + 1, 0), S - 1), (S, D, x, i1)
            # one correctly rounded float32 division: within half an ulp of 1
            assert abs(Fraction(float(w)) - frac) <= Fraction(1, 2 ** 25), (S, D, x, w, frac)


def pin_identity(o):
    """S = D: every weight is 0, so out = normalise(src) element-wise."""
    frames = synth.frames_uniform(11, 2, 23, 37)
    out = o.preprocess(frames, 37, 23, 37, 23)
    for b in range(2):
        img = frames[b].reshape(23, 37, 3).transpose(2, 0, 1)
        assert np.max(np.abs(out[b] - normalise_f64(img))) < 1e-6
    # and, without normalisation, the bytes themselves
    raw = o.preprocess(frames, 37, 23, 37, 23, norm="scale", scale=1.0)
    assert np.array_equal(raw, frames.reshape(2, 23, 37, 3).transpose(0, 3, 1, 2).astype(np.float32))


def pin_constant(o):
    """A constant image stays constant through any resize; padding is 114."""
    cases = [(40, 30, 64, 64, False), (1280, 720, 64, 64, True), (30, 41, 50, 50, True),
             (17, 5, 3, 9, False), (9, 9, 40, 21, True)]
    colour = np.array([200, 13, 114 + 7], dtype=np.uint8)
    for sw, sh, dw, dh, lb in cases:
        img = np.broadcast_to(colour, (1, sh, sw, 3)).copy()
        for norm in ("mean_std", "scale"):
            out = o.preprocess(img, sw, sh, dw, dh, letterbox=lb, norm=norm)[0]
            nw, nh, left, top = o.inner_box(sw, sh, dw, dh, lb)
            inside = np.zeros((dh, dw), bool)
            inside[top:top + nh, left:left + nw] = True
            for c in range(3):
                if norm == "mean_std":
                    want_in = (colour[c] / 255.0 - MEAN[c]) / STD[c]
                    want_pad = (114 / 255.0 - MEAN[c]) / STD[c]
                else:
                    want_in, want_pad = colour[c] / 255.0, 114 / 255.0
                assert np.max(np.abs(out[c][inside] - want_in)) < 1e-6, (sw, sh, dw, dh, lb, c)
                if (~inside).any():
                    assert np.max(np.abs(out[c][~inside] - want_pad)) < 1e-6, (sw, sh, c)


def pin_torch_interpolate(o):
    """Library special case: torch bilinear (half-pixel, clamped, no antialias)."""
    import torch
    import torch.nn.functional as F
    cases = [(64, 48, 23, 17), (1920, 1080, 224, 224), (37, 29, 80, 61), (224, 224, 224, 224),
             (5, 3, 11, 2), (640, 1, 7, 3)]
    for sw, sh, dw, dh in cases:
        frames = synth.frames_uniform(5 + sw, 1, sh, sw)
        out = o.preprocess(frames, sw, sh, dw, dh, norm="scale", scale=1.0)[0]
        img = torch.from_numpy(frames[0].reshape(sh, sw, 3).transpose(2, 0, 1).astype(np.float64))
        ref = F.interpolate(img[None], size=(dh, dw), mode="bilinear", align_corners=False,
                            antialias=False)[0].numpy()
        assert np.max(np.abs(out - ref)) < 1e-3, (sw, sh, dw, dh, np.max(np.abs(out - ref)))
    # letterbox: the inner box is a plain resize to (nh, nw), the rest padding;
    # landscape (rows padded) and portrait (columns padded, odd split) frames
    for sw, sh, dw, dh in ((160, 90, 64, 64), (90, 160, 64, 64), (45, 80, 67, 64)):
        frames = synth.frames_uniform(99 + sw, 1, sh, sw)
        out = o.preprocess(frames, sw, sh, dw, dh, letterbox=True, norm="scale", scale=1.0)[0]
        nw, nh, left, top = o.inner_box(sw, sh, dw, dh, True)
        img = torch.from_numpy(frames[0].reshape(sh, sw, 3).transpose(2, 0, 1).astype(np.float64))
        ref = F.interpolate(img[None], size=(nh, nw), mode="bilinear", align_corners=False,
                            antialias=False)[0].numpy()
        assert np.max(np.abs(out[:, top:top + nh, left:left + nw] - ref)) < 1e-3
        pad = np.ones((dh, dw), bool)
        pad[top:top + nh, left:left + nw] = False
        assert np.all(out[:, pad] == 114.0)


def pin_strides(o):
    """A padded row stride and frame stride read the same pixels as packed ones."""
    sw, sh = 19, 11
    packed = synth.frames_uniform(3, 3, sh, sw)
    rs, fs = 3 * sw + 13, (3 * sw + 13) * sh + 29
    buf = np.zeros(3 * fs, np.uint8)
    for b in range(3):
        for j in range(sh):
            buf[b * fs + j * rs: b * fs + j * rs + 3 * sw] = packed[b, j]
    a = o.preprocess(packed, sw, sh, 8, 30)
    b_ = o.preprocess(buf.reshape(3, fs), sw, sh, 8, 30, row_stride=rs, frame_stride=fs)
    assert np.array_equal(a, b_)
    # frames are independent: frame 1 alone gives frame 1's output
    one = o.preprocess(packed[1:2], sw, sh, 8, 30)
    assert np.array_equal(a[1], one[0])


# ---------------------------------------------------------------- Top-K

def _canon(v):
    return -math.inf if math.isnan(v) else v


def select_by_argmax(row, k):
    """Brute force: K rounds of a linear arg-max over the unselected entries."""
    taken, out = set(), []
    for _ in range(k):
        best = None
        for j, v in enumerate(row):
            if j in taken:
                continue
            if best is None or _canon(v) > _canon(row[best]):   # strict: lower index wins ties
                best = j
        taken.add(best)
        out.append(best)
    return out


def pin_topk_golden(o):
    for k, x, idx, val in read_topk_rows():
        v, i = o.topk(x, k)
        assert np.array_equal(i[0], idx), (x, i, idx)
        assert np.array_equal(v[0].view(np.uint32), val.view(np.uint32)), (x, v, val)


def pin_topk_bruteforce(o):
    base = [2.0, -0.0, 2.0, math.nan, 0.0, -math.inf, math.inf]
    perms = np.array(list(itertools.permutations(base)), dtype=np.float32)
    # keep the permutations distinct as value patterns (NaN compares unequal)
    for k in range(1, len(base) + 1):
        v, i = o.topk(perms, k)
        for r in range(0, perms.shape[0], 7):
            want = select_by_argmax(list(perms[r]), k)
            assert list(i[r]) == want, (perms[r], k, i[r], want)
            wv = np.array([_canon(perms[r][j]) for j in want], np.float32)
            assert np.array_equal(v[r].view(np.uint32), wv.view(np.uint32))


def pin_topk_torch(o):
    import torch
    rng = np.random.default_rng(7)
    x = rng.integers(-20, 20, size=(6, 3001)).astype(np.float32) / 4   # many ties
    x[0, rng.integers(0, 3001, 50)] = np.nan
    x[1, :] = 0.0
    x[1, ::3] = -0.0
    x[2, 5] = np.inf
    x[3, :] = np.nan
    for k in (1, 5, 32):
        v, i = o.topk(x, k)
        t = torch.from_numpy(np.where(np.isnan(x), -np.inf, x))
        # +0 and -0 must tie: compare on x + 0.0 (which turns -0 into +0)
        sv, si = torch.sort(t + 0.0, dim=1, descending=True, stable=True)
        assert np.array_equal(i, si[:, :k].numpy().astype(np.int32))
        want = np.take_along_axis(np.where(np.isnan(x), -np.inf, x), si[:, :k].numpy(), 1)
        assert np.array_equal(v.view(np.uint32), want.astype(np.float32).view(np.uint32))


def check_topk_invariants(x, val, idx, k):
    """Properties any exact Top-K result has; independent of how it was found."""
    xc = np.where(np.isnan(x), -np.inf, x).astype(np.float32)
    for r in range(x.shape[0]):
        key = xc[r]
        assert len(set(idx[r].tolist())) == k                          # unique
        assert np.array_equal(val[r].view(np.uint32), key[idx[r]].view(np.uint32))
        assert np.all(val[r][:-1] >= val[r][1:])                        # non-increasing (-inf >= -inf)
        cut = val[r][-1]
        assert np.count_nonzero(key > cut) <= k - 1                    # fewer than K above the cut
        # ties at the cut: the lowest indices among the tied values were taken
        tied = np.nonzero(key == cut)[0]
        chosen = sorted(j for j in idx[r] if key[j] == cut)
        assert chosen == sorted(tied[:len(chosen)].tolist())
        # equal values appear in index order
        for a in range(k - 1):
            if val[r][a] == val[r][a + 1]:
                assert idx[r][a] < idx[r][a + 1]


def pin_topk_invariants(o):
    rng = np.random.default_rng(3)
    x = synth.logits_with_ties(123, 4, 20000, frac=0.2)
    x[0, rng.integers(0, 20000, 500)] = np.nan
    x[2, :] = np.round(x[2, :] * 2) / 2
    for k in (1, 7, 32):
        v, i = o.topk(x, k)
        check_topk_invariants(x, v, i, k)


PRE_PINS = [pin_bilinear_golden, pin_letterbox_boxes, pin_axis_taps, pin_identity,
            pin_constant, pin_torch_interpolate, pin_strides]
TOPK_PINS = [pin_topk_golden, pin_topk_bruteforce, pin_topk_torch, pin_topk_invariants]
ALL_PINS = PRE_PINS + TOPK_PINS


# ---------------------------------------------------------------- detection

def pin_anchor_geometry(o):
    """Hand-computed anchor centres: 640x640 with strides 8, 16, 32 (80x80,
    40x40 and 20x20 cells = 8400 anchors) and a 320x192 input."""
    cases = [((0, 640, 640), (4.0, 4.0, 8)), ((79, 640, 640), (636.0, 4.0, 8)),
             ((80, 640, 640), (4.0, 12.0, 8)), ((6399, 640, 640), (636.0, 636.0, 8)),
             ((6400, 640, 640), (8.0, 8.0, 16)), ((8000, 640, 640), (16.0, 16.0, 32)),
             ((8399, 640, 640), (624.0, 624.0, 32)), ((41, 320, 192), (12.0, 12.0, 8)),
             ((960, 320, 192), (8.0, 8.0, 16)), ((1259, 320, 192), (304.0, 176.0, 32))]
    for (a, w, h), want in cases:
        assert o.anchor(a, w, h, (8, 16, 32)) == want, (a, w, h)
    try:
        o.anchor(8400, 640, 640, (8, 16, 32))
    except ValueError:
        pass
    else:
        raise AssertionError("anchor 8400 of 8400 accepted")


def _head(A, R=16, C=4):
    return np.zeros((4 * R + C, A), np.float32)


def pin_dfl_closed_forms(o):
    """Uniform bins decode to the middle bin (R-1)/2; a dominant bin to its
    index; two equal dominant bins to their midpoint.  Class arg-max takes the
    lower class on ties; the threshold is strict."""
    R, C, strides = 16, 4, (8, 16, 32)
    A = 8400
    head = _head(A, R, C)
    head[4 * R:] = -10.0
    # anchor 0 (stride 8, centre 4,4): uniform bins -> 7.5 on every side
    head[4 * R + 2, 0] = 1.0
    # anchor 6400 (stride 16, centre 8,8): left bin 3, top bin 0, right bin 15, bottom bins 2 and 6
    for side, b in ((0, 3), (1, 0), (2, 15)):
        head[side * R + b, 6400] = 100.0
    head[3 * R + 2, 6400] = 100.0
    head[3 * R + 6, 6400] = 100.0
    head[4 * R + 3, 6400] = 2.0            # ties between classes 1 and 3: class 1
    head[4 * R + 1, 6400] = 2.0
    # anchor 8399: logit exactly at the threshold -> not a candidate
    head[4 * R + 0, 8399] = 0.5
    d = o.decode(head, R, C, 640, 640, strides, 0.5)
    assert list(d["anchors"]) == [0, 6400], d["anchors"]
    assert np.array_equal(d["boxes"][0], np.float32([4 - 7.5 * 8, 4 - 7.5 * 8, 4 + 7.5 * 8, 4 + 7.5 * 8]))
    assert np.allclose(d["boxes"][1], [8 - 3 * 16, 8 - 0 * 16, 8 + 15 * 16, 8 + 4 * 16], atol=1e-4)
    assert list(d["classes"]) == [2, 1]
    assert d["logits"][0] == 1.0 and d["logits"][1] == 2.0
    assert abs(d["scores"][1] - 1 / (1 + math.exp(-2.0))) < 1e-7
    assert d["total"] == 2


def pin_dfl_torch(o):
    """Library special case: softmax expectation with torch in float64."""
    import torch
    head = synth.yolo_head(4, 1, 320, 192, num_classes=6, cls_mu=0.0)[0]
    R = 16
    d = o.decode(head, R, 6, 320, 192, synth.YOLO_STRIDES, -1e30)
    A = head.shape[1]
    assert d["total"] == A
    z = torch.from_numpy(head[:4 * R].astype(np.float64)).reshape(4, R, A)
    dist = (torch.softmax(z, dim=1) * torch.arange(R, dtype=torch.float64)[None, :, None]).sum(1)
    for n in range(0, A, 37):
        cx, cy, s = o.anchor(n, 320, 192, synth.YOLO_STRIDES)
        want = [cx - dist[0, n] * s, cy - dist[1, n] * s, cx + dist[2, n] * s, cy + dist[3, n] * s]
        assert np.allclose(d["boxes"][n], np.array(want, np.float64), rtol=0, atol=1e-4), n


def read_nms_cases():
    cases, cur = [], None
    for line in open(os.path.join(GOLDEN, "nms_hand.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        tok = line.split()
        if tok[0] == "case":
            cur = dict(thr=float(tok[1]), max_det=int(tok[2]), max_cand=int(tok[3]) if len(tok) > 3 else 1 << 30,
                       rows=[])
            cases.append(cur)
        elif tok[0] == "keep":
            cur["keep"] = [int(t) for t in tok[1:]]
        else:
            cur["rows"].append([float(t) for t in tok])
    return cases


def pin_nms_golden(o):
    for c in read_nms_cases():
        r = np.array(c["rows"], np.float64)
        keep = o.nms(r[:, :4], r[:, 4], r[:, 5].astype(np.int32), r[:, 6].astype(np.int32), c["thr"], c["max_det"],
                     c["max_cand"])
        assert [int(r[i, 6]) for i in keep] == c["keep"], (c, keep)


def _iou_above_f32(a, b, thr):
    f = np.float32
    iw = max(f(0), f(min(a[2], b[2])) - f(max(a[0], b[0])))
    ih = max(f(0), f(min(a[3], b[3])) - f(max(a[1], b[1])))
    inter = f(iw) * f(ih)
    ua = f(a[2] - a[0]) * f(a[3] - a[1])
    ub = f(b[2] - b[0]) * f(b[3] - b[1])
    return inter > f(thr) * f(f(ua + ub) - inter)


def pin_nms_bruteforce(o):
    """Greedy NMS returns the lexicographically first maximal conflict-free
    set (in score order): found here by enumerating every subset."""
    rng = np.random.default_rng(11)
    for trial in range(40):
        n = int(rng.integers(1, 11))
        xy = rng.integers(0, 12, size=(n, 2)).astype(np.float32)
        wh = rng.integers(1, 9, size=(n, 2)).astype(np.float32)
        boxes = np.concatenate([xy, xy + wh], 1).astype(np.float32)
        logits = rng.integers(0, 4, n).astype(np.float32)        # ties on purpose
        classes = rng.integers(0, 2, n).astype(np.int32)
        anchors = rng.permutation(50)[:n].astype(np.int32)
        thr = float(rng.choice([0.1, 0.3, 0.5, 0.7]))
        order = sorted(range(n), key=lambda i: (-logits[i], anchors[i]))
        conflict = [[classes[i] == classes[j] and i != j and _iou_above_f32(boxes[i], boxes[j], thr)
                     for j in range(n)] for i in range(n)]
        best = None
        for mask in range(1 << n):
            chosen = [order[p] for p in range(n) if mask >> (n - 1 - p) & 1]
            if any(conflict[a][b] for a in chosen for b in chosen):
                continue
            key = tuple(1 if (mask >> (n - 1 - p)) & 1 else 0 for p in range(n))
            if best is None or key > best[0]:
                best = (key, chosen)
        keep = o.nms(boxes, logits, classes, anchors, thr, 100)
        assert list(keep) == best[1], (trial, list(keep), best[1])


def pin_nan_and_signed_zero(o):
    """NaN class logits rank as -inf and -0 equals +0, as in the Top-K: a NaN
    class 0 does not hide a later class; an all-NaN anchor is no candidate;
    between -0 and +0 the lower class wins with its own bits.  In NMS a NaN
    logit sorts after every number, and -0 / +0 tie on the lower anchor."""
    R, C = 2, 4
    head = _head(21, R, C)          # 32x32 input: 16 + 4 + 1 anchors
    head[4 * R:] = -10.0
    head[4 * R + 0, 0] = np.nan
    head[4 * R + 2, 0] = 3.0
    head[4 * R:, 1] = np.nan
    head[4 * R + 1, 2] = -0.0
    head[4 * R + 3, 2] = 0.0
    d = o.decode(head, R, C, 32, 32, (8, 16, 32), -1.0)
    assert list(d["anchors"]) == [0, 2] and list(d["classes"]) == [2, 1]
    assert d["logits"][0] == 3.0 and np.signbit(d["logits"][1])
    box = np.float32([0, 0, 4, 4])
    # the same box four times, one class: only the first in order survives
    for logits, anchors, first in (([np.nan, -5.0], [0, 1], 1),       # NaN last although its anchor is lower
                                   ([0.0, -0.0], [3, 2], 1),          # -0 == +0: anchor 2 first
                                   ([-np.inf, np.nan], [5, 4], 1)):   # NaN == -inf: anchor 4 first
        keep = o.nms(np.stack([box, box]), np.float32(logits), np.int32([0, 0]), np.int32(anchors), 0.5, 10)
        assert list(keep) == [first], (logits, anchors, keep)


DET_PINS = [pin_anchor_geometry, pin_dfl_closed_forms, pin_dfl_torch, pin_nms_golden, pin_nms_bruteforce,
            pin_nan_and_signed_zero]
ALL_PINS = ALL_PINS + DET_PINS
