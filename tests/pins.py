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
