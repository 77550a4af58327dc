"""Plant plausible mistakes in copies of the oracle; the pins must catch each.

Each mutant is the oracle source with one textual change, compiled on the CPU
into a temporary library.  The test passes only when at least one pin in
tests/pins.py fails against the mutant.  This shows the pins are strong
enough that a dropped term, a wrong sign or index, or a transposed operand
in the oracle cannot go unnoticed.
"""
import os

import pytest

import oracle as oracle_pkg
import pins

MUTATIONS = [
    ("coordinate sign", "(2 * x + 1) * S - D", "(2 * x + 1) * S + D"),
    ("dropped half-pixel term", "(2 * x + 1) * S - D", "(2 * x) * S - D"),
    ("second tap index", "*i1 = clamp64(x0 + 1, 0, S - 1);", "*i1 = clamp64(x0, 0, S - 1);"),
    ("no clamp at the low edge", "*i0 = clamp64(x0, 0, S - 1);", "*i0 = clamp64(x0, -1, S - 1) < 0 ? 1 : x0;"),
    ("x weight on y", "const float t = p00 + wx * (p01 - p00);", "const float t = p00 + wy * (p01 - p00);"),
    ("y weight on x", "v = t + wy * (u - t);", "v = t + wx * (u - t);"),
    ("transposed neighbour", "const float p01 = (float)frame[j0 * row_stride + 3 * i1 + c];",
     "const float p01 = (float)frame[j1 * row_stride + 3 * i0 + c];"),
    ("channel swap in mean", "M[c] = (float)(255.0 * (double)mean[c]);",
     "M[c] = (float)(255.0 * (double)mean[2 - c]);"),
    ("mean sign", "if (norm == 0) out = (v - M[c]) * R[c];", "if (norm == 0) out = (v + M[c]) * R[c];"),
    ("frame stride", "src + (int64_t)b * frame_stride", "src + (int64_t)b * row_stride"),
    ("letterbox offset dropped", "axis_tap(x - left, src_w, nw, &i0, &i1, &wx);",
     "axis_tap(x, src_w, nw, &i0, &i1, &wx);"),
    ("odd padding side", "*left = (int)((DW - w) / 2);", "*left = (int)((DW - w + 1) / 2);"),
    ("box rounding", "h = (2 * SH * DW + SW) / (2 * SW);", "h = (SH * DW) / SW;"),
    ("tie to higher index", "return a.index < b.index;", "return a.index > b.index;"),
    ("NaN kept as NaN in the key", "v[(size_t)j].key = std::isnan(row[j]) ? ninf : row[j];",
     "v[(size_t)j].key = std::isnan(row[j]) ? 0.0f : row[j];"),
    ("NaN written out", "out_val[r * k + i] = std::isnan(row[j]) ? ninf : row[j];",
     "out_val[r * k + i] = row[j];"),
    ("signed zero lost", "out_val[r * k + i] = std::isnan(row[j]) ? ninf : row[j];",
     "out_val[r * k + i] = std::isnan(row[j]) ? ninf : row[j] + 0.0f;"),
    ("anchor centre offset", "*cx = ((double)(k % gw) + 0.5) * s;", "*cx = ((double)(k % gw)) * s;"),
    ("box sides swapped", "boxes[4 * n + 0] = (float)(cx - dist[0] * s);",
     "boxes[4 * n + 0] = (float)(cx - dist[2] * s);"),
    ("DFL bin index off by one", "e += w * i;", "e += w * (i + 1);"),
    ("class tie to higher index", "if (v > bl) { bl = v; best = c; }", "if (v >= bl) { bl = v; best = c; }"),
    ("threshold not strict", "if (!(bl > logit_thr)) continue;", "if (!(bl >= logit_thr)) continue;"),
    ("IoU test not strict", "return inter > thr * uni;", "return inter >= thr * uni;"),
    ("union without the overlap", "const float uni = area_a + area_b - inter;",
     "const float uni = area_a + area_b;"),
    ("class-agnostic suppression", "if (classes[j] == classes[i] && iou_above(", "if (iou_above("),
    ("NMS tie to higher anchor", "return anchor_idx[a] < anchor_idx[b];", "return anchor_idx[a] > anchor_idx[b];"),
    ("candidate cap ignored", "const int entering = std::min(n, max_cand);", "const int entering = n;"),
    ("NaN class logit taken raw", "float bl = nan_as_ninf(head[(int64_t)(4 * reg_max) * anchors + a]);",
     "float bl = head[(int64_t)(4 * reg_max) * anchors + a];"),
    ("NaN logit sorted raw", "const float la = nan_as_ninf(logits[a]), lb = nan_as_ninf(logits[b]);",
     "const float la = logits[a], lb = logits[b];"),
]


@pytest.fixture(scope="module")
def source():
    return open(oracle_pkg.SOURCE).read()


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(tmp_path, source, name, old, new):
    assert source.count(old) >= 1, f"mutation target not found: {old}"
    src = tmp_path / "mutant.cpp"
    src.write_text(source.replace(old, new, 1))
    lib = oracle_pkg.build(str(src), str(tmp_path / "libmutant.so"), force=True)
    mutant = oracle_pkg.Oracle(lib)
    failures = []
    for pin in pins.ALL_PINS:
        try:
            pin(mutant)
        except AssertionError:
            failures.append(pin.__name__)
            break
        except ValueError:
            failures.append(pin.__name__)
            break
    assert failures, f"no pin caught the mutation '{name}'"
