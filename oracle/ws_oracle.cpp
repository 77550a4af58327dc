// ws_oracle.cpp -- the oracle: a plain, slow, obviously correct CPU definition
// of the fused RGB8 -> FP32 NCHW preprocess, the exact Top-K, and the
// detection decode + greedy NMS.
//
// TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
// CPU-baseline leg load this library.  It shares no code, header, table or
// helper with the CUDA path, and the CUDA path never calls it.
//
// Built with -O2 -ffp-contract=off (no fused multiply-add, no fast-math), so
// every float operation below is one IEEE-754 rounding, in the order written.
//
// What it follows:
//  * "Inside WarpStream TRT", fused-preprocessing section and its data-flow
//    figure: one destination pixel at a time, a centre-aligned source
//    coordinate, the four bilinear neighbours of each RGB channel,
//    interpolation, normalisation by a per-channel mean and inverse standard
//    deviation, and a store to destination[channel][y][x] of the NCHW tensor.
//  * yolo.cu README, "Two ways to use it" (embedded C API): the same
//    preprocess as an aspect-preserving letterbox into the network input.
//  * "Inside WarpStream TRT", Top-K section: exact selection of the K largest
//    logits, ties to the lower class index, NaN taken as negative infinity.
//
// Readings where the pages are silent (each is listed in the design notes):
//  * half-pixel centres: source coordinate = (x + 1/2) * S / D - 1/2, held as
//    the exact rational num/den with num = (2x+1)S - D and den = 2D; the
//    fractional weight is one correctly rounded float division rem/den;
//  * clamp-to-edge: both neighbour indices are clamped into [0, S-1];
//  * no antialias prefilter on downscale (only the four neighbours);
//  * normalisation in byte units: out = (v - M_c) * R_c with
//    M_c = float(255 * mean_c) and R_c = float(1 / (255 * std_c)), both
//    evaluated in double and rounded once; the "scale" mode is out = v * scale;
//  * letterbox: the inner box keeps the aspect ratio, its short side is the
//    round-half-up integer of the scaled length (at least 1), it is centred
//    with the odd pixel of padding going to the bottom / right, sampling
//    inside the box uses S / (box size), and the padding value is stored as a
//    byte value that goes through the same normalisation;
//  * Top-K output is in rank order; an output value is the input's own bits
//    (so -0.0 stays -0.0) except that NaN is written as -inf.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <algorithm>
#include <vector>

namespace {

// Floor division for a positive divisor.
int64_t floor_div(int64_t a, int64_t b) {
    int64_t q = a / b;
    if ((a % b != 0) && (a < 0)) q -= 1;
    return q;
}

int64_t clamp64(int64_t v, int64_t lo, int64_t hi) {
    return v < lo ? lo : (v > hi ? hi : v);
}

// One axis of the bilinear tap: destination coordinate x in [0, D) of a box
// of D pixels, sampled from S source pixels.
void axis_tap(int64_t x, int64_t S, int64_t D, int64_t* i0, int64_t* i1, float* w) {
    const int64_t num = (2 * x + 1) * S - D;
    const int64_t den = 2 * D;
    const int64_t x0 = floor_div(num, den);
    const int64_t rem = num - x0 * den;       // in [0, den)
    *w = (float)rem / (float)den;
    *i0 = clamp64(x0, 0, S - 1);
    *i1 = clamp64(x0 + 1, 0, S - 1);
}

void inner_box(int sw, int sh, int dw, int dh, int letterbox,
               int* nw, int* nh, int* left, int* top) {
    if (!letterbox) {
        *nw = dw; *nh = dh; *left = 0; *top = 0;
        return;
    }
    const int64_t SW = sw, SH = sh, DW = dw, DH = dh;
    int64_t w, h;
    if (DW * SH <= DH * SW) {          // width-limited: scale = DW / SW
        w = DW;
        h = (2 * SH * DW + SW) / (2 * SW);
    } else {                           // height-limited: scale = DH / SH
        h = DH;
        w = (2 * SW * DH + SH) / (2 * SH);
    }
    if (w < 1) w = 1;
    if (h < 1) h = 1;
    *nw = (int)w; *nh = (int)h;
    *left = (int)((DW - w) / 2);
    *top = (int)((DH - h) / 2);
}

struct Cand {
    float key;      // the value, with NaN replaced by -inf
    int64_t index;
};

}  // namespace

extern "C" {

// Inner box of the destination that the source image covers.
// Returns 0, or -1 on invalid sizes.
int oracle_inner_box(int src_w, int src_h, int dst_w, int dst_h, int letterbox,
                     int* nw, int* nh, int* left, int* top) {
    if (src_w <= 0 || src_h <= 0 || dst_w <= 0 || dst_h <= 0) return -1;
    inner_box(src_w, src_h, dst_w, dst_h, letterbox, nw, nh, left, top);
    return 0;
}

// Taps (i0, i1, weight) of destination coordinate x of a D-pixel box sampled
// from S source pixels.
int oracle_axis_tap(int64_t x, int64_t S, int64_t D, int64_t* i0, int64_t* i1, float* w) {
    if (S <= 0 || D <= 0 || x < 0 || x >= D) return -1;
    axis_tap(x, S, D, i0, i1, w);
    return 0;
}

// Fused preprocess.
//   src:   batch frames of interleaved RGB8; byte (b, j, i, c) lives at
//          src[b * frame_stride + j * row_stride + 3 * i + c]
//   dst:   float [batch][3][dst_h][dst_w]
//   letterbox: 0 = stretch to the whole destination, 1 = letterbox
//   norm:  0 = mean/std, 1 = scale
// Returns 0, or -1 on invalid arguments.
int oracle_preprocess(const uint8_t* src, int64_t row_stride, int64_t frame_stride,
                      int src_w, int src_h, int batch,
                      int dst_w, int dst_h, int letterbox, int pad_value,
                      int norm, const float* mean, const float* stdv, float scale,
                      float* dst) {
    if (!src || !dst || src_w <= 0 || src_h <= 0 || dst_w <= 0 || dst_h <= 0 || batch <= 0)
        return -1;
    if (row_stride < 3LL * src_w || frame_stride < row_stride * src_h) return -1;
    if (pad_value < 0 || pad_value > 255) return -1;

    float M[3], R[3];
    for (int c = 0; c < 3; ++c) {
        if (norm == 0) {
            M[c] = (float)(255.0 * (double)mean[c]);
            R[c] = (float)(1.0 / (255.0 * (double)stdv[c]));
        } else {
            M[c] = 0.0f;
            R[c] = scale;
        }
    }

    int nw, nh, left, top;
    inner_box(src_w, src_h, dst_w, dst_h, letterbox, &nw, &nh, &left, &top);

    for (int b = 0; b < batch; ++b) {
        const uint8_t* frame = src + (int64_t)b * frame_stride;
        for (int c = 0; c < 3; ++c) {
            for (int y = 0; y < dst_h; ++y) {
                for (int x = 0; x < dst_w; ++x) {
                    float v;
                    const bool inside = (x >= left && x < left + nw && y >= top && y < top + nh);
                    if (!inside) {
                        v = (float)pad_value;
                    } else {
                        int64_t i0, i1, j0, j1;
                        float wx, wy;
                        axis_tap(x - left, src_w, nw, &i0, &i1, &wx);
                        axis_tap(y - top, src_h, nh, &j0, &j1, &wy);
                        const float p00 = (float)frame[j0 * row_stride + 3 * i0 + c];
                        const float p01 = (float)frame[j0 * row_stride + 3 * i1 + c];
                        const float p10 = (float)frame[j1 * row_stride + 3 * i0 + c];
                        const float p11 = (float)frame[j1 * row_stride + 3 * i1 + c];
                        const float t = p00 + wx * (p01 - p00);
                        const float u = p10 + wx * (p11 - p10);
                        v = t + wy * (u - t);
                    }
                    float out;
                    if (norm == 0) out = (v - M[c]) * R[c];
                    else           out = v * R[c];
                    dst[(((int64_t)b * 3 + c) * dst_h + y) * dst_w + x] = out;
                }
            }
        }
    }
    return 0;
}

// Exact Top-K of each row of x [rows][cols]: the K entries with the largest
// values, ties to the lower index, NaN ordered as -inf; written in rank order.
// Returns 0, or -1 on invalid arguments.
int oracle_topk(const float* x, int64_t rows, int64_t cols, int k,
                float* out_val, int32_t* out_idx) {
    if (!x || !out_val || !out_idx || rows <= 0 || cols <= 0 || k <= 0 || k > cols ||
        cols > 2147483647LL)
        return -1;
    const float ninf = -std::numeric_limits<float>::infinity();
    std::vector<Cand> v((size_t)cols);
    for (int64_t r = 0; r < rows; ++r) {
        const float* row = x + r * cols;
        for (int64_t j = 0; j < cols; ++j) {
            v[(size_t)j].key = std::isnan(row[j]) ? ninf : row[j];
            v[(size_t)j].index = j;
        }
        std::sort(v.begin(), v.end(), [](const Cand& a, const Cand& b) {
            if (a.key > b.key) return true;
            if (a.key < b.key) return false;
            return a.index < b.index;     // equal values (+0 == -0): lower index first
        });
        for (int i = 0; i < k; ++i) {
            const int64_t j = v[(size_t)i].index;
            out_idx[r * k + i] = (int32_t)j;
            out_val[r * k + i] = std::isnan(row[j]) ? ninf : row[j];
        }
    }
    return 0;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Detection decode and non-maximum suppression.
//
// What it follows: yolo.cu README ("Why is it this fast?", GPU-resident NMS,
// and the end-to-end pipeline: DFL decode, then NMS with a bitonic sort sized
// to the live candidate count and greedy suppression) and "Inside WarpStream
// TRT" (next steps: detection decode and NMS).  The pages name the steps but
// not their formulas; the readings taken:
//  * head layout [batch][4 * R + C][A] (R DFL bins per box side, C classes,
//    A anchors), FP32 logits;
//  * anchors run level by level (strides given, e.g. 8, 16, 32), row-major
//    within a level; anchor (x, y) of a level with stride s has its centre
//    at ((x + 1/2) s, (y + 1/2) s) in input pixels;
//  * DFL: the distance of each side (left, top, right, bottom) is the
//    expectation sum_i i * softmax(z)_i over its R bins, in units of the
//    stride; box = (cx - l s, cy - t s, cx + r s, cy + b s);
//  * the class is the arg-max of the class logits (lower class on ties, NaN
//    ranked as -inf and -0 equal to +0, as in the Top-K); an
//    anchor is a candidate when that logit exceeds a logit threshold (the
//    caller passes logit(conf) so the decision needs no transcendental); its
//    score is the logistic of the logit;
//  * greedy NMS per image, class-aware: candidates in order of logit
//    (higher first, the same NaN / -0 rule, lower anchor on ties), of which only the first max_cand
//    enter (a per-image cap, this library's reading); a candidate is kept unless an
//    already kept box of the same class has IoU > iou_thr with it, tested as
//    inter > iou_thr * union in FP32 with the operation order below; at most
//    max_det are kept.
// ---------------------------------------------------------------------------

namespace {

float nan_as_ninf(float v) { return std::isnan(v) ? -std::numeric_limits<float>::infinity() : v; }

// IoU test in FP32 (no fused operations: the file is built with
// -ffp-contract=off).  Boxes are x1, y1, x2, y2.
bool iou_above(const float* a, const float* b, float thr) {
    const float iw = std::max(0.0f, std::min(a[2], b[2]) - std::max(a[0], b[0]));
    const float ih = std::max(0.0f, std::min(a[3], b[3]) - std::max(a[1], b[1]));
    const float inter = iw * ih;
    const float area_a = (a[2] - a[0]) * (a[3] - a[1]);
    const float area_b = (b[2] - b[0]) * (b[3] - b[1]);
    const float uni = area_a + area_b - inter;
    return inter > thr * uni;
}

}  // namespace

extern "C" {

// Anchor centre and stride of anchor a for an input of in_w x in_h pixels
// and the given strides.  Returns 0, or -1 if a is out of range.
int oracle_anchor(int64_t a, int in_w, int in_h, const int* strides, int nlevels,
                  double* cx, double* cy, int* stride) {
    int64_t off = 0;
    for (int l = 0; l < nlevels; ++l) {
        const int s = strides[l];
        const int64_t gw = in_w / s, gh = in_h / s;
        if (a < off + gw * gh) {
            const int64_t k = a - off;
            *cx = ((double)(k % gw) + 0.5) * s;
            *cy = ((double)(k / gw) + 0.5) * s;
            *stride = s;
            return 0;
        }
        off += gw * gh;
    }
    return -1;
}

// Decode of one image: candidates (box, logit, score, class, anchor) for every
// anchor whose best class logit exceeds logit_thr, in anchor order.
// Returns the number of candidates written (at most max_cand; the true count
// goes to *total), or -1 on invalid arguments.  DFL arithmetic in double.
int oracle_decode(const float* head, int64_t anchors, int reg_max, int num_classes,
                  int in_w, int in_h, const int* strides, int nlevels, float logit_thr,
                  int max_cand, float* boxes, float* logits, float* scores, int32_t* classes,
                  int32_t* anchor_idx, int* total) {
    if (!head || anchors <= 0 || reg_max <= 0 || num_classes <= 0 || max_cand < 0) return -1;
    int64_t count_levels = 0;
    for (int l = 0; l < nlevels; ++l) count_levels += (int64_t)(in_w / strides[l]) * (in_h / strides[l]);
    if (count_levels != anchors) return -1;
    int n = 0, all = 0;
    for (int64_t a = 0; a < anchors; ++a) {
        // arg-max with NaN ranked as -inf (as in the Top-K), the first class on ties
        int best = 0;
        float bl = nan_as_ninf(head[(int64_t)(4 * reg_max) * anchors + a]);
        for (int c = 1; c < num_classes; ++c) {
            const float v = nan_as_ninf(head[(int64_t)(4 * reg_max + c) * anchors + a]);
            if (v > bl) { bl = v; best = c; }
        }
        if (!(bl > logit_thr)) continue;
        ++all;
        if (n >= max_cand) continue;
        double cx, cy;
        int s;
        oracle_anchor(a, in_w, in_h, strides, nlevels, &cx, &cy, &s);
        double dist[4];
        for (int side = 0; side < 4; ++side) {
            double m = -1e300;
            for (int i = 0; i < reg_max; ++i) m = std::max(m, (double)head[(int64_t)(side * reg_max + i) * anchors + a]);
            double z = 0.0, e = 0.0;
            for (int i = 0; i < reg_max; ++i) {
                const double w = std::exp((double)head[(int64_t)(side * reg_max + i) * anchors + a] - m);
                z += w;
                e += w * i;
            }
            dist[side] = e / z;
        }
        boxes[4 * n + 0] = (float)(cx - dist[0] * s);
        boxes[4 * n + 1] = (float)(cy - dist[1] * s);
        boxes[4 * n + 2] = (float)(cx + dist[2] * s);
        boxes[4 * n + 3] = (float)(cy + dist[3] * s);
        logits[n] = bl;
        scores[n] = (float)(1.0 / (1.0 + std::exp(-(double)bl)));
        classes[n] = best;
        anchor_idx[n] = (int32_t)a;
        ++n;
    }
    if (total) *total = all;
    return n;
}

// Greedy class-aware NMS of n candidates (any order), of which the first
// max_cand in sorted order enter.  Writes the indices
// (into the candidate arrays) of the kept boxes, in keep order; returns how
// many were kept (at most max_det), or -1 on invalid arguments.
int oracle_nms(const float* boxes, const float* logits, const int32_t* classes, const int32_t* anchor_idx,
               int n, float iou_thr, int max_cand, int max_det, int32_t* keep) {
    if (n < 0 || max_det < 0 || max_cand < 0 ||
        (n > 0 && (!boxes || !logits || !classes || !anchor_idx || !keep)))
        return -1;
    std::vector<int> order((size_t)n);
    for (int i = 0; i < n; ++i) order[(size_t)i] = i;
    // higher logit first (NaN as -inf, -0 equal to +0), then the lower anchor
    std::sort(order.begin(), order.end(), [&](int a, int b) {
        const float la = nan_as_ninf(logits[a]), lb = nan_as_ninf(logits[b]);
        if (la > lb) return true;
        if (la < lb) return false;
        return anchor_idx[a] < anchor_idx[b];
    });
    int kept = 0;
    const int entering = std::min(n, max_cand);
    for (int oi = 0; oi < entering && kept < max_det; ++oi) {
        const int i = order[(size_t)oi];
        bool ok = true;
        for (int q = 0; q < kept && ok; ++q) {
            const int j = keep[q];
            if (classes[j] == classes[i] && iou_above(boxes + 4 * j, boxes + 4 * i, iou_thr)) ok = false;
        }
        if (ok) keep[kept++] = i;
    }
    return kept;
}

}  // extern "C"
