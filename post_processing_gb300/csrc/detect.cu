// detect.cu -- DFL box decode and class-aware greedy NMS of a YOLO-style
// detection head, sm_103a.
//
// What it computes (yolo.cu README, "Why is it this fast?": GPU-resident NMS,
// candidates sorted by a bitonic sort sized to the live candidate count, then
// greedy suppression, all inside the graph; "Inside WarpStream TRT", next
// steps: detection decode and NMS).  The readings where the pages give no
// formula are stated in include/ws.h next to ws_detect_desc.
//
// How:
//  * decode: one thread per anchor.  The class logits of consecutive anchors
//    are consecutive in memory, so the arg-max scan over the classes is
//    coalesced; only anchors whose best logit clears the threshold (about 2 %
//    of them) go on to the DFL softmax expectations and are appended to their
//    image's candidate buffer.
//  * NMS: one block per image.  If the image has more than max_cand
//    candidates, a radix select on the 64-bit keys (logit order bits, then
//    the complemented anchor) keeps the best max_cand.  The survivors are
//    bitonic-sorted in shared memory, every pair's suppression test (same
//    class, IoU > threshold) is evaluated in parallel into a bit matrix, and
//    one warp walks the sorted list keeping a running "removed" bit set, so
//    the greedy pass costs one step per candidate.  The IoU test is FP32 with
//    every operation rounded separately (no fused multiply-add), so given the
//    same boxes the decisions are exactly those of the definition.
#include <algorithm>
#include <cmath>

#include "ws_internal.cuh"

namespace ws {
namespace {

constexpr int kDecodeThreads = 256;
constexpr int kNmsThreads = 512;
constexpr int kMaxCand = 1024;
constexpr int kMaxLevels = 4;
constexpr unsigned kFull = 0xffffffffu;

struct DetParams {
    const float* head;
    long long A;
    int R, C, ch;                     // ch = 4 R + C
    int nlevels;
    int stride[kMaxLevels];
    int gw[kMaxLevels];
    long long off[kMaxLevels + 1];    // first anchor of each level
    float logit_thr, iou_thr;
    int max_cand, max_det;
    ws_candidate* cand;               // [batch][A]
    int* count;                       // [batch]
    ws_detection* out;                // [batch][max_det]
    int* out_count;                   // [batch]
    // NMS shared-memory layout
    int P;                            // power of two >= max_cand
    int W;                            // 64-bit words per mask row
    int off_idx, off_box, off_cls, off_logit, off_anchor, off_mask, off_keep, off_hist;
};

__device__ __forceinline__ uint32_t order_bits(float f) {
    const uint32_t b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned long long cand_key(const ws_candidate& c) {
    return ((unsigned long long)order_bits(c.logit) << 32) | (uint32_t)(~(uint32_t)c.anchor);
}

__global__ void __launch_bounds__(kDecodeThreads) detect_decode_kernel(const __grid_constant__ DetParams p) {
    const int b = blockIdx.y;
    const long long a = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (a >= p.A) return;
    const float* hb = p.head + (size_t)b * p.ch * p.A;
    const float* cl = hb + (size_t)(4 * p.R) * p.A + a;
    float best = __ldg(cl);
    int bc = 0;
    for (int c = 1; c < p.C; ++c) {
        const float v = __ldg(cl + (size_t)c * p.A);
        if (v > best) {
            best = v;
            bc = c;
        }
    }
    if (!(best > p.logit_thr)) return;

    int l = 0;
    while (l + 1 < p.nlevels && a >= p.off[l + 1]) ++l;
    const long long k = a - p.off[l];
    const float s = (float)p.stride[l];
    const float cx = ((float)(k % p.gw[l]) + 0.5f) * s;
    const float cy = ((float)(k / p.gw[l]) + 0.5f) * s;
    float dist[4];
#pragma unroll
    for (int side = 0; side < 4; ++side) {
        const float* z = hb + (size_t)(side * p.R) * p.A + a;
        float m = -INFINITY;
        for (int i = 0; i < p.R; ++i) m = fmaxf(m, __ldg(z + (size_t)i * p.A));
        float zs = 0.f, es = 0.f;
        for (int i = 0; i < p.R; ++i) {
            const float w = expf(__ldg(z + (size_t)i * p.A) - m);
            zs += w;
            es += w * (float)i;
        }
        dist[side] = es / zs;
    }
    ws_candidate c;
    c.x1 = cx - dist[0] * s;
    c.y1 = cy - dist[1] * s;
    c.x2 = cx + dist[2] * s;
    c.y2 = cy + dist[3] * s;
    c.logit = best;
    c.cls = bc;
    c.anchor = (int32_t)a;
    c.pad_ = 0;
    const int slot = atomicAdd(&p.count[b], 1);
    if (slot < p.A) p.cand[(size_t)b * p.A + slot] = c;
}

// IoU(a, b) > thr, as inter > thr * union, every operation rounded on its own.
__device__ __forceinline__ bool iou_above(const float4 a, const float4 b, float thr) {
    const float iw = fmaxf(0.f, __fsub_rn(fminf(a.z, b.z), fmaxf(a.x, b.x)));
    const float ih = fmaxf(0.f, __fsub_rn(fminf(a.w, b.w), fmaxf(a.y, b.y)));
    const float inter = __fmul_rn(iw, ih);
    const float area_a = __fmul_rn(__fsub_rn(a.z, a.x), __fsub_rn(a.w, a.y));
    const float area_b = __fmul_rn(__fsub_rn(b.z, b.x), __fsub_rn(b.w, b.y));
    const float uni = __fsub_rn(__fadd_rn(area_a, area_b), inter);
    return inter > __fmul_rn(thr, uni);
}

__global__ void __launch_bounds__(kNmsThreads) detect_nms_kernel(const __grid_constant__ DetParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long* s_key = reinterpret_cast<unsigned long long*>(smem);   // [P]
    int* s_idx = reinterpret_cast<int*>(smem + p.off_idx);                     // [P] candidate slot
    float4* s_box = reinterpret_cast<float4*>(smem + p.off_box);                // [max_cand] sorted
    int* s_cls = reinterpret_cast<int*>(smem + p.off_cls);
    float* s_logit = reinterpret_cast<float*>(smem + p.off_logit);
    int* s_anchor = reinterpret_cast<int*>(smem + p.off_anchor);
    unsigned long long* s_mask = reinterpret_cast<unsigned long long*>(smem + p.off_mask);  // [max_cand][W]
    int* s_keep = reinterpret_cast<int*>(smem + p.off_keep);
    uint32_t* s_hist = reinterpret_cast<uint32_t*>(smem + p.off_hist);         // [256] + 4 words
    uint32_t* s_misc = s_hist + 256;

    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const ws_candidate* cb = p.cand + (size_t)b * p.A;
    const int n = (int)min((long long)p.count[b], p.A);
    const int m = min(n, p.max_cand);
    if (tid == 0) s_misc[0] = 0;
    for (int i = tid; i < p.P; i += kNmsThreads) s_key[i] = 0ull;   // padding sorts last
    __syncthreads();

    // 1. the best m candidates' keys into shared memory
    unsigned long long kth = 0;
    if (n > m) {
        // exact radix select of the m-th largest key (8 passes of 8 bits)
        unsigned long long prefix = 0, mask = 0;
        uint32_t remaining = (uint32_t)m;
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += kNmsThreads) s_hist[i] = 0;
            __syncthreads();
            for (int i = tid; i < n; i += kNmsThreads) {
                const unsigned long long key = cand_key(cb[i]);
                if ((key & mask) == prefix) atomicAdd(&s_hist[(key >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (tid == 0) {
                uint32_t acc = 0;
                for (int d = 255; d >= 0; --d) {
                    if (acc + s_hist[d] >= remaining) {
                        s_misc[1] = (uint32_t)d;
                        s_misc[2] = remaining - acc;
                        break;
                    }
                    acc += s_hist[d];
                }
            }
            __syncthreads();
            prefix |= (unsigned long long)s_misc[1] << shift;
            mask |= 0xffull << shift;
            remaining = s_misc[2];
            __syncthreads();
        }
        kth = prefix;   // keys are unique (anchors are), so exactly m are >= kth
    }
    for (int i = tid; i < n; i += kNmsThreads) {
        const unsigned long long key = cand_key(cb[i]);
        if (key >= kth) {
            const uint32_t pos = atomicAdd(&s_misc[0], 1u);
            if (pos < (uint32_t)m) {
                s_key[pos] = key;
                s_idx[pos] = i;
            }
        }
    }
    __syncthreads();

    // 2. bitonic sort, descending (padding keys 0 go last)
    for (int k = 2; k <= p.P; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < p.P; i += kNmsThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const unsigned long long a = s_key[i], c = s_key[ixj];
                    const bool desc = (i & k) == 0;
                    if (desc ? (a < c) : (a > c)) {
                        s_key[i] = c;
                        s_key[ixj] = a;
                        const int t = s_idx[i];
                        s_idx[i] = s_idx[ixj];
                        s_idx[ixj] = t;
                    }
                }
            }
            __syncthreads();
        }
    }

    // 3. the sorted candidates
    for (int q = tid; q < m; q += kNmsThreads) {
        const ws_candidate c = cb[s_idx[q]];
        s_box[q] = make_float4(c.x1, c.y1, c.x2, c.y2);
        s_cls[q] = c.cls;
        s_logit[q] = c.logit;
        s_anchor[q] = c.anchor;
    }
    __syncthreads();

    // 4. suppression bits: word w of row i holds j = 64 w + bit, j > i
    const int W = p.W;
    for (int t = tid; t < m * W; t += kNmsThreads) {
        const int i = t / W, w = t - i * W;
        const float4 bi = s_box[i];
        const int ci = s_cls[i];
        unsigned long long bits = 0;
        const int j0 = w * 64;
        const int j1 = min(m, j0 + 64);
        for (int j = max(j0, i + 1); j < j1; ++j)
            if (s_cls[j] == ci && iou_above(bi, s_box[j], p.iou_thr)) bits |= 1ull << (j - j0);
        s_mask[(size_t)i * W + w] = bits;
    }
    __syncthreads();

    // 5. greedy walk by one warp; lane w holds removed-word w
    if (warp == 0) {
        unsigned long long rem = 0;
        int nk = 0;
        for (int i = 0; i < m && nk < p.max_det; ++i) {
            const unsigned long long word = __shfl_sync(kFull, rem, i >> 6);
            if (!((word >> (i & 63)) & 1ull)) {
                if (lane == 0) s_keep[nk] = i;
                ++nk;
                if (lane < W) rem |= s_mask[(size_t)i * W + lane];
            }
        }
        if (lane == 0) s_misc[3] = (uint32_t)nk;
    }
    __syncthreads();

    // 6. detections in keep order
    const int nk = (int)s_misc[3];
    for (int q = tid; q < nk; q += kNmsThreads) {
        const int i = s_keep[q];
        ws_detection d;
        const float4 bx = s_box[i];
        d.x1 = bx.x;
        d.y1 = bx.y;
        d.x2 = bx.z;
        d.y2 = bx.w;
        d.score = 1.0f / (1.0f + expf(-s_logit[i]));
        d.cls = s_cls[i];
        d.anchor = s_anchor[i];
        d.pad_ = 0;
        p.out[(size_t)b * p.max_det + q] = d;
    }
    if (tid == 0) {
        p.out_count[b] = nk;
        p.count[b] = 0;   // ready for the next decode / replay
    }
}

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

ws_status fill_params(const ws_detect_desc* d, int32_t batch, DetParams& p) {
    if (!d) return fail(WS_ERR_INVALID_ARGUMENT, "descriptor is NULL");
    if (batch < 1 || batch > 65535) return fail(WS_ERR_INVALID_ARGUMENT, "batch %d outside 1..65535", batch);
    if (d->in_w < 1 || d->in_h < 1) return fail(WS_ERR_INVALID_ARGUMENT, "input size %dx%d", d->in_w, d->in_h);
    if (d->nlevels < 1 || d->nlevels > kMaxLevels)
        return fail(WS_ERR_INVALID_ARGUMENT, "levels %d outside 1..%d", d->nlevels, kMaxLevels);
    if (d->reg_max < 1 || d->reg_max > 32) return fail(WS_ERR_INVALID_ARGUMENT, "reg_max %d outside 1..32", d->reg_max);
    if (d->num_classes < 1 || d->num_classes > 4096)
        return fail(WS_ERR_INVALID_ARGUMENT, "num_classes %d outside 1..4096", d->num_classes);
    if (d->max_cand < 1 || d->max_cand > kMaxCand)
        return fail(WS_ERR_INVALID_ARGUMENT, "max_cand %d outside 1..%d", d->max_cand, kMaxCand);
    if (d->max_det < 1 || d->max_det > d->max_cand)
        return fail(WS_ERR_INVALID_ARGUMENT, "max_det %d outside 1..max_cand", d->max_det);
    if (!std::isfinite(d->iou_thr) || std::isnan(d->logit_thr))
        return fail(WS_ERR_INVALID_ARGUMENT, "thresholds must be numbers");
    p = DetParams{};
    long long A = 0;
    for (int l = 0; l < d->nlevels; ++l) {
        const int s = d->strides[l];
        if (s < 1 || d->in_w % s || d->in_h % s)
            return fail(WS_ERR_INVALID_ARGUMENT, "stride %d does not divide %dx%d", s, d->in_w, d->in_h);
        p.stride[l] = s;
        p.gw[l] = d->in_w / s;
        p.off[l] = A;
        A += (long long)(d->in_w / s) * (d->in_h / s);
    }
    p.off[d->nlevels] = A;
    if (A > (1LL << 24)) return fail(WS_ERR_INVALID_ARGUMENT, "%lld anchors > 2^24", A);
    p.A = A;
    p.nlevels = d->nlevels;
    p.R = d->reg_max;
    p.C = d->num_classes;
    p.ch = 4 * d->reg_max + d->num_classes;
    p.logit_thr = d->logit_thr;
    p.iou_thr = d->iou_thr;
    p.max_cand = d->max_cand;
    p.max_det = d->max_det;
    p.P = 1;
    while (p.P < d->max_cand) p.P <<= 1;
    p.W = (d->max_cand + 63) / 64;
    size_t o = (size_t)p.P * 8;
    p.off_idx = (int)o;        o = align16(o + (size_t)p.P * 4);
    p.off_box = (int)o;        o = align16(o + (size_t)d->max_cand * 16);
    p.off_cls = (int)o;        o = align16(o + (size_t)d->max_cand * 4);
    p.off_logit = (int)o;      o = align16(o + (size_t)d->max_cand * 4);
    p.off_anchor = (int)o;     o = align16(o + (size_t)d->max_cand * 4);
    p.off_mask = (int)o;       o = align16(o + (size_t)d->max_cand * p.W * 8);
    p.off_keep = (int)o;       o = align16(o + (size_t)d->max_cand * 4);
    p.off_hist = (int)o;
    return WS_OK;
}

size_t nms_smem(const DetParams& p) { return (size_t)p.off_hist + (256 + 4) * 4; }

size_t det_workspace(const DetParams& p, int32_t batch) {
    return (size_t)(batch * 4 + 255) / 256 * 256 + (size_t)batch * p.A * sizeof(ws_candidate);
}

bool g_nms_attr_set[64];

ws_status launch_decode(const DetParams& p, int32_t batch, cudaStream_t stream) {
    const dim3 grid((unsigned)((p.A + kDecodeThreads - 1) / kDecodeThreads), (unsigned)batch);
    detect_decode_kernel<<<grid, kDecodeThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return WS_OK;
}

ws_status launch_nms(const DetParams& p, int32_t batch, cudaStream_t stream) {
    int dev;
    const DeviceInfo* info;
    ws_status st = current_device_info(&dev, &info);
    if (st != WS_OK) return st;
    const size_t smem = nms_smem(p);
    if (smem > (size_t)info->max_smem_optin) return fail(WS_ERR_UNSUPPORTED, "NMS needs %zu bytes of shared memory", smem);
    if (!g_nms_attr_set[dev]) {
        WS_TRY_CUDA(cudaFuncSetAttribute(detect_nms_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info->max_smem_optin));
        g_nms_attr_set[dev] = true;
    }
    detect_nms_kernel<<<batch, kNmsThreads, smem, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "NMS launch");
    return WS_OK;
}

}  // namespace
}  // namespace ws

extern "C" {

ws_status ws_detect_validate(const ws_detect_desc* desc, int32_t batch, int64_t* anchors) {
    ws::clear_error();
    ws::DetParams p;
    ws_status st = ws::fill_params(desc, batch, p);
    if (st == WS_OK && anchors) *anchors = p.A;
    return st;
}

ws_status ws_detect_workspace_bytes(const ws_detect_desc* desc, int32_t batch, size_t* bytes) {
    ws::clear_error();
    if (!bytes) return ws::fail(WS_ERR_INVALID_ARGUMENT, "bytes is NULL");
    ws::DetParams p;
    ws_status st = ws::fill_params(desc, batch, p);
    if (st != WS_OK) return st;
    *bytes = ws::det_workspace(p, batch);
    return WS_OK;
}

ws_status ws_detect_workspace_init(void* workspace, size_t bytes, cudaStream_t stream) {
    ws::clear_error();
    if (bytes == 0) return WS_OK;
    if (!workspace) return ws::fail(WS_ERR_INVALID_ARGUMENT, "workspace is NULL");
    WS_TRY_CUDA(cudaMemsetAsync(workspace, 0, bytes, stream));
    return WS_OK;
}

ws_status ws_detect_decode(const ws_detect_desc* desc, const float* head, int32_t batch, ws_candidate* cand,
                           int32_t* count, cudaStream_t stream) {
    ws::clear_error();
    ws::DetParams p;
    ws_status st = ws::fill_params(desc, batch, p);
    if (st != WS_OK) return st;
    if (!head || !cand || !count) return ws::fail(WS_ERR_INVALID_ARGUMENT, "head, cand or count is NULL");
    p.head = head;
    p.cand = cand;
    p.count = count;
    return ws::launch_decode(p, batch, stream);
}

ws_status ws_detect_nms(const ws_detect_desc* desc, ws_candidate* cand, int32_t* count, int32_t batch,
                        ws_detection* out, int32_t* out_count, cudaStream_t stream) {
    ws::clear_error();
    ws::DetParams p;
    ws_status st = ws::fill_params(desc, batch, p);
    if (st != WS_OK) return st;
    if (!cand || !count || !out || !out_count)
        return ws::fail(WS_ERR_INVALID_ARGUMENT, "cand, count, out or out_count is NULL");
    p.cand = cand;
    p.count = count;
    p.out = out;
    p.out_count = out_count;
    return ws::launch_nms(p, batch, stream);
}

ws_status ws_detect(const ws_detect_desc* desc, const float* head, int32_t batch, ws_detection* out,
                    int32_t* out_count, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    ws::clear_error();
    ws::DetParams p;
    ws_status st = ws::fill_params(desc, batch, p);
    if (st != WS_OK) return st;
    if (!head || !out || !out_count) return ws::fail(WS_ERR_INVALID_ARGUMENT, "head, out or out_count is NULL");
    const size_t need = ws::det_workspace(p, batch);
    if (!workspace || workspace_bytes < need)
        return ws::fail(WS_ERR_INVALID_ARGUMENT, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if ((uintptr_t)workspace % 256 != 0) return ws::fail(WS_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");
    p.head = head;
    p.count = static_cast<int*>(workspace);
    p.cand = reinterpret_cast<ws_candidate*>(static_cast<char*>(workspace) + (size_t)(batch * 4 + 255) / 256 * 256);
    p.out = out;
    p.out_count = out_count;
    if ((st = ws::launch_decode(p, batch, stream)) != WS_OK) return st;
    return ws::launch_nms(p, batch, stream);
}

}  // extern "C"
