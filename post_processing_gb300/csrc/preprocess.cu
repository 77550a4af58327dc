// preprocess.cu -- fused RGB8 -> FP32 NCHW preprocess for sm_103a.
//
// What it computes ("Inside WarpStream TRT", fused-preprocessing section and
// its data-flow figure; yolo.cu README, "Two ways to use it", for the
// letterbox): every destination pixel takes a centre-aligned bilinear sample
// of the interleaved RGB8 frame, each channel is normalised by a mean and an
// inverse standard deviation (or one scale), and the value goes straight into
// its channel plane of the NCHW tensor.  Nothing else is materialised.
//
// How (GB300 design, not the page's one-thread-per-pixel gather):
//  * Staged kernel (16-byte aligned rows).  A block owns one frame and a band
//    of output rows.  One thread works out which source rows the band needs
//    (two per output row on a downscale, fewer on an upscale, none for
//    letterbox padding rows) and pulls each whole row into shared memory
//    with one bulk copy (cp.async.bulk, completion counted on an mbarrier).
//    On a 4-9x downscale the bilinear taps of a row touch every 32-byte
//    sector, so streaming whole rows is the least DRAM traffic any reader
//    can have; the bulk copy engine moves them without spending registers.
//    While the copies fly, the threads build the column tap table (byte
//    offsets and weights) in shared memory.  Each thread then produces four
//    consecutive x of one output row and writes them as one 16-byte store per
//    channel plane, so the NCHW planes are written fully coalesced.
//  * Direct kernel (any alignment): one thread per output pixel with plain
//    byte loads; same arithmetic, same results.
//
// Arithmetic (the reading where the pages are silent): half-pixel centres as
// the exact rational ((2x+1) S - D) / (2D); floor gives the lower neighbour,
// the remainder over 2D (one correctly rounded division) the weight; both
// neighbours clamped to [0, S-1]; three FP32 lerps; out = (v - M_c) * R_c.
#include <algorithm>
#include <cmath>

#include "ws_internal.cuh"

namespace ws {
namespace {

constexpr int kPreThreads = 256;
constexpr int kMaxBand = 16;
constexpr int kMaxSlots = 2 * kMaxBand;
constexpr int kSmemTarget = 56 * 1024;     // about four blocks per SM
constexpr int kMaxTableCols = 8192;
constexpr int kHeaderBytes = 16 + 4 * (3 * kMaxBand + kMaxSlots + 1);
constexpr int kOffCols = (kHeaderBytes + 15) / 16 * 16;
constexpr unsigned long long kWaitLimitNs = 1ull << 30;   // ~1.07 s

struct PreParams {
    const uint8_t* src;
    long long row_stride, frame_stride;
    int sw, sh, dw, dh;
    int nw, nh, left, top;    // inner box (the whole destination when stretching)
    float M[3], R[3];         // out = (v - M) * R
    float pad;                // padding byte value
    float* dst;
    int band;                 // staged: output rows per block
    int slot_bytes;           // staged: shared bytes per staged source row (multiple of 16)
    int bulk_bytes;           // staged: leading bytes of a row moved by the bulk copy
    int row_bytes;            // 3 * sw
    int off_slots;            // staged: shared offset of the row slots
    uint32_t* err;            // device error word
};

// Taps of destination coordinate x of a D-pixel box sampled from S pixels.
__device__ __forceinline__ void axis_taps(int x, int S, int D, int& lo, int& hi, float& w) {
    const long long num = (2LL * x + 1) * S - D;
    const long long den = 2LL * D;
    long long q = num / den;                  // truncates toward zero
    if (num < 0 && q * den != num) --q;       // floor
    const long long rem = num - q * den;      // 0 <= rem < den
    w = __fdiv_rn((float)rem, (float)den);
    lo = (int)(q < 0 ? 0 : (q > S - 1 ? S - 1 : q));
    const long long q1 = q + 1;
    hi = (int)(q1 < 0 ? 0 : (q1 > S - 1 ? S - 1 : q1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// One bulk copy global -> this block's shared memory, completion on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for phase `parity` of `bar`, giving up after `limit_ns`.
__device__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, unsigned long long limit_ns) {
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_ns() - t0 > limit_ns) return false;
    }
    return true;
}

__device__ __forceinline__ int find_or_add(int* rows, int& n, int j) {
    for (int s = 0; s < n; ++s)
        if (rows[s] == j) return s;
    rows[n] = j;
    return n++;
}

template <bool kVecStore>
__global__ void __launch_bounds__(kPreThreads) pre_staged_kernel(const __grid_constant__ PreParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem);
    int* s_slot_a = reinterpret_cast<int*>(smem + 16);   // [kMaxBand] slot of the upper row, -1 = padding row
    int* s_slot_b = s_slot_a + kMaxBand;                  // [kMaxBand] slot of the lower row
    float* s_wy = reinterpret_cast<float*>(s_slot_b + kMaxBand);  // [kMaxBand]
    int* s_rows = reinterpret_cast<int*>(s_wy + kMaxBand);        // [kMaxSlots] source row per slot
    int* s_nslots = s_rows + kMaxSlots;
    int* s_off0 = reinterpret_cast<int*>(smem + kOffCols);        // [dw] byte offset of the left tap
    int* s_off1 = s_off0 + p.dw;                                  // [dw] byte offset of the right tap
    float* s_wx = reinterpret_cast<float*>(s_off1 + p.dw);        // [dw]
    unsigned char* slots = smem + p.off_slots;

    const int tid = threadIdx.x;
    const int b = blockIdx.y;
    const int y0 = blockIdx.x * p.band;
    const int nrows = min(p.band, p.dh - y0);
    const uint8_t* frame = p.src + (long long)b * p.frame_stride;

    if (tid == 0) {
        int n = 0;
        for (int r = 0; r < nrows; ++r) {
            const int y = y0 + r;
            int a = -1, c = -1;
            float wy = 0.f;
            if (y >= p.top && y < p.top + p.nh) {
                int j0, j1;
                axis_taps(y - p.top, p.sh, p.nh, j0, j1, wy);
                a = find_or_add(s_rows, n, j0);
                // a zero weight needs no second row (v = t exactly)
                c = (wy != 0.f && j1 != j0) ? find_or_add(s_rows, n, j1) : a;
            }
            s_slot_a[r] = a;
            s_slot_b[r] = c;
            s_wy[r] = wy;
        }
        *s_nslots = n;
        if (n > 0 && p.bulk_bytes > 0) {
            mbar_init(bar, 1);
            mbar_arrive_expect_tx(bar, (uint32_t)n * (uint32_t)p.bulk_bytes);
            for (int s = 0; s < n; ++s)
                bulk_g2s(slots + (size_t)s * p.slot_bytes, frame + (long long)s_rows[s] * p.row_stride,
                         (uint32_t)p.bulk_bytes, bar);
        }
    }

    // Column taps while the rows are in flight.
    for (int x = tid; x < p.dw; x += kPreThreads) {
        int i0 = 0, i1 = 0;
        float wx = 0.f;
        if (x >= p.left && x < p.left + p.nw) axis_taps(x - p.left, p.sw, p.nw, i0, i1, wx);
        s_off0[x] = 3 * i0;
        s_off1[x] = 3 * i1;
        s_wx[x] = wx;
    }
    __syncthreads();

    const int nslots = *s_nslots;
    const int tail = p.row_bytes - p.bulk_bytes;   // < 16 trailing bytes moved by plain loads
    if (tail > 0) {
        for (int i = tid; i < nslots * tail; i += kPreThreads) {
            const int s = i / tail, t = p.bulk_bytes + i % tail;
            slots[(size_t)s * p.slot_bytes + t] = frame[(long long)s_rows[s] * p.row_stride + t];
        }
    }
    int ok = 1;
    if (nslots > 0 && p.bulk_bytes > 0) ok = mbar_wait_bounded(bar, 0, kWaitLimitNs) ? 1 : 0;
    if (!__syncthreads_and(ok)) {
        // A copy never completed: report it, give copies in flight a last
        // bounded chance to land in this block's memory, and leave.
        if (tid == 0) atomicOr(p.err, kDevErrBulkCopyTimeout);
        if (!ok) mbar_wait_bounded(bar, 0, kWaitLimitNs);
        return;
    }

    float padn[3];
#pragma unroll
    for (int c = 0; c < 3; ++c) padn[c] = (p.pad - p.M[c]) * p.R[c];

    const int groups = (p.dw + 3) >> 2;
    const int items = nrows * groups;
    const size_t plane = (size_t)p.dh * p.dw;
    float* out_b = p.dst + (size_t)b * 3 * plane;

    for (int it = tid; it < items; it += kPreThreads) {
        const int r = it / groups;
        const int x0 = (it - r * groups) * 4;
        const int y = y0 + r;
        float o[3][4];
        const int sa = s_slot_a[r];
        if (sa < 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int c = 0; c < 3; ++c) o[c][q] = padn[c];
        } else {
            const unsigned char* A = slots + (size_t)sa * p.slot_bytes;
            const unsigned char* B = slots + (size_t)s_slot_b[r] * p.slot_bytes;
            const float wy = s_wy[r];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int x = x0 + q;
                if (x < p.dw && x >= p.left && x < p.left + p.nw) {
                    const int o0 = s_off0[x], o1 = s_off1[x];
                    const float wx = s_wx[x];
#pragma unroll
                    for (int c = 0; c < 3; ++c) {
                        const float p00 = A[o0 + c], p01 = A[o1 + c];
                        const float p10 = B[o0 + c], p11 = B[o1 + c];
                        const float t = p00 + wx * (p01 - p00);
                        const float u = p10 + wx * (p11 - p10);
                        const float v = t + wy * (u - t);
                        o[c][q] = (v - p.M[c]) * p.R[c];
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 3; ++c) o[c][q] = padn[c];
                }
            }
        }
        float* row0 = out_b + (size_t)y * p.dw + x0;
        if (kVecStore) {
#pragma unroll
            for (int c = 0; c < 3; ++c)
                *reinterpret_cast<float4*>(row0 + c * plane) = make_float4(o[c][0], o[c][1], o[c][2], o[c][3]);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (x0 + q < p.dw)
#pragma unroll
                    for (int c = 0; c < 3; ++c) row0[c * plane + q] = o[c][q];
        }
    }
}

// One thread per destination pixel, plain byte loads; any alignment.
__global__ void __launch_bounds__(256) pre_direct_kernel(const __grid_constant__ PreParams p, long long total) {
    const size_t plane = (size_t)p.dh * p.dw;
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const int x = (int)(i % p.dw);
        const long long t = i / p.dw;
        const int y = (int)(t % p.dh);
        const long long b = t / p.dh;
        float v[3];
        if (x >= p.left && x < p.left + p.nw && y >= p.top && y < p.top + p.nh) {
            int i0, i1, j0, j1;
            float wx, wy;
            axis_taps(x - p.left, p.sw, p.nw, i0, i1, wx);
            axis_taps(y - p.top, p.sh, p.nh, j0, j1, wy);
            const uint8_t* f = p.src + b * p.frame_stride;
            const uint8_t* A = f + (long long)j0 * p.row_stride;
            const uint8_t* B = f + (long long)j1 * p.row_stride;
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                const float p00 = __ldg(A + 3 * i0 + c), p01 = __ldg(A + 3 * i1 + c);
                const float p10 = __ldg(B + 3 * i0 + c), p11 = __ldg(B + 3 * i1 + c);
                const float tt = p00 + wx * (p01 - p00);
                const float u = p10 + wx * (p11 - p10);
                v[c] = tt + wy * (u - tt);
            }
        } else {
            v[0] = v[1] = v[2] = p.pad;
        }
        float* o = p.dst + (size_t)b * 3 * plane + (size_t)y * p.dw + x;
#pragma unroll
        for (int c = 0; c < 3; ++c) o[c * plane] = (v[c] - p.M[c]) * p.R[c];
    }
}

// Inner box of the destination covered by the frame (same reading as the
// header states: round half up, at least one pixel, odd pad at bottom/right).
void inner_box(const ws_preprocess_desc& d, int* nw, int* nh, int* left, int* top) {
    if (d.resize == WS_RESIZE_STRETCH) {
        *nw = d.dst_w; *nh = d.dst_h; *left = 0; *top = 0;
        return;
    }
    const long long sw = d.src_w, sh = d.src_h, dw = d.dst_w, dh = d.dst_h;
    long long w, h;
    if (dw * sh <= dh * sw) {
        w = dw;
        h = (2 * sh * dw + sw) / (2 * sw);
    } else {
        h = dh;
        w = (2 * sw * dh + sh) / (2 * sh);
    }
    w = std::max(w, 1LL);
    h = std::max(h, 1LL);
    *nw = (int)w; *nh = (int)h;
    *left = (int)((dw - w) / 2);
    *top = (int)((dh - h) / 2);
}

bool g_staged_attr_set[64][2];

}  // namespace

ws_status validate_preprocess(const ws_preprocess_desc* d, int32_t batch) {
    if (!d) return fail(WS_ERR_INVALID_ARGUMENT, "descriptor is NULL");
    if (batch < 1) return fail(WS_ERR_INVALID_ARGUMENT, "batch %d < 1", batch);
    if (d->src_w < 1 || d->src_h < 1 || d->src_w > 65535 || d->src_h > 65535)
        return fail(WS_ERR_INVALID_ARGUMENT, "source size %dx%d outside 1..65535", d->src_w, d->src_h);
    if (d->dst_w < 1 || d->dst_h < 1 || d->dst_w > 65535 || d->dst_h > 65535)
        return fail(WS_ERR_INVALID_ARGUMENT, "destination size %dx%d outside 1..65535", d->dst_w, d->dst_h);
    if (d->src_row_stride < 3LL * d->src_w)
        return fail(WS_ERR_INVALID_ARGUMENT, "row stride %lld < 3 * width", (long long)d->src_row_stride);
    if (d->src_row_stride > (1LL << 40))
        return fail(WS_ERR_INVALID_ARGUMENT, "row stride %lld too large", (long long)d->src_row_stride);
    if (d->src_frame_stride < d->src_row_stride * d->src_h)
        return fail(WS_ERR_INVALID_ARGUMENT, "frame stride %lld < row stride * height",
                    (long long)d->src_frame_stride);
    if (d->src_frame_stride > (1LL << 46) / batch)
        return fail(WS_ERR_INVALID_ARGUMENT, "batch * frame stride overflows");
    if (d->resize != WS_RESIZE_STRETCH && d->resize != WS_RESIZE_LETTERBOX)
        return fail(WS_ERR_INVALID_ARGUMENT, "resize mode %d", d->resize);
    if (d->pad_value < 0 || d->pad_value > 255)
        return fail(WS_ERR_INVALID_ARGUMENT, "pad value %d outside 0..255", d->pad_value);
    if (d->channel_order != WS_ORDER_RGB)
        return fail(WS_ERR_UNSUPPORTED, "channel order %d", d->channel_order);
    if (d->norm == WS_NORM_MEAN_STD) {
        for (int c = 0; c < 3; ++c) {
            if (!(d->std[c] > 0.f) || !std::isfinite(d->std[c]) || !std::isfinite(d->mean[c]))
                return fail(WS_ERR_INVALID_ARGUMENT, "mean/std of channel %d", c);
        }
    } else if (d->norm == WS_NORM_SCALE) {
        if (!std::isfinite(d->scale)) return fail(WS_ERR_INVALID_ARGUMENT, "scale is not finite");
    } else {
        return fail(WS_ERR_INVALID_ARGUMENT, "normalisation mode %d", d->norm);
    }
    if ((long long)batch * 3 * d->dst_w * d->dst_h > (1LL << 40))
        return fail(WS_ERR_INVALID_ARGUMENT, "destination too large");
    return WS_OK;
}

}  // namespace ws

extern "C" {

ws_status ws_preprocess_validate(const ws_preprocess_desc* desc, int32_t batch) {
    ws::clear_error();
    return ws::validate_preprocess(desc, batch);
}

ws_status ws_preprocess(const ws_preprocess_desc* d, const uint8_t* src, int32_t batch, float* dst,
                        cudaStream_t stream) {
    using namespace ws;
    clear_error();
    ws_status st = validate_preprocess(d, batch);
    if (st != WS_OK) return st;
    if (!src || !dst) return fail(WS_ERR_INVALID_ARGUMENT, "src or dst is NULL");

    int dev;
    const DeviceInfo* info;
    st = current_device_info(&dev, &info);
    if (st != WS_OK) return st;

    PreParams p{};
    p.src = src;
    p.row_stride = d->src_row_stride;
    p.frame_stride = d->src_frame_stride;
    p.sw = d->src_w; p.sh = d->src_h; p.dw = d->dst_w; p.dh = d->dst_h;
    inner_box(*d, &p.nw, &p.nh, &p.left, &p.top);
    for (int c = 0; c < 3; ++c) {
        if (d->norm == WS_NORM_MEAN_STD) {
            p.M[c] = (float)(255.0 * (double)d->mean[c]);
            p.R[c] = (float)(1.0 / (255.0 * (double)d->std[c]));
        } else {
            p.M[c] = 0.f;
            p.R[c] = d->scale;
        }
    }
    p.pad = (float)d->pad_value;
    p.dst = dst;
    p.row_bytes = 3 * d->src_w;
    p.err = device_error_word();

    const bool aligned = ((uintptr_t)src % 16 == 0) && (d->src_row_stride % 16 == 0) &&
                         (batch == 1 || d->src_frame_stride % 16 == 0);
    const int slot_bytes = (p.row_bytes + 15) / 16 * 16;
    const int off_slots = kOffCols + (12 * d->dst_w + 15) / 16 * 16;
    const long long min_smem = (long long)off_slots + 2LL * slot_bytes;
    if (aligned && d->dst_w <= kMaxTableCols && min_smem <= info->max_smem_optin) {
        int band = 1;
        while (band < kMaxBand && off_slots + 2LL * (band + 1) * slot_bytes <= kSmemTarget) ++band;
        // keep at least two blocks per SM in the grid
        while (band > 1 && (long long)((d->dst_h + band - 1) / band) * batch < 2LL * info->sm_count) band /= 2;
        p.band = band;
        p.slot_bytes = slot_bytes;
        p.bulk_bytes = p.row_bytes / 16 * 16;
        p.off_slots = off_slots;
        const size_t smem = (size_t)off_slots + 2ull * band * slot_bytes;
        const bool vec = (d->dst_w % 4 == 0) && ((uintptr_t)dst % 16 == 0);
        if (!g_staged_attr_set[dev][vec]) {
            if (vec)
                WS_TRY_CUDA(cudaFuncSetAttribute(pre_staged_kernel<true>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 info->max_smem_optin));
            else
                WS_TRY_CUDA(cudaFuncSetAttribute(pre_staged_kernel<false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 info->max_smem_optin));
            g_staged_attr_set[dev][vec] = true;
        }
        const dim3 grid((d->dst_h + band - 1) / band, batch);
        if (grid.y > 65535) return fail(WS_ERR_UNSUPPORTED, "batch %d > 65535", batch);
        if (vec)
            pre_staged_kernel<true><<<grid, kPreThreads, smem, stream>>>(p);
        else
            pre_staged_kernel<false><<<grid, kPreThreads, smem, stream>>>(p);
    } else {
        const long long total = (long long)batch * d->dst_h * d->dst_w;
        const long long blocks = std::min<long long>((total + 255) / 256, (long long)info->sm_count * 16);
        pre_direct_kernel<<<(unsigned)blocks, 256, 0, stream>>>(p, total);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "preprocess launch");
    return WS_OK;
}

}  // extern "C"
