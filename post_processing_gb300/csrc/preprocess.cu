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
//  * Ring kernel, persistent.  The work is cut into
//    units of (frame, band of output rows); each resident block walks its
//    share of units.  Warp 0 plans a unit (one lane per output row works out
//    its two source rows and weight) and pulls each needed source row, whole,
//    into a stage of a shared-memory ring with one bulk copy (cp.async.bulk)
//    of its 16-byte window, completion counted on the stage's mbarrier; any
//    base and stride work.  While the block computes
//    unit i from its stage, the copies of the next units are already in
//    flight, so HBM sees a steady stream instead of load-then-compute bursts.
//    On a 4-9x downscale the taps of a row touch every 32-byte sector, so
//    whole rows are also the least DRAM traffic any reader can have.  The
//    column tap table (byte offsets and weights) is built once per block.
//    Each thread produces four consecutive x of one output row and writes one
//    16-byte store per channel plane: the NCHW planes are written coalesced.
//  * Direct kernel: one thread per output pixel with plain byte loads; same
//    arithmetic, same results.  Small outputs, where the ring's per-block
//    set-up is not amortised.
//
// Arithmetic (the reading where the pages are silent): half-pixel centres as
// the exact rational ((2x+1) S - D) / (2D); floor gives the lower neighbour,
// the remainder over 2D (one correctly rounded division) the weight; both
// neighbours clamped to [0, S-1]; three FP32 lerps; out = (v - M_c) * R_c.
#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ws_internal.cuh"
#include "ws_ptx.cuh"

namespace ws {

// Tuning of one launch of the ring kernel.
struct PreTuning {
    int band, stages, blocks_per_sm, threads;
};

namespace {

constexpr int kMaxBand = 8;            // output rows per unit
constexpr int kMaxStages = 8;
constexpr int kMaxThreads = 512;
constexpr int kMaxTableCols = 8192;
// Threads of the ring kernel an SM holds by registers (about 64 a thread).
constexpr int kRingThreadsPerSM = 65536 / 64;
// AUTO: outputs of at most this many pixels (batch x dst_w x dst_h) take the
// direct kernel.  One-launch graphs on GB300 (events around the replay) put
// the crossover between 409,600 px (one 640x640 letterbox: 9.2 us either
// way; 8 x 224x224 from 1080p, 401K px: direct 11.3, staged 12.6) and
// 524,288 px (2 x 4K -> 512x512: direct 13.0, staged 11.2).
constexpr long long kDirectMaxPixels = 460000;
constexpr unsigned kFull = 0xffffffffu;

struct StagePlan {
    int frame, y0, nrows, pad_;
    int a[kMaxBand];     // byte offset in the stage of output row r's upper source row, -1 = padding row
    int b[kMaxBand];     // ... of its lower source row
    float wy[kMaxBand];
};

struct PreParams {
    const uint8_t* src;
    long long row_stride, frame_stride;
    int sw, sh, dw, dh;
    int nw, nh, left, top;    // inner box (the whole destination when stretching)
    float M[3], R[3];         // out = (v - M) * R
    float pad;                // padding byte value
    int cmap[3];              // byte of a source pixel that feeds output plane c (RGB or BGR)
    void* dst;                // [batch][3][dh][dw] of the output type
    // ring kernel
    int band;                 // output rows per unit
    int stages;               // ring depth
    int slot_bytes;           // shared bytes per staged source row (multiple of 16; room for its 16-byte window)
    int row_bytes;            // 3 * sw
    int stage_bytes;          // 2 * band * slot_bytes
    int off_plan, off_cols, off_slots;
    int nbands;               // units per frame
    long long units;          // batch * nbands
    uint32_t* err;            // device error word
};

// Taps of destination coordinate x of a D-pixel box sampled from S pixels:
// the source coordinate is num / den with num = (2x + 1) S - D and den = 2D;
// lo = floor(num / den), rem = num - lo den in [0, den), w = rem / den in one
// correctly rounded division; both taps clamped to [0, S - 1].  32-bit
// arithmetic whenever num fits (every size up to about 23,000 pixels; 64-bit
// conversions and compares are slow), 64-bit otherwise.
__device__ __forceinline__ void axis_taps(int x, int S, int D, int& lo, int& hi, float& w) {
    const long long num = (2LL * x + 1) * S - D;
    const int den = 2 * D;   // at most 131,070
    int q, rem;
    if (num >= (long long)INT_MIN && num <= (long long)INT_MAX) {
        const int n = (int)num;
        q = n / den;               // truncates toward zero
        rem = n - q * den;
        if (rem < 0) {             // floor for negative num
            --q;
            rem += den;
        }
    } else {
        long long q64 = num / den;
        long long r64 = num - q64 * den;
        if (r64 < 0) {
            --q64;
            r64 += den;
        }
        // only the clamped taps are needed: [-1, S] keeps them
        q = (int)(q64 < -1 ? -1 : (q64 > S ? S : q64));
        rem = (int)r64;
    }
    // 0 <= rem < den
    w = __fdiv_rn((float)rem, (float)den);
    lo = min(max(q, 0), S - 1);
    hi = min(max(q + 1, 0), S - 1);
}

// Output element conversion (round to nearest even for the half types).
template <typename OutT> __device__ __forceinline__ OutT to_out(float v);
template <> __device__ __forceinline__ float to_out<float>(float v) { return v; }
template <> __device__ __forceinline__ __half to_out<__half>(float v) { return __float2half_rn(v); }
template <> __device__ __forceinline__ __nv_bfloat16 to_out<__nv_bfloat16>(float v) { return __float2bfloat16_rn(v); }

// Four consecutive outputs of one plane in one store (16 bytes for float,
// 8 for the half types); the address is aligned to the store's size.
template <typename OutT>
__device__ __forceinline__ void store4(OutT* dst, float a, float b, float c, float d) {
    if constexpr (sizeof(OutT) == 4) {
        *reinterpret_cast<float4*>(dst) = make_float4(a, b, c, d);
    } else {
        union { OutT h[4]; uint2 u; } pk;
        pk.h[0] = to_out<OutT>(a);
        pk.h[1] = to_out<OutT>(b);
        pk.h[2] = to_out<OutT>(c);
        pk.h[3] = to_out<OutT>(d);
        *reinterpret_cast<uint2*>(dst) = pk.u;
    }
}

// Warp 0: plan unit `u` into stage `s` and start its copies.  Lane r handles
// output row r of the unit; its rows go to slots 2r and 2r+1 of the stage.
// Each row is copied as its 16-byte window: from the 16-byte boundary at or
// below the row's first byte to the one at or above its end, so that any base
// and any stride work.  The extra bytes (at most 15 on each side) lie in the
// same 16-byte blocks as bytes of the row, hence in pages the row itself
// occupies; they are copied and never used.  The plan records where in the
// slot the row starts.
__device__ void issue_unit(const PreParams& p, long long u, uint64_t* bar, StagePlan* plan,
                           unsigned char* stage) {
    const int lane = threadIdx.x & 31;
    const int frame = (int)(u / p.nbands);
    const int y0 = (int)(u - (long long)frame * p.nbands) * p.band;
    const int nrows = min(p.band, p.dh - y0);
    const uint8_t* fr = p.src + (long long)frame * p.frame_stride;
    const uint8_t* wa = nullptr;
    const uint8_t* wb = nullptr;
    uint32_t na = 0, nb = 0;
    if (lane < nrows) {
        const int y = y0 + lane;
        const int pl = WS_CHECKED(lane, 0, kMaxBand, p.err);   // the plan's row slot
        int a = -1, b = -1;
        float wy = 0.f;
        if (y >= p.top && y < p.top + p.nh) {
            int j0, j1;
            axis_taps(y - p.top, p.sh, p.nh, j0, j1, wy);
            j0 = WS_CHECKED(j0, 0, p.sh, p.err);
            j1 = WS_CHECKED(j1, 0, p.sh, p.err);
            const uint8_t* ra = fr + (long long)j0 * p.row_stride;
            const int oa = (int)((uintptr_t)ra & 15u);
            wa = ra - oa;
            na = (uint32_t)((oa + p.row_bytes + 15) & ~15);
            a = 2 * lane * p.slot_bytes + oa;
            if (wy != 0.f && j1 != j0) {   // a zero weight needs no second row (v = t exactly)
                const uint8_t* rb = fr + (long long)j1 * p.row_stride;
                const int ob = (int)((uintptr_t)rb & 15u);
                wb = rb - ob;
                nb = (uint32_t)((ob + p.row_bytes + 15) & ~15);
                b = (2 * lane + 1) * p.slot_bytes + ob;
            } else {
                b = a;
            }
#ifdef WS_BOUNDS_CHECK
            // each row's window fits its slot, and the slots fit the stage
            if (na > (uint32_t)p.slot_bytes || nb > (uint32_t)p.slot_bytes ||
                (2 * lane + 2) * p.slot_bytes > p.stage_bytes) {
                atomicOr(p.err, (uint32_t)kDevErrBounds);
                na = nb = 0;   // nothing copied; the row reads the slot as it is
                a = b = 2 * (lane % max(1, p.stage_bytes / (2 * p.slot_bytes))) * p.slot_bytes;
            }
            a = WS_CHECKED(a, 0, p.stage_bytes - p.row_bytes + 1, p.err);
            b = WS_CHECKED(b, 0, p.stage_bytes - p.row_bytes + 1, p.err);
#endif
        }
        plan->a[pl] = a;
        plan->b[pl] = b;
        plan->wy[pl] = wy;
    }
    if (lane == 0) {
        plan->frame = frame;
        plan->y0 = y0;
        plan->nrows = nrows;
    }
    uint32_t bytes = na + nb;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) bytes += __shfl_xor_sync(kFull, bytes, o);
    // The expected bytes are registered (with the one arrival) before any copy
    // can complete; a band of padding rows completes the phase at once.
    if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
    __syncwarp();
    if (na) bulk_g2s(stage + 2 * lane * p.slot_bytes, wa, na, bar);
    if (nb) bulk_g2s(stage + (2 * lane + 1) * p.slot_bytes, wb, nb, bar);
}

// Column taps: the byte offset of the left tap in a staged row, with kTapSame
// set when the right tap is the same pixel (clamped at an edge; otherwise it
// is the next pixel, 3 bytes on), and the weight's bits: one 8-byte entry
// per output column, one shared load per pixel instead of three.
constexpr int kTapSame = 1 << 30;

template <typename OutT, bool kVecStore>
__device__ __forceinline__ void compute_unit(const PreParams& p, const StagePlan& plan, const unsigned char* stage,
                                             const int2* s_tap, const float (&padn)[3]) {
    const int groups = (p.dw + 3) >> 2;
    const int items = plan.nrows * groups;
    const size_t plane = (size_t)p.dh * p.dw;
    OutT* out_b = static_cast<OutT*>(p.dst) + (size_t)plan.frame * 3 * plane;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
        const int r = WS_CHECKED(it / groups, 0, kMaxBand, p.err);
        const int x0 = (it - r * groups) * 4;
        const int y = plan.y0 + r;
        float o[3][4];
        const int sa = plan.a[r];
        if (sa < 0) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
#pragma unroll
                for (int c = 0; c < 3; ++c) o[c][q] = padn[c];
        } else {
            const unsigned char* A = stage + WS_CHECKED(sa, 0, p.stage_bytes - p.row_bytes + 1, p.err);
            const unsigned char* B = stage + WS_CHECKED(plan.b[r], 0, p.stage_bytes - p.row_bytes + 1, p.err);
            const float wy = plan.wy[r];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int x = x0 + q;
                if (x < p.dw && x >= p.left && x < p.left + p.nw) {
                    const int2 tap = s_tap[WS_CHECKED(x, 0, p.dw, p.err)];
                    const bool same = (tap.x & kTapSame) != 0;
                    const int o0 = WS_CHECKED(tap.x & ~kTapSame, 0, p.row_bytes - 2, p.err);
                    const float wx = __int_as_float(tap.y);
                    const int o1 = WS_CHECKED(same ? o0 : o0 + 3, 0, p.row_bytes - 2, p.err);
#pragma unroll
                    for (int c = 0; c < 3; ++c) {
                        const int sc = p.cmap[c];
                        const float p00 = A[o0 + sc], p01 = A[o1 + sc];
                        const float p10 = B[o0 + sc], p11 = B[o1 + sc];
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
        OutT* row0 = out_b + (size_t)y * p.dw + x0;
        if (kVecStore) {
#pragma unroll
            for (int c = 0; c < 3; ++c) store4<OutT>(row0 + c * plane, o[c][0], o[c][1], o[c][2], o[c][3]);
        } else {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (x0 + q < p.dw)
#pragma unroll
                    for (int c = 0; c < 3; ++c) row0[c * plane + q] = to_out<OutT>(o[c][q]);
        }
    }
}

template <typename OutT, bool kVecStore>
__global__ void __launch_bounds__(kMaxThreads) pre_ring_kernel(const __grid_constant__ PreParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem);                    // [stages]
    StagePlan* plans = reinterpret_cast<StagePlan*>(smem + p.off_plan);   // [stages]
    int2* s_tap = reinterpret_cast<int2*>(smem + p.off_cols);             // [dw] left-tap offset | same, weight
    unsigned char* slots = smem + p.off_slots;

    // Let a programmatic dependent (the Top-K) be launched now; it waits for
    // this grid's completion before it reads anything.  This grid is itself
    // a programmatic dependent of the previous kernel on the stream: nothing
    // global is read or written before that kernel has finished.
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int tid = threadIdx.x;
    const long long G = gridDim.x;
    const long long first = blockIdx.x;
    const int n_my = p.units > first ? (int)((p.units - 1 - first) / G + 1) : 0;

    if (tid < 32) {
        if (tid == 0) {
            for (int s = 0; s < p.stages; ++s) mbar_init(&bars[s], 1);
            fence_mbar_init();
        }
        __syncwarp();
        const int pre = min(p.stages, n_my);
        for (int i = 0; i < pre; ++i)
            issue_unit(p, first + i * G, &bars[i], &plans[i], slots + (size_t)i * p.stage_bytes);
    }
    // Column taps, once per block, while the first rows are in flight.
    for (int x = tid; x < p.dw; x += blockDim.x) {
        int i0 = 0, i1 = 0;
        float wx = 0.f;
        if (x >= p.left && x < p.left + p.nw) axis_taps(x - p.left, p.sw, p.nw, i0, i1, wx);
        i0 = WS_CHECKED(i0, 0, p.sw, p.err);
        i1 = WS_CHECKED(i1, 0, p.sw, p.err);
        s_tap[WS_CHECKED(x, 0, p.dw, p.err)] = make_int2(3 * i0 | (i1 == i0 ? kTapSame : 0), __float_as_int(wx));
    }
    float padn[3];
#pragma unroll
    for (int c = 0; c < 3; ++c) padn[c] = (p.pad - p.M[c]) * p.R[c];
    __syncthreads();

    for (int i = 0; i < n_my; ++i) {
        const int s = i % p.stages;
        const uint32_t parity = (uint32_t)(i / p.stages) & 1u;
        const bool ok = mbar_wait_bounded(&bars[s], parity, kWaitLimitNs);
        if (ok)
            compute_unit<OutT, kVecStore>(p, plans[s], slots + (size_t)s * p.stage_bytes, s_tap, padn);
        // Everyone is done with stage s (and agrees on whether a copy hung).
        if (__syncthreads_or(!ok)) {
            if (tid == 0) {
                atomicOr(p.err, kDevErrBulkCopyTimeout);
                // let the copies still in flight land in this block's memory
                for (int j = i; j < min(n_my, i + p.stages); ++j)
                    mbar_wait_bounded(&bars[j % p.stages], (uint32_t)(j / p.stages) & 1u, kWaitLimitNs);
            }
            return;
        }
        if (tid < 32 && i + p.stages < n_my)
            issue_unit(p, first + (long long)(i + p.stages) * G, &bars[s], &plans[s],
                       slots + (size_t)s * p.stage_bytes);
    }
}

// One thread per destination pixel, plain byte loads; any alignment.  A 3-D
// grid: x from the block column and thread, output row blockIdx.y (its taps
// are the same for the whole block), frame blockIdx.z (frames beyond the
// grid's z extent loop).  No index divisions: the loads are issued after a
// few dozen instructions.
template <typename OutT>
__global__ void __launch_bounds__(256) pre_direct_kernel(const __grid_constant__ PreParams p, int batch) {
    asm volatile("griddepcontrol.launch_dependents;");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int x = blockIdx.x * blockDim.x + threadIdx.x;
    const int y = blockIdx.y;
    if (x >= p.dw) return;
    const size_t plane = (size_t)p.dh * p.dw;
    const bool in_x = x >= p.left && x < p.left + p.nw;
    const bool in_y = y >= p.top && y < p.top + p.nh;
    int i0 = 0, i1 = 0, j0 = 0, j1 = 0;
    float wx = 0.f, wy = 0.f;
    if (in_x && in_y) {
        axis_taps(x - p.left, p.sw, p.nw, i0, i1, wx);
        axis_taps(y - p.top, p.sh, p.nh, j0, j1, wy);
        i0 = WS_CHECKED(i0, 0, p.sw, p.err);
        i1 = WS_CHECKED(i1, 0, p.sw, p.err);
        j0 = WS_CHECKED(j0, 0, p.sh, p.err);
        j1 = WS_CHECKED(j1, 0, p.sh, p.err);
    }
    for (int b = blockIdx.z; b < batch; b += gridDim.z) {
        float v[3];
        if (in_x && in_y) {
            const uint8_t* f = p.src + (long long)b * p.frame_stride;
            const uint8_t* A = f + (long long)j0 * p.row_stride;
            const uint8_t* Bq = f + (long long)j1 * p.row_stride;
            float q[3][4];
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                const int sc = p.cmap[c];
                q[c][0] = __ldg(A + 3 * i0 + sc);
                q[c][1] = __ldg(A + 3 * i1 + sc);
                q[c][2] = __ldg(Bq + 3 * i0 + sc);
                q[c][3] = __ldg(Bq + 3 * i1 + sc);
            }
#pragma unroll
            for (int c = 0; c < 3; ++c) {
                const float tt = q[c][0] + wx * (q[c][1] - q[c][0]);
                const float u = q[c][2] + wx * (q[c][3] - q[c][2]);
                v[c] = tt + wy * (u - tt);
            }
        } else {
            v[0] = v[1] = v[2] = p.pad;
        }
        OutT* o = static_cast<OutT*>(p.dst) + (size_t)b * 3 * plane + (size_t)y * p.dw + x;
#pragma unroll
        for (int c = 0; c < 3; ++c) o[c * plane] = to_out<OutT>((v[c] - p.M[c]) * p.R[c]);
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

size_t align16(size_t v) { return (v + 15) / 16 * 16; }

// Shared-memory layout of the ring kernel for a tuning; returns total bytes.
size_t ring_layout(PreParams& p, const PreTuning& t) {
    p.band = t.band;
    p.stages = t.stages;
    p.stage_bytes = 2 * t.band * p.slot_bytes;
    p.off_plan = (int)align16(8 * kMaxStages);
    p.off_cols = (int)align16(p.off_plan + sizeof(StagePlan) * kMaxStages);
    p.off_slots = (int)align16(p.off_cols + 8 * (size_t)p.dw);
    return (size_t)p.off_slots + (size_t)t.stages * p.stage_bytes;
}

// Default tuning, from sweeps on GB300 of blocks per SM, output rows per unit
// and ring depth over ten geometries (1080p, 720p, 1366x768, 640x480,
// 320x240 and 4K sources; 224 to 640 wide outputs).  What decides is the
// output per source byte, r = dst_w / (6 src_w): with little output per byte
// (strong downscales) the kernel is HBM-bound and needs only enough copies in
// flight, with more it is bound by its per-pixel work and needs more warps to
// hide that work's latency.  The best setting had about 800 r warps per SM
// (8 .. 32), blocks of about 128 threads while r < 0.025 and about 256
// above, and a ring of two stages.  For example (batch, source -> output:
// blocks per SM x rows per unit x stages, us): 64, 1080p -> 224: 4 x 2 x 2,
// 33.7; 8, 4K -> 512: 4 x 1 x 2, 20.7; 64, 1280x720 -> 224: 3 x 4 x 2, 26.7
// (the earlier fixed 3 blocks of 128 threads and a 3-stage ring: 35.7);
// 256, 640x480 -> 224: 4 x 4 x 2, 74.9 (185.3); 16, 1080p -> 640:
// 6 x 1 x 2, 36.9 (62.2).  Single-frame work is spread thin for latency.
PreTuning default_tuning(const PreParams& p, int batch, const DeviceInfo& info) {
    const int groups = (p.dw + 3) / 4;
    const size_t fixed = align16(8 * kMaxStages) + sizeof(StagePlan) * kMaxStages + align16(8 * (size_t)p.dw) + 64;
    const double r = (double)p.dw / (6.0 * (double)p.sw);
    const int warps_per_sm = std::max(8, std::min(32, (int)std::lround(800.0 * r)));
    const int target_threads = r < 0.025 ? 128 : 256;
    auto threads_for = [&](int band) { return std::min(kMaxThreads, std::max(64, (band * groups + 31) / 32 * 32)); };
    int band0 = std::max(1, std::min(kMaxBand, target_threads / std::max(groups, 1)));
    while (band0 > 1 && band0 * groups > kMaxThreads) --band0;
    for (int band = band0; band >= 1; band = band > 1 ? band / 2 : 0) {
        const int threads = threads_for(band);
        int want = std::max(1, std::min(8, (int)std::lround((double)warps_per_sm / (threads / 32))));
        want = std::min(want, kRingThreadsPerSM / threads);
        for (int bps = want; bps >= 1; --bps) {
            const size_t budget =
                std::min<size_t>((size_t)info.smem_per_sm / bps - 1024, (size_t)info.max_smem_optin);
            int b = band;
            // keep at least ~2 units per resident block when the batch is large enough
            const long long slots_total = (long long)info.sm_count * bps;
            while (b > 1 && (long long)batch * ((p.dh + b - 1) / b) < 2 * slots_total) b /= 2;
            const size_t stage = 2ull * b * p.slot_bytes;
            if (budget < fixed + 2 * stage) continue;
            PreTuning t{};
            t.band = b;
            t.stages = 2;
            t.blocks_per_sm = bps;
            t.threads = threads_for(b);
            // blocks that get a single unit (small batches) are latency-bound:
            // more threads build the column table and issue the loads sooner
            if ((long long)batch * ((p.dh + b - 1) / b) <= slots_total) t.threads = std::max(t.threads, 128);
            return t;
        }
    }
    // very wide rows: one block per SM with a single stage when even two do not fit
    PreTuning t{};
    t.band = 1;
    t.blocks_per_sm = 1;
    t.threads = threads_for(1);
    const size_t budget = std::min<size_t>((size_t)info.smem_per_sm - 1024, (size_t)info.max_smem_optin);
    t.stages = budget >= fixed + 4ull * p.slot_bytes ? 2 : 1;
    return t;
}

std::atomic<bool> g_ring_attr_set[64][3][2];

// Both preprocess kernels launch as programmatic dependents of the kernel
// before them and wait in griddepcontrol.wait before their first read.
template <typename Kernel, typename... Args>
ws_status pdl_launch(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaError_t e = launch_pdl(kernel, grid, block, smem, stream, args...);
    if (e != cudaSuccess) return cuda_fail(e, "preprocess launch");
    return WS_OK;
}

template <typename OutT, bool kVec>
ws_status launch_ring(const PreParams& p, int dev, const DeviceInfo& info, unsigned blocks, int threads, size_t smem,
                      int type_slot, cudaStream_t stream) {
    if (!g_ring_attr_set[dev][type_slot][kVec].load(std::memory_order_acquire)) {
        WS_TRY_CUDA(cudaFuncSetAttribute(pre_ring_kernel<OutT, kVec>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info.max_smem_optin));
        g_ring_attr_set[dev][type_slot][kVec].store(true, std::memory_order_release);
    }
    // The kernel is persistent: a grid larger than what is resident would run
    // a second, mostly idle wave.  Clamp it to the resident blocks.
    int resident = 0;
    WS_TRY_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&resident, pre_ring_kernel<OutT, kVec>, threads, smem));
    if (resident < 1) return fail(WS_ERR_UNSUPPORTED, "preprocess: no ring block fits an SM (%zu bytes)", smem);
    blocks = std::min<unsigned>(blocks, (unsigned)resident * (unsigned)info.sm_count);
    return pdl_launch(pre_ring_kernel<OutT, kVec>, dim3(blocks), dim3(threads), smem, stream, p);
}

std::atomic<bool> g_direct_attr_set[64][3];

template <typename OutT>
ws_status launch_any(const PreParams& p, bool ring, bool vec, int dev, const DeviceInfo& info, unsigned blocks,
                     int threads, size_t smem, int type_slot, long long total, cudaStream_t stream) {
    if (ring)
        return vec ? launch_ring<OutT, true>(p, dev, info, blocks, threads, smem, type_slot, stream)
                   : launch_ring<OutT, false>(p, dev, info, blocks, threads, smem, type_slot, stream);
    // The direct kernel needs no shared memory, but the kernels that follow it
    // (Top-K stages a 32 KB chunk, NMS far more) do.  Left to its default, an
    // SM runs it with the largest L1 and must drain and re-partition before
    // the next kernel's blocks fit: measured as ~2 us added to a batch-1
    // 640x640 letterbox + Top-5 over 672K graph.  Asking for the shared-heavy
    // split keeps one partition across the sequence at no cost to this kernel.
    if (!g_direct_attr_set[dev][type_slot].load(std::memory_order_acquire)) {
        WS_TRY_CUDA(cudaFuncSetAttribute(pre_direct_kernel<OutT>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared));
        g_direct_attr_set[dev][type_slot].store(true, std::memory_order_release);
    }
    // x across blocks of up to 256 threads, one output row per blockIdx.y,
    // frames across blockIdx.z (the kernel loops over frames beyond it)
    const int tx = std::min(256, (p.dw + 31) / 32 * 32);
    const dim3 grid((unsigned)((p.dw + tx - 1) / tx), (unsigned)p.dh, (unsigned)std::min<long long>(total, 65535));
    return pdl_launch(pre_direct_kernel<OutT>, grid, dim3(tx), 0, stream, p, (int)total);
}

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
    if (d->channel_order != WS_ORDER_RGB && d->channel_order != WS_ORDER_BGR)
        return fail(WS_ERR_INVALID_ARGUMENT, "channel order %d", d->channel_order);
    if (d->dst_type != WS_DTYPE_F32 && d->dst_type != WS_DTYPE_F16 && d->dst_type != WS_DTYPE_BF16)
        return fail(WS_ERR_INVALID_ARGUMENT, "destination type %d", d->dst_type);
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

// Launch with an explicit ring tuning (NULL = the default policy).
ws_status preprocess_launch(const ws_preprocess_desc* d, const uint8_t* src, int32_t batch, void* dst,
                            cudaStream_t stream, const PreTuning* tuning, int32_t path) {
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
    for (int c = 0; c < 3; ++c) p.cmap[c] = d->channel_order == WS_ORDER_BGR ? 2 - c : c;
    p.dst = dst;
    p.row_bytes = 3 * d->src_w;
    // A row's 16-byte window is align16(row_bytes) long when every row starts
    // on a 16-byte boundary, and up to 16 bytes longer otherwise.
    const bool aligned = ((uintptr_t)src % 16 == 0) && (d->src_row_stride % 16 == 0) &&
                         (batch == 1 || d->src_frame_stride % 16 == 0);
    p.slot_bytes = (int)align16(p.row_bytes) + (aligned ? 0 : 16);
    p.err = device_error_word();
    PreTuning t = tuning ? *tuning : default_tuning(p, batch, *info);
    const size_t smem = ring_layout(p, t);
    // The staged ring pays a fixed set-up per block (barriers, plan, column
    // table, a copy round trip): small outputs (a single 224x224 frame)
    // finish sooner one thread per pixel.
    const bool small = (long long)batch * d->dst_w * d->dst_h <= kDirectMaxPixels;
    const bool want_ring = path == WS_PRE_PATH_STAGED || (path == WS_PRE_PATH_AUTO && !small);
    const bool ring_ok = want_ring && d->dst_w <= kMaxTableCols && t.band >= 1 && t.band <= kMaxBand &&
                         t.stages >= 1 && t.stages <= kMaxStages && t.threads >= 32 &&
                         t.threads <= kMaxThreads && smem <= (size_t)info->max_smem_optin;
    bool vec = false;
    unsigned blocks;
    long long total = 0;
    if (ring_ok) {
        p.nbands = (d->dst_h + t.band - 1) / t.band;
        p.units = (long long)batch * p.nbands;
        vec = (d->dst_w % 4 == 0) && ((uintptr_t)dst % 16 == 0);
        blocks = (unsigned)std::min<long long>(p.units, (long long)info->sm_count * t.blocks_per_sm);
    } else {
        total = batch;   // the per-pixel kernel's grid is set up in launch_any
        blocks = 0;
    }
    switch (d->dst_type) {
        case WS_DTYPE_F16:
            st = launch_any<__half>(p, ring_ok, vec, dev, *info, blocks, t.threads, smem, 1, total, stream);
            break;
        case WS_DTYPE_BF16:
            st = launch_any<__nv_bfloat16>(p, ring_ok, vec, dev, *info, blocks, t.threads, smem, 2, total, stream);
            break;
        default:
            st = launch_any<float>(p, ring_ok, vec, dev, *info, blocks, t.threads, smem, 0, total, stream);
    }
    if (st != WS_OK) return st;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "preprocess launch");
    return WS_OK;
}

}  // namespace ws

extern "C" {

ws_status ws_preprocess_validate(const ws_preprocess_desc* desc, int32_t batch) {
    ws::clear_error();
    return ws::validate_preprocess(desc, batch);
}

ws_status ws_preprocess(const ws_preprocess_desc* d, const uint8_t* src, int32_t batch, void* dst,
                        cudaStream_t stream) {
    ws::clear_error();
    return ws::preprocess_launch(d, src, batch, dst, stream, nullptr, WS_PRE_PATH_AUTO);
}

ws_status ws_preprocess_path(const ws_preprocess_desc* d, const uint8_t* src, int32_t batch, void* dst,
                             int32_t path, cudaStream_t stream) {
    ws::clear_error();
    if (path < WS_PRE_PATH_AUTO || path > WS_PRE_PATH_DIRECT)
        return ws::fail(WS_ERR_INVALID_ARGUMENT, "preprocess path %d", path);
    return ws::preprocess_launch(d, src, batch, dst, stream, nullptr, path);
}

}  // extern "C"
