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
//  * decode: one warp per tile of 128 consecutive anchors (4 per lane).  The
//    warp scans every class row of its tile with coalesced 512-byte row
//    segments (16 bytes a lane, 8 rows in flight), so the arg-max needs no
//    merge across warps and no block barrier.  One atomic reserves slots for
//    the anchors whose best logit clears the threshold (about 2 % of them),
//    and the same warp then takes their DFL: four lanes per candidate, one
//    per side, load that side's reg_max logits and take the softmax
//    expectation.  All tiles stream at once; a warp's scattered DFL loads
//    overlap the other warps' class rows.
//  * NMS: one block per image, launched as a programmatic dependent of the
//    decode kernel so its launch overlaps the decode's tail.  If the image has more
//    than max_cand candidates, their 64-bit keys (logit order bits, then the
//    complemented anchor) are held in registers and a radix select
//    (warp-aggregated histogram counts, early exit once a digit bin closes
//    the count) keeps the best max_cand.  The survivors are ranked by counting
//    when there are few, else bitonic-sorted at the next power of two of the
//    live count (shuffles within a warp's 64 elements, shared memory above).  Every pair's suppression test (same class, IoU > threshold)
//    is evaluated in parallel into a bit matrix, a thread per (row, 64-bit
//    word), the IoU only where a class-bucket table shows a match, and one
//    warp walks the sorted list a 64-candidate word at a time,
//    deciding at each step every candidate that nothing live can still
//    suppress.  The IoU test is FP32 with every operation rounded
//    separately (no fused multiply-add), so given the same boxes the
//    decisions are exactly those of the definition.
#include <algorithm>
#include <atomic>
#include <cmath>


#include "ws_internal.cuh"

namespace ws {
namespace {

constexpr int kDecodeAnchors = 128;                    // anchors per decode tile: 4 per lane
constexpr int kLaneAnchors = 4;
constexpr int kWarpScanWarps = 4;                      // warps (tiles) per decode block
constexpr int kWarpScanLoads = 8;                      // class rows in flight per lane
constexpr int kDecodeSplit = 4;                        // warps per tile when tiles are few
constexpr long long kDecodeSplitTiles = 1100;          // up to this many tiles in all (16 640x640 heads)
constexpr int kNmsThreads = 512;
constexpr int kNmsWarps = kNmsThreads / 32;
constexpr int kMaxCand = 1024;
constexpr int kMaxLevels = 4;
constexpr int kMaxRegMax = 32;
constexpr int kKeysPerThread = 32;    // candidate keys a thread holds in registers for the cap selection
constexpr int kBuckets = 256;         // class buckets of the match table
constexpr int kCountSortMax = 256;    // rank by counting up to this many candidates, bitonic above
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
    int Pcap;                         // power of two >= max_cand
    int off_idx, off_box, off_cls, off_logit, off_anchor, off_keep, off_hist, off_u;
    int off_tab;                      // match table, from off_u
    int u_bytes;                      // per-warp histograms, later the suppression matrix and match table
};

// Class logits and NMS keys: NaN ranks as -inf and -0 equals +0, as in the
// Top-K.
__device__ __forceinline__ float nan_as_ninf(float v) { return v != v ? -INFINITY : v; }

__device__ __forceinline__ uint32_t order_bits(float f) {
    uint32_t b = __float_as_uint(nan_as_ninf(f));
    if (b == 0x80000000u) b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ unsigned long long cand_key(const ws_candidate* c) {
    return ((unsigned long long)order_bits(c->logit) << 32) | (uint32_t)(~(uint32_t)c->anchor);
}

// Running arg-max of a lane's four anchors over one class row (NaN counts
// as -inf; a strictly larger logit replaces, so the lower class keeps a tie).
__device__ __forceinline__ void take4(float (&best)[kLaneAnchors], int (&bc)[kLaneAnchors], const float4 v4, int c) {
    const float v[4] = {nan_as_ninf(v4.x), nan_as_ninf(v4.y), nan_as_ninf(v4.z), nan_as_ninf(v4.w)};
#pragma unroll
    for (int e = 0; e < 4; ++e)
        if (v[e] > best[e]) {
            best[e] = v[e];
            bc[e] = c;
        }
}

// Decode with one warp per 128-anchor tile: the warp scans every class row of
// its tile (lane l holds anchors 4l .. 4l + 3, one 16-byte word per class
// row, kWarpScanLoads rows in flight), so the arg-max needs no merge across
// warps and no block barrier; the warp then reserves its candidates' slots
// with one atomic and decodes their DFL boxes itself, four lanes per
// candidate (one per side).  Every tile streams at once, and the scattered
// DFL loads of a warp overlap other warps' class rows.
// kSplit > 1 (few tiles, e.g. one image): a block of kSplit warps takes one
// tile, each warp a contiguous range of classes, and warp 0 merges their
// arg-maxes (value, then the lower class) through shared memory before it
// goes on alone.  A warp's chain of dependent class-row loads is then
// kSplit times shorter.
template <bool kVec, int kSplit>
__global__ void __launch_bounds__(32 * (kSplit == 1 ? kWarpScanWarps : kSplit))
    detect_decode_warp_kernel(const __grid_constant__ DetParams p) {
    constexpr int kTilesPerBlock = kSplit == 1 ? kWarpScanWarps : 1;
    __shared__ int s_loc[kTilesPerBlock][kDecodeAnchors];   // tile offset of each local candidate
    __shared__ float s_v[kSplit][kDecodeAnchors];          // per-warp arg-max values (kSplit > 1)
    __shared__ int s_c[kSplit][kDecodeAnchors];            // and classes
    asm volatile("griddepcontrol.wait;" ::: "memory");   // the head and the counters are the previous kernels'
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5, b = blockIdx.y;
    const int tw = kSplit == 1 ? w : 0;                     // this warp's tile in the block
    const long long a0 = ((long long)blockIdx.x * kTilesPerBlock + tw) * kDecodeAnchors;
    if (a0 >= p.A) return;   // whole warp (whole block when kSplit > 1)
    const int cbeg = kSplit == 1 ? 0 : p.C * w / kSplit;
    const int cend = kSplit == 1 ? p.C : p.C * (w + 1) / kSplit;
    const float* hb = p.head + (size_t)b * p.ch * p.A;
    const float* cl = hb + (size_t)(4 * p.R) * p.A;
    float best[kLaneAnchors];
    int bc[kLaneAnchors];
#pragma unroll
    for (int e = 0; e < kLaneAnchors; ++e) {
        best[e] = -INFINITY;
        bc[e] = 0;
    }
    // Classes in increasing order with a strict comparison: the lower class
    // keeps a tie.
    if (kVec) {   // A % 4 == 0: a word's four anchors all exist or none does
        const bool live = a0 + 4 * lane < p.A;
        const float* col = cl + a0 + 4 * lane;
        auto load = [&](int c) -> float4 {
            return live ? __ldg(reinterpret_cast<const float4*>(col + (size_t)c * p.A))
                        : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        };
        int c = cbeg;
        for (; c + kWarpScanLoads <= cend; c += kWarpScanLoads) {
            float4 v4[kWarpScanLoads];
#pragma unroll
            for (int u = 0; u < kWarpScanLoads; ++u) v4[u] = load(c + u);
#pragma unroll
            for (int u = 0; u < kWarpScanLoads; ++u) take4(best, bc, v4[u], c + u);
        }
        for (; c < cend; ++c) take4(best, bc, load(c), c);
    } else {
#pragma unroll 2
        for (int c = cbeg; c < cend; ++c) {
            const float* row = cl + (size_t)c * p.A;
#pragma unroll
            for (int e = 0; e < kLaneAnchors; ++e) {
                const long long a = a0 + 4 * lane + e;
                if (a < p.A) {
                    const float v = nan_as_ninf(__ldg(row + a));
                    if (v > best[e]) {
                        best[e] = v;
                        bc[e] = c;
                    }
                }
            }
        }
    }

    if (kSplit > 1) {
        // An all -inf range reports class 0, which is the arg-max exactly
        // when every class of the anchor is -inf.
#pragma unroll
        for (int e = 0; e < kLaneAnchors; ++e) {
            s_v[w][4 * lane + e] = best[e];
            s_c[w][4 * lane + e] = bc[e];
        }
        __syncthreads();
        if (w != 0) return;
#pragma unroll
        for (int e = 0; e < kLaneAnchors; ++e) {
#pragma unroll
            for (int q = 1; q < kSplit; ++q) {
                const float v = s_v[q][4 * lane + e];
                const int c = s_c[q][4 * lane + e];
                if (v > best[e] || (v == best[e] && c < bc[e])) {
                    best[e] = v;
                    bc[e] = c;
                }
            }
        }
    }

    // candidates: one ballot per anchor position, slots from one atomic
    const unsigned lt = (1u << lane) - 1u;
    unsigned m[kLaneAnchors];
    int total = 0;
#pragma unroll
    for (int e = 0; e < kLaneAnchors; ++e) {
        m[e] = __ballot_sync(kFull, a0 + 4 * lane + e < p.A && best[e] > p.logit_thr);
        total += __popc(m[e]);
    }
    if (total == 0) {
        asm volatile("griddepcontrol.launch_dependents;");
        return;
    }
    int base = 0;
    if (lane == 0) base = atomicAdd(&p.count[b], total);
    base = __shfl_sync(kFull, base, 0);
    ws_candidate* cb = p.cand + (size_t)b * p.A;
    int before = 0;
#pragma unroll
    for (int e = 0; e < kLaneAnchors; ++e) {
        if ((m[e] >> lane) & 1u) {
            const int q = before + __popc(m[e] & lt);
            s_loc[tw][q] = 4 * lane + e;
            const int slot = base + q;
            if (slot < p.A)
                reinterpret_cast<float4*>(cb + slot)[1] =
                    make_float4(best[e], __int_as_float(bc[e]), __int_as_float((int)(a0 + 4 * lane + e)), 0.f);
        }
        before += __popc(m[e]);
    }
    __syncwarp();

    // DFL boxes: lane 4q + side takes side `side` of local candidate q
    for (int t0 = 0; t0 < 4 * total; t0 += 32) {
        const int t = t0 + lane, q = t >> 2, side = t & 3;
        float dist = 0.f;
        long long a = 0;
        if (q < total) {
            a = a0 + s_loc[tw][q];
            const float* z = hb + (size_t)(side * p.R) * p.A + a;
            float v[kMaxRegMax];
#pragma unroll
            for (int i = 0; i < kMaxRegMax; ++i) v[i] = i < p.R ? __ldg(z + (size_t)i * p.A) : -INFINITY;
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kMaxRegMax; ++i) mx = fmaxf(mx, v[i]);
            float zs = 0.f, es = 0.f;
#pragma unroll
            for (int i = 0; i < kMaxRegMax; ++i) {
                if (i < p.R) {
                    const float wgt = expf(v[i] - mx);
                    zs += wgt;
                    es += wgt * (float)i;
                }
            }
            dist = es / zs;
        }
        const float d1 = __shfl_down_sync(kFull, dist, 1), d2 = __shfl_down_sync(kFull, dist, 2),
                    d3 = __shfl_down_sync(kFull, dist, 3);
        if (q < total && side == 0 && base + q < p.A) {
            int l = 0;
            while (l + 1 < p.nlevels && a >= p.off[l + 1]) ++l;
            const long long k = a - p.off[l];
            const float s = (float)p.stride[l];
            const float cx = ((float)(k % p.gw[l]) + 0.5f) * s;
            const float cy = ((float)(k / p.gw[l]) + 0.5f) * s;
            reinterpret_cast<float4*>(cb + base + q)[0] = make_float4(cx - dist * s, cy - d1 * s, cx + d2 * s, cy + d3 * s);
        }
    }
    asm volatile("griddepcontrol.launch_dependents;");
}

__device__ __forceinline__ unsigned long long or_all(unsigned long long v) {
    const unsigned lo = __reduce_or_sync(kFull, (unsigned)v);
    const unsigned hi = __reduce_or_sync(kFull, (unsigned)(v >> 32));
    return ((unsigned long long)hi << 32) | lo;
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

__device__ __forceinline__ void put_sorted(const ws_candidate* cb, int from, int to,
                                           float4* s_box, int* s_cls, float* s_logit, int* s_anchor) {
    const float4* c = reinterpret_cast<const float4*>(cb + from);
    const float4 box = __ldcg(c);
    const float4 rest = __ldcg(c + 1);
    s_box[to] = box;
    s_logit[to] = rest.x;
    s_cls[to] = __float_as_int(rest.y);
    s_anchor[to] = __float_as_int(rest.z);
}

__global__ void __launch_bounds__(kNmsThreads) detect_nms_kernel(const __grid_constant__ DetParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long* s_key = reinterpret_cast<unsigned long long*>(smem);   // [Pcap]
    int* s_idx = reinterpret_cast<int*>(smem + p.off_idx);                     // [Pcap] candidate slot
    float4* s_box = reinterpret_cast<float4*>(smem + p.off_box);                // [max_cand] sorted
    int* s_cls = reinterpret_cast<int*>(smem + p.off_cls);
    float* s_logit = reinterpret_cast<float*>(smem + p.off_logit);
    int* s_anchor = reinterpret_cast<int*>(smem + p.off_anchor);
    int* s_keep = reinterpret_cast<int*>(smem + p.off_keep);
    uint32_t* s_hist = reinterpret_cast<uint32_t*>(smem + p.off_hist);         // [256]
    uint32_t* s_misc = s_hist + 256;                                            // [8]
    unsigned char* s_u = smem + p.off_u;

    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid < 8) s_misc[tid] = 0;
    // the candidates and their count come from the kernel this one may overlap
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const ws_candidate* cb = p.cand + (size_t)b * p.A;
    const int n = (int)min((long long)__ldcg(p.count + b), p.A);
    const int m = min(n, p.max_cand);
    __syncthreads();

    const int Wl = (m + 63) >> 6;
    const int RS = Wl | 1;
    unsigned long long* s_m = reinterpret_cast<unsigned long long*>(s_u);
    unsigned long long* s_tab = reinterpret_cast<unsigned long long*>(s_u + p.off_tab);   // [Wl][kBuckets]
    // Few candidates (the usual case): each thread reads its candidate's
    // 32-byte record once and keeps it in registers; its rank by counting
    // then places the record and sets its class-table bit directly.
    const bool fast = n <= p.max_cand && n <= kCountSortMax;
    if (fast) {
        float4 box = make_float4(0.f, 0.f, 0.f, 0.f), rest = box;
        unsigned long long key = 0ull;
        if (tid < n) {
            const float4* c = reinterpret_cast<const float4*>(cb + tid);
            box = __ldcg(c);
            rest = __ldcg(c + 1);
            key = ((unsigned long long)order_bits(rest.x) << 32) | (uint32_t)(~(uint32_t)__float_as_int(rest.z));
            s_key[tid] = key;
        }
        // the histograms of the cap selection are not used on this path, so
        // the match table can be cleared now
        for (int q = tid; q < Wl * kBuckets; q += kNmsThreads) s_tab[q] = 0ull;
        __syncthreads();
        if (tid < n) {
            int r = 0;
#pragma unroll 4
            for (int j = 0; j < n; ++j) r += s_key[j] > key;
            s_box[r] = box;
            s_logit[r] = rest.x;
            s_cls[r] = __float_as_int(rest.y);
            s_anchor[r] = __float_as_int(rest.z);
            atomicOr(&s_tab[(r >> 6) * kBuckets + (__float_as_int(rest.y) & (kBuckets - 1))], 1ull << (r & 63));
        }
    }

    // 1. the best m candidates' keys
    if (fast) {
    } else if (n <= p.max_cand) {
        for (int i = tid; i < n; i += kNmsThreads) {
            s_key[i] = cand_key(cb + i);
            s_idx[i] = i;
        }
    } else {
        // exact radix select of the m-th largest key, 8 bits a pass; up to
        // kKeysPerThread keys a thread are held in registers, more are re-read
        const bool in_regs = n <= kNmsThreads * kKeysPerThread;
        const int iters = (n + kNmsThreads - 1) / kNmsThreads;
        unsigned long long kr[kKeysPerThread];
        if (in_regs) {
#pragma unroll
            for (int r = 0; r < kKeysPerThread; ++r) {
                const int i = r * kNmsThreads + tid;
                kr[r] = (r < iters && i < n) ? cand_key(cb + i) : 0ull;
            }
        }
        unsigned long long prefix = 0, mask = 0;
        uint32_t remaining = (uint32_t)m;
        uint32_t* s_whist = reinterpret_cast<uint32_t*>(s_u) + warp * 256;   // this warp's histogram
        for (int shift = 56; shift >= 0; shift -= 8) {
            for (int i = tid; i < kNmsWarps * 256; i += kNmsThreads) reinterpret_cast<uint32_t*>(s_u)[i] = 0;
            __syncthreads();
            // Histogram counts, per warp and aggregated over it: up to three times the
            // lanes sharing the first remaining lane's digit add once (the
            // leading passes see only a few distinct digits), then any lanes
            // left add one each.
            auto count = [&](unsigned long long k, bool valid) {
                unsigned act = __ballot_sync(kFull, valid && (k & mask) == prefix);
                const uint32_t d = (uint32_t)(k >> shift) & 255u;
                for (int r = 0; r < 3 && act != 0u; ++r) {
                    const int leader = __ffs(act) - 1;
                    const uint32_t lead = __shfl_sync(kFull, d, leader);
                    const unsigned same = __ballot_sync(kFull, ((act >> lane) & 1u) && d == lead);
                    if (lane == leader) atomicAdd(&s_whist[lead], (uint32_t)__popc(same));
                    act &= ~same;
                }
                if ((act >> lane) & 1u) atomicAdd(&s_whist[d], 1u);
            };
            if (in_regs) {
#pragma unroll
                for (int r = 0; r < kKeysPerThread; ++r)
                    if (r < iters) count(kr[r], r * kNmsThreads + tid < n);
            } else {
                for (int r = 0; r < iters; ++r) {
                    const int i = r * kNmsThreads + tid;
                    count(i < n ? cand_key(cb + i) : 0ull, i < n);
                }
            }
            __syncthreads();
            for (int d = tid; d < 256; d += kNmsThreads) {
                uint32_t h = 0;
#pragma unroll
                for (int w = 0; w < kNmsWarps; ++w) h += reinterpret_cast<const uint32_t*>(s_u)[w * 256 + d];
                s_hist[d] = h;
            }
            __syncthreads();
            if (warp == 0) {
                // lane l holds bins 255 - 8 l .. 248 - 8 l; a scan from the top finds
                // the bin holding the remaining-th largest key
                uint32_t h[8], sum = 0;
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    h[e] = s_hist[255 - 8 * lane - e];
                    sum += h[e];
                }
                uint32_t incl = sum;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const uint32_t v = __shfl_up_sync(kFull, incl, o);
                    if (lane >= o) incl += v;
                }
                uint32_t acc = incl - sum;
                if (acc < remaining && incl >= remaining) {
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (acc + h[e] >= remaining) {
                            s_misc[1] = (uint32_t)(255 - 8 * lane - e);
                            s_misc[2] = remaining - acc;
                            s_misc[4] = (acc + h[e] == remaining);   // the whole bin is in: done
                            break;
                        }
                        acc += h[e];
                    }
                }
            }
            __syncthreads();
            prefix |= (unsigned long long)s_misc[1] << shift;
            mask |= 0xffull << shift;
            remaining = s_misc[2];
            const bool done = s_misc[4] != 0;
            __syncthreads();
            if (done) break;
        }
        // keys are distinct (anchors are), so exactly m keys are >= prefix
        auto place = [&](unsigned long long k, bool valid, int i) {   // called by whole warps
            const bool in = valid && k >= prefix;
            const unsigned bal = __ballot_sync(kFull, in);
            uint32_t base = 0;
            if (lane == 0 && bal) base = atomicAdd(&s_misc[0], (uint32_t)__popc(bal));
            base = __shfl_sync(kFull, base, 0);
            const uint32_t pos = base + (uint32_t)__popc(bal & ((1u << lane) - 1u));
            if (in && pos < (uint32_t)m) {
                s_key[pos] = k;
                s_idx[pos] = i;
            }
        };
        if (in_regs) {
#pragma unroll
            for (int r = 0; r < kKeysPerThread; ++r) {
                const int i = r * kNmsThreads + tid;
                if (r < iters) place(kr[r], i < n, i);
            }
        } else {
            for (int r = 0; r < iters; ++r) {
                const int i = r * kNmsThreads + tid;
                place(i < n ? cand_key(cb + i) : 0ull, i < n, i);
            }
        }
    }
    if (!fast) __syncthreads();

    // 2. descending order: rank by counting when few, else a bitonic sort at
    //    the next power of two of the live count
    if (fast) {
    } else if (m <= kCountSortMax) {
        for (int t = tid; t < m; t += kNmsThreads) {
            const unsigned long long k = s_key[t];
            int r = 0;
#pragma unroll 4
            for (int j = 0; j < m; ++j) r += s_key[j] > k;
            put_sorted(cb, s_idx[t], r, s_box, s_cls, s_logit, s_anchor);
        }
    } else {
        int P = 1;
        while (P < m) P <<= 1;   // 512 or 1024
        for (int i = m + tid; i < P; i += kNmsThreads) s_key[i] = 0ull;   // padding sorts last
        __syncthreads();
        // Warp w holds elements 64 w + lane and 64 w + 32 + lane in registers;
        // stages with j >= 64 go through shared memory, the rest use shuffles.
        const bool active = 64 * warp < P;
        const int e0 = 64 * warp + lane, e1 = e0 + 32;
        unsigned long long x0 = 0, x1 = 0;
        int i0 = 0, i1 = 0;
        if (active) {
            x0 = s_key[e0];
            i0 = s_idx[e0];
            x1 = s_key[e1];
            i1 = s_idx[e1];
        }
        for (int k = 2; k <= P; k <<= 1) {
            if (k >= 128) {
                if (active) {
                    s_key[e0] = x0;
                    s_idx[e0] = i0;
                    s_key[e1] = x1;
                    s_idx[e1] = i1;
                }
                __syncthreads();
                for (int j = k >> 1; j >= 64; j >>= 1) {
                    for (int t = tid; t < (P >> 1); t += kNmsThreads) {
                        const int i = ((t & ~(j - 1)) << 1) | (t & (j - 1));
                        const int ixj = i + j;
                        const unsigned long long x = s_key[i], y = s_key[ixj];
                        const bool desc = (i & k) == 0;
                        if (desc ? (x < y) : (x > y)) {
                            s_key[i] = y;
                            s_key[ixj] = x;
                            const int tmp = s_idx[i];
                            s_idx[i] = s_idx[ixj];
                            s_idx[ixj] = tmp;
                        }
                    }
                    __syncthreads();
                }
                if (active) {
                    x0 = s_key[e0];
                    i0 = s_idx[e0];
                    x1 = s_key[e1];
                    i1 = s_idx[e1];
                }
            }
            if (active) {
                for (int j = min(k >> 1, 32); j >= 1; j >>= 1) {
                    if (j == 32) {
                        const bool desc = (e0 & k) == 0;
                        if (desc ? (x0 < x1) : (x0 > x1)) {
                            const unsigned long long tx = x0;
                            x0 = x1;
                            x1 = tx;
                            const int ti = i0;
                            i0 = i1;
                            i1 = ti;
                        }
                    } else {
                        const unsigned long long y0 = __shfl_xor_sync(kFull, x0, j), y1 = __shfl_xor_sync(kFull, x1, j);
                        const int j0 = __shfl_xor_sync(kFull, i0, j), j1 = __shfl_xor_sync(kFull, i1, j);
                        // the lower element of a pair keeps the larger key when the run is descending
                        const bool hi0 = ((e0 & j) == 0) == ((e0 & k) == 0);
                        const bool hi1 = ((e1 & j) == 0) == ((e1 & k) == 0);
                        if (hi0 ? (y0 > x0) : (y0 < x0)) {
                            x0 = y0;
                            i0 = j0;
                        }
                        if (hi1 ? (y1 > x1) : (y1 < x1)) {
                            x1 = y1;
                            i1 = j1;
                        }
                    }
                }
            }
        }
        if (active) {
            if (e0 < m) put_sorted(cb, i0, e0, s_box, s_cls, s_logit, s_anchor);
            if (e1 < m) put_sorted(cb, i1, e1, s_box, s_cls, s_logit, s_anchor);
        }
    }
    __syncthreads();

    // 3. suppression bits: row i holds bit j (j > i, same class, IoU above the
    //    threshold) in word j / 64; words below i / 64 are never read.  A table
    //    holds, per word and class bucket (class mod kBuckets), the mask of the
    //    word's candidates in that bucket, so a (row, word) task finds its
    //    class matches with one load and takes the IoU only for those.  The
    //    odd row stride keeps the row-parallel stores apart.
    if (!fast) {
        for (int q = tid; q < Wl * kBuckets; q += kNmsThreads) s_tab[q] = 0ull;
        __syncthreads();
        for (int q = tid; q < m; q += kNmsThreads)
            atomicOr(&s_tab[(q >> 6) * kBuckets + (s_cls[q] & (kBuckets - 1))], 1ull << (q & 63));
        __syncthreads();
    }
    for (int t = tid; t < m * Wl; t += kNmsThreads) {
        const int w = t / m, i = t - w * m;
        if (w < (i >> 6)) continue;
        const int ci = s_cls[i];
        const int lo = i + 1 - 64 * w;   // bits lo .. 63 (the table holds no bit at or above m)
        unsigned long long match = lo >= 64 ? 0ull : s_tab[w * kBuckets + (ci & (kBuckets - 1))];
        if (lo > 0) match &= ~((1ull << lo) - 1ull);
        unsigned long long bits = 0;
        if (match != 0ull) {
            const float4 bi = s_box[i];
            while (match != 0ull) {
                const int bit = __ffsll((long long)match) - 1;
                match &= match - 1ull;
                const int j = 64 * w + bit;
                if (s_cls[j] == ci && iou_above(bi, s_box[j], p.iou_thr)) bits |= 1ull << bit;
            }
        }
        s_m[(size_t)i * RS + w] = bits;
    }
    __syncthreads();

    // 4. greedy walk by one warp, a 64-candidate word at a time.  A word
    //    starts with the bits that the boxes kept so far suppress in it (each
    //    lane ORs that word of every 32nd kept row).  Then, every live
    //    candidate that no live candidate of the word suppresses is kept
    //    (nothing before it that could still be kept removes it); those
    //    remove what they suppress, and the step repeats until the word is
    //    decided -- the greedy result, in as many steps as the longest chain
    //    of suppressions inside the word.  Lane l holds the word's rows l and
    //    l + 32.
    if (warp == 0) {
        int nk = 0;
        for (int w = 0; w < Wl && nk < p.max_det; ++w) {
            const int r0 = 64 * w + lane, r1 = r0 + 32;
            const unsigned long long d0 = r0 < m ? s_m[(size_t)r0 * RS + w] : 0ull;
            const unsigned long long d1 = r1 < m ? s_m[(size_t)r1 * RS + w] : 0ull;
            unsigned long long mine = 0;
            for (int q = lane; q < nk; q += 32) mine |= s_m[(size_t)s_keep[q] * RS + w];
            unsigned long long cur = ~or_all(mine);
            const int live = m - 64 * w;
            if (live < 64) cur &= (1ull << live) - 1ull;
            unsigned long long kept = 0;
            while (cur != 0ull) {
                mine = (((cur >> lane) & 1ull) ? d0 : 0ull) | (((cur >> (lane + 32)) & 1ull) ? d1 : 0ull);
                const unsigned long long sure = cur & ~or_all(mine);
                mine = (((sure >> lane) & 1ull) ? d0 : 0ull) | (((sure >> (lane + 32)) & 1ull) ? d1 : 0ull);
                const unsigned long long gone = or_all(mine);
                kept |= sure;
                cur &= ~(sure | gone);
            }
            // kept boxes in order, at most max_det in all
            if ((kept >> lane) & 1ull) {
                const int pos = nk + __popcll(kept & ((1ull << lane) - 1ull));
                if (pos < p.max_det) s_keep[pos] = r0;
            }
            if ((kept >> (lane + 32)) & 1ull) {
                const int pos = nk + __popcll(kept & ((1ull << (lane + 32)) - 1ull));
                if (pos < p.max_det) s_keep[pos] = r1;
            }
            __syncwarp();
            nk = min(nk + __popcll(kept), p.max_det);
        }
        if (lane == 0) s_misc[3] = (uint32_t)nk;
    }
    __syncthreads();

    // 5. detections in keep order
    const int nk = (int)s_misc[3];
    for (int q = tid; q < nk; q += kNmsThreads) {
        const int i = s_keep[q];
        float4* dst = reinterpret_cast<float4*>(p.out + (size_t)b * p.max_det + q);
        dst[0] = s_box[i];
        dst[1] = make_float4(1.0f / (1.0f + expf(-s_logit[i])), __int_as_float(s_cls[i]), __int_as_float(s_anchor[i]),
                             0.f);
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
    p.Pcap = 2;
    while (p.Pcap < d->max_cand) p.Pcap <<= 1;
    size_t o = (size_t)p.Pcap * 8;
    p.off_idx = (int)o;        o = align16(o + (size_t)p.Pcap * 4);
    p.off_box = (int)o;        o = align16(o + (size_t)d->max_cand * 16);
    p.off_cls = (int)o;        o = align16(o + (size_t)d->max_cand * 4);
    p.off_logit = (int)o;      o = align16(o + (size_t)d->max_cand * 4);
    p.off_anchor = (int)o;     o = align16(o + (size_t)d->max_cand * 4);
    p.off_keep = (int)o;       o = align16(o + (size_t)d->max_cand * 4);
    p.off_hist = (int)o;       o = align16(o + (256 + 8) * 4);
    p.off_u = (int)o;
    // the suppression matrix: max_cand rows of ceil(max_cand / 64) words, the
    // row stride made odd; then the class-bucket match table
    const int W = (d->max_cand + 63) / 64;
    p.off_tab = (int)align16((size_t)d->max_cand * (W | 1) * 8);
    p.u_bytes = p.off_tab + W * kBuckets * 8;
    // the cap selection's per-warp histograms share this area
    p.u_bytes = std::max(p.u_bytes, kNmsWarps * 256 * 4);
    return WS_OK;
}

size_t nms_smem(const DetParams& p) { return (size_t)p.off_u + (size_t)p.u_bytes; }

size_t det_workspace(const DetParams& p, int32_t batch) {
    return (size_t)(batch * 4 + 255) / 256 * 256 + (size_t)batch * p.A * sizeof(ws_candidate);
}

std::atomic<bool> g_nms_attr_set[64];

// Few tiles in all: split each tile's classes over kDecodeSplit warps.
bool decode_split(int tiles, int32_t batch) { return (long long)tiles * batch <= kDecodeSplitTiles; }

ws_status launch_decode(DetParams p, int32_t batch, cudaStream_t stream) {
    const int tiles = (int)((p.A + kDecodeAnchors - 1) / kDecodeAnchors);
    const bool vec = p.A % 4 == 0 && (uintptr_t)p.head % 16 == 0;
    // one kernel, a programmatic dependent of whatever wrote the head
    cudaError_t e;
    if (decode_split(tiles, batch)) {
        const dim3 grid((unsigned)tiles, (unsigned)batch);
        e = vec ? launch_pdl(detect_decode_warp_kernel<true, kDecodeSplit>, grid, dim3(32 * kDecodeSplit), 0, stream, p)
                : launch_pdl(detect_decode_warp_kernel<false, kDecodeSplit>, grid, dim3(32 * kDecodeSplit), 0, stream, p);
    } else {
        const dim3 grid((unsigned)((tiles + kWarpScanWarps - 1) / kWarpScanWarps), (unsigned)batch);
        e = vec ? launch_pdl(detect_decode_warp_kernel<true, 1>, grid, dim3(32 * kWarpScanWarps), 0, stream, p)
                : launch_pdl(detect_decode_warp_kernel<false, 1>, grid, dim3(32 * kWarpScanWarps), 0, stream, p);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return WS_OK;
}

// The NMS is a programmatic dependent launch ("Streams, concurrency and CUDA
// Graphs", PDL section): it may be scheduled while the decode drains and
// waits in griddepcontrol.wait for the decode's results.
ws_status launch_nms(const DetParams& p, int32_t batch, cudaStream_t stream) {
    int dev;
    const DeviceInfo* info;
    ws_status st = current_device_info(&dev, &info);
    if (st != WS_OK) return st;
    const size_t smem = nms_smem(p);
    if (smem > (size_t)info->max_smem_optin) return fail(WS_ERR_UNSUPPORTED, "NMS needs %zu bytes of shared memory", smem);
    if (dev < 0 || dev >= 64) return fail(WS_ERR_UNSUPPORTED, "device ordinal %d", dev);
    if (!g_nms_attr_set[dev].load(std::memory_order_acquire)) {
        WS_TRY_CUDA(cudaFuncSetAttribute(detect_nms_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         info->max_smem_optin));
        g_nms_attr_set[dev].store(true, std::memory_order_release);
    }
    const cudaError_t e = launch_pdl(detect_nms_kernel, dim3((unsigned)batch), dim3(kNmsThreads), smem, stream, p);
    if (e != cudaSuccess) return cuda_fail(e, "NMS launch");
    return WS_OK;
}

}  // namespace
}  // namespace ws

extern "C" {

ws_status ws_detect_validate(const ws_detect_desc* desc, int32_t batch, int64_t* anchors) {
    ws::clear_error();
    ws::DetParams p{};
    ws_status st = ws::fill_params(desc, batch, p);
    if (st == WS_OK && anchors) *anchors = p.A;
    return st;
}

ws_status ws_detect_workspace_bytes(const ws_detect_desc* desc, int32_t batch, size_t* bytes) {
    ws::clear_error();
    if (!bytes) return ws::fail(WS_ERR_INVALID_ARGUMENT, "bytes is NULL");
    ws::DetParams p{};
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
    ws::DetParams p{};
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
    ws::DetParams p{};
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
    ws::DetParams p{};
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
