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
//    numbered in anchor order, and the same warp then takes their DFL: four
//    lanes per candidate, one per side, load that side's reg_max logits and
//    take the softmax expectation.  All tiles stream at once; a warp's
//    scattered DFL loads overlap the other warps' class rows.  With few tiles
//    a block of four warps splits a tile's classes and then its DFL work.
//  * NMS: launched as a programmatic dependent of the decode kernel so its
//    launch overlaps the decode's tail; a thread-block cluster of up to 8
//    CTAs per image when the batch leaves room.  An image with at most 256
//    candidates runs on one CTA: two threads rank each candidate by counting.
//    Above that, one CTA alone (large batches) takes a radix select of the
//    best max_cand keys (64-bit: logit order bits, then the complemented
//    anchor) and a bitonic sort; a cluster shares the work: the radix select
//    sums its histograms over distributed shared memory, each CTA sorts its
//    run of the kept keys, a key's rank is its position summed over the
//    sorted runs, and the suppression matrix is split between the CTAs.
//    Every pair's suppression test (same class, IoU > threshold) is evaluated
//    in parallel into a word-major bit matrix, a thread per (row, 64-bit
//    word), the IoU only where a class-bucket table shows a match, and one
//    warp walks the sorted list a 64-candidate word at a time, deciding at
//    each step every candidate that nothing live can still suppress.  The IoU
//    test is FP32 with every operation rounded separately (no fused
//    multiply-add), so given the same boxes the decisions are exactly those of
//    the definition.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>


#include "ws_internal.cuh"
#include "ws_ptx.cuh"

namespace ws {
namespace {

constexpr int kDecodeAnchors = 128;                    // anchors per decode tile: 4 per lane
constexpr int kLaneAnchors = 4;
constexpr int kWarpScanWarps = 4;                      // warps (tiles) per decode block
constexpr int kWarpScanLoads = 8;                      // class rows in flight per lane
constexpr int kWideLoads = 20;                         // ... in the one-block-per-SM split form
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
// arg-maxes (value, then the lower class) through shared memory and reserves
// the candidates' slots; then all kSplit warps share the DFL work.  A warp's
// chain of dependent loads (class rows, then DFL rounds) is then kSplit times
// shorter.
// kWide (with kSplit > 1, when the launch has at most one block per SM, e.g.
// one 640x640 image): each warp loads up to kWideLoads class rows at once, one
// round trip for a quarter of 80 classes, at up to 128 registers.
template <bool kVec, int kSplit, int kR, bool kWide = false>
__global__ void __launch_bounds__(32 * (kSplit == 1 ? kWarpScanWarps : kSplit), kWide ? 4 : 8)
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
        if constexpr (kWide) {
            for (int c = cbeg; c < cend; c += kWideLoads) {
                float4 v4[kWideLoads];
#pragma unroll
                for (int u = 0; u < kWideLoads; ++u)
                    v4[u] = c + u < cend ? load(c + u) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
#pragma unroll
                for (int u = 0; u < kWideLoads; ++u)
                    if (c + u < cend) take4(best, bc, v4[u], c + u);
            }
        } else {
            int c = cbeg;
            for (; c + kWarpScanLoads <= cend; c += kWarpScanLoads) {
                float4 v4[kWarpScanLoads];
#pragma unroll
                for (int u = 0; u < kWarpScanLoads; ++u) v4[u] = load(c + u);
#pragma unroll
                for (int u = 0; u < kWarpScanLoads; ++u) take4(best, bc, v4[u], c + u);
            }
            for (; c < cend; ++c) take4(best, bc, load(c), c);
        }
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
        if (w == 0) {
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
    }

    // candidates: one ballot per anchor position, slots from one atomic (warp
    // 0 of the block when kSplit > 1)
    __shared__ int s_total, s_base;
    ws_candidate* cb = p.cand + (size_t)b * p.A;
    int total = 0, base = 0;
    if (kSplit == 1 || w == 0) {
        const unsigned lt = (1u << lane) - 1u;
        unsigned m[kLaneAnchors];
#pragma unroll
        for (int e = 0; e < kLaneAnchors; ++e) {
            m[e] = __ballot_sync(kFull, a0 + 4 * lane + e < p.A && best[e] > p.logit_thr);
            total += __popc(m[e]);
        }
        if (total > 0) {
            if (lane == 0) base = atomicAdd(&p.count[b], total);
            base = __shfl_sync(kFull, base, 0);
            // candidates numbered in anchor order (the lower lanes' anchors,
            // then this lane's lower ones), so that neighbouring DFL tasks
            // read neighbouring anchors
            int q = 0;
#pragma unroll
            for (int e = 0; e < kLaneAnchors; ++e) q += __popc(m[e] & lt);
#pragma unroll
            for (int e = 0; e < kLaneAnchors; ++e) {
                if ((m[e] >> lane) & 1u) {
                    s_loc[tw][q] = 4 * lane + e;
                    const int slot = base + q;
                    if (slot < p.A)
                        reinterpret_cast<float4*>(cb + slot)[1] =
                            make_float4(best[e], __int_as_float(bc[e]), __int_as_float((int)(a0 + 4 * lane + e)), 0.f);
                    ++q;
                }
            }
        }
        if (kSplit > 1 && lane == 0) {
            s_total = total;
            s_base = base;
        }
        __syncwarp();
    }
    if (kSplit > 1) {   // every warp of the block takes a share of the DFL work
        __syncthreads();
        total = s_total;
        base = s_base;
    }
    if (total == 0) {
        asm volatile("griddepcontrol.launch_dependents;");
        return;
    }

    // DFL boxes: lane 4q + side takes side `side` of local candidate q; with
    // kSplit > 1 the block's warps take turns of 32 (candidate, side) tasks
    for (int t0 = (kSplit > 1 ? w : 0) * 32; t0 < 4 * total; t0 += 32 * kSplit) {
        const int t = t0 + lane, q = t >> 2, side = t & 3;
        float dist = 0.f;
        long long a = 0;
        if (q < total) {
            a = a0 + s_loc[tw][q];
            const float* z = hb + (size_t)(side * p.R) * p.A + a;
            float v[kR];
#pragma unroll
            for (int i = 0; i < kR; ++i) v[i] = i < p.R ? __ldg(z + (size_t)i * p.A) : -INFINITY;
            float mx = -INFINITY;
#pragma unroll
            for (int i = 0; i < kR; ++i) mx = fmaxf(mx, v[i]);
            float zs = 0.f, es = 0.f;
#pragma unroll
            for (int i = 0; i < kR; ++i) {
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

// One key per lane into a radix-select histogram (whole warps call it):
// the lanes whose key matches the prefix so far count its digit at `shift`.
// Up to three times, the lanes sharing the first remaining lane's digit add
// once (the leading passes see only a few distinct digits); any lanes left
// add one each.
__device__ __forceinline__ void hist_count(uint32_t* h, unsigned long long k, bool valid, unsigned long long mask,
                                           unsigned long long prefix, int shift, int lane) {
    unsigned act = __ballot_sync(kFull, valid && (k & mask) == prefix);
    const uint32_t d = (uint32_t)(k >> shift) & 255u;
    for (int r = 0; r < 3 && act != 0u; ++r) {
        const int leader = __ffs(act) - 1;
        const uint32_t lead = __shfl_sync(kFull, d, leader);
        const unsigned same = __ballot_sync(kFull, ((act >> lane) & 1u) && d == lead);
        if (lane == leader) atomicAdd(&h[lead], (uint32_t)__popc(same));
        act &= ~same;
    }
    if ((act >> lane) & 1u) atomicAdd(&h[d], 1u);
}

// Warp 0: the bin of the 256-bin histogram `hist` that holds the
// remaining-th largest key.  Writes the digit to misc[1], the count still
// wanted inside that bin to misc[2], and misc[4] = 1 when the whole bin is
// in (the selection is then complete).  Lane l holds bins 255 - 8 l ..
// 248 - 8 l, so a scan from the top finds it.
__device__ __forceinline__ void find_digit(const uint32_t* hist, uint32_t remaining, uint32_t* misc, int lane) {
    uint32_t h[8], sum = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        h[e] = hist[255 - 8 * lane - e];
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
                misc[1] = (uint32_t)(255 - 8 * lane - e);
                misc[2] = remaining - acc;
                misc[4] = (acc + h[e] == remaining);
                break;
            }
            acc += h[e];
        }
    }
}

// Word w of row i of the suppression matrix: bit j - 64 w set when sorted
// candidate j (j > i) has i's class and IoU(i, j) above the threshold.  The
// class-bucket table holds, per 64-candidate word and bucket (class mod
// kBuckets), the mask of the word's candidates in the bucket, so a task finds
// its class matches with one load and takes the IoU only for those.
__device__ __forceinline__ unsigned long long suppress_word(const float4* s_box, const int* s_cls,
                                                           const unsigned long long* s_tab, int i, int w, float thr) {
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
            if (s_cls[j] == ci && iou_above(bi, s_box[j], thr)) bits |= 1ull << bit;
        }
    }
    return bits;
}

// A CTA's NMS shared memory (the same layout in every CTA of a cluster).
struct NmsSmem {
    unsigned long long* key;   // [Pcap]
    int* idx;                  // [Pcap] candidate slot
    float4* box;               // [max_cand] sorted
    int* cls;
    float* logit;
    int* anchor;
    int* keep;
    uint32_t* hist;            // [256]
    uint32_t* misc;            // [8]
    unsigned char* u;          // histograms, later the suppression matrix, and the match table
};

// The sum of a shared word over the cluster's CTAs 0 .. ranks - 1 (at most
// kMaxCluster): every remote load is issued before the first is used.
constexpr int kMaxCluster = 8;
// Cluster NMS: runs of at least kSplitRun keys on average (2 CTAs an image,
// up to 1024 keys) are sorted in sub-runs of kSubRun keys; shorter runs are
// sorted whole, so a key is ranked against G sorted runs.  Measured on GB300
// (every anchor a candidate, ws_detect): sub-runs of 256 at 2 CTAs an image
// 130.9 -> 125.5 us at batch 64; sub-runs at 4 or 8 CTAs an image (runs of
// about 256 and 128 keys, often split one key past the length) cost more
// ranking lanes than the sort saves (batch 1: 36.6 -> 38.0 us with sub-runs
// of 128).
constexpr int kSubRun = 256;
constexpr int kSplitRun = 384;
__device__ __forceinline__ uint32_t sum_over_cluster(const uint32_t* p, int ranks) {
    uint32_t v[kMaxCluster];
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) v[c] = c < ranks ? ld_cluster_u32(cluster_map(p, (uint32_t)c)) : 0u;
    uint32_t t = 0;
#pragma unroll
    for (int c = 0; c < kMaxCluster; ++c) t += v[c];
    return t;
}

// Number of keys above k in a run sorted in descending order (keys distinct).
__device__ __forceinline__ int count_above(const unsigned long long* run, int len, unsigned long long k) {
    int lo = 0, hi = len;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (run[mid] > k)
            lo = mid + 1;
        else
            hi = mid;
    }
    return lo;
}

// Steps 1-3 for an image with more than kCountSortMax candidates, by the G
// CTAs of its cluster (rank 0 then walks the matrix and writes the result).
//  1. The best m keys as G runs, one per CTA.  Selection (n > max_cand): CTA
//     r holds the keys of candidate slots [r n / G, (r + 1) n / G) in
//     registers.  Each radix pass counts them into the CTA's histogram (two
//     buffers, by pass parity); after a cluster barrier every CTA sums the G
//     histograms through distributed shared memory, so all take the same
//     digit.  CTA r's run is then its keys at or above the selected prefix
//     (exactly m over the cluster), at list positions after the lower ranks'
//     runs.  With n <= max_cand every CTA reads all n keys, and CTA r's run is
//     list positions [r m / G, (r + 1) m / G).
//  2. Order.  Each CTA sorts its run, whole or (long runs) in sub-runs of
//     kSubRun keys, by counting within each (1 .. 32 threads per key), and
//     writes it back in place;
//     every CTA then copies the other runs (coalesced remote loads), so all
//     hold the same list of sorted sub-runs.  A key's rank is the number of
//     keys above it summed over the sub-runs (a binary search in each, one
//     lane per sub-run); each CTA ranks its own run's keys, then reads the
//     other CTAs' ranks, so it knows the candidate slot at every sorted
//     position, and loads the sorted records from global memory itself.
//  3. Suppression matrix: each CTA builds the class-bucket table and computes
//     a contiguous G-th of the (row, word) tasks in word order, storing them
//     into rank 0's matrix (word-major, so a warp's stores are consecutive).
// Every CTA passes the same sequence of cluster barriers: n, m and each
// pass's summed histogram are the same in all of them.  Remote shared memory
// is only touched between barriers that its owner also passes, so no CTA
// reads or writes one that has exited.
__device__ __forceinline__ void nms_cluster_build(const DetParams& p, const NmsSmem& s, const ws_candidate* cb,
                                                  int n, int m, int G, int rank) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    int bound[kMaxCluster + 1];   // run c holds list positions bound[c] .. bound[c + 1] - 1
    const unsigned long long* run_key;   // this CTA's run, unsorted
    const int* run_idx;
    if (n <= p.max_cand) {
        for (int i = tid; i < n; i += kNmsThreads) {
            s.key[i] = cand_key(cb + i);
            s.idx[i] = i;
        }
#pragma unroll
        for (int c = 0; c <= kMaxCluster; ++c) bound[c] = (int)((long long)m * min(c, G) / G);
        const int r0 = (int)((long long)m * rank / G);
        run_key = s.key + r0;
        run_idx = s.idx + r0;
    } else {
        const int lo = (int)((long long)n * rank / G);
        const int cnt = (int)((long long)n * (rank + 1) / G) - lo;
        const bool in_regs = cnt <= kNmsThreads * kKeysPerThread;
        const int iters = (cnt + kNmsThreads - 1) / kNmsThreads;
        unsigned long long kr[kKeysPerThread];
        if (in_regs) {
#pragma unroll
            for (int r = 0; r < kKeysPerThread; ++r) {
                const int i = r * kNmsThreads + tid;
                kr[r] = (r < iters && i < cnt) ? cand_key(cb + lo + i) : 0ull;
            }
        }
        uint32_t* hbuf = reinterpret_cast<uint32_t*>(s.u);
        unsigned long long prefix = 0, mask = 0;
        uint32_t remaining = (uint32_t)m;
        int pass = 0;
        // pass 0's histogram is cleared here; each later pass's in the pass
        // before it (below)
        for (int d = tid; d < 256; d += kNmsThreads) hbuf[d] = 0;
        __syncthreads();
        for (int shift = 56; shift >= 0; shift -= 8, ++pass) {
            uint32_t* h = hbuf + (pass & 1) * 256;
            if (in_regs) {
#pragma unroll
                for (int r = 0; r < kKeysPerThread; ++r)
                    if (r < iters) hist_count(h, kr[r], r * kNmsThreads + tid < cnt, mask, prefix, shift, lane);
            } else {
                for (int r = 0; r < iters; ++r) {
                    const int i = r * kNmsThreads + tid;
                    hist_count(h, i < cnt ? cand_key(cb + lo + i) : 0ull, i < cnt, mask, prefix, shift, lane);
                }
            }
            cluster_sync();
            // Every CTA has read the other buffer (the previous pass's sums
            // came before this barrier): clear it for the next pass.  The
            // barriers below order the clear before the next pass's counts,
            // and this pass's reads of s.misc before the next pass's
            // find_digit (after its cluster barrier).
            for (int d = tid; d < 256; d += kNmsThreads) hbuf[((pass + 1) & 1) * 256 + d] = 0;
            if (tid < 256) s.hist[tid] = sum_over_cluster(h + tid, G);
            __syncthreads();
            if (warp == 0) find_digit(s.hist, remaining, s.misc, lane);
            __syncthreads();
            prefix |= (unsigned long long)s.misc[1] << shift;
            mask |= 0xffull << shift;
            remaining = s.misc[2];
            if (s.misc[4] != 0) break;
        }
        // this CTA's kept keys per warp (s.hist is free after the last pass)
        int wcount = 0;
        if (in_regs) {
#pragma unroll
            for (int r = 0; r < kKeysPerThread; ++r)
                if (r < iters) wcount += __popc(__ballot_sync(kFull, r * kNmsThreads + tid < cnt && kr[r] >= prefix));
        } else {
            for (int r = 0; r < iters; ++r) {
                const int i = r * kNmsThreads + tid;
                wcount += __popc(__ballot_sync(kFull, i < cnt && cand_key(cb + lo + i) >= prefix));
            }
        }
        if (lane == 0) s.hist[warp] = (uint32_t)wcount;
        __syncthreads();
        uint32_t pos = 0, ctot = 0;
#pragma unroll
        for (int w = 0; w < kNmsWarps; ++w) {
            const uint32_t c = s.hist[w];
            pos += w < warp ? c : 0u;
            ctot += c;
        }
        if (tid == 0) s.misc[5] = ctot;
        cluster_sync();
        {
            uint32_t v[kMaxCluster];
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) v[c] = c < G ? ld_cluster_u32(cluster_map(&s.misc[5], (uint32_t)c)) : 0u;
            bound[0] = 0;
#pragma unroll
            for (int c = 0; c < kMaxCluster; ++c) bound[c + 1] = bound[c] + (int)v[c];
        }
        // the run, unsorted, into the (now free) histogram area: warp by
        // warp, key slot by key slot, lanes in order
        unsigned long long* st_key = reinterpret_cast<unsigned long long*>(s.u);
        int* st_idx = reinterpret_cast<int*>(s.u + (size_t)8 * p.max_cand);
        auto stage = [&](unsigned long long k, bool in, int i) {   // called by whole warps
            const unsigned bal = __ballot_sync(kFull, in);
            if (in) {
                const uint32_t at = pos + (uint32_t)__popc(bal & lt);
                st_key[at] = k;
                st_idx[at] = lo + i;
            }
            pos += (uint32_t)__popc(bal);
        };
        if (in_regs) {
#pragma unroll
            for (int r = 0; r < kKeysPerThread; ++r) {
                const int i = r * kNmsThreads + tid;
                if (r < iters) stage(kr[r], i < cnt && kr[r] >= prefix, i);
            }
        } else {
            for (int r = 0; r < iters; ++r) {
                const int i = r * kNmsThreads + tid;
                const unsigned long long k = i < cnt ? cand_key(cb + lo + i) : 0ull;
                stage(k, i < cnt && k >= prefix, i);
            }
        }
        run_key = st_key;
        run_idx = st_idx;
    }
    __syncthreads();

    // 2. this CTA's run, list positions bound[rank] .. bound[rank + 1] - 1,
    //    sorted whole or in sub-runs of kSubRun keys (by counting within each)
    const bool split = m / G >= kSplitRun;   // the same in every CTA
    const int sub = split ? kSubRun : kMaxCand;   // a power of two at least L when the runs are whole
    int off = 0, L = 0;
#pragma unroll
    for (int d = 0; d < kMaxCluster; ++d)
        if (d == rank) {
            off = bound[d];
            L = bound[d + 1] - bound[d];
        }
    {
        int tpk = 1;   // threads per key (consecutive lanes); part p counts keys p, p + tpk, ...
        while (tpk < 32 && 2 * tpk * L <= kNmsThreads) tpk <<= 1;
        const int part = tid & (tpk - 1), per = kNmsThreads / tpk;
        // at most two rounds: L <= m <= 1024 keys, and tpk >= 2 only when tpk L <= 256
        unsigned long long hk[2];
        int hx[2], hr[2];
#pragma unroll
        for (int it = 0; it < 2; ++it) {
            const int e = it * per + tid / tpk;
            const bool act = e < L;
            const unsigned long long k = act ? run_key[e] : 0ull;
            const int sb = e & ~(sub - 1);   // this key's sub-run: sb .. sb + sub - 1
            int r = 0;
            if (act) {
                const int se = min(L, sb + sub);
#pragma unroll 4
                for (int q = sb + part; q < se; q += tpk) r += run_key[q] > k;
            }
            for (int o = 1; o < tpk; o <<= 1) r += __shfl_xor_sync(kFull, r, o);
            hk[it] = k;
            hx[it] = act ? run_idx[e] : 0;
            hr[it] = act && part == 0 ? sb + r : -1;
        }
        __syncthreads();   // the run is read; the direct case writes it back in place
#pragma unroll
        for (int it = 0; it < 2; ++it)
            if (hr[it] >= 0) {
                s.key[off + hr[it]] = hk[it];
                s.idx[off + hr[it]] = hx[it];
            }
    }
    cluster_sync();
    // the other runs, from their CTAs (coalesced remote loads)
    for (int q = tid; q < m; q += kNmsThreads) {
        int c = 0;
#pragma unroll
        for (int d = 1; d < kMaxCluster; ++d) c += (d < G && q >= bound[d]) ? 1 : 0;
        if (c != rank) {
            s.key[q] = ld_cluster_u64(cluster_map(s.key + q, (uint32_t)c));
            s.idx[q] = (int)ld_cluster_u32(cluster_map(s.idx + q, (uint32_t)c));
        }
    }
    const int Wl = (m + 63) >> 6, MS = (m + 1) & ~1;
    unsigned long long* s_tab = reinterpret_cast<unsigned long long*>(s.u + p.off_tab);   // [Wl][kBuckets]
    for (int q = tid; q < Wl * kBuckets; q += kNmsThreads) s_tab[q] = 0ull;   // the staging area is done with
    __syncthreads();
    // Ranks of this run's keys: a key's rank is the number of larger keys summed
    // over the sorted runs (whole runs: G lanes per key, lane c searching run
    // c) or over every sorted sub-run of every CTA's run (at most 12: m <= 1024
    // keys in sub-runs of 256 plus one partial sub-run per CTA; lpk lanes per
    // key, lane q searching sub-run q).
    int* rank_of = s.keep;         // [m] ranks of this CTA's list positions (read by the other CTAs)
    int* sorted_slot = s.anchor;   // [m] the candidate slot at each sorted position
    if (!split) {
        for (int t0 = 0; t0 < L * G; t0 += kNmsThreads) {   // the same trip count in every thread
            const int t = t0 + tid, e = t / G, c = t - e * G;
            const bool act = e < L;
            int r = 0;
            if (act) {
                int b0 = 0, b1 = 0;
#pragma unroll
                for (int d = 0; d < kMaxCluster; ++d)
                    if (d == c) {
                        b0 = bound[d];
                        b1 = bound[d + 1];
                    }
                r = count_above(s.key + b0, b1 - b0, s.key[off + e]);
            }
            for (int o = 1; o < G; o <<= 1) r += __shfl_xor_sync(kFull, r, o);
            if (act && c == 0) rank_of[off + e] = r;
        }
    } else {
        constexpr int kSubShift = 8;   // log2(kSubRun)
        static_assert((1 << kSubShift) == kSubRun, "sub-run shift");
        int nsub[kMaxCluster];
        int nr = 0;
#pragma unroll
        for (int c = 0; c < kMaxCluster; ++c) {
            nsub[c] = (bound[c + 1] - bound[c] + kSubRun - 1) >> kSubShift;
            nr += nsub[c];
        }
        int lpk = 1;   // lanes per key
        while (lpk < nr) lpk <<= 1;
        for (int t0 = 0; t0 < L * lpk; t0 += kNmsThreads) {   // the same trip count in every thread
            const int t = t0 + tid, e = t / lpk, q = t - e * lpk;
            int r = 0;
            if (e < L && q < nr) {
                int b0 = 0, b1 = 0, j = q;   // sub-run q: of run c, its sub-run j
#pragma unroll
                for (int c = 0; c < kMaxCluster; ++c) {
                    if (j >= 0 && j < nsub[c]) {
                        b0 = bound[c] + (j << kSubShift);
                        b1 = min(bound[c + 1], b0 + kSubRun);
                    }
                    j -= nsub[c];
                }
                r = count_above(s.key + b0, b1 - b0, s.key[off + e]);
            }
            for (int o = 1; o < lpk; o <<= 1) r += __shfl_xor_sync(kFull, r, o);
            if (e < L && q == 0) rank_of[off + e] = r;
        }
    }
    cluster_sync();
    for (int j = tid; j < m; j += kNmsThreads) {
        int c = 0;
#pragma unroll
        for (int d = 1; d < kMaxCluster; ++d) c += (d < G && j >= bound[d]) ? 1 : 0;
        sorted_slot[ld_cluster_u32(cluster_map(rank_of + j, (uint32_t)c))] = s.idx[j];
    }
    __syncthreads();
    // the sorted records (rank 0 also keeps logits and anchors for the output;
    // a thread reads sorted_slot[q] before it writes the anchor there)
    for (int q = tid; q < m; q += kNmsThreads) {
        const float4* c4 = reinterpret_cast<const float4*>(cb + sorted_slot[q]);
        const float4 box = __ldcg(c4);
        const float4 rest = __ldcg(c4 + 1);
        s.box[q] = box;
        s.cls[q] = __float_as_int(rest.y);
        if (rank == 0) {
            s.logit[q] = rest.x;
            s.anchor[q] = __float_as_int(rest.z);
        }
    }
    __syncthreads();

    // 3. the match table, then this CTA's share of the tasks into rank 0's matrix
    for (int q = tid; q < m; q += kNmsThreads)
        atomicOr(&s_tab[(q >> 6) * kBuckets + (s.cls[q] & (kBuckets - 1))], 1ull << (q & 63));
    __syncthreads();
    // The tasks (i, w) with i < min(m, 64 (w + 1)), word by word, split into G
    // contiguous ranges: a warp takes consecutive rows of one word.
    unsigned long long* s_m = reinterpret_cast<unsigned long long*>(s.u);
    int total = 0;
    for (int w = 0; w < Wl; ++w) total += min(m, 64 * (w + 1));
    const int t1 = (int)((long long)total * (rank + 1) / G);
    int w = 0, first = 0;   // the word of task t and its first task
    for (int t = (int)((long long)total * rank / G) + tid; t < t1; t += kNmsThreads) {
        while (t >= first + min(m, 64 * (w + 1))) {
            first += min(m, 64 * (w + 1));
            ++w;
        }
        const int i = t - first;
        st_cluster_u64(cluster_map(s_m + (size_t)w * MS + i, 0u), suppress_word(s.box, s.cls, s_tab, i, w, p.iou_thr));
    }
    cluster_sync();
}

// One image per cluster of G CTAs (G = 1 without a cluster launch).  Rank 0
// owns the image: it runs the whole NMS alone when the image has at most
// kCountSortMax candidates (the other ranks leave at once), and otherwise
// after the cluster has built the sorted list and the suppression matrix
// (nms_cluster_build).
__global__ void __launch_bounds__(kNmsThreads) detect_nms_kernel(const __grid_constant__ DetParams p) {
    extern __shared__ __align__(16) unsigned char smem[];
    NmsSmem S;
    S.key = reinterpret_cast<unsigned long long*>(smem);
    S.idx = reinterpret_cast<int*>(smem + p.off_idx);
    S.box = reinterpret_cast<float4*>(smem + p.off_box);
    S.cls = reinterpret_cast<int*>(smem + p.off_cls);
    S.logit = reinterpret_cast<float*>(smem + p.off_logit);
    S.anchor = reinterpret_cast<int*>(smem + p.off_anchor);
    S.keep = reinterpret_cast<int*>(smem + p.off_keep);
    S.hist = reinterpret_cast<uint32_t*>(smem + p.off_hist);
    S.misc = S.hist + 256;
    S.u = smem + p.off_u;
    unsigned long long* s_key = S.key;
    int* s_idx = S.idx;
    float4* s_box = S.box;
    int* s_cls = S.cls;
    float* s_logit = S.logit;
    int* s_anchor = S.anchor;
    int* s_keep = S.keep;
    uint32_t* s_hist = S.hist;
    uint32_t* s_misc = S.misc;
    unsigned char* s_u = S.u;

    const int b = blockIdx.y, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int G = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
    if ((int)blockIdx.x != rank) return;   // launched without its cluster: block 0 alone takes the image
    if (tid < 8) s_misc[tid] = 0;
    // the candidates and their count come from the kernel this one may overlap
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const ws_candidate* cb = p.cand + (size_t)b * p.A;
    const int n = (int)min((long long)__ldcg(p.count + b), p.A);
    const int m = min(n, p.max_cand);
    // Every CTA of the cluster reads the count before rank 0 resets it: the
    // arrival here, the matching wait before the reset (or at once).
    if (G > 1) cluster_arrive();
    __syncthreads();
    const bool coop = G > 1 && n > kCountSortMax;
    if (coop) {
        cluster_wait();
        nms_cluster_build(p, S, cb, n, m, G, rank);
        if (rank != 0) return;
    } else if (rank != 0) {
        cluster_wait();
        return;
    }

    const int Wl = (m + 63) >> 6;
    const int MS = (m + 1) & ~1;   // the matrix is word-major: word w of row i at w * MS + i
    unsigned long long* s_m = reinterpret_cast<unsigned long long*>(s_u);
    unsigned long long* s_tab = reinterpret_cast<unsigned long long*>(s_u + p.off_tab);   // [Wl][kBuckets]
    if (!coop) {
        // Few candidates (the usual case): two threads per candidate read its
        // 32-byte record once and keep it in registers, each counts the larger
        // keys in half of the list (16-byte loads, summed by a shuffle), and
        // the rank then places the record and sets its class-table bit
        // directly.  Two threads per candidate instead of one: batch-1
        // ws_detect 11.1 -> 10.1 us, batch 64 46.2 -> 45.1 us.
        const bool fast = n <= p.max_cand && n <= kCountSortMax;
        if (fast) {
            float4 box = make_float4(0.f, 0.f, 0.f, 0.f), rest = box;
            unsigned long long key = 0ull;
            const int ci = tid >> 1, part = tid & 1;   // two threads per candidate
            if (ci < n) {
                const float4* c = reinterpret_cast<const float4*>(cb + ci);
                box = __ldcg(c);
                rest = __ldcg(c + 1);
                key = ((unsigned long long)order_bits(rest.x) << 32) | (uint32_t)(~(uint32_t)__float_as_int(rest.z));
                if (part == 0) s_key[ci] = key;
            }
            if (tid == 0 && (n & 1)) s_key[n] = 0ull;   // pads the list to pairs (below every key)
            // the histograms of the cap selection are not used on this path, so
            // the match table can be cleared now
            for (int q = tid; q < Wl * kBuckets; q += kNmsThreads) s_tab[q] = 0ull;
            __syncthreads();
            int r = 0;
            if (ci < n) {
                const ulonglong2* key2 = reinterpret_cast<const ulonglong2*>(s_key);
                const int pairs = (n + 1) >> 1;
#pragma unroll 4
                for (int q = part; q < pairs; q += 2) {
                    const ulonglong2 kk = key2[q];
                    r += (kk.x > key) + (kk.y > key);
                }
            }
            r += __shfl_xor_sync(kFull, r, 1);
            if (ci < n && part == 0) {
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
                if (in_regs) {
#pragma unroll
                    for (int r = 0; r < kKeysPerThread; ++r)
                        if (r < iters) hist_count(s_whist, kr[r], r * kNmsThreads + tid < n, mask, prefix, shift, lane);
                } else {
                    for (int r = 0; r < iters; ++r) {
                        const int i = r * kNmsThreads + tid;
                        hist_count(s_whist, i < n ? cand_key(cb + i) : 0ull, i < n, mask, prefix, shift, lane);
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
                if (warp == 0) find_digit(s_hist, remaining, s_misc, lane);
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
        //    matrix is word-major, so a warp's stores are consecutive words.
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
            s_m[(size_t)w * MS + i] = suppress_word(s_box, s_cls, s_tab, i, w, p.iou_thr);
        }
        __syncthreads();
    }

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
            const unsigned long long d0 = r0 < m ? s_m[(size_t)w * MS + r0] : 0ull;
            const unsigned long long d1 = r1 < m ? s_m[(size_t)w * MS + r1] : 0ull;
            unsigned long long mine = 0;
            for (int q = lane; q < nk; q += 32) mine |= s_m[(size_t)w * MS + s_keep[q]];
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
    if (G > 1 && !coop) cluster_wait();
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
    // the suppression matrix: ceil(max_cand / 64) words of max_cand rows (an
    // even number), word-major; then the class-bucket match table
    const int W = (d->max_cand + 63) / 64;
    p.off_tab = (int)align16((size_t)W * ((d->max_cand + 1) & ~1) * 8);
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
    int dev;
    const DeviceInfo* info;
    const ws_status st = current_device_info(&dev, &info);
    if (st != WS_OK) return st;
    const int tiles = (int)((p.A + kDecodeAnchors - 1) / kDecodeAnchors);
    const bool vec = p.A % 4 == 0 && (uintptr_t)p.head % 16 == 0;
    // one kernel, a programmatic dependent of whatever wrote the head
    cudaError_t e;
    // the DFL bins of a side in registers: 16 (the usual reg_max) or up to 32
    const bool r16 = p.R <= 16;
    if ((long long)tiles * batch <= info->sm_count) {
        // at most one block per SM: every warp loads its classes' rows at once.
        // Measured on one 640x640 image (a detection lane, GPU p50): 20.8 ->
        // 19.5 us; with more blocks the wider registers cost occupancy (batch
        // 16: 15.7 -> 17.3 us) and back-to-back calls overlap less (batch 4:
        // 11.5 -> 11.85 us), so those keep the narrower forms.
        const dim3 grid((unsigned)tiles, (unsigned)batch), block(32 * kDecodeSplit);
        e = vec ? (r16 ? launch_pdl(detect_decode_warp_kernel<true, kDecodeSplit, 16, true>, grid, block, 0, stream, p)
                       : launch_pdl(detect_decode_warp_kernel<true, kDecodeSplit, kMaxRegMax, true>, grid, block, 0, stream, p))
                : (r16 ? launch_pdl(detect_decode_warp_kernel<false, kDecodeSplit, 16, true>, grid, block, 0, stream, p)
                       : launch_pdl(detect_decode_warp_kernel<false, kDecodeSplit, kMaxRegMax, true>, grid, block, 0, stream, p));
    } else if (decode_split(tiles, batch)) {
        const dim3 grid((unsigned)tiles, (unsigned)batch), block(32 * kDecodeSplit);
        e = vec ? (r16 ? launch_pdl(detect_decode_warp_kernel<true, kDecodeSplit, 16>, grid, block, 0, stream, p)
                       : launch_pdl(detect_decode_warp_kernel<true, kDecodeSplit, kMaxRegMax>, grid, block, 0, stream, p))
                : (r16 ? launch_pdl(detect_decode_warp_kernel<false, kDecodeSplit, 16>, grid, block, 0, stream, p)
                       : launch_pdl(detect_decode_warp_kernel<false, kDecodeSplit, kMaxRegMax>, grid, block, 0, stream, p));
    } else {
        const dim3 grid((unsigned)((tiles + kWarpScanWarps - 1) / kWarpScanWarps), (unsigned)batch),
            block(32 * kWarpScanWarps);
        e = vec ? (r16 ? launch_pdl(detect_decode_warp_kernel<true, 1, 16>, grid, block, 0, stream, p)
                       : launch_pdl(detect_decode_warp_kernel<true, 1, kMaxRegMax>, grid, block, 0, stream, p))
                : (r16 ? launch_pdl(detect_decode_warp_kernel<false, 1, 16>, grid, block, 0, stream, p)
                       : launch_pdl(detect_decode_warp_kernel<false, 1, kMaxRegMax>, grid, block, 0, stream, p));
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode launch");
    return WS_OK;
}

// CTAs per image for the NMS: the largest of 8, 4 and 2 for which the
// batch's clusters fit on the GPU at once (one wave), else 1.  The cluster
// only works on images with more than kCountSortMax candidates; on the others
// rank 0 runs alone and the other ranks leave at once.  Asked of the runtime
// once per device, shared-memory size and cluster size.
int nms_cluster_ctas(int32_t batch, size_t smem, int dev, int sm_count) {
    static std::mutex mu;
    static std::map<std::tuple<int, size_t, int>, int> fits;   // clusters resident at once
    for (int G = 8; G >= 2; G >>= 1) {
        if ((long long)batch * G > sm_count) continue;
        int n = 0;
        {
            std::lock_guard<std::mutex> lock(mu);
            const auto key = std::make_tuple(dev, smem, G);
            auto it = fits.find(key);
            if (it == fits.end()) {
                cudaLaunchConfig_t cfg{};
                cfg.gridDim = dim3((unsigned)G, (unsigned)batch);
                cfg.blockDim = dim3(kNmsThreads);
                cfg.dynamicSmemBytes = smem;
                cudaLaunchAttribute attr[1];
                attr[0].id = cudaLaunchAttributeClusterDimension;
                attr[0].val.clusterDim.x = (unsigned)G;
                attr[0].val.clusterDim.y = 1;
                attr[0].val.clusterDim.z = 1;
                cfg.attrs = attr;
                cfg.numAttrs = 1;
                if (cudaOccupancyMaxActiveClusters(&n, detect_nms_kernel, &cfg) == cudaSuccess) {
                    fits.emplace(key, n);
                } else {
                    (void)cudaGetLastError();   // not kept: asked again next time
                    n = 0;
                }
            } else {
                n = it->second;
            }
        }
        if (batch <= n) return G;
    }
    return 1;
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
    const int G = nms_cluster_ctas(batch, smem, dev, info->sm_count);
    cudaError_t e;
    if (G > 1) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3((unsigned)G, (unsigned)batch);
        cfg.blockDim = dim3(kNmsThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = (unsigned)G;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = pdl_enabled() ? 2 : 1;
        e = cudaLaunchKernelEx(&cfg, detect_nms_kernel, p);
        if (e == cudaSuccess) e = cudaGetLastError();
    } else {
        e = launch_pdl(detect_nms_kernel, dim3(1u, (unsigned)batch), dim3(kNmsThreads), smem, stream, p);
    }
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
