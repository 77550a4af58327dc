// topk.cu -- exact row-wise Top-K (K <= 32) over device FP32 logits, sm_103a.
//
// What it computes ("Inside WarpStream TRT", Top-K section): per row the K
// largest values, exact, ties to the lower index, NaN ranked as -inf, and only
// the K value/index pairs are written.  The page's own kernel repeats a
// block-wide arg-max K times (work ~ classes x K) and says large label spaces
// need hierarchical or radix selection instead; this kernel is built for both.
//
// Keys.  Each element becomes one 64-bit key: the upper word maps the float
// (NaN -> -inf, -0 -> +0) to an unsigned integer with the same order, the
// lower word is the bitwise complement of the index, so a larger key is a
// larger value or, for equal values, a lower index.  Keys are unique, the
// order is total and the Top-K set is unique: results are bit-exact.
//
// One block per (row, chunk of up to 8192 elements; 16384 where the 8192 cut
// would give more than 16 chunks a row or more than two blocks per SM):
//  1. The chunk is staged in shared memory (four bulk copies of consecutive
//     quarters when the row is 16-byte aligned, each with its own barrier,
//     else coalesced loads); each thread keeps the maxima of its 4-element
//     groups in registers, and their maximum (a "delegate"), reading each
//     quarter as soon as it has landed.
//  2. Threshold without sorting: each warp finds the kw-th largest of its
//     delegates with warp max-reductions (kw = ceil(K/8) when all 256
//     threads hold one, more on short chunks); t = the minimum over the warps
//     that hold kw.  Those warps own kw distinct elements >= t each, at least
//     K in all, so the chunk's Top-K are all among the elements >= t.
//  3. Elements >= t (typically a few dozen) are appended to shared memory
//     (slots from one shared counter).
//  4. Each candidate's rank is the number of candidates with a larger key
//     (keys are unique, so ranks are distinct): rank < K is written in place.
//  If more than 2048 elements pass the threshold (adversarial inputs, e.g. a
//  constant row), an exact radix select on the 64-bit keys (8 passes of 8
//  bits, warp-aggregated shared histograms) finds the K-th key instead; with
//  385 to 2048 candidates (many ties at the top) the same select runs over
//  the candidates, and only the K keys at or above the K-th are ranked.
// Rows longer than one chunk: every chunk writes its K keys, sorted, to a
// workspace; the last block of the row to finish (an atomic ticket, reset by
// that block so the workspace is ready for the next call or graph replay)
// merges the sorted lists: its warps fold them into at most eight sorted
// lists with bitonic merges in registers, and every key of those is ranked by
// binary searches in all eight at once (its rank is the number of larger
// keys); ranks below K are the row's result, in rank order.  On a direct call
// a row of 2 to 8 chunks is instead one thread-block cluster: each block
// stores its list into rank 0's shared memory (distributed shared memory),
// and one cluster barrier hands rank 0 all of them (no ticket, fence or
// global round trip); lanes keep the ticket, which shares SMs better with
// other lanes.
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

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVpt = 32;                       // values per thread
constexpr int kChunk = kThreads * kVpt;        // 8192 elements per block
constexpr int kCap = 2048;                     // shared candidate capacity
constexpr int kRankMax = 384;                  // candidates ranked by counting; more take a radix select first
constexpr int kMaxK = 32;
constexpr int kBigChunk = 2 * kChunk;          // 16384: the chunk of rows cut into many chunks
constexpr int kFoldBatch = 6;                  // chunk lists a warp loads per round of the merge
constexpr int kMinChunk = 2048;                // shortest chunk a long row is cut into
constexpr int kCutChunks = 16;                 // most blocks per row when a row is cut finer than 8192
constexpr unsigned kFull = 0xffffffffu;

struct TopkParams {
    const float* x;
    long long cols;
    int k;
    int nchunks;
    int chunk;                    // elements per block (a multiple of 4, <= kBigChunk)
    float* out_val;
    int* out_idx;
    unsigned int* tickets;        // [rows]
    unsigned long long* keys;     // [rows][nchunks][k]
    uint32_t* err;                // device error word
    int cluster;                  // 1: a row's blocks form a thread-block cluster and merge through it
    int kw, kw_last;              // delegates each warp vouches for: full chunks, the row's last chunk
};

__device__ __forceinline__ uint32_t order_bits(float f) {
    uint32_t b = __float_as_uint(f);
    if ((b & 0x7fffffffu) > 0x7f800000u) b = 0xff800000u;   // NaN -> -inf
    if (b == 0x80000000u) b = 0u;                            // -0 -> +0 (ordering only)
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// Inverse of order_bits on the canonical value: the float bits of a key's
// value.  Only the sign of a zero is lost, so zeros are read back from x.
__device__ __forceinline__ float key_value(unsigned long long key, const float* xr) {
    const uint32_t u = (uint32_t)(key >> 32);
    const uint32_t b = (u & 0x80000000u) ? (u & 0x7fffffffu) : ~u;
    if (b == 0u) return xr[~(uint32_t)(key & 0xffffffffull)];   // +0 or -0 as stored
    return __uint_as_float(b);                                   // NaN came in as -inf
}

__device__ __forceinline__ unsigned long long make_key(uint32_t u, uint32_t idx) {
    return ((unsigned long long)u << 32) | (uint32_t)(~idx);
}

__device__ __forceinline__ uint32_t key_index(unsigned long long key) {
    return ~(uint32_t)(key & 0xffffffffull);
}

// Top 32 of two 32-key lists, each sorted descending across the warp (lane
// 0 largest): the lane-wise maximum of one list and the other reversed is a
// bitonic sequence holding the 32 largest keys, and five half-cleaner
// stages sort it descending.
__device__ __forceinline__ unsigned long long merge_top32(unsigned long long a, unsigned long long b) {
    const int lane = threadIdx.x & 31;
    const unsigned long long br = __shfl_sync(kFull, b, 31 - lane);
    unsigned long long c = a > br ? a : br;
#pragma unroll
    for (int j = 16; j >= 1; j >>= 1) {
        const unsigned long long o = __shfl_xor_sync(kFull, c, j);
        c = (lane & j) == 0 ? (c > o ? c : o) : (c < o ? c : o);
    }
    return c;
}

struct __align__(16) Shared {
    unsigned long long cand[kCap + kThreads];   // candidates, then one spare slot per thread
    unsigned long long wlist[kWarps][32];       // merge: each warp's top-K list
    unsigned long long red[kWarps];
    uint32_t hist[256];
    uint32_t warp_t[kWarps];
    uint32_t cnt;
    uint32_t sel[2];
    int last;
};

constexpr int kSharedBytes = (int)((sizeof(Shared) + 127) / 128 * 128);
constexpr int kDynSmem = kSharedBytes + kChunk * 4;
constexpr int kDynSmemBig = kSharedBytes + kBigChunk * 4;

// Exact kth-largest (1-based) of n unique 64-bit keys by radix select.
template <class KeyAt>
__device__ unsigned long long block_kth_largest(KeyAt key_at, int n, int kth, Shared& s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    unsigned long long prefix = 0, mask = 0;
    uint32_t remaining = (uint32_t)kth;
    for (int shift = 56; shift >= 0; shift -= 8) {
        for (int i = tid; i < 256; i += kThreads) s.hist[i] = 0;
        __syncthreads();
        for (int base = warp * 32; base < n; base += kThreads) {
            const int i = base + lane;
            uint32_t bin = 256;
            if (i < n) {
                const unsigned long long key = key_at(i);
                if ((key & mask) == prefix) bin = (uint32_t)(key >> shift) & 255u;
            }
            const unsigned peers = __match_any_sync(kFull, bin);
            if (bin < 256 && lane == __ffs(peers) - 1) atomicAdd(&s.hist[bin], (uint32_t)__popc(peers));
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 255-8l down to 248-8l
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = s.hist[255 - 8 * lane - j];
                sum += c[j];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += v;
            }
            const uint32_t excl = incl - sum;
            if (excl < remaining && remaining <= incl) {
                uint32_t acc = excl;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (acc < remaining && remaining <= acc + c[j]) {
                        s.sel[0] = 255u - 8u * lane - j;
                        s.sel[1] = remaining - acc;
                    }
                    acc += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= (unsigned long long)s.sel[0] << shift;
        mask |= 0xffull << shift;
        remaining = s.sel[1];
        __syncthreads();
    }
    return prefix;
}

// Ranks the `cnt` unique candidates in keys[] (shared memory) and calls
// emit(rank, key) for ranks below `kk`; a candidate's rank is the number of
// larger keys.  One thread per candidate: splitting a candidate's count over
// several threads measured slower on GB300 (64 x 1000: 4.0 against 3.3 us).
template <class Emit>
__device__ __forceinline__ void rank_and_emit(const unsigned long long* keys, uint32_t cnt, int kk, Emit emit) {
    for (uint32_t i = threadIdx.x; i < cnt; i += kThreads) {
        const unsigned long long key = keys[i];
        int rank = 0;
#pragma unroll 8
        for (uint32_t j = 0; j < cnt; ++j) rank += (keys[j] > key) ? 1 : 0;
        if (rank < kk) emit(rank, key);
    }
}

// Takes the row's ticket once this block's list is written: true for the
// row's last block, which then merges.  Thread 0 counts the block in with
// one acquire-release atomic at GPU scope: its release covers the whole
// block's writes (the block barrier orders the other threads' writes before
// it), and in the last block its acquire orders the reads of the other
// blocks' lists after every earlier block's release on the same counter; the
// second block barrier carries that order to the other threads.  (A fence
// before and after a relaxed atomic did the same, 0.2-0.5 us slower per
// launch on rows of 16 to 62 chunks.)
__device__ __forceinline__ bool take_ticket(const TopkParams& p, long long row, Shared& s) {
    __syncthreads();
    if (threadIdx.x == 0) {
        unsigned prev;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(prev) : "l"(&p.tickets[row]) : "memory");
        s.last = (prev == (unsigned)p.nchunks - 1u);
    }
    __syncthreads();
    return s.last != 0;
}

// The row's last block: the row's Top-K from the chunks' sorted lists, and
// the row's ticket reset for the next call or graph replay.  Warp w folds the
// lists w, w + 8, ... into one sorted list with bitonic merges in registers
// (lane i holding the i-th key; 0 past a list's K keys, and every real key is
// larger than 0), a batch of lists at a time with the next batch's loads in
// flight.  Then every key of the (at most eight) folded lists is ranked: the
// lists are sorted, so the number of larger keys in each is found by a
// branch-free binary search in shared memory, all eight searches in lockstep
// so that their loads overlap (the key's own list holds exactly `lane`
// larger keys).  Keys are unique, so the K keys of rank below K are written
// once each, in rank order.
__device__ __forceinline__ void merge_chunk_lists(const TopkParams& p, long long row, const float* xr, Shared& s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = p.k, nch = p.nchunks;
    const unsigned long long* all = p.keys + row * nch * k;
    unsigned long long acc = 0ull;
    if (warp < nch) {
        auto load_batch = [&](int c0, unsigned long long (&kb)[kFoldBatch]) {
#pragma unroll
            for (int r = 0; r < kFoldBatch; ++r) {
                const int c = c0 + r * kWarps;
                kb[r] = (c < nch && lane < k) ? __ldcg(all + (long long)c * k + lane) : 0ull;
            }
        };
        unsigned long long cur[kFoldBatch], nxt[kFoldBatch];
        load_batch(warp, cur);
        for (int c0 = warp; c0 < nch; c0 += kWarps * kFoldBatch) {
            const int cn = c0 + kWarps * kFoldBatch;
            if (cn < nch) load_batch(cn, nxt);
#pragma unroll
            for (int step = 1; step < kFoldBatch; step *= 2)
#pragma unroll
                for (int r = 0; r + step < kFoldBatch; r += 2 * step)
                    if (c0 + (r + step) * kWarps < nch) cur[r] = merge_top32(cur[r], cur[r + step]);
            acc = c0 == warp ? cur[0] : merge_top32(acc, cur[0]);
#pragma unroll
            for (int r = 0; r < kFoldBatch; ++r) cur[r] = nxt[r];
        }
    }
    s.wlist[warp][lane] = acc;   // zero keys for warps without a list
    __syncthreads();
    if (tid == 0) p.tickets[row] = 0u;   // ready for the next call / replay
    if (acc == 0ull) return;             // padding
    int lo[kWarps];
#pragma unroll
    for (int c = 0; c < kWarps; ++c) lo[c] = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1)
#pragma unroll
        for (int c = 0; c < kWarps; ++c) lo[c] += s.wlist[c][lo[c] + step - 1] > acc ? step : 0;
    int rank = 0;
#pragma unroll
    for (int c = 0; c < kWarps; ++c) rank += lo[c] + (s.wlist[c][lo[c]] > acc ? 1 : 0);
    if (rank < k) {
        p.out_val[row * k + rank] = key_value(acc, xr);
        p.out_idx[row * k + rank] = (int)key_index(acc);
    }
}

// The row's blocks as one thread-block cluster (at most 8 chunks).  Every
// block arrives once on the cluster barrier as it starts; once that phase is
// complete (cluster_push_begin) all of the cluster's blocks exist, and each
// block stores its chunk's sorted list straight into rank 0's shared memory
// (s.wlist[chunk], zero keys past the list) with remote stores.  One cluster
// barrier (release / acquire) then hands rank 0 every list, with no ticket,
// fence, global round trip or remote load; the other blocks leave, and rank
// 0 ranks every key as merge_chunk_lists does.
__device__ __forceinline__ uint32_t cluster_push_begin(int chunk, Shared& s) {
    cluster_wait();   // the phase every block arrived on at its start
    return cluster_map(&s.wlist[chunk][0], 0u);
}

__device__ __forceinline__ void cluster_merge(const TopkParams& p, long long row, const float* xr, Shared& s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int k = p.k, nch = p.nchunks;
    const bool lead = cluster_ctarank() == 0;
    if (lead)   // zero keys for the rows of absent chunks
        for (int i = nch * 32 + tid; i < kWarps * 32; i += kThreads) s.wlist[i >> 5][i & 31] = 0ull;
    cluster_arrive();
    cluster_wait();   // every list is in rank 0's shared memory
    if (!lead) return;
    const unsigned long long acc = s.wlist[warp][lane];
    if (acc == 0ull) return;
    int lo[kWarps];
#pragma unroll
    for (int c = 0; c < kWarps; ++c) lo[c] = 0;
#pragma unroll
    for (int step = 16; step >= 1; step >>= 1)
#pragma unroll
        for (int c = 0; c < kWarps; ++c) lo[c] += s.wlist[c][lo[c] + step - 1] > acc ? step : 0;
    int rank = 0;
#pragma unroll
    for (int c = 0; c < kWarps; ++c) rank += lo[c] + (s.wlist[c][lo[c]] > acc ? 1 : 0);
    if (rank < k) {
        p.out_val[row * k + rank] = key_value(acc, xr);
        p.out_idx[row * k + rank] = (int)key_index(acc);
    }
}

// kG: 4-element groups a thread (8 for chunks of up to 8192 elements, 16 for
// up to 16384).
template <bool kVec, int kG>
__global__ void __launch_bounds__(kThreads, kG == 8 ? 4 : 2) topk_kernel(const __grid_constant__ TopkParams p) {
    extern __shared__ __align__(128) unsigned char dsmem[];
    Shared& s = *reinterpret_cast<Shared*>(dsmem);
    float* sx = reinterpret_cast<float*>(dsmem + kSharedBytes);   // [chunk] the staged chunk
    // 4 parts of the staged chunk, one bulk copy and one barrier each
    constexpr int kParts = 4;
    constexpr int kPartGroups = kG / kParts;                 // a thread's 4-element groups in one part
    constexpr int kPartElems = kThreads * 4 * kPartGroups;   // elements of one part
    __shared__ uint64_t bar[kParts];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (kVec) {
        // The part barriers are initialised, and the block barrier makes
        // that visible, before the wait below: on a programmatic launch this
        // overlaps the previous grid's tail.
        if (tid == 0) {
#pragma unroll
            for (int q = 0; q < kParts; ++q) mbar_init(&bar[q], 1);
            fence_mbar_init();
        }
        __syncthreads();
    }
    // Launched as a programmatic dependent of the previous kernel on the
    // stream: wait here until that grid has finished and its writes (the
    // logits) are visible.  A no-op for an ordinary launch.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (tid == 0) s.cnt = 0u;   // the candidate counter (read after the next barriers)
    // a cluster merge needs the launch's clusters to be the rows
    if (p.cluster) {
        if ((int)cluster_nctarank() != p.nchunks) {
            if (tid == 0) atomicOr(p.err, kDevErrBadLaunch);
            return;
        }
        cluster_arrive_relaxed();   // this block has started (see cluster_merge)
    }
    const long long row = blockIdx.x / p.nchunks;
    const int chunk = (int)(blockIdx.x - row * p.nchunks);
    const long long c0 = (long long)chunk * p.chunk;
    const int n = (int)min((long long)p.chunk, p.cols - c0);
    const float* xr = p.x + row * p.cols;
    const int k = p.k;

    // 1. stage the chunk in shared memory: four bulk copies of consecutive
    // parts (16-byte aligned rows), each completing its own barrier, else
    // coalesced loads.  The delegate pass below reads each part as soon as
    // it has landed, so its shared-memory reads overlap the later parts'
    // transfer.
    if (kVec) {
        if (tid == 0) {
#pragma unroll
            for (int q = 0; q < kParts; ++q) {
                const int e0 = q * kPartElems;
                if (e0 < n) {
                    const uint32_t bytes = (uint32_t)min(kPartElems, n - e0) * 4u;
                    mbar_arrive_expect_tx(&bar[q], bytes);
                    bulk_g2s(sx + e0, xr + c0 + e0, bytes, &bar[q]);
                }
            }
        }
    } else {
        for (int i = tid; i < n; i += kThreads) sx[i] = __ldcs(xr + c0 + i);
        __syncthreads();
    }
    // Thread tid owns the 4-element groups tid, tid + 256, ... of the chunk
    // (the last group padded with NaN), and keeps each group's maximum in a
    // register: the candidate pass then re-reads only the rare groups whose
    // maximum reaches the threshold.  Group g * 256 + tid lies in part
    // g / kPartGroups; a thread's successful wait on that part's barrier is
    // its acquire of the bytes the part's copy wrote.  A wait that runs out
    // leaves ok false; the block leaves through the error path at the
    // threshold's barrier (the values read meanwhile are not used).
    const int ng = (n + 3) >> 2;
    const float qnan = __int_as_float(0x7fffffff);
    const float4* sx4 = reinterpret_cast<const float4*>(sx);
    auto group = [&](int i) -> float4 {
        if (kVec) return sx4[i];   // n is a multiple of 4 on this path
        const int e = 4 * i;
        return make_float4(e < n ? sx[e] : qnan, e + 1 < n ? sx[e + 1] : qnan, e + 2 < n ? sx[e + 2] : qnan,
                           e + 3 < n ? sx[e + 3] : qnan);
    };
    bool ok = true;
    float gmax[kG];
    float dm = -INFINITY;   // the delegate: fmaxf skips NaN, so a NaN counts as -inf
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        if (kVec && g % kPartGroups == 0) {
            const int q = g / kPartGroups;
            if (ok && q * kPartElems < n) ok = mbar_wait_bounded(&bar[q], 0, kWaitLimitNs);
        }
        const int i = g * kThreads + tid;
        float mx = qnan;
        if (i < ng) {
            const float4 f = group(i);
            mx = fmaxf(fmaxf(f.x, f.y), fmaxf(f.z, f.w));
        }
        gmax[g] = mx;
        dm = fmaxf(dm, mx);
    }
    uint32_t d = tid < ng ? order_bits(dm) : 0u;   // threads without elements have no delegate

    // 2. threshold: min over warps of each warp's kw-th largest delegate
    // (kw from delegate_rounds() on the host, by the chunk's length).
    const int kw = chunk + 1 == p.nchunks ? p.kw_last : p.kw;
    uint32_t tw = 0;
    for (int r = 0; r < kw; ++r) {
        const uint32_t m = __reduce_max_sync(kFull, d);
        tw = m;
        if (m == 0) break;
        const unsigned who = __ballot_sync(kFull, d == m);
        if (lane == __ffs(who) - 1) d = 0;
    }
    if (lane == 0) s.warp_t[warp] = tw;
    if (__syncthreads_or(!ok)) {
        // A part's copy did not land in time.
        if (tid == 0) {
            atomicOr(p.err, kDevErrBulkCopyTimeout);
#pragma unroll
            for (int q = 0; q < kParts; ++q)   // let the copies land before leaving
                if (q * kPartElems < n) mbar_wait_bounded(&bar[q], 0, kWaitLimitNs);
        }
        if (p.nchunks == 1) return;
        // A row split over several blocks: this chunk contributes an empty
        // list (padding keys) but still takes part in the merge (the
        // cluster's barriers, or the row's ticket, so that the row's last
        // block merges and resets the ticket and the workspace is ready for
        // the next call).  The error bit says the row's result is not to be
        // used.
        if (p.cluster) {
            const uint32_t dst = cluster_push_begin(chunk, s);
            if (tid < 32) st_cluster_u64(dst + 8u * tid, 0ull);
            cluster_merge(p, row, xr, s);
            return;
        }
        unsigned long long* kr = p.keys + (row * p.nchunks + chunk) * k;
        for (int r = tid; r < k; r += kThreads) kr[r] = 0ull;
        if (!take_ticket(p, row, s)) return;
        merge_chunk_lists(p, row, xr, s);
        return;
    }
    // Warps that hold kw delegates each vouch for kw elements >= their own
    // threshold; the minimum over enough such warps is a valid threshold.
    uint32_t t = 0xffffffffu;
    int vouching = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
        const uint32_t tv = s.warp_t[w];
        if (tv != 0) {
            t = min(t, tv);
            ++vouching;
        }
    }

    // 3. candidates.  Each thread marks the groups whose maximum reaches the
    // threshold (usually none or one) and visits only those, once to count
    // and once to write; a shared counter gives every candidate its slot.
    // Above -inf the threshold is tested as a float (NaN fails it,
    // +0 and -0 both pass a zero).  Too few vouching warps, or a threshold of
    // -inf, make every element a candidate (the chunk then usually takes the
    // radix select below).
    const uint32_t kOrderNegInf = 0x007fffffu;   // order_bits(-inf)
    const bool by_value = vouching * kw >= k && t > kOrderNegInf;
    const float tf = __uint_as_float((t & 0x80000000u) ? (t & 0x7fffffffu) : ~t);
    unsigned hits = 0;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
        const int i = g * kThreads + tid;
        if (i < ng && (!by_value || gmax[g] >= tf)) hits |= 1u << g;
    }
    int mine = 0;
    for (unsigned m = hits; m; m &= m - 1) {
        const int i = (__ffs(m) - 1) * kThreads + tid;
        const float4 f = group(i);
        if (by_value) {
            mine += (f.x >= tf) + (f.y >= tf) + (f.z >= tf) + (f.w >= tf);
        } else {
            mine += min(4, n - 4 * i);
        }
    }
    // Slots from one shared counter: a thread with candidates takes its run
    // with one atomic.  Their order does not matter (ranks are counted), and
    // this replaced a warp scan and a block scan with its barrier (measured
    // 1-3 % faster on every shape).  A thread whose run would pass kCap
    // writes nothing; the count then sends the chunk to the radix select.
    int pos = mine ? (int)atomicAdd(&s.cnt, (uint32_t)mine) : 0;
    if (pos + mine <= kCap) {
        // Branch-free: an element not taken goes to the thread's spare slot.
        unsigned long long* spare = &s.cand[kCap + tid];
        for (unsigned m = hits; m; m &= m - 1) {
            const int i = (__ffs(m) - 1) * kThreads + tid;
            const float4 f = group(i);
            const float e[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const bool take = by_value ? e[c] >= tf : 4 * i + c < n;
                *(take ? &s.cand[pos] : spare) = make_key(order_bits(e[c]), (uint32_t)(c0 + 4 * i + c));
                pos += take ? 1 : 0;
            }
        }
    }
    __syncthreads();
    uint32_t cnt = s.cnt;
    const int kk = min(k, n);
    const unsigned long long* ck = s.cand;   // the keys step 4 ranks
    if (cnt > kCap) {
        // exact fallback: radix select over the chunk's keys
        auto key_at = [&](int i) { return make_key(order_bits(sx[i]), (uint32_t)(c0 + i)); };
        const unsigned long long kth = block_kth_largest(key_at, n, kk, s);
        if (tid == 0) s.cnt = 0;
        __syncthreads();
        for (int i = tid; i < n; i += kThreads) {
            const unsigned long long key = key_at(i);
            if (key >= kth) s.cand[atomicAdd(&s.cnt, 1u)] = key;   // exactly kk keys
        }
        __syncthreads();
        cnt = s.cnt;
    } else if (cnt > (uint32_t)kRankMax) {
        // Many candidates (ties at the top of the chunk): ranking each against
        // all is quadratic (1500 candidates of an 8000-entry row took 68 us).
        // The kk-th largest candidate by radix select instead, and the kk keys
        // at or above it, copied past the candidates, are ranked.
        const unsigned long long kth = block_kth_largest([&](int i) { return s.cand[i]; }, (int)cnt, kk, s);
        if (tid == 0) s.cnt = 0;
        __syncthreads();
        for (uint32_t i = tid; i < cnt; i += kThreads) {
            const unsigned long long key = s.cand[i];
            if (key >= kth) s.cand[kCap + atomicAdd(&s.cnt, 1u)] = key;   // exactly kk keys
        }
        __syncthreads();
        cnt = s.cnt;
        ck = s.cand + kCap;
    }

    // 4. rank and emit
    if (p.nchunks == 1) {
        rank_and_emit(ck, cnt, kk, [&](int rank, unsigned long long key) {
            p.out_val[row * k + rank] = key_value(key, xr);
            p.out_idx[row * k + rank] = (int)key_index(key);
        });
        return;
    }
    if (p.cluster) {
        const uint32_t dst = cluster_push_begin(chunk, s);
        rank_and_emit(ck, cnt, kk, [&](int rank, unsigned long long key) { st_cluster_u64(dst + 8u * rank, key); });
        for (int r = kk + tid; r < 32; r += kThreads) st_cluster_u64(dst + 8u * r, 0ull);   // past the list
        cluster_merge(p, row, xr, s);
        return;
    }
    unsigned long long* kr = p.keys + (row * p.nchunks + chunk) * k;
    rank_and_emit(ck, cnt, kk, [&](int rank, unsigned long long key) { kr[rank] = key; });
    for (int r = kk + tid; r < k; r += kThreads) kr[r] = 0ull;   // chunk shorter than K

    // Last block of the row merges.
    if (!take_ticket(p, row, s)) return;
    merge_chunk_lists(p, row, xr, s);
}

// ---------------------------------------------------------------------------
// Many short rows (at most kWarpMaxCols entries; see use_warp_kernel): one
// warp per row, no block-wide barrier.  The row sits in the warp's registers (V values per lane); the
// selection is the same threshold / candidates / rank scheme as above, with
// warp-wide steps only:
//  1. delegates: the maximum of each 4-value group (NaN and padding count as
//     -inf); V / 4 per lane.
//  2. threshold t: a value with at least K delegates >= t, found by
//     bisection between the smallest and the largest delegate, counting with
//     redux.sync.  Those delegates are K distinct elements >= t, so every
//     element of the row's Top-K is >= t.
//  3. the elements >= t (typically K plus a few) go to the warp's slice of
//     shared memory as 64-bit keys, each lane's slots from a warp scan.
//  4. each candidate's rank is the number of candidates with a larger key.
// Without K delegates above -inf, every element is a candidate.  If more than
// kWarpCap elements are candidates (a constant row, many NaN), an exact
// selection replaces steps 2-4: the K-th largest value is built bit by bit
// from warp counts, the elements above it are taken, and the ties at it are
// taken in index order, lowest first.
// ---------------------------------------------------------------------------
constexpr int kWarpMaxCols = 2048;
constexpr int kWarpCap = 256;          // candidate keys per warp in shared memory
constexpr int kWarpSlots = kWarpCap;
constexpr int kWarpRounds = 4;         // threshold search rounds (3 pivots each: 4x narrower)

struct TopkWarpParams {
    const float* x;
    long long rows;
    int cols;
    int k;
    float* out_val;
    int* out_idx;
};

// Element index of a lane's i-th register: 16-byte loads put 4 consecutive
// elements in each lane (a warp covers 128 per load); scalar loads 1 (32).
template <bool kVec>
__device__ __forceinline__ int warp_elem(int i, int lane) {
    return kVec ? 128 * (i >> 2) + 4 * lane + (i & 3) : 32 * i + lane;
}

__device__ __forceinline__ uint32_t warp_scan_excl(uint32_t v, uint32_t& total) {
    const int lane = threadIdx.x & 31;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
    }
    total = __shfl_sync(kFull, incl, 31);
    return incl - v;
}

template <int V, bool kVec>
__global__ void __launch_bounds__(128) topk_warp_kernel(const __grid_constant__ TopkWarpParams p) {
    extern __shared__ __align__(16) unsigned long long wsm[];   // [warps][kWarpSlots]
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const long long row = (long long)blockIdx.x * (blockDim.x >> 5) + w;
    if (row >= p.rows) return;
    unsigned long long* cand = wsm + w * kWarpSlots;
    const int n = p.cols, k = p.k;
    const float* xr = p.x + row * (long long)n;
    const float qnan = __int_as_float(0x7fffffff);

    float v[V];
    if (kVec) {
#pragma unroll
        for (int j = 0; j < V / 4; ++j) {
            const int e = 128 * j + 4 * lane;   // n % 4 == 0: a group is whole or absent
            const float4 f = e < n ? __ldg(reinterpret_cast<const float4*>(xr + e)) : make_float4(qnan, qnan, qnan, qnan);
            v[4 * j] = f.x;
            v[4 * j + 1] = f.y;
            v[4 * j + 2] = f.z;
            v[4 * j + 3] = f.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < V; ++i) {
            const int e = 32 * i + lane;
            v[i] = e < n ? __ldg(xr + e) : qnan;
        }
    }

    // 1-2. delegates and the bisected threshold
    constexpr int G = V / 4;
    float d[G];
    uint32_t nvalid = 0, dmin = 0xffffffffu, dmax = 0u;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        d[g] = fmaxf(fmaxf(fmaxf(-INFINITY, v[4 * g]), fmaxf(v[4 * g + 1], v[4 * g + 2])), v[4 * g + 3]);
        const uint32_t ob = order_bits(d[g]);
        const bool valid = d[g] > -INFINITY;
        nvalid += valid ? 1u : 0u;
        dmin = min(dmin, valid ? ob : 0xffffffffu);
        dmax = max(dmax, ob);
    }
    nvalid = __reduce_add_sync(kFull, nvalid);
    bool by_value = nvalid >= (uint32_t)k;
    float t = -INFINITY;
    if (by_value) {
        dmin = __reduce_min_sync(kFull, dmin);
        dmax = __reduce_max_sync(kFull, dmax);
        auto value_of = [](uint32_t u) { return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u); };
        float lo = value_of(dmin);                  // count(d >= lo) = nvalid >= K
        float hi = fminf(value_of(dmax), 3.402823466e38f);
        // Only lo must keep at least K delegates at or above it; hi only
        // narrows the search.  Each round counts three pivots at once (their
        // warp sums are independent, so their latencies overlap).
        for (int r = 0; r < kWarpRounds; ++r) {
            const float q1 = 0.75f * lo + 0.25f * hi, q2 = 0.5f * lo + 0.5f * hi, q3 = 0.25f * lo + 0.75f * hi;
            if (!(q2 > lo && q2 < hi)) break;
            uint32_t c1 = 0, c2 = 0, c3 = 0;
#pragma unroll
            for (int g = 0; g < G; ++g) {
                c1 += d[g] >= q1 ? 1u : 0u;
                c2 += d[g] >= q2 ? 1u : 0u;
                c3 += d[g] >= q3 ? 1u : 0u;
            }
            c1 = __reduce_add_sync(kFull, c1);
            c2 = __reduce_add_sync(kFull, c2);
            c3 = __reduce_add_sync(kFull, c3);
            const uint32_t kk = (uint32_t)k;
            // counts fall as the pivot rises: take the highest pivot that keeps K
            const float nlo = c3 >= kk ? q3 : c2 >= kk ? q2 : c1 >= kk ? q1 : lo;
            const float nhi = c1 < kk ? q1 : c2 < kk ? q2 : c3 < kk ? q3 : hi;
            lo = fmaxf(lo, nlo);
            hi = nhi;
        }
        t = lo;
    }

    // 3. candidates: elements >= t (every present element without a threshold)
    unsigned long long taken = 0;   // bit i: register i is a candidate
#pragma unroll
    for (int i = 0; i < V; ++i) {
        const bool take = by_value ? v[i] >= t : warp_elem<kVec>(i, lane) < n;
        taken |= (unsigned long long)(take ? 1u : 0u) << i;
    }
    uint32_t total;
    uint32_t pos = warp_scan_excl((uint32_t)__popcll(taken), total);
    if (total <= (uint32_t)kWarpCap) {
        // A lane visits only its own candidates (usually none or one) and
        // re-reads each by index from the cached row.
        for (; taken; taken &= taken - 1) {
            const int e = warp_elem<kVec>(__ffsll(taken) - 1, lane);
            cand[pos++] = make_key(order_bits(__ldg(xr + e)), (uint32_t)e);
        }
    } else {
        // Exact selection.  ob[i]: order bits, 0 for padding (below every
        // element, NaN included, which maps to -inf).
        uint32_t ob[V];
#pragma unroll
        for (int i = 0; i < V; ++i) ob[i] = warp_elem<kVec>(i, lane) < n ? order_bits(v[i]) : 0u;
        uint32_t T = 0;   // the K-th largest order bits: the largest T with count(ob >= T) >= K
        for (int b = 31; b >= 0; --b) {
            const uint32_t c_try = T | (1u << b);
            uint32_t c = 0;
#pragma unroll
            for (int i = 0; i < V; ++i) c += ob[i] >= c_try ? 1u : 0u;
            if (__reduce_add_sync(kFull, c) >= (uint32_t)k) T = c_try;
        }
        uint32_t gt = 0;
#pragma unroll
        for (int i = 0; i < V; ++i) gt += ob[i] > T ? 1u : 0u;
        uint32_t ngt;
        pos = warp_scan_excl(gt, ngt);   // ngt < K
#pragma unroll
        for (int i = 0; i < V; ++i)
            if (ob[i] > T) cand[pos++] = make_key(ob[i], (uint32_t)warp_elem<kVec>(i, lane));
        // ties at T, lowest indices first: registers in index order, a tile
        // (one register group across the warp) at a time
        const uint32_t need = (uint32_t)k - ngt;
        uint32_t ties = 0;                   // ties taken so far (warp-uniform)
        constexpr int kPer = kVec ? 4 : 1;   // registers of one lane in a tile
#pragma unroll
        for (int j = 0; j < V / kPer; ++j) {
            if (ties < need) {
                uint32_t eq = 0;
#pragma unroll
                for (int c = 0; c < kPer; ++c) eq += ob[kPer * j + c] == T ? 1u : 0u;
                uint32_t tile_total;
                uint32_t slot = ngt + ties + warp_scan_excl(eq, tile_total);
#pragma unroll
                for (int c = 0; c < kPer; ++c) {
                    const int i = kPer * j + c;
                    if (ob[i] == T && slot < (uint32_t)k)
                        cand[slot++] = make_key(T, (uint32_t)warp_elem<kVec>(i, lane));
                }
                ties += tile_total;
            }
        }
        total = (uint32_t)k;
    }
    __syncwarp();

    // 4. rank and emit: each lane ranks two candidates per pass over the list
    for (uint32_t base = 0; base < total; base += 64) {
        const uint32_t i0 = base + lane, i1 = base + 32 + lane;
        const unsigned long long a = i0 < total ? cand[i0] : ~0ull;
        const unsigned long long b = i1 < total ? cand[i1] : ~0ull;
        int ra = 0, rb = 0;
#pragma unroll 4
        for (uint32_t j = 0; j < total; ++j) {
            const unsigned long long c = cand[j];
            ra += c > a ? 1 : 0;
            rb += c > b ? 1 : 0;
        }
        if (i0 < total && ra < k) {
            p.out_val[row * k + ra] = key_value(a, xr);
            p.out_idx[row * k + ra] = (int)key_index(a);
        }
        if (i1 < total && rb < k) {
            p.out_val[row * k + rb] = key_value(b, xr);
            p.out_idx[row * k + rb] = (int)key_index(b);
        }
    }
}

// The one-warp-per-row kernel has fewer steps per row but a longer serial
// chain per warp than the block kernel.  Measured on GB300 (back-to-back
// launches): it wins from about two rows per SM (608 x 1000: 4.1 against
// 5.1 us; 4096 x 1000: 8.8 against 24.0 us) and on rows of at most 512
// entries (304 x 256: 3.2 against 5.5 us); with fewer, longer rows the block
// kernel's wider fan-out is faster (64 x 1000: 3.3 against 4.0 us).
// A row cut into 2 .. 8 chunks merges through a thread-block cluster of its
// blocks (cluster_merge) when the runtime can place clusters of that many of
// these blocks; asked once per device, kernel variant, shared-memory size and
// cluster size.
template <bool kVec, int kG>
bool topk_cluster_fits(int dev, int nch, size_t smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, size_t, int>, bool> fits;
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, smem, nch);
    auto it = fits.find(key);
    if (it != fits.end()) return it->second;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)nch);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nch;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, topk_kernel<kVec, kG>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();   // not kept: asked again next time
        return false;
    }
    fits.emplace(key, n > 0);
    return n > 0;
}

template <bool kVec, int kG>
cudaError_t launch_topk_block(const TopkParams& p, long long blocks, size_t smem, cudaStream_t stream) {
    if (!p.cluster) return launch_pdl(topk_kernel<kVec, kG>, dim3((unsigned)blocks), dim3(kThreads), smem, stream, p);
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)p.nchunks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, topk_kernel<kVec, kG>, p);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

bool use_warp_kernel(int64_t rows, int64_t cols, int sm_count) {
    return cols <= kWarpMaxCols && (cols <= 512 || rows >= 2LL * sm_count);
}

template <int V>
cudaError_t launch_warp_v(const TopkWarpParams& p, bool vec, int warps, cudaStream_t stream) {
    const long long blocks = (p.rows + warps - 1) / warps;
    const size_t smem = (size_t)warps * kWarpSlots * sizeof(unsigned long long);
    return vec ? launch_pdl(topk_warp_kernel<V, true>, dim3((unsigned)blocks), dim3(32 * warps), smem, stream, p)
               : launch_pdl(topk_warp_kernel<V, false>, dim3((unsigned)blocks), dim3(32 * warps), smem, stream, p);
}

// Rows of at most kWarpMaxCols entries: one warp per row, the row in
// V = 8 .. 64 registers per lane.
cudaError_t launch_topk_warp(const TopkWarpParams& p, bool vec, int sm_count, cudaStream_t stream) {
    // one warp per block while the rows alone do not fill the SMs, four after
    const int warps = p.rows <= sm_count ? 1 : 4;
    if (p.cols <= 256) return launch_warp_v<8>(p, vec, warps, stream);
    if (p.cols <= 512) return launch_warp_v<16>(p, vec, warps, stream);
    if (p.cols <= 1024) return launch_warp_v<32>(p, vec, warps, stream);
    return launch_warp_v<64>(p, vec, warps, stream);
}

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

std::atomic<bool> g_topk_attr_set[64];

}  // namespace

ws_status validate_topk(int64_t rows, int64_t cols, int32_t k) {
    if (rows < 1) return fail(WS_ERR_INVALID_ARGUMENT, "rows %lld < 1", (long long)rows);
    if (cols < 1 || cols > 2147483647LL)
        return fail(WS_ERR_INVALID_ARGUMENT, "cols %lld outside 1 .. 2^31-1", (long long)cols);
    if (k < 1 || k > kMaxK) return fail(WS_ERR_INVALID_ARGUMENT, "k %d outside 1..%d", k, kMaxK);
    if (k > cols) return fail(WS_ERR_INVALID_ARGUMENT, "k %d > cols %lld", k, (long long)cols);
    if (rows > (1LL << 40) / cols) return fail(WS_ERR_INVALID_ARGUMENT, "rows * cols too large");
    return WS_OK;
}

// Most blocks a row of `cols` elements is cut into: 8192-element blocks, or
// up to kCutChunks blocks of at least kMinChunk elements.
long long max_blocks_per_row(int64_t cols) {
    const long long base = (cols + kChunk - 1) / kChunk;
    return std::max<long long>(base, std::min<long long>((cols + kMinChunk - 1) / kMinChunk, kCutChunks));
}

// Blocks per row.  Rows up to kChunk elements take one block.  Longer rows
// take 8192-element blocks, except that when that leaves SMs without a block
// the rows are cut finer, down to kMinChunk elements and at most kCutChunks
// blocks per row, until there is about one block per SM.  Both limits were
// measured on GB300.  More blocks per SM: a block's phases are chains of
// short steps and block barriers, and blocks sharing an SM slow each other's
// chains about as much as they shorten them ([16,131072]: one block per SM,
// 16 chunks, 7.6 us; four per SM, 38 chunks, 9.5 us).  More blocks per row:
// the last block has more lists to merge ([2,100000]: 16 chunks 6.5 us, 49
// chunks 7.3 us; [4,65536]: 16 chunks 6.5 us, 32 chunks 6.8 us).
int blocks_per_row(int64_t rows, int64_t cols, int sm_count) {
    const long long base = (cols + kChunk - 1) / kChunk;
    if (base <= 1) return 1;
    const long long cap = max_blocks_per_row(cols);
    const long long want = (long long)sm_count / std::max<int64_t>(rows, 1);
    return (int)std::min<long long>(cap, std::max<long long>(base, want));
}

// Delegates each warp of a block vouches for in the threshold step, for a
// chunk of n elements: the least kw for which the warps holding at least kw
// delegates (a thread holds one if it has an element) own K elements between
// them.  ceil(K/8) when all 256 threads hold a delegate (n >= 1024); more on
// shorter chunks, where fewer warps hold delegates: a 576-element chunk has
// four full warps and one of 16, so kw = 7 for K = 32, where ceil(K/8) = 4
// would leave too few vouching warps and make every element a candidate
// (ranked against every other: [1,576] took 14.5 us instead of 2.9).
// Chunks too short for any kw fall back to every element being a candidate.
int delegate_rounds(long long n, int k) {
    const long long ng = (n + 3) / 4;
    const int full = (int)std::min<long long>(kWarps, ng / 32);   // warps whose 32 threads hold one
    const int part = ng < kThreads ? (int)(ng % 32) : 0;           // delegates of the one partial warp
    int kw = (k + kWarps - 1) / kWarps;
    if ((full + (part >= kw ? 1 : 0)) * kw < k) {
        const int w = full + (part > 0 ? 1 : 0);
        kw = (k + w - 1) / w;
        if (part > 0 && part < kw && full > 0) kw = (k + full - 1) / full;
    }
    return std::min(kw, 32);
}

// Chunk length for a number of blocks per row: a multiple of 4 elements.
int chunk_len(int64_t cols, int nchunks, int max_chunk) {
    const long long c = (cols + nchunks - 1) / nchunks;
    return (int)std::min<long long>(max_chunk, (c + 3) / 4 * 4);
}

// How a row longer than one block is cut: blocks_per_row() chunks of at most
// 8192 elements, except where that would give more than kCutChunks chunks in
// a row or more than two blocks per SM; those take chunks of up to 16384 (half
// the blocks, half the lists for the last block to merge, and each thread's
// fixed per-block steps spread over twice the elements).  Measured on GB300,
// K = 32, back-to-back launches: [32,131072] 9.3 -> 8.0 us, [64,131072] 14.7
// -> 13.3 us, [1,1000000] 9.9 -> 8.0 us; inside the 8 x 4K -> 512 lanes the
// step went 21.6 -> 20.9 us with lanes on their own streams and 34.5 -> 33.7
// us on one stream.  Chunks of 32768 (one block per SM) were faster alone
// ([32,131072] 7.6 us) but slowed the own-stream step to 21.4 us.
struct ChunkPlan {
    int nchunks, chunk, groups;   // groups: 4-element groups a thread (8 or 16)
};

ChunkPlan plan_chunks(int64_t rows, int64_t cols, int sm_count) {
    ChunkPlan c{};
    const long long base = (cols + kChunk - 1) / kChunk;
    if (base > kCutChunks || rows * base > 2LL * sm_count) {
        c.groups = 16;
        c.nchunks = (int)((cols + kBigChunk - 1) / kBigChunk);
        c.chunk = chunk_len(cols, c.nchunks, kBigChunk);
    } else {
        c.groups = 8;
        c.nchunks = blocks_per_row(rows, cols, sm_count);
        c.chunk = chunk_len(cols, c.nchunks, kChunk);
    }
    c.nchunks = (int)((cols + c.chunk - 1) / c.chunk);
    return c;
}

size_t topk_workspace_size(int64_t rows, int64_t cols, int32_t k) {
    // Upper bound over every launch shape blocks_per_row() can choose, so it
    // depends on (rows, cols, k) only.
    const long long base = (cols + kChunk - 1) / kChunk;
    if (base <= 1) return 0;
    const long long nchunks = max_blocks_per_row(cols);
    return round_up((size_t)rows * 4, 256) + (size_t)rows * nchunks * k * 8;
}

}  // namespace ws

extern "C" {

ws_status ws_topk_validate(int64_t rows, int64_t cols, int32_t k) {
    ws::clear_error();
    return ws::validate_topk(rows, cols, k);
}

ws_status ws_topk_workspace_bytes(int64_t rows, int64_t cols, int32_t k, size_t* bytes) {
    ws::clear_error();
    if (!bytes) return ws::fail(WS_ERR_INVALID_ARGUMENT, "bytes is NULL");
    ws_status st = ws::validate_topk(rows, cols, k);
    if (st != WS_OK) return st;
    *bytes = ws::topk_workspace_size(rows, cols, k);
    return WS_OK;
}

ws_status ws_topk_workspace_init(void* workspace, size_t bytes, cudaStream_t stream) {
    ws::clear_error();
    if (bytes == 0) return WS_OK;
    if (!workspace) return ws::fail(WS_ERR_INVALID_ARGUMENT, "workspace is NULL");
    WS_TRY_CUDA(cudaMemsetAsync(workspace, 0, bytes, stream));
    return WS_OK;
}

ws_status ws_topk(const float* x, int64_t rows, int64_t cols, int32_t k, float* out_val, int32_t* out_idx,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream) {
    ws::clear_error();
    return ws::topk_enqueue(x, rows, cols, k, out_val, out_idx, workspace, workspace_bytes, stream, true);
}

}  // extern "C"

namespace ws {

ws_status topk_enqueue(const float* x, int64_t rows, int64_t cols, int32_t k, float* out_val, int32_t* out_idx,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream, bool cluster_merge_ok) {
    ws_status st = validate_topk(rows, cols, k);
    if (st != WS_OK) return st;
    if (!x || !out_val || !out_idx) return fail(WS_ERR_INVALID_ARGUMENT, "x, out_val or out_idx is NULL");
    const size_t need = topk_workspace_size(rows, cols, k);
    if (need > 0 && (!workspace || workspace_bytes < need))
        return fail(WS_ERR_INVALID_ARGUMENT, "workspace of %zu bytes, %zu needed", workspace_bytes, need);
    if (need > 0 && (uintptr_t)workspace % 256 != 0)
        return fail(WS_ERR_INVALID_ARGUMENT, "workspace must be 256-byte aligned");

    int dev;
    const DeviceInfo* info;
    st = current_device_info(&dev, &info);
    if (st != WS_OK) return st;
    const bool vec = (cols % 4 == 0) && ((uintptr_t)x % 16 == 0);
    if (use_warp_kernel(rows, cols, info->sm_count)) {
        if ((rows + 3) / 4 > 2147483647LL) return fail(WS_ERR_UNSUPPORTED, "too many rows");
        const TopkWarpParams wp{x, rows, (int)cols, k, out_val, out_idx};
        const cudaError_t e = launch_topk_warp(wp, vec, info->sm_count, stream);
        if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
        return WS_OK;
    }

    TopkParams p{};
    p.x = x;
    p.cols = cols;
    p.k = k;
    const ChunkPlan plan = plan_chunks(rows, cols, info->sm_count);
    p.nchunks = plan.nchunks;
    p.chunk = plan.chunk;
    p.kw = delegate_rounds(std::min<long long>(plan.chunk, cols), k);
    p.kw_last = delegate_rounds(cols - (long long)(plan.nchunks - 1) * plan.chunk, k);
    p.out_val = out_val;
    p.out_idx = out_idx;
    if (need > 0) {
        p.tickets = static_cast<unsigned int*>(workspace);
        p.keys = reinterpret_cast<unsigned long long*>(static_cast<char*>(workspace) +
                                                       round_up((size_t)rows * 4, 256));
    }
    const long long blocks = rows * p.nchunks;
    if (blocks > 2147483647LL) return fail(WS_ERR_UNSUPPORTED, "too many blocks");
    // Programmatic dependent launch ("Streams, concurrency and CUDA Graphs",
    // PDL section): the grid may be launched while the previous kernel on the
    // stream is still running and waits in griddepcontrol.wait, which hides
    // the launch gap between the preprocess and the Top-K.
    if (!g_topk_attr_set[dev].load(std::memory_order_acquire)) {
        WS_TRY_CUDA(cudaFuncSetAttribute(topk_kernel<true, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem));
        WS_TRY_CUDA(cudaFuncSetAttribute(topk_kernel<false, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem));
        WS_TRY_CUDA(
            cudaFuncSetAttribute(topk_kernel<true, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemBig));
        WS_TRY_CUDA(
            cudaFuncSetAttribute(topk_kernel<false, 16>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmemBig));
        g_topk_attr_set[dev].store(true, std::memory_order_release);
    }
    p.err = device_error_word();
    // the staged chunk only needs the chunk's length when the chunk is short
    const size_t smem = (size_t)kSharedBytes + (size_t)(p.chunk + 3) / 4 * 16;
    if (cluster_merge_ok && p.nchunks >= 2 && p.nchunks <= 8)
        p.cluster = (plan.groups == 16 ? (vec ? topk_cluster_fits<true, 16>(dev, p.nchunks, smem)
                                              : topk_cluster_fits<false, 16>(dev, p.nchunks, smem))
                                       : (vec ? topk_cluster_fits<true, 8>(dev, p.nchunks, smem)
                                              : topk_cluster_fits<false, 8>(dev, p.nchunks, smem)))
                        ? 1
                        : 0;
    cudaError_t e;
    if (plan.groups == 16)
        e = vec ? launch_topk_block<true, 16>(p, blocks, smem, stream) : launch_topk_block<false, 16>(p, blocks, smem, stream);
    else
        e = vec ? launch_topk_block<true, 8>(p, blocks, smem, stream) : launch_topk_block<false, 8>(p, blocks, smem, stream);
    if (e != cudaSuccess) return cuda_fail(e, "top-k launch");
    return WS_OK;
}

}  // namespace ws

// ---------------------------------------------------------------------------
// ws_topk_noalloc: the same Top-K for callers that cannot allocate device
// memory.  Its scratch (row tickets + per-block keys, laid out exactly like a
// ws_topk workspace) is this fixed array in the library's device image: every
// GPU that loads the library holds it until the process exits.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = 1u << 20;   // 1 MiB per device
static __device__ __align__(256) unsigned char g_topk_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64];

// Device address of this device's scratch array.  The array's name is only a
// host-side stand-in in host code, so the address is looked up once per
// device, with that device current, and cached.
ws_status noalloc_scratch(void** out) {
    int dev;
    const ws::DeviceInfo* info;
    ws_status st = ws::current_device_info(&dev, &info);
    if (st != WS_OK) return st;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_topk_noalloc_scratch);
        if (e != cudaSuccess) return ws::cuda_fail(e, "cudaGetSymbolAddress of the Top-K scratch array");
        g_noalloc_ptr[dev] = p;
    }
    *out = g_noalloc_ptr[dev];
    return WS_OK;
}

}  // namespace

extern "C" ws_status ws_topk_noalloc(const float* x, int64_t rows, int64_t cols, int32_t k, float* out_val,
                                     int32_t* out_idx, cudaStream_t stream) {
    ws::clear_error();
    ws_status st = ws::validate_topk(rows, cols, k);
    if (st != WS_OK) return st;
    // Refuse bad pointers before anything is enqueued (the ticket clearing
    // below is stream work).
    if (!x || !out_val || !out_idx) return ws::fail(WS_ERR_INVALID_ARGUMENT, "x, out_val or out_idx is NULL");
    const size_t need = ws::topk_workspace_size(rows, cols, k);
    if (need > kNoAllocScratchBytes)
        return ws::fail(WS_ERR_UNSUPPORTED,
                        "rows=%lld cols=%lld k=%d needs %zu bytes of scratch; ws_topk_noalloc has a fixed "
                        "%zu-byte array (use ws_topk with a caller workspace)",
                        (long long)rows, (long long)cols, k, need, kNoAllocScratchBytes);
    void* scratch = nullptr;
    if (need > 0) {
        if ((st = noalloc_scratch(&scratch)) != WS_OK) return st;
        // The array keeps the previous call's contents; the row tickets must
        // start at zero.
        cudaError_t e = cudaMemsetAsync(scratch, 0, (size_t)rows * sizeof(unsigned int), stream);
        if (e != cudaSuccess) return ws::cuda_fail(e, "clearing the Top-K scratch tickets");
    }
    return ws_topk(x, rows, cols, k, out_val, out_idx, scratch, need > 0 ? kNoAllocScratchBytes : 0, stream);
}
