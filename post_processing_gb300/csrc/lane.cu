// lane.cu -- fixed-shape execution lanes: preallocated buffers, one CUDA
// Graph per lane, an explicit FREE -> ACQUIRED -> IN_FLIGHT -> FREE state
// machine and event-timed submit / wait.
//
// Follows "Inside WarpStream TRT" (lane and CUDA Graph sections): every lane
// owns its buffers, two timing events and a non-blocking stream; the work is
// captured once (thread-local capture mode) and replayed with one launch;
// submit records an event, launches the graph and records completion; the
// application synchronises only in wait; a lane is never submitted unless
// acquired nor reused while busy.  And "Streams, concurrency and CUDA Graphs"
// (CUDA handbook, CUDA Graphs section): fixed addresses, capture once,
// instantiate once, nothing synchronising inside the graph.  The network
// between the two stages is not part of this library: its slot in the graph
// is the logits buffer, which the caller fills.  The post-processing stage is
// the Top-K of the logits or, for a detection lane (yolo.cu README: decode,
// bitonic sort and greedy suppression inside the graph), the DFL decode and
// NMS of the head held in that slot.
#include <chrono>
#include <cstring>
#include <new>

#include <nvtx3/nvToolsExt.h>

#include "ws_internal.cuh"

constexpr int kMaxBuckets = 17;   // batch sizes 1, 2, 4, ..., 2^15 and the lane's own

struct ws_lane {
    ws_lane_desc d{};
    int state = WS_LANE_FREE;
    bool fake = false;
    int fake_left = 0;

    cudaStream_t stream = nullptr;
    bool own_stream = false;

    void* in_host = nullptr;       // MAPPED / COPY: host view
    void* in_dev = nullptr;        // what the preprocess reads
    // what the lane allocated itself (freed at destroy); in_host, in_dev and
    // logits are the current bindings, which ws_lane_rebind may change
    void* owned_in_host = nullptr;
    void* owned_in_dev = nullptr;
    void* tensor = nullptr;
    bool own_tensor = false;
    float* logits = nullptr;
    float* owned_logits = nullptr;
    // result slots: Top-K values / indices, or detections / per-image counts
    void* rv_host = nullptr;
    void* ri_host = nullptr;
    void* rv_dev = nullptr;
    void* ri_dev = nullptr;
    size_t rv_bytes = 0, ri_bytes = 0;
    bool own_r_host = false, own_r_dev = false;
    // one post-processing workspace per bucket: a call with a smaller batch
    // lays its workspace out differently, and each layout must keep its own
    // counters at zero between calls
    void* ws[kMaxBuckets] = {};
    size_t ws_bytes[kMaxBuckets] = {};

    size_t input_bytes = 0, tensor_bytes = 0, logits_bytes = 0, result_bytes = 0;

    cudaEvent_t ev_start = nullptr, ev_end = nullptr;
    cudaEvent_t ev_pre0 = nullptr, ev_pre1 = nullptr, ev_post1 = nullptr;
    // batch buckets: bucket i replays bucket_batch[i] frames (the last is the
    // lane's batch); one captured graph and one executable graph per bucket
    int nbuckets = 1;
    int bucket_batch[kMaxBuckets] = {};
    cudaGraph_t graph[kMaxBuckets] = {};
    cudaGraphExec_t exec[kMaxBuckets] = {};
    std::chrono::steady_clock::time_point t_submit;
    // this lane's error word (mapped pinned): its kernels set bits in it when
    // a bounded wait gives up; wait reads and clears it
    uint32_t* err_host = nullptr;
    uint32_t* err_dev = nullptr;
    // a failed rebind could not restore the previous graphs: only destroy
    bool broken = false;
};

namespace ws {
namespace {

bool stage_timing(const ws_lane* L) { return (L->d.flags & WS_LANE_FLAG_STAGE_TIMING) != 0; }
bool submit_timing(const ws_lane* L) { return (L->d.flags & WS_LANE_FLAG_NO_TIMING) == 0; }
bool use_graph(const ws_lane* L) { return (L->d.flags & WS_LANE_FLAG_NO_GRAPH) == 0; }
bool detecting(const ws_lane* L) { return L->d.post == WS_POST_DETECT; }

// NVTX ranges in the "ws" domain (WS_LANE_FLAG_NVTX): host-side spans of the
// lane calls, visible to a profiler that is attached; a no-op otherwise.
nvtxDomainHandle_t nvtx_domain() {
    static nvtxDomainHandle_t d = nvtxDomainCreateA("ws");
    return d;
}

struct NvtxRange {
    bool on;
    NvtxRange(const ws_lane* L, const char* name) : on(L && (L->d.flags & WS_LANE_FLAG_NVTX)) {
        if (!on) return;
        nvtxEventAttributes_t a{};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(nvtx_domain(), &a);
    }
    ~NvtxRange() {
        if (on) nvtxDomainRangePop(nvtx_domain());
    }
};

// Rows of the logits a bucket of nb frames post-processes: per-frame rows
// scale with the batch; a lane that is not bucketed always takes all rows.
int64_t bucket_rows(const ws_lane* L, int nb) {
    return nb == L->d.batch ? L->d.rows : L->d.rows / L->d.batch * nb;
}

// Every CUDA resource a lane makes or frees goes through these helpers: each
// creation first passes a fault point (host-side fault injection, see
// ws_debug_inject_failure) and the live resources are counted.
ws_status alloc_dev(void** p, size_t bytes, const char* what) {
    *p = nullptr;
    if (fault_point()) return fail(WS_ERR_OUT_OF_MEMORY, "injected failure: cudaMalloc of %zu bytes for %s", bytes, what);
    cudaError_t e = cudaMalloc(p, bytes);
    if (e == cudaErrorMemoryAllocation) {
        cudaGetLastError();
        return fail(WS_ERR_OUT_OF_MEMORY, "cudaMalloc of %zu bytes for %s", bytes, what);
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    count_resource(kResDevice, +1);
    return WS_OK;
}

ws_status alloc_host(void** p, size_t bytes, unsigned flags, const char* what) {
    *p = nullptr;
    if (fault_point()) return fail(WS_ERR_OUT_OF_MEMORY, "injected failure: cudaHostAlloc of %zu bytes for %s", bytes, what);
    cudaError_t e = cudaHostAlloc(p, bytes, flags);
    if (e == cudaErrorMemoryAllocation) {
        cudaGetLastError();
        return fail(WS_ERR_OUT_OF_MEMORY, "cudaHostAlloc of %zu bytes for %s", bytes, what);
    }
    if (e != cudaSuccess) return cuda_fail(e, what);
    count_resource(kResHost, +1);
    return WS_OK;
}

void free_dev(void* p) {
    if (!p) return;
    cudaFree(p);
    count_resource(kResDevice, -1);
}

void free_host(void* p) {
    if (!p) return;
    cudaFreeHost(p);
    count_resource(kResHost, -1);
}

ws_status make_event(cudaEvent_t* ev, unsigned flags) {
    *ev = nullptr;
    if (fault_point()) return fail(WS_ERR_CUDA, "injected failure: cudaEventCreateWithFlags");
    WS_TRY_CUDA(cudaEventCreateWithFlags(ev, flags));
    count_resource(kResEvent, +1);
    return WS_OK;
}

void destroy_event(cudaEvent_t ev) {
    if (!ev) return;
    cudaEventDestroy(ev);
    count_resource(kResEvent, -1);
}

ws_status memset_async(void* p, size_t bytes, cudaStream_t s, const char* what) {
    if (fault_point()) return fail(WS_ERR_CUDA, "injected failure: cudaMemsetAsync of %s", what);
    cudaError_t e = cudaMemsetAsync(p, 0, bytes, s);
    if (e != cudaSuccess) return cuda_fail(e, what);
    return WS_OK;
}

void destroy_graph(cudaGraph_t g) {
    if (!g) return;
    cudaGraphDestroy(g);
    count_resource(kResGraph, -1);
}

void destroy_exec(cudaGraphExec_t x) {
    if (!x) return;
    cudaGraphExecDestroy(x);
    count_resource(kResExec, -1);
}

void release_all(ws_lane* L) {
    if (L->fake) return;
    for (int i = 0; i < kMaxBuckets; ++i) {
        destroy_exec(L->exec[i]);
        destroy_graph(L->graph[i]);
        free_dev(L->ws[i]);
        L->exec[i] = nullptr;
        L->graph[i] = nullptr;
        L->ws[i] = nullptr;
    }
    for (cudaEvent_t e : {L->ev_start, L->ev_end, L->ev_pre0, L->ev_pre1, L->ev_post1}) destroy_event(e);
    if (L->own_r_dev) {
        free_dev(L->rv_dev);
        free_dev(L->ri_dev);
    }
    if (L->own_r_host) {
        free_host(L->rv_host);
        free_host(L->ri_host);
    }
    free_dev(L->owned_logits);
    if (L->own_tensor) free_dev(L->tensor);
    free_dev(L->owned_in_dev);
    free_host(L->owned_in_host);
    free_host(L->err_host);
    if (L->own_stream) {
        cudaStreamDestroy(L->stream);
        count_resource(kResStream, -1);
    }
}

ws_status device_view(void* host, void** dev, const char* what) {
    cudaError_t e = cudaHostGetDevicePointer(dev, host, 0);
    if (e != cudaSuccess)
        return fail(WS_ERR_INVALID_ARGUMENT, "%s is not mapped pinned memory (%s)", what, cudaGetErrorName(e));
    return WS_OK;
}

ws_status record(cudaEvent_t ev, cudaStream_t s, bool capturing) {
    WS_TRY_CUDA(cudaEventRecordWithFlags(ev, s, capturing ? cudaEventRecordExternal : cudaEventRecordDefault));
    return WS_OK;
}

// The lane's whole path for bucket bi (its first bucket_batch[bi] frames),
// enqueued on its stream: captured once into the bucket's graph, and also
// used directly for the warm-up and NO_GRAPH lanes.
ws_status enqueue_path(ws_lane* L, bool capturing, int bi) {
    ws_status st;
    const NoPdlScope no_pdl((L->d.flags & WS_LANE_FLAG_NO_PDL) != 0);
    const ErrWordScope err_word(L->err_dev);   // the lane's kernels report into its own word
    const int nb = L->bucket_batch[bi];
    const int64_t rows = bucket_rows(L, nb);
    if (L->d.input_mode == WS_INPUT_COPY)
        WS_TRY_CUDA(cudaMemcpyAsync(L->in_dev, L->in_host, L->input_bytes / L->d.batch * nb, cudaMemcpyHostToDevice,
                                    L->stream));
    if (stage_timing(L) && (st = record(L->ev_pre0, L->stream, capturing)) != WS_OK) return st;
    st = ws_preprocess(&L->d.pre, static_cast<const uint8_t*>(L->in_dev), nb, L->tensor, L->stream);
    if (st != WS_OK) return st;
    if (stage_timing(L) && (st = record(L->ev_pre1, L->stream, capturing)) != WS_OK) return st;
    size_t rv = L->rv_bytes, ri = L->ri_bytes;
    if (detecting(L)) {
        st = ws_detect(&L->d.detect, L->logits, nb, static_cast<ws_detection*>(L->rv_dev),
                       static_cast<int32_t*>(L->ri_dev), L->ws[bi], L->ws_bytes[bi], L->stream);
        rv = rv / L->d.batch * nb;
        ri = ri / L->d.batch * nb;
    } else {
        // the row ticket, not a cluster merge: lanes share the GPU with other lanes' kernels
        st = topk_enqueue(L->logits, rows, L->d.cols, L->d.k, static_cast<float*>(L->rv_dev),
                          static_cast<int32_t*>(L->ri_dev), L->ws[bi], L->ws_bytes[bi], L->stream, false);
        rv = ri = (size_t)rows * L->d.k * sizeof(float);
    }
    if (st != WS_OK) return st;
    if (stage_timing(L) && (st = record(L->ev_post1, L->stream, capturing)) != WS_OK) return st;
    if (L->d.result_mode == WS_RESULT_COPY) {
        WS_TRY_CUDA(cudaMemcpyAsync(L->rv_host, L->rv_dev, rv, cudaMemcpyDeviceToHost, L->stream));
        WS_TRY_CUDA(cudaMemcpyAsync(L->ri_host, L->ri_dev, ri, cudaMemcpyDeviceToHost, L->stream));
    }
    // The completion event is part of the path (an event-record node in a
    // captured graph), so a submit is a single graph launch.
    return record(L->ev_end, L->stream, capturing);
}

// Capture bucket bi's path into a new graph (its buffers as bound now).
ws_status capture_bucket(ws_lane* L, int bi, cudaGraph_t* out) {
    *out = nullptr;
    if (fault_point()) return fail(WS_ERR_CAPTURE, "injected failure: begin capture");
    cudaError_t e = cudaStreamBeginCapture(L->stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return fail(WS_ERR_CAPTURE, "begin capture: %s", cudaGetErrorName(e));
    ws_status st = enqueue_path(L, true, bi);
    cudaGraph_t g = nullptr;
    // the real end of capture always runs, so the stream leaves capture mode
    const bool injected = fault_point();
    e = cudaStreamEndCapture(L->stream, &g);
    if (g) count_resource(kResGraph, +1);
    if (st != WS_OK || e != cudaSuccess || injected) {
        destroy_graph(g);
        cudaGetLastError();
        if (st != WS_OK) return st;
        if (injected) return fail(WS_ERR_CAPTURE, "injected failure: end capture");
        return fail(WS_ERR_CAPTURE, "end capture: %s", cudaGetErrorName(e));
    }
    *out = g;
    return WS_OK;
}

// An executable graph of g, uploaded once so the first submit pays no
// first-launch set-up.  *out is NULL on failure.
ws_status instantiate_graph(cudaGraph_t g, cudaGraphExec_t* out, cudaStream_t stream) {
    *out = nullptr;
    if (fault_point()) return fail(WS_ERR_CAPTURE, "injected failure: instantiate");
    cudaGraphExec_t x = nullptr;
    cudaError_t e = cudaGraphInstantiateWithFlags(&x, g, 0);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(WS_ERR_CAPTURE, "instantiate: %s", cudaGetErrorName(e));
    }
    count_resource(kResExec, +1);
    if (fault_point()) {
        destroy_exec(x);
        return fail(WS_ERR_CAPTURE, "injected failure: upload");
    }
    e = cudaGraphUpload(x, stream);
    if (e != cudaSuccess) {
        destroy_exec(x);
        cudaGetLastError();
        return fail(WS_ERR_CAPTURE, "upload: %s", cudaGetErrorName(e));
    }
    *out = x;
    return WS_OK;
}

// In-place update of executable graph x to graph g's parameters; false when
// refused (the executable graph is then unchanged).
bool exec_update(cudaGraphExec_t x, cudaGraph_t g) {
    if (fault_point()) return false;
    cudaGraphExecUpdateResultInfo info;
    if (cudaGraphExecUpdate(x, g, &info) == cudaSuccess) return true;
    cudaGetLastError();
    return false;
}

ws_status build(ws_lane* L) {
    const ws_lane_desc& d = L->d;
    ws_status st;
    if (d.stream) {
        L->stream = d.stream;
    } else {
        if (fault_point()) return fail(WS_ERR_CUDA, "injected failure: cudaStreamCreateWithFlags");
        WS_TRY_CUDA(cudaStreamCreateWithFlags(&L->stream, cudaStreamNonBlocking));
        L->own_stream = true;
        count_resource(kResStream, +1);
    }
    // the lane's error word: zero, read by the host after each submit
    if ((st = alloc_host((void**)&L->err_host, 64, cudaHostAllocMapped, "error word")) != WS_OK) return st;
    *(volatile uint32_t*)L->err_host = 0u;
    WS_TRY_CUDA(cudaHostGetDevicePointer((void**)&L->err_dev, L->err_host, 0));
    L->input_bytes = (size_t)d.batch * (size_t)d.pre.src_frame_stride;
    const size_t elem = d.pre.dst_type == WS_DTYPE_F32 ? 4 : 2;
    L->tensor_bytes = (size_t)d.batch * 3 * d.pre.dst_h * d.pre.dst_w * elem;
    void* borrowed_rv = d.result_val;
    void* borrowed_ri = d.result_idx;
    if (detecting(L)) {
        int64_t A = 0;
        if ((st = ws_detect_validate(&d.detect, d.batch, &A)) != WS_OK) return st;
        L->logits_bytes = (size_t)d.batch * (4 * d.detect.reg_max + d.detect.num_classes) * (size_t)A * sizeof(float);
        L->rv_bytes = (size_t)d.batch * d.detect.max_det * sizeof(ws_detection);
        L->ri_bytes = (size_t)d.batch * sizeof(int32_t);
        borrowed_rv = d.detections;
        borrowed_ri = d.det_count;
    } else {
        L->logits_bytes = (size_t)d.rows * d.cols * sizeof(float);
        L->rv_bytes = L->ri_bytes = (size_t)d.rows * d.k * sizeof(float);
    }
    L->result_bytes = L->rv_bytes;

    // producer slot
    switch (d.input_mode) {
        case WS_INPUT_DEVICE:
            if (d.input) {
                L->in_dev = d.input;
            } else {
                if ((st = alloc_dev(&L->in_dev, L->input_bytes, "input")) != WS_OK) return st;
                L->owned_in_dev = L->in_dev;
            }
            break;
        case WS_INPUT_MAPPED:
            if (d.input) {
                L->in_host = d.input;
            } else {
                if ((st = alloc_host(&L->in_host, L->input_bytes, cudaHostAllocMapped, "input")) != WS_OK)
                    return st;
                L->owned_in_host = L->in_host;
            }
            if ((st = device_view(L->in_host, &L->in_dev, "input")) != WS_OK) return st;
            break;
        case WS_INPUT_COPY:
            if (d.input) {
                L->in_host = d.input;
            } else {
                if ((st = alloc_host(&L->in_host, L->input_bytes, cudaHostAllocDefault, "input")) != WS_OK)
                    return st;
                L->owned_in_host = L->in_host;
            }
            if ((st = alloc_dev(&L->in_dev, L->input_bytes, "input copy")) != WS_OK) return st;
            L->owned_in_dev = L->in_dev;
            break;
        default:
            return fail(WS_ERR_INVALID_ARGUMENT, "input mode %d", d.input_mode);
    }

    if (d.tensor) {
        L->tensor = d.tensor;
    } else {
        if ((st = alloc_dev(&L->tensor, L->tensor_bytes, "tensor")) != WS_OK) return st;
        L->own_tensor = true;
    }
    if (d.logits) {
        L->logits = d.logits;
    } else {
        if ((st = alloc_dev((void**)&L->logits, L->logits_bytes, "logits")) != WS_OK) return st;
        L->owned_logits = L->logits;
        if ((st = memset_async(L->logits, L->logits_bytes, L->stream, "logits")) != WS_OK) return st;
    }

    // result slot
    switch (d.result_mode) {
        case WS_RESULT_DEVICE:
            if (borrowed_rv) {
                L->rv_dev = borrowed_rv;
                L->ri_dev = borrowed_ri;
            } else {
                if ((st = alloc_dev(&L->rv_dev, L->rv_bytes, "result")) != WS_OK) return st;
                if ((st = alloc_dev(&L->ri_dev, L->ri_bytes, "result")) != WS_OK) {
                    free_dev(L->rv_dev);
                    L->rv_dev = nullptr;
                    return st;
                }
                L->own_r_dev = true;
            }
            break;
        case WS_RESULT_MAPPED:
        case WS_RESULT_COPY: {
            const unsigned flags = d.result_mode == WS_RESULT_MAPPED ? cudaHostAllocMapped : cudaHostAllocDefault;
            if (borrowed_rv) {
                L->rv_host = borrowed_rv;
                L->ri_host = borrowed_ri;
            } else {
                if ((st = alloc_host(&L->rv_host, L->rv_bytes, flags, "result")) != WS_OK) return st;
                if ((st = alloc_host(&L->ri_host, L->ri_bytes, flags, "result")) != WS_OK) {
                    free_host(L->rv_host);
                    L->rv_host = nullptr;
                    return st;
                }
                L->own_r_host = true;
            }
            if (d.result_mode == WS_RESULT_MAPPED) {
                if ((st = device_view(L->rv_host, &L->rv_dev, "result")) != WS_OK) return st;
                if ((st = device_view(L->ri_host, &L->ri_dev, "result")) != WS_OK) return st;
            } else {
                if ((st = alloc_dev(&L->rv_dev, L->rv_bytes, "result")) != WS_OK) return st;
                if ((st = alloc_dev(&L->ri_dev, L->ri_bytes, "result")) != WS_OK) {
                    free_dev(L->rv_dev);
                    L->rv_dev = nullptr;
                    return st;
                }
                L->own_r_dev = true;
            }
            break;
        }
        default:
            return fail(WS_ERR_INVALID_ARGUMENT, "result mode %d", d.result_mode);
    }

    // batch buckets
    L->nbuckets = 0;
    if (d.flags & WS_LANE_FLAG_BUCKETS)
        for (int nb = 1; nb < d.batch && L->nbuckets < kMaxBuckets - 1; nb *= 2) L->bucket_batch[L->nbuckets++] = nb;
    L->bucket_batch[L->nbuckets++] = d.batch;
    for (int bi = 0; bi < L->nbuckets; ++bi) {
        const int nb = L->bucket_batch[bi];
        if (detecting(L)) {
            if ((st = ws_detect_workspace_bytes(&d.detect, nb, &L->ws_bytes[bi])) != WS_OK) return st;
        } else {
            L->ws_bytes[bi] = topk_workspace_size(bucket_rows(L, nb), d.cols, d.k);
        }
        if (L->ws_bytes[bi]) {   // cudaMalloc's alignment covers both workspaces' 256-byte rule
            if ((st = alloc_dev(&L->ws[bi], L->ws_bytes[bi], "post-processing workspace")) != WS_OK) return st;
            if ((st = memset_async(L->ws[bi], L->ws_bytes[bi], L->stream, "post-processing workspace")) != WS_OK)
                return st;
        }
    }

    if (submit_timing(L)) {
        if ((st = make_event(&L->ev_start, cudaEventDefault)) != WS_OK) return st;
        if ((st = make_event(&L->ev_end, cudaEventDefault)) != WS_OK) return st;
    } else {
        // completion only: a timing-disabled event is the lightest marker
        if ((st = make_event(&L->ev_end, cudaEventDisableTiming)) != WS_OK) return st;
    }
    if (stage_timing(L)) {
        if ((st = make_event(&L->ev_pre0, cudaEventDefault)) != WS_OK) return st;
        if ((st = make_event(&L->ev_pre1, cudaEventDefault)) != WS_OK) return st;
        if ((st = make_event(&L->ev_post1, cudaEventDefault)) != WS_OK) return st;
    }

    // Warm direct runs: settle lazy module loading and kernel attributes
    // before anything is captured.
    for (int bi = 0; bi < L->nbuckets; ++bi)
        if ((st = enqueue_path(L, false, bi)) != WS_OK) return st;
    WS_TRY_CUDA(cudaStreamSynchronize(L->stream));

    if (use_graph(L)) {
        for (int bi = 0; bi < L->nbuckets; ++bi) {
            if ((st = capture_bucket(L, bi, &L->graph[bi])) != WS_OK) return st;
            if ((st = instantiate_graph(L->graph[bi], &L->exec[bi], L->stream)) != WS_OK) return st;
        }
        WS_TRY_CUDA(cudaStreamSynchronize(L->stream));
    }
    return WS_OK;
}

ws_status validate_lane(const ws_lane_desc* d) {
    if (!d) return fail(WS_ERR_INVALID_ARGUMENT, "descriptor is NULL");
    ws_status st = validate_preprocess(&d->pre, d->batch);
    if (st != WS_OK) return st;
    if (d->post == WS_POST_DETECT) {
        if ((st = ws_detect_validate(&d->detect, d->batch, nullptr)) != WS_OK) return st;
        if (d->result_val || d->result_idx)
            return fail(WS_ERR_INVALID_ARGUMENT, "a detection lane takes detections / det_count, not result_val / result_idx");
        if ((d->detections == nullptr) != (d->det_count == nullptr))
            return fail(WS_ERR_INVALID_ARGUMENT, "detections and det_count must both be given or both NULL");
    } else if (d->post == WS_POST_TOPK) {
        if ((st = validate_topk(d->rows, d->cols, d->k)) != WS_OK) return st;
        if ((d->result_val == nullptr) != (d->result_idx == nullptr))
            return fail(WS_ERR_INVALID_ARGUMENT, "result_val and result_idx must both be given or both NULL");
    } else {
        return fail(WS_ERR_INVALID_ARGUMENT, "post-processing kind %d", d->post);
    }
    if (d->input_mode < WS_INPUT_DEVICE || d->input_mode > WS_INPUT_COPY)
        return fail(WS_ERR_INVALID_ARGUMENT, "input mode %d", d->input_mode);
    if (d->result_mode < WS_RESULT_DEVICE || d->result_mode > WS_RESULT_COPY)
        return fail(WS_ERR_INVALID_ARGUMENT, "result mode %d", d->result_mode);
    const uint32_t known = WS_LANE_FLAG_NO_GRAPH | WS_LANE_FLAG_STAGE_TIMING | WS_LANE_FLAG_NO_TIMING |
                           WS_LANE_FLAG_NO_DEVICE | WS_LANE_FLAG_NVTX | WS_LANE_FLAG_BUCKETS |
                           WS_LANE_FLAG_NO_PDL;
    if (d->flags & ~known) return fail(WS_ERR_INVALID_ARGUMENT, "unknown flags 0x%x", d->flags & ~known);
    if ((d->flags & WS_LANE_FLAG_NO_DEVICE) && d->fake_polls < 0)
        return fail(WS_ERR_INVALID_ARGUMENT, "fake_polls %d < 0", d->fake_polls);
    if ((d->flags & WS_LANE_FLAG_BUCKETS) && d->post == WS_POST_TOPK && d->rows % d->batch != 0)
        return fail(WS_ERR_INVALID_ARGUMENT, "bucketed Top-K lane needs rows (%lld) a multiple of batch (%d)",
                    (long long)d->rows, d->batch);
    return WS_OK;
}

}  // namespace
}  // namespace ws

extern "C" {

ws_status ws_lane_create(const ws_lane_desc* desc, ws_lane** out) {
    using namespace ws;
    clear_error();
    if (!out) return fail(WS_ERR_INVALID_ARGUMENT, "lane output pointer is NULL");
    *out = nullptr;
    ws_status st = validate_lane(desc);
    if (st != WS_OK) return st;
    ws_lane* L = new (std::nothrow) ws_lane();
    if (!L) return fail(WS_ERR_OUT_OF_MEMORY, "lane object");
    L->d = *desc;
    NvtxRange r(L, "ws_lane_create");
    if (desc->flags & WS_LANE_FLAG_NO_DEVICE) {
        L->fake = true;
        *out = L;
        return WS_OK;
    }
    st = build(L);
    if (st != WS_OK) {
        // keep the message of the failure, not of the cleanup
        release_all(L);
        delete L;
        cudaGetLastError();
        return st;
    }
    *out = L;
    return WS_OK;
}

ws_status ws_lane_get_buffers(const ws_lane* L, ws_lane_buffers* b) {
    ws::clear_error();
    if (!L || !b) return ws::fail(WS_ERR_INVALID_ARGUMENT, "lane or buffers is NULL");
    std::memset(b, 0, sizeof *b);
    b->input_host = L->in_host;
    b->input_device = L->in_dev;
    b->tensor = L->tensor;
    b->logits = L->logits;
    if (L->d.post == WS_POST_DETECT) {
        b->detections_host = static_cast<ws_detection*>(L->rv_host);
        b->det_count_host = static_cast<int32_t*>(L->ri_host);
        b->detections_device = static_cast<ws_detection*>(L->rv_dev);
        b->det_count_device = static_cast<int32_t*>(L->ri_dev);
    } else {
        b->result_val_host = static_cast<float*>(L->rv_host);
        b->result_idx_host = static_cast<int32_t*>(L->ri_host);
        b->result_val_device = static_cast<float*>(L->rv_dev);
        b->result_idx_device = static_cast<int32_t*>(L->ri_dev);
    }
    b->input_bytes = L->input_bytes;
    b->tensor_bytes = L->tensor_bytes;
    b->logits_bytes = L->logits_bytes;
    b->result_bytes = L->result_bytes;
    b->stream = L->stream;
    return WS_OK;
}

ws_status ws_lane_acquire(ws_lane* L) {
    ws::clear_error();
    if (!L) return ws::fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    if (L->state != WS_LANE_FREE)
        return ws::fail(WS_ERR_LANE_BUSY, "lane is %s", L->state == WS_LANE_ACQUIRED ? "acquired" : "in flight");
    L->state = WS_LANE_ACQUIRED;
    return WS_OK;
}

ws_status ws_lane_submit_n(ws_lane* L, int32_t n) {
    using namespace ws;
    clear_error();
    if (!L) return fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    NvtxRange r(L, "ws_lane_submit");
    if (L->state != WS_LANE_ACQUIRED)
        return fail(WS_ERR_LANE_STATE, "submit needs an acquired lane (state %d)", L->state);
    if (n < 1 || n > L->d.batch) return fail(WS_ERR_INVALID_ARGUMENT, "%d frames for a lane of %d", n, L->d.batch);
    if (L->broken) return fail(WS_ERR_CAPTURE, "the lane's graphs could not be restored after a failed rebind; destroy it");
    L->t_submit = std::chrono::steady_clock::now();
    if (L->fake) {
        L->fake_left = L->d.fake_polls;
        L->state = WS_LANE_IN_FLIGHT;
        return WS_OK;
    }
    int bi = 0;   // the smallest bucket that holds n frames
    while (L->bucket_batch[bi] < n) ++bi;
    cudaError_t e = cudaSuccess;
    if (submit_timing(L)) {
        e = cudaEventRecord(L->ev_start, L->stream);
        if (e != cudaSuccess) return cuda_fail(e, "record start event");
    }
    if (use_graph(L)) {
        e = cudaGraphLaunch(L->exec[bi], L->stream);
        if (e != cudaSuccess) return cuda_fail(e, "graph launch");
    } else {
        ws_status st = enqueue_path(L, false, bi);
        if (st != WS_OK) return st;
    }
    L->state = WS_LANE_IN_FLIGHT;
    return WS_OK;
}

ws_status ws_lane_submit(ws_lane* L) {
    if (!L) {
        ws::clear_error();
        return ws::fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    }
    return ws_lane_submit_n(L, L->d.batch);
}

ws_status ws_lane_rebind(ws_lane* L, void* input, float* logits, int32_t* reinstantiated) {
    using namespace ws;
    clear_error();
    if (reinstantiated) *reinstantiated = 0;
    if (!L) return fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    NvtxRange r(L, "ws_lane_rebind");
    if (L->state == WS_LANE_IN_FLIGHT) return fail(WS_ERR_LANE_BUSY, "lane is in flight; wait first");
    if (L->broken) return fail(WS_ERR_CAPTURE, "the lane's graphs could not be restored after a failed rebind; destroy it");
    if (!input && !logits) return WS_OK;
    if (L->fake) {
        if (input) L->d.input = input;
        if (logits) L->d.logits = logits;
        return WS_OK;
    }
    // the new slot addresses
    void* in_host = L->in_host;
    void* in_dev = L->in_dev;
    if (input) {
        switch (L->d.input_mode) {
            case WS_INPUT_DEVICE: in_dev = input; break;
            case WS_INPUT_MAPPED: {
                in_host = input;
                ws_status st = device_view(input, &in_dev, "input");
                if (st != WS_OK) return st;
                break;
            }
            default: in_host = input; break;   // COPY: the graph's copy source
        }
    }
    void* const old_in_host = L->in_host;
    void* const old_in_dev = L->in_dev;
    float* const old_logits = L->logits;
    L->in_host = in_host;
    L->in_dev = in_dev;
    if (logits) L->logits = logits;
    if (!use_graph(L)) return WS_OK;
    // Re-capture each bucket with the new addresses and update its executable
    // graph in place ("Streams, concurrency and CUDA Graphs", CUDA Graphs:
    // cudaGraphExecUpdate instead of re-instantiation); re-instantiate only if
    // the update is refused.  All or nothing: every bucket is captured before
    // any executable graph changes, and on a later failure the graphs already
    // updated are put back to their previous parameters.
    cudaGraph_t ng[kMaxBuckets] = {};
    cudaGraphExec_t nx[kMaxBuckets] = {};
    bool updated[kMaxBuckets] = {};
    auto undo = [&](ws_status st) {
        for (int bi = 0; bi < L->nbuckets; ++bi) {
            if (updated[bi]) {
                cudaGraphExecUpdateResultInfo info;
                if (cudaGraphExecUpdate(L->exec[bi], L->graph[bi], &info) != cudaSuccess) {
                    cudaGetLastError();
                    L->broken = true;
                }
            }
            destroy_exec(nx[bi]);
            destroy_graph(ng[bi]);
        }
        L->in_host = old_in_host;
        L->in_dev = old_in_dev;
        L->logits = old_logits;
        return st;
    };
    for (int bi = 0; bi < L->nbuckets; ++bi) {
        ws_status st = capture_bucket(L, bi, &ng[bi]);
        if (st != WS_OK) return undo(st);
    }
    for (int bi = 0; bi < L->nbuckets; ++bi) {
        if (exec_update(L->exec[bi], ng[bi])) {
            updated[bi] = true;
            continue;
        }
        ws_status st = instantiate_graph(ng[bi], &nx[bi], L->stream);
        if (st != WS_OK) return undo(st);
    }
    for (int bi = 0; bi < L->nbuckets; ++bi) {
        if (nx[bi]) {
            destroy_exec(L->exec[bi]);
            L->exec[bi] = nx[bi];
            if (reinstantiated) *reinstantiated = 1;
        }
        destroy_graph(L->graph[bi]);
        L->graph[bi] = ng[bi];
    }
    return WS_OK;
}

ws_status ws_lane_wait(ws_lane* L, int64_t timeout_us, ws_lane_timing* timing) {
    using namespace ws;
    clear_error();
    if (!L) return fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    NvtxRange r(L, "ws_lane_wait");
    if (L->state != WS_LANE_IN_FLIGHT) return fail(WS_ERR_LANE_STATE, "wait needs a lane in flight");
    const auto t0 = std::chrono::steady_clock::now();
    if (!L->fake && timeout_us < 0) {
        // no deadline: the driver's own wait on the completion event reacts
        // faster than polling cudaEventQuery
        cudaError_t e = cudaEventSynchronize(L->ev_end);
        if (e != cudaSuccess) {
            L->state = WS_LANE_FREE;
            return cuda_fail(e, "lane work");
        }
    }
    for (;;) {
        cudaError_t e;
        if (L->fake) {
            e = L->fake_left > 0 ? cudaErrorNotReady : cudaSuccess;
            if (L->fake_left > 0) --L->fake_left;
        } else {
            e = cudaEventQuery(L->ev_end);
        }
        if (e == cudaSuccess) break;
        if (e != cudaErrorNotReady) {
            L->state = WS_LANE_FREE;
            return cuda_fail(e, "lane work");
        }
        if (timeout_us >= 0) {
            const auto waited =
                std::chrono::duration_cast<std::chrono::microseconds>(std::chrono::steady_clock::now() - t0);
            if (waited.count() >= timeout_us) return fail(WS_ERR_TIMEOUT, "lane still in flight");
        }
    }
    const auto t1 = std::chrono::steady_clock::now();
    // The work has completed, so whatever its kernels wrote into the mapped
    // error word is visible here.
    const uint32_t dev_err = L->fake ? 0u : *(volatile uint32_t*)L->err_host;
    if (timing) {
        timing->host_us = std::chrono::duration<double, std::micro>(t1 - L->t_submit).count();
        timing->gpu_us = timing->preprocess_us = timing->post_us = -1.f;
        if (!L->fake) {
            float ms = 0.f;
            if (submit_timing(L) && cudaEventElapsedTime(&ms, L->ev_start, L->ev_end) == cudaSuccess)
                timing->gpu_us = ms * 1000.f;
            if (stage_timing(L)) {
                if (cudaEventElapsedTime(&ms, L->ev_pre0, L->ev_pre1) == cudaSuccess)
                    timing->preprocess_us = ms * 1000.f;
                if (cudaEventElapsedTime(&ms, L->ev_pre1, L->ev_post1) == cudaSuccess)
                    timing->post_us = ms * 1000.f;
            }
            cudaGetLastError();
        }
    }
    L->state = WS_LANE_FREE;
    if (dev_err) {
        *(volatile uint32_t*)L->err_host = 0u;   // the next submit starts clean
        return fail(WS_ERR_DEVICE,
                    "a kernel of this lane reported an error (bits 0x%x%s%s); this submit's results are undefined",
                    dev_err, (dev_err & kDevErrBulkCopyTimeout) ? ": a bulk copy did not complete in time" : "",
                    (dev_err & kDevErrBadLaunch) ? ": a launch did not match its parameters" : "");
    }
    return WS_OK;
}

ws_status ws_lane_selftest_wait_timeout(ws_lane* L, uint32_t limit_us) {
    using namespace ws;
    clear_error();
    if (!L) return fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    if (L->fake) return fail(WS_ERR_UNSUPPORTED, "a host-only lane has no GPU error word");
    if (L->state == WS_LANE_IN_FLIGHT) return fail(WS_ERR_LANE_BUSY, "lane is in flight; wait first");
    return launch_selftest_wait(L->err_dev, limit_us, L->stream);
}

ws_status ws_lane_release(ws_lane* L) {
    ws::clear_error();
    if (!L) return ws::fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    if (L->state != WS_LANE_ACQUIRED) return ws::fail(WS_ERR_LANE_STATE, "release needs an acquired lane");
    L->state = WS_LANE_FREE;
    return WS_OK;
}

ws_status ws_lane_destroy(ws_lane* L) {
    ws::clear_error();
    if (!L) return ws::fail(WS_ERR_INVALID_ARGUMENT, "lane is NULL");
    if (L->state == WS_LANE_IN_FLIGHT) return ws::fail(WS_ERR_LANE_BUSY, "lane is in flight; wait first");
    ws::release_all(L);
    delete L;
    return WS_OK;
}

int32_t ws_lane_state(const ws_lane* L) { return L ? L->state : -1; }

}  // extern "C"
