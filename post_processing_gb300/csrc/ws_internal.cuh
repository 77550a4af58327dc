// ws_internal.cuh -- helpers shared by the library's translation units:
// per-thread error text, status shorthands and a per-device property cache.
#pragma once

#include <cstdarg>
#include <cstdint>
#include <cstdio>

#include <cuda_runtime.h>

#include "ws.h"

namespace ws {

// Records a message for ws_last_error() and returns `status`.
ws_status fail(ws_status status, const char* fmt, ...);
// Clears the thread's message (called on entry of each public call).
void clear_error();
// WS_ERR_CUDA with the CUDA error name, or WS_OK.
ws_status cuda_fail(cudaError_t err, const char* what);

#define WS_TRY_CUDA(expr)                                        \
    do {                                                         \
        cudaError_t ws_e_ = (expr);                              \
        if (ws_e_ != cudaSuccess) return ws::cuda_fail(ws_e_, #expr); \
    } while (0)

struct DeviceInfo {
    int sm_count;
    int max_smem_optin;     // bytes of dynamic shared memory a block may opt in to
    int smem_per_sm;
};
// Properties of the current device, queried once per device.
ws_status current_device_info(int* device, const DeviceInfo** info);

// Host-side argument checks shared by the entry points and the lanes.
ws_status validate_preprocess(const ws_preprocess_desc* d, int32_t batch);
ws_status validate_topk(int64_t rows, int64_t cols, int32_t k);
size_t topk_workspace_size(int64_t rows, int64_t cols, int32_t k);
// The Top-K launch behind ws_topk (same arguments and checks).  With
// cluster_merge_ok a row cut into 2 .. 8 chunks merges through a thread-block
// cluster of its blocks instead of the row ticket, which is faster when the
// Top-K has the GPU to itself; the lanes pass false, because beside other
// lanes' kernels a cluster waits for all its block slots in one GPC at once.
ws_status topk_enqueue(const float* x, int64_t rows, int64_t cols, int32_t k, float* out_val, int32_t* out_idx,
                       void* workspace, size_t workspace_bytes, cudaStream_t stream, bool cluster_merge_ok);

// Error bits kernels raise instead of waiting forever (see ws_device_error).
enum : uint32_t {
    kDevErrBulkCopyTimeout = 1u,
    kDevErrBadLaunch = 2u,   // a kernel's launch did not match its parameters: it did nothing
    kDevErrBounds = 4u,      // checked build: an index was out of range and was clamped
};

// Checked build (compiled with WS_BOUNDS_CHECK): an index tested against its
// buffer; out of range it sets kDevErrBounds in `err` and is clamped into
// [lo, hi), so nothing outside the buffer is read or written.  Without the
// macro the check is the index itself.
#ifdef WS_BOUNDS_CHECK
__device__ __forceinline__ int checked_index(int i, int lo, int hi, uint32_t* err) {
    if (i < lo || i >= hi) {
        atomicOr(err, (uint32_t)kDevErrBounds);
        i = i < lo ? lo : hi - 1;
    }
    return i;
}
#define WS_CHECKED(i, lo, hi, err) checked_index((i), (lo), (hi), (err))
#else
#define WS_CHECKED(i, lo, hi, err) (i)
#endif
// Device address of the error word the calling thread's kernels report
// into: a lane's own word while that lane enqueues or captures its path (see
// ErrWordScope), else the current device's word.  Kernels receive it as a
// parameter (no relocatable device code, so they cannot name it directly).
uint32_t* device_error_word();
// While alive, kernels enqueued by this thread report into `word` (NULL keeps
// the current choice).
struct ErrWordScope {
    uint32_t* prev;
    explicit ErrWordScope(uint32_t* word);
    ~ErrWordScope();
};
// Enqueues the bounded-wait self-test kernel (see ws_selftest_wait_timeout)
// reporting into `word`.
ws_status launch_selftest_wait(uint32_t* word, uint32_t limit_us, cudaStream_t stream);

// Host-side fault injection for the lanes' and the pool's cleanup paths (see
// ws_debug_inject_failure): true when the fault point reached now is to fail.
// Every internal call that can fail during lane creation or re-binding passes
// through one before the CUDA call it guards.
bool fault_point();
// Live CUDA resources the library made (see ws_debug_get_counters).
enum Resource { kResDevice = 0, kResHost, kResGraph, kResExec, kResEvent, kResStream, kResCount };
void count_resource(Resource r, int delta);

// Programmatic dependent launch of the stream-ordered kernels (preprocess,
// Top-K, class scan, DFL, NMS): on unless the calling thread is inside a
// NoPdlScope (a lane with WS_LANE_FLAG_NO_PDL enqueuing or capturing its path).
bool pdl_enabled();
struct NoPdlScope {
    bool prev;
    explicit NoPdlScope(bool active);
    ~NoPdlScope();
};

// Launches `kernel` as a programmatic dependent of the previous kernel on the
// stream ("Streams, concurrency and CUDA Graphs", PDL section) when
// pdl_enabled(), else as an ordinary launch.  Every kernel launched this way
// executes griddepcontrol.wait before its first global-memory access.
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, args...);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace ws
