// ws_core.cu -- status strings, per-thread error text, version, the device
// property cache and the device error word.
#include <atomic>
#include <cstring>
#include <mutex>
#include <string>

#include "ws_internal.cuh"
#include "ws_ptx.cuh"

// Error bits raised by kernels whose bounded waits ran out; one copy per
// device, zero at module load.
__device__ uint32_t g_dev_error_flags;

namespace ws {

namespace {
thread_local std::string t_error;

constexpr int kMaxDevices = 64;
DeviceInfo g_info[kMaxDevices];
bool g_have[kMaxDevices];
uint32_t* g_err_word[kMaxDevices];
std::mutex g_mu;
}  // namespace

ws_status fail(ws_status status, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    t_error = buf;
    return status;
}

void clear_error() { t_error.clear(); }

ws_status cuda_fail(cudaError_t err, const char* what) {
    return fail(WS_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(err), cudaGetErrorString(err));
}

ws_status current_device_info(int* device, const DeviceInfo** info) {
    int dev = 0;
    WS_TRY_CUDA(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return fail(WS_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_have[dev]) {
        DeviceInfo d{};
        WS_TRY_CUDA(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev));
        WS_TRY_CUDA(cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
        WS_TRY_CUDA(cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev));
        // Device address of this device's error word (no allocation).
        uint32_t* w = nullptr;
        WS_TRY_CUDA(cudaGetSymbolAddress((void**)&w, g_dev_error_flags));
        g_err_word[dev] = w;
        g_info[dev] = d;
        g_have[dev] = true;
    }
    *device = dev;
    *info = &g_info[dev];
    return WS_OK;
}

namespace {
thread_local bool t_no_pdl = false;
}

bool pdl_enabled() { return !t_no_pdl; }

NoPdlScope::NoPdlScope(bool active) : prev(t_no_pdl) {
    if (active) t_no_pdl = true;
}

NoPdlScope::~NoPdlScope() { t_no_pdl = prev; }

namespace {
thread_local uint32_t* t_err_word = nullptr;
}

ErrWordScope::ErrWordScope(uint32_t* word) : prev(t_err_word) {
    if (word) t_err_word = word;
}

ErrWordScope::~ErrWordScope() { t_err_word = prev; }

uint32_t* device_error_word() {
    if (t_err_word) return t_err_word;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    return g_err_word[dev];
}

// ---- host-side fault injection and resource counters -----------------------
namespace {
std::atomic<long long> g_fault_reached{0};   // fault points reached since the last arming
std::atomic<long long> g_fault_first{0};     // first failing point (1-based), 0 = off
std::atomic<long long> g_fault_count{0};     // consecutive points that fail
std::atomic<long long> g_live[kResCount];
}  // namespace

bool fault_point() {
    const long long first = g_fault_first.load(std::memory_order_relaxed);
    const long long n = g_fault_reached.fetch_add(1, std::memory_order_relaxed) + 1;
    return first > 0 && n >= first && n < first + g_fault_count.load(std::memory_order_relaxed);
}

void count_resource(Resource r, int delta) { g_live[r].fetch_add(delta, std::memory_order_relaxed); }

}  // namespace ws

extern "C" {

const char* ws_status_string(ws_status s) {
    switch (s) {
        case WS_OK: return "WS_OK";
        case WS_ERR_INVALID_ARGUMENT: return "WS_ERR_INVALID_ARGUMENT";
        case WS_ERR_UNSUPPORTED: return "WS_ERR_UNSUPPORTED";
        case WS_ERR_CUDA: return "WS_ERR_CUDA";
        case WS_ERR_OUT_OF_MEMORY: return "WS_ERR_OUT_OF_MEMORY";
        case WS_ERR_LANE_STATE: return "WS_ERR_LANE_STATE";
        case WS_ERR_LANE_BUSY: return "WS_ERR_LANE_BUSY";
        case WS_ERR_TIMEOUT: return "WS_ERR_TIMEOUT";
        case WS_ERR_CAPTURE: return "WS_ERR_CAPTURE";
        case WS_ERR_DEVICE: return "WS_ERR_DEVICE";
        default: return "WS_ERR_UNKNOWN";
    }
}

}  // extern "C"

namespace ws {

// An mbarrier armed for 16 bytes that no copy will deliver: the bounded wait
// runs out, the kernel records the timeout in the device error word and
// returns -- the path every kernel takes when a bulk copy never lands.
__global__ void selftest_wait_kernel(uint32_t* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(&bar, 16u);
    if (!mbar_wait_bounded(&bar, 0, limit_ns)) atomicOr(err, kDevErrBulkCopyTimeout);
}

ws_status launch_selftest_wait(uint32_t* word, uint32_t limit_us, cudaStream_t stream) {
    if (limit_us < 1 || limit_us > 1000000) return fail(WS_ERR_INVALID_ARGUMENT, "limit %u us outside 1..1e6", limit_us);
    if (!word) return fail(WS_ERR_INVALID_ARGUMENT, "no error word");
    selftest_wait_kernel<<<1, 32, 0, stream>>>(word, 1000ull * limit_us);
    WS_TRY_CUDA(cudaGetLastError());
    return WS_OK;
}

}  // namespace ws

extern "C" {

const char* ws_last_error(void) { return ws::t_error.c_str(); }

int32_t ws_version(void) { return 100; }  // 0.1.0

int32_t ws_build_features(void) {
#ifdef WS_BOUNDS_CHECK
    return WS_FEATURE_BOUNDS_CHECK;
#else
    return 0;
#endif
}

ws_status ws_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream) {
    ws::clear_error();
    int dev;
    const ws::DeviceInfo* info;
    ws_status st = ws::current_device_info(&dev, &info);
    if (st != WS_OK) return st;
    return ws::launch_selftest_wait(ws::device_error_word(), limit_us, stream);
}

ws_status ws_debug_inject_failure(int32_t nth, int32_t count) {
    ws::clear_error();
    if (count < 0) return ws::fail(WS_ERR_INVALID_ARGUMENT, "count %d < 0", count);
    ws::g_fault_first.store(0, std::memory_order_relaxed);
    ws::g_fault_count.store(count, std::memory_order_relaxed);
    ws::g_fault_reached.store(0, std::memory_order_relaxed);
    ws::g_fault_first.store(nth > 0 && count > 0 ? nth : 0, std::memory_order_relaxed);
    return WS_OK;
}

ws_status ws_debug_get_counters(ws_debug_counters* c) {
    ws::clear_error();
    if (!c) return ws::fail(WS_ERR_INVALID_ARGUMENT, "counters is NULL");
    c->device_allocs = ws::g_live[ws::kResDevice].load();
    c->host_allocs = ws::g_live[ws::kResHost].load();
    c->graphs = ws::g_live[ws::kResGraph].load();
    c->graph_execs = ws::g_live[ws::kResExec].load();
    c->events = ws::g_live[ws::kResEvent].load();
    c->streams = ws::g_live[ws::kResStream].load();
    c->fault_points = ws::g_fault_reached.load();
    return WS_OK;
}

ws_status ws_device_error(uint32_t* flags, int32_t clear) {
    ws::clear_error();
    if (!flags) return ws::fail(WS_ERR_INVALID_ARGUMENT, "flags is NULL");
    int dev;
    const ws::DeviceInfo* info;
    ws_status st = ws::current_device_info(&dev, &info);
    if (st != WS_OK) return st;
    uint32_t* w = ws::device_error_word();
    uint32_t v = 0;
    WS_TRY_CUDA(cudaMemcpy(&v, w, sizeof v, cudaMemcpyDeviceToHost));
    if (clear) {
        const uint32_t zero = 0;
        WS_TRY_CUDA(cudaMemcpy(w, &zero, sizeof zero, cudaMemcpyHostToDevice));
    }
    *flags = v;
    return WS_OK;
}

}  // extern "C"
