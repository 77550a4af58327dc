// pool.cu -- a pool of identical lanes with a producer / consumer hand-off.
//
// "Inside WarpStream TRT" (lane and state-machine sections): several lanes
// keep the GPU busy while the host fills some and drains others; a lane is
// never reused while its results are still being read, and when every lane
// is busy the producer is told so (back-pressure) instead of blocking the
// GPU.  The pool adds to the lane's own FREE -> ACQUIRED -> IN_FLIGHT cycle
// two host-side stages: submitted lanes are completed in submission order,
// and a completed lane is held (its results readable) until the consumer
// recycles it.  Built only on the public lane calls.
#include <chrono>
#include <condition_variable>
#include <deque>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include "ws_internal.cuh"

namespace {

enum Where { kFree = 0, kAcquired = 1, kSubmitted = 2, kHeld = 3 };

}  // namespace

struct ws_pool {
    std::vector<ws_lane*> lanes;
    std::vector<int> where;             // per lane: Where
    std::deque<int> free_q;             // lanes ready to be acquired
    std::deque<int> sub_q;              // submitted lanes, oldest first
    bool completing = false;            // a consumer is waiting on sub_q.front()
    std::mutex mu;
    std::condition_variable cv_free, cv_sub;
};

namespace {

int index_of(const ws_pool* P, const ws_lane* L) {
    for (size_t i = 0; i < P->lanes.size(); ++i)
        if (P->lanes[i] == L) return (int)i;
    return -1;
}

// Waits on cv until pred() holds; timeout_us < 0 waits without limit.
template <typename Pred>
bool wait_until(std::unique_lock<std::mutex>& lk, std::condition_variable& cv, int64_t timeout_us, Pred pred) {
    if (timeout_us < 0) {
        cv.wait(lk, pred);
        return true;
    }
    return cv.wait_for(lk, std::chrono::microseconds(timeout_us), pred);
}

void destroy_lanes(ws_pool* P) {
    for (ws_lane* L : P->lanes)
        if (L) ws_lane_destroy(L);
    P->lanes.clear();
}

}  // namespace

extern "C" {

ws_status ws_pool_create(const ws_lane_desc* desc, int32_t nlanes, ws_pool** out) {
    using namespace ws;
    clear_error();
    if (!out) return fail(WS_ERR_INVALID_ARGUMENT, "pool output pointer is NULL");
    *out = nullptr;
    if (!desc) return fail(WS_ERR_INVALID_ARGUMENT, "descriptor is NULL");
    if (nlanes < 1 || nlanes > 64) return fail(WS_ERR_INVALID_ARGUMENT, "%d lanes outside 1..64", nlanes);
    if (desc->input || desc->tensor || desc->logits || desc->result_val || desc->result_idx || desc->detections ||
        desc->det_count)
        return fail(WS_ERR_INVALID_ARGUMENT, "pool lanes own their buffers: leave the buffer pointers NULL");
    ws_pool* P = new (std::nothrow) ws_pool();
    if (!P) return fail(WS_ERR_OUT_OF_MEMORY, "pool object");
    for (int i = 0; i < nlanes; ++i) {
        ws_lane* L = nullptr;
        ws_status st = ws_lane_create(desc, &L);
        if (st != WS_OK) {
            // destroying the lanes already made clears the thread's message:
            // keep the failing lane's
            const std::string msg = ws_last_error();
            destroy_lanes(P);
            delete P;
            return fail(st, "lane %d of %d: %s", i, nlanes, msg.c_str());
        }
        P->lanes.push_back(L);
        P->where.push_back(kFree);
        P->free_q.push_back(i);
    }
    *out = P;
    return WS_OK;
}

ws_status ws_pool_lane(const ws_pool* P, int32_t i, ws_lane** lane) {
    ws::clear_error();
    if (!P || !lane) return ws::fail(WS_ERR_INVALID_ARGUMENT, "pool or lane pointer is NULL");
    if (i < 0 || i >= (int32_t)P->lanes.size()) return ws::fail(WS_ERR_INVALID_ARGUMENT, "lane %d out of range", i);
    *lane = P->lanes[(size_t)i];
    return WS_OK;
}

ws_status ws_pool_acquire(ws_pool* P, int64_t timeout_us, ws_lane** lane) {
    using namespace ws;
    clear_error();
    if (!P || !lane) return fail(WS_ERR_INVALID_ARGUMENT, "pool or lane pointer is NULL");
    *lane = nullptr;
    int i;
    {
        std::unique_lock<std::mutex> lk(P->mu);
        if (!wait_until(lk, P->cv_free, timeout_us, [P] { return !P->free_q.empty(); }))
            return fail(WS_ERR_TIMEOUT, "every lane is busy");
        i = P->free_q.front();
        P->free_q.pop_front();
        P->where[(size_t)i] = kAcquired;
    }
    ws_status st = ws_lane_acquire(P->lanes[(size_t)i]);
    if (st != WS_OK) {   // cannot happen for a lane only the pool hands out; give it back
        std::lock_guard<std::mutex> lk(P->mu);
        P->where[(size_t)i] = kFree;
        P->free_q.push_front(i);
        P->cv_free.notify_one();
        return st;
    }
    *lane = P->lanes[(size_t)i];
    return WS_OK;
}

ws_status ws_pool_submit(ws_pool* P, ws_lane* L, int32_t n) {
    using namespace ws;
    clear_error();
    if (!P || !L) return fail(WS_ERR_INVALID_ARGUMENT, "pool or lane is NULL");
    const int i = index_of(P, L);
    if (i < 0) return fail(WS_ERR_INVALID_ARGUMENT, "lane is not in this pool");
    {
        std::lock_guard<std::mutex> lk(P->mu);
        if (P->where[(size_t)i] != kAcquired) return fail(WS_ERR_LANE_STATE, "submit needs a lane acquired from the pool");
    }
    ws_status st = ws_lane_submit_n(L, n);
    if (st != WS_OK) return st;   // the lane stays acquired
    std::lock_guard<std::mutex> lk(P->mu);
    P->where[(size_t)i] = kSubmitted;
    P->sub_q.push_back(i);
    P->cv_sub.notify_all();
    return WS_OK;
}

ws_status ws_pool_complete(ws_pool* P, int64_t timeout_us, ws_lane** lane, ws_lane_timing* timing) {
    using namespace ws;
    clear_error();
    if (!P || !lane) return fail(WS_ERR_INVALID_ARGUMENT, "pool or lane pointer is NULL");
    *lane = nullptr;
    const auto t0 = std::chrono::steady_clock::now();
    int i;
    {
        std::unique_lock<std::mutex> lk(P->mu);
        if (!wait_until(lk, P->cv_sub, timeout_us, [P] { return !P->sub_q.empty() && !P->completing; }))
            return fail(WS_ERR_TIMEOUT, "nothing completed");
        i = P->sub_q.front();
        P->completing = true;
    }
    int64_t left = timeout_us;
    if (timeout_us >= 0) {
        const int64_t spent =
            std::chrono::duration_cast<std::chrono::microseconds>(std::chrono::steady_clock::now() - t0).count();
        left = spent >= timeout_us ? 0 : timeout_us - spent;
    }
    ws_status st = ws_lane_wait(P->lanes[(size_t)i], left, timing);
    std::lock_guard<std::mutex> lk(P->mu);
    P->completing = false;
    P->cv_sub.notify_all();
    if (st == WS_ERR_TIMEOUT) return st;   // still in flight, still first in line
    // done (or failed on the GPU: the lane is FREE, its results undefined)
    P->sub_q.pop_front();
    P->where[(size_t)i] = kHeld;
    *lane = P->lanes[(size_t)i];
    return st;
}

ws_status ws_pool_recycle(ws_pool* P, ws_lane* L) {
    using namespace ws;
    clear_error();
    if (!P || !L) return fail(WS_ERR_INVALID_ARGUMENT, "pool or lane is NULL");
    const int i = index_of(P, L);
    if (i < 0) return fail(WS_ERR_INVALID_ARGUMENT, "lane is not in this pool");
    std::lock_guard<std::mutex> lk(P->mu);
    if (P->where[(size_t)i] == kAcquired) {   // acquired but never submitted: give it back
        ws_status st = ws_lane_release(L);
        if (st != WS_OK) return st;
    } else if (P->where[(size_t)i] != kHeld) {
        return fail(WS_ERR_LANE_STATE, "recycle takes a completed (or unsubmitted) lane");
    }
    P->where[(size_t)i] = kFree;
    P->free_q.push_back(i);
    P->cv_free.notify_one();
    return WS_OK;
}

ws_status ws_pool_destroy(ws_pool* P) {
    using namespace ws;
    clear_error();
    if (!P) return fail(WS_ERR_INVALID_ARGUMENT, "pool is NULL");
    {
        std::lock_guard<std::mutex> lk(P->mu);
        if (!P->sub_q.empty() || P->completing) return fail(WS_ERR_LANE_BUSY, "lanes are in flight; complete them first");
    }
    for (size_t i = 0; i < P->lanes.size(); ++i)
        if (P->where[i] == kAcquired) ws_lane_release(P->lanes[i]);
    destroy_lanes(P);
    delete P;
    return WS_OK;
}

}  // extern "C"
