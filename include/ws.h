/* ws.h -- C ABI of the GB300 fused RGB8 -> FP32 NCHW preprocess and the
 * exact Top-K, plus the fixed-shape lanes that replay both as one CUDA Graph.
 *
 * Sources of the operations (page title, then section):
 *  - "Inside WarpStream TRT", problem-statement table: interleaved RGB8
 *    producer, fixed-shape FP32 NCHW network input, fixed-size FP32 logits,
 *    exact Top-K with K <= 32, fixed preallocated lanes, no allocation in
 *    the submit/wait path.
 *  - "Inside WarpStream TRT", fused-preprocessing section and its data-flow
 *    figure: per destination pixel a centre-aligned bilinear sample, scaling
 *    to [0,1], (value - mean) * inverse_std per channel, stored straight into
 *    the channel plane of the NCHW tensor; no intermediate image exists.
 *  - yolo.cu README, "Two ways to use it": the same preprocess as a letterbox
 *    into the network input, and a small handle-based C API.
 *  - "Inside WarpStream TRT", Top-K section: exact selection, ties to the
 *    lower class index, NaN treated as negative infinity, only K score/index
 *    pairs written back.
 *  - "Inside WarpStream TRT", lane and CUDA Graph sections: each lane owns
 *    fixed buffers, events, a non-blocking stream and one instantiated graph
 *    (preprocess, network, Top-K captured once); submit records an event,
 *    launches the graph and records completion; a lane cannot be submitted
 *    unless acquired nor reused while busy, so backpressure is part of the API.
 *  - "Streams, concurrency and CUDA Graphs" (CUDA handbook), CUDA Graphs
 *    section: capture once, instantiate once, one launch per replay; fixed
 *    addresses and shapes; nothing synchronising inside the graph.
 *
 * Conventions (apply to every call):
 *  - Every call returns a ws_status; no exception crosses the ABI.  Outputs
 *    are defined only when the call returns WS_OK.  On an error,
 *    ws_last_error() returns a message for the calling thread.
 *  - Arguments are validated on the host before anything is enqueued; a
 *    rejected call enqueues nothing.
 *  - ws_preprocess and ws_topk are asynchronous and stream-ordered; they
 *    allocate nothing and never synchronise, so they may be captured into a
 *    CUDA Graph.  A device fault shows up later, at a stream or event
 *    synchronisation, as WS_ERR_CUDA.
 *  - Pointers are plain addresses: "device" means memory the GPU reads or
 *    writes (cudaMalloc, or the device view of mapped pinned memory), "host"
 *    means CPU memory.  The caller owns every pointer it passes; the library
 *    only keeps borrowed pointers inside a lane, and those must stay valid,
 *    at the same address, until the lane is destroyed.
 *  - Calls on one lane are not thread-safe; different lanes are independent.
 *  - The library computes everything on the GPU.  There is no CPU fallback:
 *    without a usable CUDA device the compute calls return WS_ERR_CUDA.
 */
#ifndef WS_H
#define WS_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ------------------------------------------------------------------ status */

typedef int32_t ws_status;
#define WS_OK                   0
#define WS_ERR_INVALID_ARGUMENT 1  /* a size, pointer, mode or stride was rejected          */
#define WS_ERR_UNSUPPORTED      2  /* valid request this build or device cannot serve        */
#define WS_ERR_CUDA             3  /* a CUDA runtime call failed (message names the error)   */
#define WS_ERR_OUT_OF_MEMORY    4  /* a lane could not allocate its buffers                  */
#define WS_ERR_LANE_STATE       5  /* lane call made in the wrong state (e.g. submit unacquired) */
#define WS_ERR_LANE_BUSY        6  /* lane is acquired or in flight and cannot be taken      */
#define WS_ERR_TIMEOUT          7  /* ws_lane_wait deadline passed; the lane stays in flight */
#define WS_ERR_CAPTURE          8  /* graph capture or instantiation failed                  */
#define WS_ERR_DEVICE           9  /* a kernel's bounded wait gave up (see ws_device_error)  */

/* Static name of a status ("WS_OK", ...); never NULL. */
const char* ws_status_string(ws_status status);

/* Message of the last failed call made by this thread ("" if none).  The
 * pointer stays valid until this thread's next ws_* call. */
const char* ws_last_error(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int32_t ws_version(void);

/* Features of the loaded build, a bit mask.  WS_FEATURE_BOUNDS_CHECK: the
 * checked build (libws_bounds.so, the same sources compiled with
 * WS_BOUNDS_CHECK), whose preprocess kernels test every index into their
 * shared stage slots and column-tap table and every source tap; an index out
 * of range sets device error bit 0x4 (ws_device_error) and is clamped into
 * its buffer, so the kernel neither traps nor touches memory outside it.  The
 * checks cost time; the default build has none. */
#define WS_FEATURE_BOUNDS_CHECK 1
int32_t ws_build_features(void);

/* Error bits that kernels set on the current device instead of hanging or
 * faulting: 0x1 when a bounded wait (an mbarrier wait on a bulk copy) runs
 * out, 0x2 when a kernel finds its launch inconsistent with its parameters
 * (a cluster shape it was not built for) and does nothing, 0x4 in the checked
 * build when an index was out of range and was clamped (ws_build_features).
 * Reads the flags synchronously; clears them when clear != 0.  *flags == 0
 * means none. */
ws_status ws_device_error(uint32_t* flags, int32_t clear);

/* Diagnostic of that path: launches one thread that arms an mbarrier for 16
 * bytes no copy will deliver and waits for it at most limit_us (1 .. 1e6)
 * microseconds; when the wait runs out it sets the timeout bit in the device
 * error word and returns, as a kernel whose bulk copy never landed does.
 * Asynchronous on `stream`; read the result with ws_device_error. */
ws_status ws_selftest_wait_timeout(uint32_t limit_us, cudaStream_t stream);

/* Host-side fault injection for the cleanup paths of ws_lane_create,
 * ws_lane_rebind and ws_pool_create (a test hook; the pages' lane section asks
 * that failures be explicit, never a silent leak or a half-built lane).  Each
 * internal call of those paths that can fail (a stream, event, device or
 * pinned allocation, a memset, a graph capture, instantiation, upload or
 * update) first passes a fault point.  After this call, fault points number
 * nth, nth + 1, ..., nth + count - 1 counted from now (1-based, over all
 * threads) fail without calling CUDA, with the status the real failure would
 * give: WS_ERR_OUT_OF_MEMORY for an allocation, WS_ERR_CAPTURE for a graph
 * step, WS_ERR_CUDA otherwise.  An end of capture is the one exception: the
 * real call is made, so the stream leaves capture mode, and its graph is then
 * discarded.  nth <= 0 or count == 0 disarms it.  Nothing runs on the GPU. */
ws_status ws_debug_inject_failure(int32_t nth, int32_t count);

/* CUDA resources the library holds now, and the fault points reached since
 * the last ws_debug_inject_failure (for leak checks after a failure). */
typedef struct ws_debug_counters {
    int64_t device_allocs;        /* cudaMalloc blocks                              */
    int64_t host_allocs;          /* cudaHostAlloc blocks                           */
    int64_t graphs, graph_execs;  /* captured and executable graphs                 */
    int64_t events, streams;
    int64_t fault_points;         /* fault points reached since the last arming     */
} ws_debug_counters;
ws_status ws_debug_get_counters(ws_debug_counters* counters);

/* -------------------------------------------------------------- preprocess */

#define WS_RESIZE_STRETCH   0  /* bilinear resize of the whole frame to dst_w x dst_h   */
#define WS_RESIZE_LETTERBOX 1  /* aspect-preserving resize, centred, rest = pad_value  */

#define WS_NORM_MEAN_STD 0     /* out = (v - 255 mean_c) / (255 std_c)                  */
#define WS_NORM_SCALE    1     /* out = v * scale                                       */

#define WS_ORDER_RGB 0         /* source bytes are R, G, B; planes are written R, G, B  */
#define WS_ORDER_BGR 1         /* source bytes are B, G, R; planes are still written R, G, B
                                  (yolo.cu README: its engine takes BGR frames) */

#define WS_DTYPE_F32  0        /* destination float32                                    */
#define WS_DTYPE_F16  1        /* destination IEEE half, the FP32 value rounded to nearest even */
#define WS_DTYPE_BF16 2        /* destination bfloat16, the FP32 value rounded to nearest even  */

/* Geometry and normalisation of the fused preprocess.
 *
 * Resize convention (the pages say only "centre-aligned"; this is the
 * reading taken): destination pixel x of a box of D pixels samples source
 * coordinate (x + 1/2) * S / D - 1/2 (half-pixel centres), held as the exact
 * rational ((2x+1) S - D) / (2 D); the lower neighbour is its floor, the
 * weight is the remainder divided by 2D in one correctly rounded float
 * division, and both neighbours are clamped to [0, S-1] (clamp to edge).
 * Four neighbours, no antialias prefilter.  Interpolation and normalisation
 * are FP32.  Letterbox: scale min(dst_w/src_w, dst_h/src_h); the short side of
 * the inner box is the scaled length rounded half up (at least 1 pixel); the
 * box is centred with the odd padding pixel at the bottom / right; pixels
 * outside it take pad_value, normalised like a source byte. */
typedef struct ws_preprocess_desc {
    int32_t src_w, src_h;         /* source frame size in pixels, 1 .. 65535          */
    int64_t src_row_stride;       /* bytes between source rows, >= 3 * src_w         */
    int64_t src_frame_stride;     /* bytes between frames, >= row_stride * src_h    */
    int32_t dst_w, dst_h;         /* destination size, 1 .. 65535                    */
    int32_t resize;               /* WS_RESIZE_*                                     */
    int32_t pad_value;            /* 0 .. 255, letterbox padding byte (e.g. 114)     */
    int32_t norm;                 /* WS_NORM_*                                       */
    float   mean[3];              /* WS_NORM_MEAN_STD, in [0,1] units, per channel   */
    float   std[3];               /* WS_NORM_MEAN_STD, > 0, in [0,1] units           */
    float   scale;                /* WS_NORM_SCALE (e.g. 1/255)                      */
    int32_t channel_order;        /* WS_ORDER_RGB or WS_ORDER_BGR                    */
    int32_t dst_type;             /* WS_DTYPE_F32 (default 0), _F16 or _BF16 ("Inside
                                     WarpStream TRT", next steps: precision-specialised
                                     preprocessing); half outputs halve the bytes written */
} ws_preprocess_desc;

/* Host-only check of a descriptor for a batch; enqueues nothing. */
ws_status ws_preprocess_validate(const ws_preprocess_desc* desc, int32_t batch);

/* Fused preprocess of `batch` frames.
 *   src: device, uint8; byte (b, row j, column i, channel c) is at
 *        src[b * src_frame_stride + j * src_row_stride + 3 * i + c].
 *   dst: device, [batch][3][dst_h][dst_w] (NCHW, contiguous) of the element
 *        type desc->dst_type (float32, half or bfloat16).
 * One kernel launch on `stream`, a programmatic dependent of the kernel
 * before it (it reads and writes nothing until that kernel has finished).
 * Any alignment is accepted.  Outputs above 460,000 pixels (batch x dst_w x
 * dst_h, dst_w at most 8192) take the staged bulk-copy kernel, smaller
 * outputs a per-pixel kernel with the same results (see
 * ws_preprocess_path).  The staged kernel copies each needed source row as
 * its 16-byte window (from the 16-byte boundary at or below the row's first
 * byte to the one at or above its last): with a base or stride that is not a
 * multiple of 16 it reads up to 15 bytes before and after a row, always
 * inside 16-byte blocks that hold bytes of the row, and never uses them.
 * Errors: WS_ERR_INVALID_ARGUMENT (NULL pointer, batch < 1, bad descriptor),
 * WS_ERR_CUDA (launch failed). */
ws_status ws_preprocess(const ws_preprocess_desc* desc, const uint8_t* src, int32_t batch,
                        void* dst, cudaStream_t stream);

#define WS_PRE_PATH_AUTO   0  /* as ws_preprocess                                        */
#define WS_PRE_PATH_STAGED 1  /* the staged bulk-copy kernel (dst_w at most 8192)          */
#define WS_PRE_PATH_DIRECT 2  /* the per-pixel kernel                                     */

/* ws_preprocess with the kernel chosen by `path` (the results are the same;
 * for measurement and tests).  WS_ERR_INVALID_ARGUMENT for an unknown path. */
ws_status ws_preprocess_path(const ws_preprocess_desc* desc, const uint8_t* src, int32_t batch,
                             void* dst, int32_t path, cudaStream_t stream);

/* ------------------------------------------------------------------- top-k */

/* Host-only check: rows >= 1, 1 <= cols < 2^31, 1 <= k <= min(32, cols). */
ws_status ws_topk_validate(int64_t rows, int64_t cols, int32_t k);

/* Bytes of device workspace ws_topk needs for this shape (0 when every row
 * fits one block).  Depends only on (rows, cols, k). */
ws_status ws_topk_workspace_bytes(int64_t rows, int64_t cols, int32_t k, size_t* bytes);

/* Zero a workspace before its first use (one cudaMemsetAsync on `stream`).
 * Every completed ws_topk leaves it ready for the next call, so this is not
 * needed between calls or graph replays. */
ws_status ws_topk_workspace_init(void* workspace, size_t bytes, cudaStream_t stream);

/* Exact Top-K of each row.
 *   x:       device, float32 [rows][cols], read only.
 *   out_val: device (or device view of mapped memory), float32 [rows][k].
 *   out_idx: same, int32 [rows][k].
 * Per row the k entries with the largest values in rank order; equal
 * values (+0 equals -0) go to the lower index; NaN ranks as -inf.  out_val
 * holds the input's own bits (-0.0 stays -0.0) except that NaN is written as
 * -inf.  The result is unique, so it is bit-exact.
 * workspace: device, 256-byte aligned, at least ws_topk_workspace_bytes()
 * bytes, zeroed once by ws_topk_workspace_init() (or cudaMemset) before first
 * use; it holds a ticket per row and each chunk's K keys of rows longer than
 * 8192 entries, and every completed call leaves the tickets at zero again.
 * Calls that share a workspace must not overlap on the GPU.  May be NULL when
 * the size is 0.
 * One kernel launch on `stream`.  A row cut into 2 to 8 chunks is launched
 * as one thread-block cluster per row when the GPU can place such clusters:
 * the chunks' lists then meet in shared memory and the workspace is not
 * touched (lanes use the workspace form, which shares SMs better with other
 * lanes' kernels).
 * Errors: WS_ERR_INVALID_ARGUMENT (shape, K, NULL pointer, workspace too
 * small), WS_ERR_CUDA (launch failed). */
ws_status ws_topk(const float* x, int64_t rows, int64_t cols, int32_t k,
                  float* out_val, int32_t* out_idx,
                  void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Top-K for callers that cannot allocate device memory.  Same result as
 * ws_topk (same kernel, bit-exact), but its scratch lives in a fixed 1 MiB
 * array inside the library's device image instead of a caller workspace.
 * The pages have no counterpart of this call.
 *
 * Who needs it: code that is handed only its input and output buffers and has
 * no allocator of its own (a plugin or callback running inside another
 * framework's enqueue), and latency-critical loops that must not call
 * cudaMalloc after start-up (allocation can synchronise the device and take
 * driver locks, which shows up as tail latency).  They cannot size, own or
 * free a workspace; this call needs none.
 *
 * Arguments: as ws_topk (x device [rows][cols]; out_val / out_idx device
 * [rows][k]); nothing is allocated and no workspace is passed.
 * Limits and behaviour:
 *  - The scratch a shape needs is ws_topk_workspace_bytes(rows, cols, k);
 *    shapes needing more than 1 MiB (1048576 bytes) are rejected with
 *    WS_ERR_UNSUPPORTED and a message giving both sizes; nothing is enqueued.
 *    Rows of at most 8192 entries need no scratch at all.
 *  - The array costs 1 MiB of device memory on every GPU that loads the
 *    library, held until the process exits.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, no allocation) with that device current; make that
 *    first call before any stream capture.
 *  - Every call shares the one array, which keeps the last call's contents;
 *    each call therefore clears its row tickets first (one cudaMemsetAsync of
 *    rows * 4 bytes on `stream`).  Calls that overlap on the GPU (for example
 *    on two streams at once) race on the array and give wrong results:
 *    serialise them.
 * Errors: WS_ERR_INVALID_ARGUMENT (shape, K, NULL pointer), WS_ERR_UNSUPPORTED
 * (scratch above the limit), WS_ERR_CUDA (set-up, clearing or launch failed). */
ws_status ws_topk_noalloc(const float* x, int64_t rows, int64_t cols, int32_t k,
                          float* out_val, int32_t* out_idx, cudaStream_t stream);

/* ---------------------------------------------------------------- detection
 * DFL box decode and class-aware greedy NMS of a YOLO-style head, on the GPU
 * (yolo.cu README, "Why is it this fast?": GPU-resident NMS, a bitonic sort
 * sized to the live candidate count, then greedy suppression, inside the
 * graph; "Inside WarpStream TRT", next steps: detection decode and NMS).
 * Readings where the pages give no formula:
 *  - head: float32 [batch][4 * reg_max + num_classes][A]; anchors run level
 *    by level (strides[]), row-major within a level; anchor (x, y) of a level
 *    with stride s is centred at ((x + 1/2) s, (y + 1/2) s) input pixels;
 *  - DFL: each side's distance (left, top, right, bottom) is the expectation
 *    of the bin index under the softmax of its reg_max logits, in strides;
 *    box = (cx - l s, cy - t s, cx + r s, cy + b s), FP32 on the GPU;
 *  - class = arg-max of the class logits (lower class on ties, NaN ranked as
 *    -inf, -0 equal to +0, as in the Top-K); an anchor is a candidate when
 *    that logit exceeds logit_thr (pass logit(conf)): the decision needs no
 *    transcendental, so it is exact;
 *  - candidates enter NMS in order of logit (the same NaN / -0 rule), higher
 *    first, lower anchor on ties; if an image has more than max_cand, only
 *    the first max_cand do;
 *  - greedy, class-aware: a candidate is dropped when an already kept box of
 *    its class has IoU > iou_thr with it, tested as inter > iou_thr * union in
 *    FP32 with each operation rounded separately; at most max_det are kept;
 *    score = logistic(logit). */
typedef struct ws_detect_desc {
    int32_t in_w, in_h;           /* network input size in pixels                 */
    int32_t nlevels;              /* feature levels, 1 .. 4                        */
    int32_t strides[4];           /* stride of each level; in_w, in_h divisible   */
    int32_t reg_max;              /* DFL bins per side, 1 .. 32                    */
    int32_t num_classes;          /* 1 .. 4096                                     */
    float   logit_thr;            /* candidate when best class logit > logit_thr  */
    float   iou_thr;              /* drop when IoU > iou_thr (same class)         */
    int32_t max_cand;             /* candidates entering NMS per image, 1 .. 1024 */
    int32_t max_det;              /* detections kept per image, 1 .. max_cand     */
} ws_detect_desc;

/* A candidate box (decode output, NMS input), 32 bytes. */
typedef struct ws_candidate {
    float   x1, y1, x2, y2;       /* input pixels                                  */
    float   logit;                /* best class logit                              */
    int32_t cls, anchor, pad_;
} ws_candidate;

/* A kept detection, 32 bytes. */
typedef struct ws_detection {
    float   x1, y1, x2, y2;       /* input pixels                                  */
    float   score;                /* logistic(logit)                               */
    int32_t cls, anchor, pad_;
} ws_detection;

/* Host-only check; also reports the anchor count A of the geometry. */
ws_status ws_detect_validate(const ws_detect_desc* desc, int32_t batch, int64_t* anchors);

/* Bytes of device workspace ws_detect needs (candidates of every image plus
 * per-image counters).  Zero it once with ws_detect_workspace_init(); every
 * completed ws_detect leaves the counters at zero again. */
ws_status ws_detect_workspace_bytes(const ws_detect_desc* desc, int32_t batch, size_t* bytes);
ws_status ws_detect_workspace_init(void* workspace, size_t bytes, cudaStream_t stream);

/* Decode only.  cand: device ws_candidate [batch][A] (in no particular order);
 * count: device int32 [batch], which must be zero on entry; receives each
 * image's number of candidates (at most A).  One kernel launch: a warp per
 * 128-anchor tile scans the class rows, then decodes its candidates' DFL
 * boxes.
 * Deployment note: each DFL logit is an isolated 4-byte read.  With the
 * context limit cudaLimitMaxL2FetchGranularity at 32 bytes, such a read
 * fetches one 32-byte sector instead of two (batch-64 640x640 head on GB300:
 * 194 instead of 241 MB read, 37.2 instead of 40.4 us).  The library does not
 * change the limit: it is context-wide and also affects other kernels. */
ws_status ws_detect_decode(const ws_detect_desc* desc, const float* head, int32_t batch,
                           ws_candidate* cand, int32_t* count, cudaStream_t stream);

/* NMS only.  cand / count as written by ws_detect_decode (or by the caller:
 * any order, count[b] <= A, anchors distinct within an image).  out: device
 * ws_detection [batch][max_det] in keep order; out_count: device int32
 * [batch].  count[b] is reset to zero.  One kernel launch, programmatically
 * dependent on the previous kernel in the stream (it waits for that
 * kernel's results before reading cand / count).  When the GPU can hold the
 * whole batch that way, each image gets a thread-block cluster of 2, 4 or 8
 * CTAs of about 210 KB of shared memory each (max_cand 1024): an image with
 * more than 256 candidates is selected, sorted and compared across the
 * cluster, the others run on one CTA while the rest leave at once. */
ws_status ws_detect_nms(const ws_detect_desc* desc, ws_candidate* cand, int32_t* count, int32_t batch,
                        ws_detection* out, int32_t* out_count, cudaStream_t stream);

/* Decode + NMS with the candidates in `workspace`.  Two kernel launches (the
 * decode, then the NMS as its programmatic dependent), as in
 * ws_detect_decode and ws_detect_nms.
 * Errors: WS_ERR_INVALID_ARGUMENT (descriptor, pointers, workspace too
 * small), WS_ERR_CUDA (launch failed). */
ws_status ws_detect(const ws_detect_desc* desc, const float* head, int32_t batch,
                    ws_detection* out, int32_t* out_count, void* workspace, size_t workspace_bytes,
                    cudaStream_t stream);

/* ------------------------------------------------------------------- lanes */

#define WS_INPUT_DEVICE 0   /* producer writes a device buffer                       */
#define WS_INPUT_MAPPED 1   /* producer writes mapped pinned host memory; the kernel reads it in place */
#define WS_INPUT_COPY   2   /* producer writes pinned host memory; the graph copies it to the device first */

#define WS_RESULT_DEVICE 0  /* result stays in device memory                         */
#define WS_RESULT_MAPPED 1  /* the last kernel writes straight into mapped pinned host memory */
#define WS_RESULT_COPY   2  /* result is copied into pinned host memory at the end of the graph */

#define WS_LANE_FLAG_NO_GRAPH     1u  /* replay by direct launches instead of the CUDA Graph   */
#define WS_LANE_FLAG_STAGE_TIMING 2u  /* event nodes around each stage for per-stage times   */
#define WS_LANE_FLAG_NO_TIMING    4u  /* submit records only a completion event (timing
                                         disabled) instead of the start / end timing pair:
                                         each timing event costs the GPU a short bubble, so
                                         back-to-back throughput lanes run faster without
                                         them; ws_lane_timing.gpu_us is then -1 */
#define WS_LANE_FLAG_NO_DEVICE    8u  /* host-only lane: no CUDA resource is made; submit marks
                                         it in flight and the "GPU" finishes after fake_polls
                                         completion queries.  Exercises the state machine on
                                         machines without a GPU. */
#define WS_LANE_FLAG_NVTX        16u  /* NVTX ranges (domain "ws") around create, submit, wait and
                                         rebind, for a profiler's timeline ("Inside WarpStream
                                         TRT", next steps: NVTX instrumentation) */
#define WS_LANE_FLAG_BUCKETS     32u  /* one graph per batch bucket 1, 2, 4, ... below batch, plus
                                         batch itself; ws_lane_submit_n(n) replays the smallest
                                         bucket that holds n frames ("Streams, concurrency and
                                         CUDA Graphs", CUDA Graphs: one graph per batch-size
                                         bucket, the real batch rounded up).  A Top-K lane needs
                                         rows a multiple of batch (per-frame rows scale with
                                         the bucket); a detection lane takes one head per frame. */
#define WS_LANE_FLAG_NO_PDL      64u  /* launch the lane's Top-K / DFL / NMS kernels as ordinary
                                         stream-ordered launches instead of programmatic
                                         dependent launches (to measure what PDL saves:
                                         "Streams, concurrency and CUDA Graphs", PDL section) */

#define WS_POST_TOPK   0    /* post-processing: exact Top-K of the logits (rows x cols) */
#define WS_POST_DETECT 1    /* post-processing: DFL decode + class-aware NMS of a detection head */

#define WS_LANE_FREE      0
#define WS_LANE_ACQUIRED  1
#define WS_LANE_IN_FLIGHT 2

/* Everything a lane is built from.  Shapes are fixed for the lane's life.
 * Each buffer pointer is optional: NULL makes the lane allocate (and own) it,
 * non-NULL borrows the caller's buffer, which must outlive the lane. */
typedef struct ws_lane_desc {
    ws_preprocess_desc pre;       /* preprocess geometry                            */
    int32_t  batch;               /* frames per submit                              */
    int64_t  rows, cols;          /* logits shape                                   */
    int32_t  k;                   /* Top-K per row, 1 .. 32                         */
    int32_t  input_mode;          /* WS_INPUT_*                                     */
    int32_t  result_mode;         /* WS_RESULT_*                                    */
    uint32_t flags;               /* WS_LANE_FLAG_*                                 */
    void*    input;               /* DEVICE: device buffer; MAPPED: host pointer of a
                                     cudaHostAllocMapped allocation; COPY: pinned host
                                     buffer.  batch * src_frame_stride bytes.       */
    void*    tensor;              /* device, [batch][3][dst_h][dst_w] of pre.dst_type */
    float*   logits;              /* device, [rows][cols]; the network's output slot */
    float*   result_val;          /* DEVICE: device; MAPPED: mapped host; COPY: pinned host; [rows][k] */
    int32_t* result_idx;          /* same, int32 [rows][k]                          */
    cudaStream_t stream;          /* NULL: the lane creates a non-blocking stream   */
    int32_t  fake_polls;          /* WS_LANE_FLAG_NO_DEVICE only                    */
    int32_t  post;                /* WS_POST_TOPK or WS_POST_DETECT                 */
    ws_detect_desc detect;        /* WS_POST_DETECT: geometry and thresholds.  The
                                     logits slot then holds the head, float32
                                     [batch][4 reg_max + num_classes][A]; rows, cols
                                     and k are ignored and result_val / result_idx
                                     must be NULL.                                 */
    ws_detection* detections;     /* WS_POST_DETECT result [batch][detect.max_det],
                                     memory as result_mode says (like result_val)  */
    int32_t* det_count;           /* WS_POST_DETECT, int32 [batch]: kept per image  */
} ws_lane_desc;

typedef struct ws_lane ws_lane;

/* Stable addresses of a lane's buffers (valid until ws_lane_destroy). */
typedef struct ws_lane_buffers {
    void*    input_host;          /* host view of the producer slot (MAPPED, COPY) or NULL */
    void*    input_device;        /* device buffer the preprocess reads             */
    void*    tensor;              /* device NCHW tensor (pre.dst_type elements)     */
    float*   logits;              /* device logits                                  */
    float*   result_val_host;     /* host view of the result (MAPPED, COPY) or NULL */
    int32_t* result_idx_host;
    float*   result_val_device;   /* where the Top-K kernel writes                  */
    int32_t* result_idx_device;
    size_t   input_bytes, tensor_bytes, logits_bytes, result_bytes;
    cudaStream_t stream;
    ws_detection* detections_host;   /* WS_POST_DETECT: host view (MAPPED, COPY) or NULL */
    int32_t* det_count_host;
    ws_detection* detections_device; /* where the NMS kernel writes             */
    int32_t* det_count_device;
} ws_lane_buffers;

/* Times of one completed submit. */
typedef struct ws_lane_timing {
    float  gpu_us;         /* event before the graph launch -> event after the last stage
                              (-1 on WS_LANE_FLAG_NO_TIMING lanes) */
    float  preprocess_us;  /* STAGE_TIMING lanes: preprocess kernel alone, else -1   */
    float  post_us;        /* STAGE_TIMING lanes: the post-processing stage alone
                              (Top-K, or decode + NMS), else -1                    */
    double host_us;        /* steady clock, entry of submit -> return of wait       */
} ws_lane_timing;

/* Validate, allocate or borrow every buffer, run the path once directly
 * (which settles any lazy set-up), capture copy-in -> preprocess -> Top-K (or
 * decode -> NMS) -> copy-out into one graph on the lane's stream and
 * instantiate it.  All
 * allocation of the lane's life happens here.  Must not be called while the
 * stream is being captured.  On failure everything made so far is released.
 * Errors: WS_ERR_INVALID_ARGUMENT, WS_ERR_OUT_OF_MEMORY, WS_ERR_CUDA,
 * WS_ERR_CAPTURE. */
ws_status ws_lane_create(const ws_lane_desc* desc, ws_lane** lane);

ws_status ws_lane_get_buffers(const ws_lane* lane, ws_lane_buffers* buffers);

/* FREE -> ACQUIRED; WS_ERR_LANE_BUSY if the lane is acquired or in flight. */
ws_status ws_lane_acquire(ws_lane* lane);

/* ACQUIRED -> IN_FLIGHT: record the start event (timing lanes) and launch
 * the graph (or the direct launches), whose last step records the end event.
 * No allocation, no synchronisation.
 * WS_ERR_LANE_STATE unless acquired; WS_ERR_CUDA if a launch fails (the lane
 * then returns to ACQUIRED). */
ws_status ws_lane_submit(ws_lane* lane);

/* As ws_lane_submit, for the first n frames (1 <= n <= batch): a bucketed lane
 * replays the smallest bucket of at least n frames (frames past n in it are
 * processed as they are and their results are to be ignored); otherwise the
 * whole batch is replayed.  Results for the first n frames (rows) are valid. */
ws_status ws_lane_submit_n(ws_lane* lane, int32_t n);

/* Point the lane at a new producer slot and / or logits slot without
 * rebuilding it: input is, per input_mode, a device buffer (DEVICE), the host
 * pointer of a mapped pinned allocation (MAPPED) or pinned host memory (COPY),
 * with the lane's frame layout; logits is a device buffer of the lane's
 * logits (or head) shape.  NULL keeps the current one.  The new buffers are
 * borrowed and must outlive their use.  Each bucket's graph is re-captured
 * and its executable graph updated in place with cudaGraphExecUpdate ("Streams,
 * concurrency and CUDA Graphs", CUDA Graphs); only if the update is refused is
 * it re-instantiated, which *reinstantiated (if not NULL) reports.  Buffers the
 * lane allocated itself stay allocated until ws_lane_destroy.  This is how a
 * producer that writes into its own device memory (a decoder's or camera's
 * GPUDirect buffers) registers them with a lane.
 * All or nothing: every bucket is re-captured before any executable graph
 * changes, and a failure after some graphs were updated puts those back, so
 * on an error the lane keeps its previous buffers and graphs.
 * WS_ERR_LANE_BUSY while in flight; WS_ERR_INVALID_ARGUMENT for a MAPPED input
 * that is not mapped pinned memory; WS_ERR_CAPTURE if a capture,
 * instantiation or update fails (the lane is unchanged and usable).  Only if
 * putting the previous graphs back fails as well is the lane marked broken:
 * later submits and rebinds return WS_ERR_CAPTURE and it may only be
 * destroyed. */
ws_status ws_lane_rebind(ws_lane* lane, void* input, float* logits, int32_t* reinstantiated);

/* IN_FLIGHT -> FREE once the end event has completed.  timeout_us < 0 waits
 * without limit; otherwise WS_ERR_TIMEOUT after timeout_us microseconds, with
 * the lane still IN_FLIGHT (call again).  timing may be NULL.
 * Every lane has its own error word (4 bytes of mapped pinned memory) that its
 * kernels set when a bounded wait on a bulk copy runs out ("Inside WarpStream
 * TRT", lane section: failures are explicit); wait reads it once the work has
 * completed, with no extra synchronisation.
 * WS_ERR_LANE_STATE unless in flight; WS_ERR_CUDA if the GPU work failed;
 * WS_ERR_DEVICE if one of the lane's kernels gave up a bounded wait (the
 * message names the error bits; the word is cleared, so the next submit
 * starts clean).  After either error the lane is FREE and this submit's
 * results are undefined. */
ws_status ws_lane_wait(ws_lane* lane, int64_t timeout_us, ws_lane_timing* timing);

/* Diagnostic of the lane's error path: enqueues on the lane's stream the
 * bounded wait that nothing completes (as ws_selftest_wait_timeout, 1 .. 1e6
 * microseconds), reporting into this lane's error word, so that the wait of
 * the next submit returns WS_ERR_DEVICE.  The lane must not be in flight
 * (WS_ERR_LANE_BUSY) nor host-only (WS_ERR_UNSUPPORTED). */
ws_status ws_lane_selftest_wait_timeout(ws_lane* lane, uint32_t limit_us);

/* ACQUIRED -> FREE without a submit; WS_ERR_LANE_STATE otherwise. */
ws_status ws_lane_release(ws_lane* lane);

/* Free what the lane owns.  WS_ERR_LANE_BUSY while IN_FLIGHT (wait first). */
ws_status ws_lane_destroy(ws_lane* lane);

/* WS_LANE_FREE / ACQUIRED / IN_FLIGHT, or -1 for NULL. */
int32_t ws_lane_state(const ws_lane* lane);

/* -------------------------------------------------------------- lane pool */

/* N identical lanes with a producer / consumer hand-off ("Inside WarpStream
 * TRT", lane and state-machine sections: several lanes keep the GPU busy while
 * the host fills and drains others; a busy lane is reported, not waited on).
 * A lane goes: free -> acquired (ws_pool_acquire; the producer fills its
 * input / logits slots) -> submitted (ws_pool_submit) -> completed
 * (ws_pool_complete, oldest submission first; its results are readable and it
 * is held) -> free (ws_pool_recycle).  Any number of producer threads and one
 * consumer thread at a time may call concurrently.  Timeouts: < 0 waits
 * without limit, 0 does not wait. */
typedef struct ws_pool ws_pool;

/* `lanes` (1 .. 64) lanes from one descriptor; its buffer pointers must be
 * NULL (every lane owns its buffers).  Errors as ws_lane_create. */
ws_status ws_pool_create(const ws_lane_desc* desc, int32_t lanes, ws_pool** pool);

/* Lane i of the pool (for ws_lane_get_buffers). */
ws_status ws_pool_lane(const ws_pool* pool, int32_t i, ws_lane** lane);

/* A free lane, acquired; WS_ERR_TIMEOUT if none became free in time. */
ws_status ws_pool_acquire(ws_pool* pool, int64_t timeout_us, ws_lane** lane);

/* ws_lane_submit_n on an acquired pool lane; on failure it stays acquired. */
ws_status ws_pool_submit(ws_pool* pool, ws_lane* lane, int32_t n);

/* Waits for the oldest submitted lane; *lane is it, completed and held.
 * WS_ERR_TIMEOUT if nothing completed in time; WS_ERR_CUDA or WS_ERR_DEVICE
 * (as ws_lane_wait) if its GPU work failed (it is still returned, held, its
 * results undefined). */
ws_status ws_pool_complete(ws_pool* pool, int64_t timeout_us, ws_lane** lane, ws_lane_timing* timing);

/* A held (or an acquired, unsubmitted) lane back to the free list. */
ws_status ws_pool_recycle(ws_pool* pool, ws_lane* lane);

/* Destroys every lane; WS_ERR_LANE_BUSY while any is submitted. */
ws_status ws_pool_destroy(ws_pool* pool);

#ifdef __cplusplus
}
#endif

#endif /* WS_H */
