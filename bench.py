"""Benchmark of the fused preprocess + exact Top-K hot path on GB300.

One step = one replay of a lane's CUDA Graph: preprocess a batch of RGB8
frames into the FP32 NCHW tensor, then the row-wise exact Top-K of the
logits (the network between them is out of scope; its output slot is a
fixed logits buffer).  Default workload: 64 independent 1920x1080 RGB8
frames -> 224x224 mean/std, Top-32 of [64, 1000] logits, the batched
HBM-throughput configuration.  The headline replays four lanes in
rotation, each on its own stream (one lane's preprocess overlaps the
previous lane's Top-K, as lanes run in a deployment); the same lanes on one
shared stream, every step serialised, are reported beside it.  Also measured
on every run:

* batch-1 graph-replay latency (p50 / p99 / max, GPU events and host steady
  clock, graph and no-graph) on one 1920x1080 frame -> 224x224, Top-5 of 1000;
* end-to-end throughput through the lane API with host buffers: the frames
  sit in mapped pinned host memory, which the preprocess reads in place, and
  the K pairs are written to pinned host memory (a second figure copies the
  whole frames in with a copy node of the graph);
* the roofline of the dominant kernel (the preprocess): its average launch
  duration from CUDA events around back-to-back launches on the lanes'
  buffers, against the measured HBM copy bandwidth;
* the CPU oracle on the host cores (a bounded sample), as a reported baseline;
* detection decode + NMS of a YOLO-style 640x640 head: batch-64 throughput,
  the decode kernel's HBM rate, and batch-1 latency through a detection lane;
* lane graph variants: re-binding cost (cudaGraphExecUpdate), a bucketed
  lane's 1-frame replay, and batch-1 frames/s through a pool of 1, 2, 4 lanes.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
       [--workload NAME] [--latency-samples S] [--no-cpu-baseline]
Multi-GPU (replicas, no collective on the data path) runs under torchrun.
Rank 0 prints one JSON line on stdout; everything else goes to stderr.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "frames/s + HBM GB/s (% of roofline); p50/p99 batch-1 graph-replay latency"
DEFAULT_WORKLOAD = "b64_1080p_to_224"
LATENCY_WORKLOAD = "b1_1080p_to_224"
FALLBACK_HBM_GBS = 6800.0
LANES = 4          # throughput lanes at least; more for small workloads (see n_lanes)
MAX_LANES = 64

# DRAM traffic of the preprocess kernel per launch from one ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum) of the FP32-output
# workload, keyed by the SHA-256 of the kernel source it was taken on;
# reported only for that output type and while that source is unchanged.
# Filled from the committed ncu summary under profiles/.
NCU_TRAFFIC = {
    "b64_1080p_to_224": {
        "bytes": 185_237_760,
        "source_sha": "084f6c76b3b2aa2ff2e2df4063500e9f55313b39b9971ca2bf0d538841ae7c27",
    },
    "b8_4k_to_512": {
        "bytes": 99_373_312,
        "source_sha": "084f6c76b3b2aa2ff2e2df4063500e9f55313b39b9971ca2bf0d538841ae7c27",
    },
}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


CUDA_LIMIT_MAX_L2_FETCH_GRANULARITY = 5   # cudaLimitMaxL2FetchGranularity


def _cudart():
    """The CUDA runtime torch has loaded (dlopen returns that copy), or None."""
    import glob
    import torch
    names = ["libcudart.so.13", "libcudart.so"]
    names += glob.glob(os.path.join(os.path.dirname(torch.__file__), "..", "nvidia", "*", "lib", "libcudart.so*"))
    names += glob.glob("/usr/local/cuda/lib64/libcudart.so*")
    for n in names:
        try:
            lib = ctypes.CDLL(n)
        except OSError:
            continue
        lib.cudaDeviceGetLimit.argtypes = [ctypes.POINTER(ctypes.c_size_t), ctypes.c_int]
        lib.cudaDeviceSetLimit.argtypes = [ctypes.c_int, ctypes.c_size_t]
        return lib
    return None


# ----------------------------------------------------------------- geometry
# Bytes the path must move at minimum (the algorithmic bytes): the 32-byte
# sectors of the source that taps with a non-zero weight touch, the FP32
# tensor written once, the logits read once and the K pairs written.

def _axis(S: int, D: int):
    x = np.arange(D, dtype=np.int64)
    num = (2 * x + 1) * S - D
    den = 2 * D
    q = np.floor_divide(num, den)
    rem = num - q * den
    lo = np.clip(q, 0, S - 1)
    hi = np.clip(q + 1, 0, S - 1)
    return lo, hi, rem != 0


def _box(sw, sh, dw, dh, letterbox):
    if not letterbox:
        return dw, dh
    if dw * sh <= dh * sw:
        return dw, max(1, (2 * sh * dw + sw) // (2 * sw))
    return max(1, (2 * sw * dh + sh) // (2 * sh)), dh


def algorithmic_bytes(w: dict, out_bytes: int = 4) -> dict:
    nw, nh = _box(w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], w["resize"] == "letterbox")
    lo, hi, nz = _axis(w["src_h"], nh)
    rows = np.unique(np.concatenate([lo, hi[nz]]))
    lo, hi, nz = _axis(w["src_w"], nw)
    cols = np.unique(np.concatenate([lo, hi[nz]]))
    row_bytes = 3 * w["src_w"]
    col_bytes = (3 * cols[:, None] + np.arange(3)[None, :]).reshape(-1)
    src_sectors = 0
    for j in rows:                                   # rows start at j * row_bytes in a packed frame
        src_sectors += np.unique((j * row_bytes + col_bytes) // 32).size
    src = src_sectors * 32 * w["batch"]
    dst = w["batch"] * 3 * w["dst_w"] * w["dst_h"] * out_bytes
    topk = w["rows"] * w["cols"] * 4 + w["rows"] * w["k"] * 8
    full = w["batch"] * 3 * w["src_w"] * w["src_h"] + dst     # every source byte read: a sanity bound
    return {"preprocess": int(src + dst), "source": int(src), "tensor": int(dst), "topk": int(topk),
            "total": int(src + dst + topk), "full_frame_preprocess": int(full)}


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during timed regions."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if self.gpu_id:
            cmd += ["--id=" + self.gpu_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def pump():
            for line in self.proc.stdout:
                self.lines.append(line.strip())
        self.thread = threading.Thread(target=pump, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def stop(self) -> dict | None:
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- distributed

def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a per-rank number over the job (identity on one process)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, seconds_per_rank: float, world: int, device=None) -> tuple[float, float]:
    """Units of all ranks divided by the slowest rank's time."""
    t = max_over_ranks(seconds_per_rank, world, device)
    return units_per_rank * world / t, t


# ----------------------------------------------------------------- oracle baseline

def host_cpu() -> str:
    """The host CPU as /proc/cpuinfo names it (x86: model name; Arm: the
    implementer and part codes), or the platform string."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                fields.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if fields.get("model name"):
        return fields["model name"]
    if fields.get("CPU implementer"):
        return f"{platform.machine()} implementer {fields['CPU implementer']} part {fields.get('CPU part', '?')}"
    return platform.processor() or platform.machine()


def cpu_baseline(w: dict, frames: np.ndarray, logits: np.ndarray, budget_s: float = 10.0) -> dict:
    """The oracle as it stands, single-threaded, repeated over a bounded sample."""
    import oracle as oracle_pkg
    o = oracle_pkg.Oracle()
    n_frames = 2
    lb = w["resize"] == "letterbox"
    done, t0 = 0, time.perf_counter()
    while True:
        for b in range(0, frames.shape[0], n_frames):
            o.preprocess(frames[b:b + n_frames], w["src_w"], w["src_h"], w["dst_w"], w["dst_h"],
                         letterbox=lb, norm=w["norm"])
            o.topk(logits[b:b + n_frames], w["k"])
            done += n_frames
            if time.perf_counter() - t0 >= budget_s:
                break
        if time.perf_counter() - t0 >= budget_s:
            break
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "frames/s", "cores": 1, "kind": "oracle", "cpu_model": host_cpu(),
            "sample": f"{done} frames of the workload (preprocess of the frame + Top-{w['k']} of its "
                      f"{w['cols']}-logit row), single-threaded C++ oracle, {dt:.1f} s"}


def cpu_baseline_all_cores(w: dict, frames: np.ndarray, logits: np.ndarray, budget_s: float = 5.0) -> dict:
    """The same oracle on every host core: one Python thread per core, each
    looping over frames (the oracle's C calls release the interpreter lock)."""
    import oracle as oracle_pkg
    o = oracle_pkg.Oracle()
    lb = w["resize"] == "letterbox"
    cores = os.cpu_count() or 1
    counts = [0] * cores
    deadline = time.perf_counter() + budget_s

    def work(tid):
        b = tid % frames.shape[0]
        while time.perf_counter() < deadline:
            o.preprocess(frames[b:b + 1], w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], letterbox=lb,
                         norm=w["norm"])
            o.topk(logits[b:b + 1], w["k"])
            counts[tid] += 1
            b = (b + cores) % frames.shape[0]

    t0 = time.perf_counter()
    threads = [threading.Thread(target=work, args=(i,)) for i in range(cores)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    dt = time.perf_counter() - t0
    done = sum(counts)
    return {"value": done / dt, "unit": "frames/s", "cores": cores, "kind": "oracle", "cpu_model": host_cpu(),
            "sample": f"{done} frames on {cores} threads (one per host core), {dt:.1f} s"}


def run_reference(args, w: dict) -> None:
    """--impl reference: the oracle timed on the host cores, one frame per step."""
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    import oracle as oracle_pkg
    o = oracle_pkg.Oracle()
    frames = synth.make_frames(args.workload, batch=1)
    logits = synth.make_logits(args.workload, rows=1)
    lb = w["resize"] == "letterbox"

    def step():
        o.preprocess(frames, w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], letterbox=lb, norm=w["norm"])
        o.topk(logits, w["k"])

    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    dt = time.perf_counter() - t0
    value = args.steps / dt
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic", "config": workload_config(args.workload, w),
        "cpu_baseline": {"value": value, "unit": "frames/s", "cores": 1, "kind": "oracle", "cpu_model": host_cpu(),
                         "sample": "one frame of the workload per step (its preprocess + the Top-K of its "
                                   "logit row), single-threaded C++ oracle"},
        "e2e": {"value": value, "unit": "frames/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


DETECT_BATCH = 64
DETECT_SEED = 0x57A70D00


def detect_measurements(B, Lane, device, stream, samples: int) -> dict:
    """Detection decode + NMS (the next-row extension of the hot path).

    Workload: a YOLO-style head for a 640x640 input (strides 8/16/32, 8400
    anchors, reg_max 16, 80 classes), DFL logits N(0, 2) and class logits
    N(-8, 2) -- about 2 % of the anchors clear conf 0.25; IoU 0.45,
    max_cand 1024, max_det 300.  Batch 64 for throughput and the decode
    roofline (two heads alternate, 620 MB > L2), batch 1 through a detection
    lane (720p letterbox -> 640 preprocess, decode, NMS) for latency."""
    import torch
    desc = B.detect_desc()
    st, A = B.ws_detect_validate(desc, DETECT_BATCH)
    B.check(st)
    t0 = time.perf_counter()
    head = synth.yolo_head(DETECT_SEED, DETECT_BATCH)
    heads = [torch.from_numpy(head).to(device), torch.from_numpy(head[::-1].copy()).to(device)]
    log(f"[bench] detection heads generated in {time.perf_counter() - t0:.1f} s")
    st, nws = B.ws_detect_workspace_bytes(desc, DETECT_BATCH)
    B.check(st)
    ws = torch.zeros(nws + 256, dtype=torch.uint8, device=device)
    wp = ws.data_ptr() + (-ws.data_ptr()) % 256
    out = torch.zeros((DETECT_BATCH, desc.max_det, 8), dtype=torch.int32, device=device)
    oc = torch.zeros(DETECT_BATCH, dtype=torch.int32, device=device)
    cand = torch.zeros((DETECT_BATCH, A, 8), dtype=torch.int32, device=device)
    cnt = torch.zeros(DETECT_BATCH, dtype=torch.int32, device=device)
    s = stream.cuda_stream

    def full(i):
        B.check(B.ws_detect(desc, heads[i % 2].data_ptr(), DETECT_BATCH, out.data_ptr(), oc.data_ptr(), wp, nws, s))

    def timed(fn, n):
        for i in range(8):
            fn(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / n

    n = 500
    detect_us = timed(full, n)
    # the decode kernel alone, each launch between its own events; the NMS
    # (which resets the counters) follows outside them
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    for i in range(8):
        B.check(B.ws_detect_decode(desc, heads[i % 2].data_ptr(), DETECT_BATCH, cand.data_ptr(), cnt.data_ptr(), s))
        B.check(B.ws_detect_nms(desc, cand.data_ptr(), cnt.data_ptr(), DETECT_BATCH, out.data_ptr(), oc.data_ptr(), s))
    torch.cuda.synchronize()
    for i, (a, b) in enumerate(evs):
        a.record(stream)
        B.check(B.ws_detect_decode(desc, heads[i % 2].data_ptr(), DETECT_BATCH, cand.data_ptr(), cnt.data_ptr(), s))
        b.record(stream)
        B.check(B.ws_detect_nms(desc, cand.data_ptr(), cnt.data_ptr(), DETECT_BATCH, out.data_ptr(), oc.data_ptr(), s))
    torch.cuda.synchronize()
    decode_us = statistics.mean(a.elapsed_time(b) * 1000.0 for a, b in evs)

    def decode_mean():
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(evs):
            a.record(stream)
            B.check(B.ws_detect_decode(desc, heads[i % 2].data_ptr(), DETECT_BATCH, cand.data_ptr(), cnt.data_ptr(), s))
            b.record(stream)
            B.check(B.ws_detect_nms(desc, cand.data_ptr(), cnt.data_ptr(), DETECT_BATCH, out.data_ptr(), oc.data_ptr(), s))
        torch.cuda.synchronize()
        return statistics.mean(a.elapsed_time(b) * 1000.0 for a, b in evs)

    # Deployment option: the context's L2 fetch granularity at 32 bytes makes
    # each isolated 4-byte DFL read fetch one sector instead of two.  The
    # library never sets this context-wide limit; it is set here for this one
    # measurement and put back.
    decode_us_fetch32 = None
    rt = _cudart()
    if rt is not None:
        prev = ctypes.c_size_t(0)
        if rt.cudaDeviceGetLimit(ctypes.byref(prev), CUDA_LIMIT_MAX_L2_FETCH_GRANULARITY) == 0:
            if rt.cudaDeviceSetLimit(CUDA_LIMIT_MAX_L2_FETCH_GRANULARITY, ctypes.c_size_t(32)) == 0:
                decode_us_fetch32 = decode_mean()
            rt.cudaDeviceSetLimit(CUDA_LIMIT_MAX_L2_FETCH_GRANULARITY, prev)
    # candidate count of the timed heads (decode once more, read the counters)
    with torch.cuda.stream(stream):
        B.check(B.ws_detect_decode(desc, heads[0].data_ptr(), DETECT_BATCH, cand.data_ptr(), cnt.data_ptr(), s))
        stream.synchronize()
        n_cand = int(cnt.sum())
        B.check(B.ws_detect_nms(desc, cand.data_ptr(), cnt.data_ptr(), DETECT_BATCH, out.data_ptr(), oc.data_ptr(), s))
        stream.synchronize()
    kept = int(oc.sum())
    R, C = desc.reg_max, desc.num_classes
    # class logits once, each candidate's 4 R DFL logits as the 32-byte
    # sectors they sit in (A-strided rows: one sector each), its 32-byte record
    alg_decode = DETECT_BATCH * C * A * 4 + n_cand * (4 * R * 32 + 32) + DETECT_BATCH * 4

    # Worst case: every anchor a candidate.  The same heads with the class
    # logits moved up by 13 (N(5, 2)): 8400 candidates an image, capped at
    # max_cand 1024 by the NMS's selection, 300 kept.
    shifted = head.copy()
    shifted[:, 4 * desc.reg_max:] += 13.0
    worst = {}
    for nb in (1, DETECT_BATCH):
        hw = torch.from_numpy(shifted[:nb].copy()).to(device)
        B.check(B.ws_detect_workspace_init(wp, nws, s))

        def worst_call(i, hw=hw, nb=nb):
            B.check(B.ws_detect(desc, hw.data_ptr(), nb, out.data_ptr(), oc.data_ptr(), wp, nws, s))

        worst[f"batch{nb}_us"] = timed(worst_call, 200)
        torch.cuda.synchronize()
        worst[f"batch{nb}_kept_per_image"] = int(oc[:nb].sum()) / nb
    del shifted

    # batch-1 latency through a detection lane
    pre = B.preprocess_desc(1280, 720, 640, 640, letterbox=True, norm="scale")
    frame = torch.from_numpy(synth.frames_uniform(DETECT_SEED, 1, 720, 1280)).to(device)
    head1 = torch.from_numpy(head[:1].copy()).to(device)
    lat = {}
    warm = min(200, samples)
    for label, flags in (("graph", 0), ("graph_no_timing", B.WS_LANE_FLAG_NO_TIMING)):
        d = B.lane_desc(pre, 1, 0, 0, 0, input=frame.data_ptr(), logits=head1.data_ptr(), detect=desc, flags=flags)
        with Lane(d) as lane:
            gpu, host = [], []
            for i in range(warm + samples):
                lane.acquire()
                lane.submit()
                t = lane.wait()
                if i >= warm:
                    gpu.append(t.gpu_us)
                    host.append(t.host_us)
            lat[label] = {"host_us": percentiles(host)}
            if not flags & B.WS_LANE_FLAG_NO_TIMING:
                lat[label]["gpu_us"] = percentiles(gpu)
    return {
        "workload": "YOLO-style head 640x640 (8400 anchors, reg_max 16, 80 classes), conf 0.25, IoU 0.45, "
                    "max_cand 1024, max_det 300; synthetic head DFL N(0,2), class N(-8,2)",
        "batch": DETECT_BATCH,
        "images_per_s": DETECT_BATCH / (detect_us * 1e-6),
        "detect_us": detect_us,
        "decode_us": decode_us,
        "nms_us_by_difference": detect_us - decode_us,
        "candidates_per_image": n_cand / DETECT_BATCH,
        "kept_per_image": kept / DETECT_BATCH,
        "all_candidates": dict(workload="the same heads with class logits + 13 (N(5,2)): every anchor a candidate, "
                                        "8400 -> max_cand 1024 -> 300 kept; ws_detect back to back", **worst),
        "decode_roofline": {"bound": "hbm", "kernels": "class scan + DFL boxes in one kernel (ws_detect_decode)",
                            "algorithmic_bytes_per_launch": alg_decode,
                            "bytes_rule": "class plane + 32-byte sector per DFL logit of each candidate + "
                                          "32-byte candidate record",
                            "achieved_gbs": alg_decode / (decode_us * 1e-6) / 1e9},
        "decode_l2_fetch_32": None if decode_us_fetch32 is None else {
            "decode_us": decode_us_fetch32, "achieved_gbs": alg_decode / (decode_us_fetch32 * 1e-6) / 1e9,
            "setting": "cudaLimitMaxL2FetchGranularity = 32 bytes for this measurement only (a context-wide "
                       "limit the library does not set)"},
        "latency_b1_lane": dict(lat, samples=samples, warmup=warm,
                                path="720p letterbox -> 640 preprocess, decode, NMS in one lane graph"),
    }


def lane_measurements(B, Lane, device, samples: int) -> dict:
    """Graph variants and the lane pool on the batch-1 1080p -> 224 + Top-5
    workload: the cost of re-binding a lane's producer slot (cudaGraphExecUpdate
    instead of re-instantiation), a 1-frame submit on a bucketed 64-frame lane,
    and frames/s through a pool of 1, 2 and 4 lanes, each on its own stream."""
    import torch
    lw = synth.WORKLOADS[LATENCY_WORKLOAD]
    frames = torch.from_numpy(synth.make_frames(LATENCY_WORKLOAD)).to(device)
    frames2 = frames.clone()
    logits = torch.from_numpy(synth.make_logits(LATENCY_WORKLOAD)).to(device)
    pre = B.preprocess_desc(lw["src_w"], lw["src_h"], lw["dst_w"], lw["dst_h"], norm=lw["norm"])
    out = {"workload": LATENCY_WORKLOAD}
    d = B.lane_desc(pre, 1, 1, lw["cols"], lw["k"], input=frames.data_ptr(), logits=logits.data_ptr())
    with Lane(d) as lane:
        times, reinst = [], 0
        for i in range(200):
            t0 = time.perf_counter()
            reinst += lane.rebind(input=(frames2 if i % 2 else frames).data_ptr())
            times.append((time.perf_counter() - t0) * 1e6)
            lane.acquire(); lane.submit(); lane.wait()
        out["rebind_host_us"] = percentiles(times[10:])
        out["rebind_reinstantiated"] = reinst
    # a 64-frame bucketed lane replaying its 1-frame bucket
    w64 = synth.WORKLOADS[DEFAULT_WORKLOAD]
    src64 = torch.zeros((64, lw["src_h"], 3 * lw["src_w"]), dtype=torch.uint8, device=device)
    src64[0].copy_(frames[0])
    lg64 = torch.from_numpy(synth.logits_normal(0x57A7D64, 64, lw["cols"])).to(device)
    d = B.lane_desc(pre, 64, 64, lw["cols"], w64["k"], input=src64.data_ptr(), logits=lg64.data_ptr(),
                    flags=B.WS_LANE_FLAG_BUCKETS)
    with Lane(d) as lane:
        for n in (1, 64):
            gpu = []
            for i in range(min(samples, 1000) + 50):
                lane.acquire(); lane.submit(n); t = lane.wait()
                if i >= 50:
                    gpu.append(t.gpu_us)
            out[f"bucketed_b64_lane_submit_n{n}_gpu_us"] = percentiles(gpu)
    # lane pool: batch-1 jobs, producer and consumer on this thread
    d = B.lane_desc(pre, 1, 1, lw["cols"], lw["k"], flags=B.WS_LANE_FLAG_NO_TIMING)
    pool = {}
    for nl in (1, 2, 4):
        st, P = B.ws_pool_create(d, nl)
        B.check(st)
        try:
            jobs = max(400, min(2 * samples, 8000))

            def run(n):
                # bursts: every lane submitted (each on its own stream), then
                # all completed, so the lanes' graphs can overlap on the GPU
                done = 0
                while done < n:
                    burst = []
                    for _ in range(nl):
                        st, L = B.ws_pool_acquire(P, 0)
                        B.check(st)
                        B.check(B.ws_pool_submit(P, L, 1))
                        burst.append(L)
                    for _ in burst:
                        st, L, _ = B.ws_pool_complete(P, -1)
                        B.check(st)
                        B.check(B.ws_pool_recycle(P, L))
                    done += nl

            run(100)
            t0 = time.perf_counter()
            run(jobs)
            dt = time.perf_counter() - t0
            pool[f"lanes_{nl}"] = {"frames_per_s": (jobs // nl * nl) / dt, "jobs": jobs // nl * nl}
        finally:
            B.check(B.ws_pool_destroy(P))
    out["pool_b1"] = pool
    return out


def workload_config(name: str, w: dict) -> dict:
    return {"workload": f"{w['batch']}x {w['src_w']}x{w['src_h']} RGB8 -> "
                        f"{'letterbox ' if w['resize'] == 'letterbox' else ''}{w['dst_w']}x{w['dst_h']} "
                        f"{'mean/std' if w['norm'] == 'mean_std' else '1/255'} FP32 NCHW + exact Top-{w['k']} "
                        f"of [{w['rows']},{w['cols']}] FP32 logits",
            "name": name, "batch": w["batch"], "k": w["k"], "rows": w["rows"], "cols": w["cols"]}


# ----------------------------------------------------------------- GPU arm

def percentiles(xs):
    a = np.sort(np.asarray(xs, dtype=np.float64))
    return {"p50": float(np.percentile(a, 50)), "p99": float(np.percentile(a, 99)), "max": float(a[-1]),
            "mean": float(a.mean())}


def preprocess_kernel_name(w: dict) -> str:
    """The kernel ws_preprocess launches for a workload: outputs of at most
    460,000 pixels (batch x dst_w x dst_h) take the per-pixel kernel, larger
    ones (dst_w at most 8192) the staged ring kernel."""
    small = w["batch"] * w["dst_w"] * w["dst_h"] <= 460_000
    return "pre_direct_kernel" if small or w["dst_w"] > 8192 else "pre_ring_kernel"


ROOFLINE_LAUNCHES = 1000


def kernel_times(B, torch, stream, pre, w: dict, bufs, n: int, device) -> tuple[float, float]:
    """Average launch time (us) of the preprocess and of the Top-K over n
    back-to-back launches each, through the C ABI on `stream`, rotating over
    the lanes' buffers; CUDA events on that stream around the n launches."""
    st_ws = [B.ws_topk_workspace_bytes(w["rows"], w["cols"], w["k"])[1] for _ in bufs]
    topk_ws = [torch.zeros(max(m, 1), dtype=torch.uint8, device=device) for m in st_ws]

    def time_kernel(launch):
        for i in range(8):
            launch(i)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for i in range(n):
            launch(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1000.0 / n

    def launch_pre(i):
        b = bufs[i % len(bufs)]
        B.check(B.ws_preprocess(pre, b.input_device, w["batch"], b.tensor, stream.cuda_stream))

    def launch_topk(i):
        b, ws_t, m = bufs[i % len(bufs)], topk_ws[i % len(bufs)], st_ws[i % len(bufs)]
        B.check(B.ws_topk(b.logits, w["rows"], w["cols"], w["k"], b.result_val_device, b.result_idx_device,
                          ws_t.data_ptr() if m else None, m, stream.cuda_stream))

    return time_kernel(launch_pre), time_kernel(launch_topk)


def make_lanes(B, Lane, torch, w: dict, pre, frames_dev, logits_dev, n_lanes: int, stream):
    """n_lanes throughput lanes without timing events, each with its own copy
    of the inputs: on their own streams (stream None) or sharing `stream`."""
    lanes, keep = [], []
    for _ in range(n_lanes):
        src = frames_dev.clone()
        lg = logits_dev.clone()
        keep += [src, lg]
        d = B.lane_desc(pre, w["batch"], w["rows"], w["cols"], w["k"], input=src.data_ptr(), logits=lg.data_ptr(),
                        stream=stream, flags=B.WS_LANE_FLAG_NO_TIMING)
        lanes.append(Lane(d))
    return lanes, keep


def run_steps(B, ls, n):
    """Round-robin submits over lanes `ls`; returns the lanes still in flight."""
    inflight = []
    for s_ in range(n):
        lane = ls[s_ % len(ls)]
        if lane.state == B.WS_LANE_IN_FLIGHT:
            lane.wait()
            inflight.remove(lane)
        lane.acquire()
        lane.submit()
        inflight.append(lane)
    return inflight


HOLD_CYCLES = 400_000   # about 0.2 ms of SM clock cycles


def timed_steps(B, torch, stream, ls, n):
    """Device time (s) of n steps: a start event on `stream`, which every lane
    stream waits on, and an end event after `stream` has waited on every lane
    stream's last work.  A short spin kernel on `stream` ahead of the start
    event holds the GPU while the host makes its first submissions, so that
    the interval is the GPU running the n steps rather than the host's
    latency to its first launch (every step's work is inside the interval)."""
    lane_streams = [torch.cuda.ExternalStream(lane.buffers.stream) for lane in ls]
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(HOLD_CYCLES)
    ev0.record(stream)
    for ls_ in lane_streams:
        ls_.wait_event(ev0)
    inflight = run_steps(B, ls, n)
    for ls_ in lane_streams:
        e = torch.cuda.Event()
        e.record(ls_)
        stream.wait_event(e)
    ev1.record(stream)
    for lane in inflight:
        lane.wait()
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1) / 1000.0


C5_WORKLOAD = "b8_4k_to_512"


def c5_record(B, Lane, torch, device, stream, peak: float, steps: int = 400) -> dict:
    """The second batched configuration (8 x 4K -> 512 + Top-32 of
    [32,131072] with 5 % ties): frames/s with four lanes on their own streams
    and with the same lanes' steps serialised on one stream, the step's
    algorithmic bytes per second, each kernel's average launch time and the
    roofline fraction of both against the measured copy bandwidth."""
    w = synth.WORKLOADS[C5_WORKLOAD]
    frames_dev = torch.from_numpy(synth.make_frames(C5_WORKLOAD)).to(device)
    logits_dev = torch.from_numpy(synth.make_logits(C5_WORKLOAD)).to(device)
    pre = B.preprocess_desc(w["src_w"], w["src_h"], w["dst_w"], w["dst_h"], norm=w["norm"])
    alg = algorithmic_bytes(w)
    own, keep = make_lanes(B, Lane, torch, w, pre, frames_dev, logits_dev, LANES, None)
    one, keep1 = make_lanes(B, Lane, torch, w, pre, frames_dev, logits_dev, LANES, stream.cuda_stream)
    try:
        for ls in (own, one):
            for lane in run_steps(B, ls, 20):
                lane.wait()
        t_own = timed_steps(B, torch, stream, own, steps)
        t_one = timed_steps(B, torch, stream, one, steps)
        pre_us, topk_us = kernel_times(B, torch, stream, pre, w, [lane.buffers for lane in one], ROOFLINE_LAUNCHES,
                                       device)
    finally:
        for lane in own + one:
            lane.close()
    step_own, step_one = t_own / steps, t_one / steps
    return {
        "workload": C5_WORKLOAD, "steps": steps,
        "frames_per_s": w["batch"] / step_own, "us_per_step": 1e6 * step_own,
        "step_frac": alg["total"] / step_own / 1e9 / peak,
        "one_stream_frames_per_s": w["batch"] / step_one, "one_stream_us_per_step": 1e6 * step_one,
        "one_stream_step_frac": alg["total"] / step_one / 1e9 / peak,
        "preprocess_us": pre_us, "preprocess_frac": alg["preprocess"] / (pre_us * 1e-6) / 1e9 / peak,
        "topk_us": topk_us, "topk_frac": alg["topk"] / (topk_us * 1e-6) / 1e9 / peak,
        "algorithmic_bytes_per_step": alg["total"], "peak_gbs": peak,
        "lanes": f"{LANES} lanes on their own streams; one_stream: {LANES} lanes sharing one stream",
    }


def latency_summary(latency: dict, other: dict) -> dict:
    """p50 / p99 (us) of each batch-1 configuration, compact: GPU interval
    and host clock of the timed graph replay, host clock of the graph replay
    without timing events, GPU interval and host clock of direct launches."""
    out = {}
    for rec in [latency] + list(other.values()):
        name = next(n for n, v in synth.WORKLOADS.items() if workload_config(n, v)["workload"] == rec["workload"])

        def pp(d):
            return [round(d["p50"], 2), round(d["p99"], 2)]
        out[name] = {"graph_gpu": pp(rec["graph"]["gpu_us"]), "graph_host": pp(rec["graph"]["host_us"]),
                     "graph_no_timing_host": pp(rec["graph_no_timing"]["host_us"]),
                     "no_graph_gpu": pp(rec["no_graph"]["gpu_us"]), "no_graph_host": pp(rec["no_graph"]["host_us"])}
    out["replay_floor_gpu"] = [round(latency["graph_floor"]["gpu_us"]["p50"], 2),
                               round(latency["graph_floor"]["gpu_us"]["p99"], 2)]
    out["fields"] = "[p50, p99] us; samples per entry as in latency_b1"
    return out


def source_sha(path: str) -> str:
    return hashlib.sha256(open(path, "rb").read()).hexdigest()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(synth.WORKLOADS))
    ap.add_argument("--latency-samples", type=int, default=10000)
    ap.add_argument("--e2e-steps", type=int, default=60)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-detect", action="store_true", help="skip the detection decode + NMS measurements")
    ap.add_argument("--no-c5", action="store_true", help="skip the compact 8 x 4K -> 512 record")
    ap.add_argument("--out-dtype", default="f32", choices=["f32", "f16", "bf16"],
                    help="element type of the NCHW tensor (the workloads specify FP32)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = synth.WORKLOADS[args.workload]

    if args.impl == "reference":
        run_reference(args, w)
        return

    import torch
    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    if world > 1:
        torch.distributed.barrier()
    __graft_entry__.build()
    from post_processing_gb300 import Lane
    from post_processing_gb300 import binding as B

    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20)
    try:
        gpu_id = "GPU-" + str(props.uuid)
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)

    # inputs: one seeded batch, copied into every lane's fixed buffers
    t0 = time.perf_counter()
    frames = synth.make_frames(args.workload)
    logits = synth.make_logits(args.workload)
    log(f"[bench] inputs generated in {time.perf_counter() - t0:.1f} s")
    frames_dev = torch.from_numpy(frames).to(device)
    logits_dev = torch.from_numpy(logits).to(device)

    stream = torch.cuda.Stream(device)
    dst_type = {"f32": B.WS_DTYPE_F32, "f16": B.WS_DTYPE_F16, "bf16": B.WS_DTYPE_BF16}[args.out_dtype]
    out_bytes = 4 if args.out_dtype == "f32" else 2
    pre = B.preprocess_desc(w["src_w"], w["src_h"], w["dst_w"], w["dst_h"],
                            letterbox=w["resize"] == "letterbox", norm=w["norm"], dst_type=dst_type)
    # Two sets of throughput lanes, only a completion event per submit (no
    # timing pair): each lane of the first set on its own stream, as lanes run
    # in a deployment (a lane's preprocess overlaps the previous lane's Top-K;
    # within a lane the order copy-in -> preprocess -> Top-K is unchanged) --
    # the headline; the second set sharing one stream, every step serialised
    # behind the previous one.
    # Enough lanes that one rotation touches about three times the L2, and at
    # least four: while the host waits for a lane and submits it again, three
    # others keep the GPU busy (on the 4K workload a third lane left gaps:
    # 24.2 us per step with three lanes, 21.5 with four or six; the 64-frame
    # step is 28.5 us with three, four or six).
    alg = algorithmic_bytes(w, out_bytes)
    n_lanes = max(LANES, min(MAX_LANES, -(-3 * l2 // max(1, int(alg["total"])))))
    lanes, keep = make_lanes(B, Lane, torch, w, pre, frames_dev, logits_dev, n_lanes, None)
    lanes_1s, keep1 = make_lanes(B, Lane, torch, w, pre, frames_dev, logits_dev, n_lanes, stream.cuda_stream)
    torch.cuda.synchronize()
    touched_per_rotation = n_lanes * alg["total"]

    for ls in (lanes, lanes_1s):
        for lane in run_steps(B, ls, args.warmup):
            lane.wait()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks.start()
    elapsed_s = timed_steps(B, torch, stream, lanes, args.steps)
    elapsed_1s = timed_steps(B, torch, stream, lanes_1s, args.steps)
    if world > 1:
        torch.distributed.barrier()

    # Per-kernel durations for the roofline: the same kernels on the same
    # stream and the lanes' own buffers (rotating, so inputs stay larger than
    # L2), launched back to back through the C ABI and bracketed by CUDA
    # events, right after the timed region; a fixed number of launches,
    # whatever --steps is.
    kernel_launches = ROOFLINE_LAUNCHES
    pre_avg_us, topk_avg_us = kernel_times(B, torch, stream, pre, w, [lane.buffers for lane in lanes_1s],
                                           kernel_launches, device)

    # batch-1 latency: one lane, submit -> wait, graph and direct launches.
    # "graph": the page's measurement, timing events just before the graph
    # launch and after the Top-K (GPU interval) plus the host steady clock;
    # "graph_no_timing": the same replay with only a completion event (host
    # clock); "no_graph": direct launches with the timing events;
    # "graph_no_pdl": the graph with the Top-K as an ordinary launch instead
    # of a programmatic dependent launch (what PDL saves).
    def latency_of(name, samples):
        lw = synth.WORKLOADS[name]
        lframes = torch.from_numpy(synth.make_frames(name)).to(device)
        llogits = torch.from_numpy(synth.make_logits(name)).to(device)
        lpre = B.preprocess_desc(lw["src_w"], lw["src_h"], lw["dst_w"], lw["dst_h"],
                                 letterbox=lw["resize"] == "letterbox", norm=lw["norm"])
        out = {"workload": workload_config(name, lw)["workload"], "samples": samples,
               "warmup": min(1000, samples), "input": "device-resident"}
        for label, flags in (("graph", 0), ("graph_no_timing", B.WS_LANE_FLAG_NO_TIMING),
                             ("no_graph", B.WS_LANE_FLAG_NO_GRAPH), ("graph_no_pdl", B.WS_LANE_FLAG_NO_PDL)):
            d = B.lane_desc(lpre, 1, lw["rows"], lw["cols"], lw["k"], input=lframes.data_ptr(),
                            logits=llogits.data_ptr(), flags=flags)
            with Lane(d) as lane:
                gpu, host = [], []
                for i in range(out["warmup"] + samples):
                    lane.acquire()
                    lane.submit()
                    t = lane.wait()
                    if i >= out["warmup"]:
                        gpu.append(t.gpu_us)
                        host.append(t.host_us)
                out[label] = {"host_us": percentiles(host)}
                if flags & B.WS_LANE_FLAG_NO_TIMING == 0:
                    out[label]["gpu_us"] = percentiles(gpu)
        return out

    latency = latency_of(LATENCY_WORKLOAD, args.latency_samples)

    # The fixed cost of a replay: the same two timing events around a graph
    # that holds one 1-element fill kernel (no work of this library).
    def graph_floor(samples):
        fs = torch.cuda.Stream()
        buf = torch.zeros(1, device=device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(fs):
            buf.fill_(1.0)
            fs.synchronize()
            with torch.cuda.graph(g, stream=fs):
                buf.fill_(2.0)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            vals = []
            warm = min(1000, samples)
            for i in range(warm + samples):
                e0.record(fs)
                g.replay()
                e1.record(fs)
                e1.synchronize()
                if i >= warm:
                    vals.append(e0.elapsed_time(e1) * 1000.0)
        return percentiles(vals)

    latency["graph_floor"] = {"gpu_us": graph_floor(args.latency_samples),
                              "what": "the same timing events around a graph holding one 1-element fill kernel"}
    # the other two batch-1 configurations: 224x224 identity + Top-5 of 1000,
    # and 1280x720 letterboxed to 640x640 + Top-32 of one 672,000-entry row
    latency_other = {name: latency_of(name, args.latency_samples)
                     for name in ("b1_224_identity", "b1_720p_letterbox_640")}
    detect = None
    if not args.no_detect:
        detect = detect_measurements(B, Lane, device, stream, min(2000, args.latency_samples))
    lanes_extra = lane_measurements(B, Lane, device, args.latency_samples)
    peaks_path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(peaks_path):
        peak, peak_src = float(json.load(open(peaks_path))["hbm_gbs"]), "measured"
    else:
        peak, peak_src = FALLBACK_HBM_GBS, "fallback"
    c5 = None if args.no_c5 else c5_record(B, Lane, torch, device, stream, peak)
    clk = clocks.stop()

    # End to end through the lane API with host buffers, two lanes each on its
    # own stream, host clock.  "e2e": the producer writes the frames into the
    # lane's mapped pinned input slot, the preprocess reads the rows it needs
    # in place across the host link, and the Top-K writes the K pairs straight
    # into mapped pinned host memory (the producer / result path of the
    # WarpStream write-up).  "e2e_copy_in": the other input topology the page
    # says to measure -- the graph first copies the whole frames from pinned
    # host memory into a fixed device slot, and copies the K pairs back.
    def end_to_end(input_mode, result_mode):
        import ctypes
        e_lanes = []
        for _ in range(2):
            d = B.lane_desc(pre, w["batch"], w["rows"], w["cols"], w["k"], input_mode=input_mode,
                            result_mode=result_mode, logits=logits_dev.data_ptr(), flags=B.WS_LANE_FLAG_NO_TIMING)
            lane = Lane(d)
            buf = (ctypes.c_char * frames.nbytes).from_address(lane.buffers.input_host)
            np.frombuffer(buf, dtype=np.uint8)[:] = frames.reshape(-1)
            e_lanes.append(lane)
        for lane in e_lanes:
            lane.acquire(); lane.submit(); lane.wait()
        torch.cuda.synchronize()
        if world > 1:
            torch.distributed.barrier()
        t0 = time.perf_counter()
        for s_ in range(args.e2e_steps):
            lane = e_lanes[s_ % 2]
            if lane.state == B.WS_LANE_IN_FLIGHT:
                lane.wait()
            lane.acquire()
            lane.submit()
        for lane in e_lanes:
            if lane.state == B.WS_LANE_IN_FLIGHT:
                lane.wait()
        e_dt = time.perf_counter() - t0
        for lane in e_lanes:
            lane.close()
        rate, _ = whole_job_rate(w["batch"] * args.e2e_steps, e_dt, world, device)
        return rate, e_dt

    e2e = e2e_copy = None
    if args.e2e_steps > 0:
        rate, dt = end_to_end(B.WS_INPUT_MAPPED, B.WS_RESULT_MAPPED)
        e2e = {"value": rate, "unit": "frames/s", "h2d_bytes_per_step": int(alg["source"]),
               "d2h_bytes_per_step": int(w["rows"] * w["k"] * 8),
               "path": "ws_lane_submit/wait on host buffers: input_mode=MAPPED (frames written by the host "
                       "into mapped pinned memory; the kernel reads the needed rows, h2d_bytes_per_step, "
                       "in place), result_mode=MAPPED (the K pairs written into pinned host memory); "
                       "2 lanes on their own streams; host clock",
               "frames_bytes_per_step": int(frames.nbytes),
               "link_gbs": alg["source"] * args.e2e_steps / dt / 1e9}
        rate, dt = end_to_end(B.WS_INPUT_COPY, B.WS_RESULT_COPY)
        e2e_copy = {"value": rate, "unit": "frames/s", "h2d_bytes_per_step": int(frames.nbytes),
                    "d2h_bytes_per_step": int(w["rows"] * w["k"] * 8),
                    "path": "input_mode=COPY (cudaMemcpyAsync of the whole frames into a fixed device slot "
                            "inside the graph), result_mode=COPY; 2 lanes on their own streams; host clock",
                    "link_gbs": frames.nbytes * args.e2e_steps / dt / 1e9}

    for lane in lanes + lanes_1s:
        lane.close()

    value, t_max = whole_job_rate(w["batch"] * args.steps, elapsed_s, world, device)
    value_1s, t_max_1s = whole_job_rate(w["batch"] * args.steps, elapsed_1s, world, device)
    achieved = alg["preprocess"] / (pre_avg_us * 1e-6) / 1e9
    sha = source_sha(os.path.join(ROOT, "post_processing_gb300", "csrc", "preprocess.cu"))
    traffic = NCU_TRAFFIC.get(args.workload) if args.out_dtype == "f32" else None   # captured on FP32 output
    traffic = traffic["bytes"] if traffic and traffic.get("source_sha") == sha else None

    if rank == 0:
        cpu = cpu_all = None
        if not args.no_cpu_baseline:
            cpu = cpu_baseline(w, frames, logits)
            cpu_all = cpu_baseline_all_cores(w, frames, logits)
        line = {
            "metric": METRIC, "value": value, "unit": "frames/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000.0 * t_max / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": dict(workload_config(args.workload, w), out_dtype=args.out_dtype,
                           l2=f"{n_lanes} lanes rotate, {touched_per_rotation / 1e6:.0f} MB touched per rotation "
                              f"({touched_per_rotation / l2:.1f}x the {l2 / 2 ** 20:.0f} MiB L2): inputs "
                              + ("larger than L2" if touched_per_rotation > l2 else
                                 "SMALLER than L2 (this workload's rate is L2-resident)"),
                           parallelism=f"replicas x{world}", graph=True,
                           lanes=f"{n_lanes} lanes, each on its own stream, replayed in rotation",
                           algorithmic_bytes_per_step=alg["total"]),
            "hbm_gbs_step": alg["total"] * args.steps * world / t_max / 1e9,
            "serialized_one_stream": {"value": value_1s, "ms_per_step": 1000.0 * t_max_1s / args.steps,
                                      "hbm_gbs_step": alg["total"] * args.steps * world / t_max_1s / 1e9,
                                      "lanes": f"{n_lanes} lanes sharing one stream: each step after the previous"},
            "roofline": {"bound": "hbm", "kernel": preprocess_kernel_name(w), "achieved": achieved, "peak": peak,
                         "unit": "GB/s", "frac": achieved / peak, "peak_source": peak_src,
                         "traffic": traffic, "algorithmic_bytes_per_launch": alg["preprocess"],
                         "full_frame_bytes_per_launch": alg["full_frame_preprocess"],
                         "avg_launch_us": pre_avg_us, "launches_timed": kernel_launches,
                         "timing": "CUDA events on the launching stream around back-to-back launches "
                                   "on the lanes' rotating buffers, after the timed region",
                         "topk_avg_launch_us": topk_avg_us,
                         "topk_gbs": alg["topk"] / (topk_avg_us * 1e-6) / 1e9},
            "latency_b1": latency,
            "latency_b1_other": latency_other,
            "detect": detect,
            "lanes": lanes_extra,
            "e2e": e2e,
            "e2e_copy_in": e2e_copy,
            "gpu_launches": 2 * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
        }
        # compact records last, so that a tail of the line shows them
        if c5 is not None:
            line["c5"] = {k_: (round(v_, 4) if isinstance(v_, float) else v_) for k_, v_ in c5.items()}
        line["latency_b1_summary"] = latency_summary(latency, latency_other)
        line["roofline"]["frac_note"] = "of measured" if peak_src == "measured" else "of fallback"
        if detect:
            r = detect["decode_roofline"]
            r.update(peak=peak, unit="GB/s", frac=r["achieved_gbs"] / peak,
                     frac_note="of measured" if peak_src == "measured" else "of fallback")
            if detect.get("decode_l2_fetch_32"):
                r32 = detect["decode_l2_fetch_32"]
                r32.update(frac=r32["achieved_gbs"] / peak)
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
