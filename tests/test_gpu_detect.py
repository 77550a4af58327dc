"""Detection decode + NMS on the GPU against the oracle.

Decode: the candidate set (anchors), classes and logits are exact (no
transcendental decides them); boxes agree within box_tol(), a bound derived
from the GPU's FP32 softmax against the oracle's double one.  NMS: given the same candidates
the kept list is exact -- the IoU test is FP32 with every operation rounded
separately on both sides.  End to end, ws_detect equals the oracle's NMS of
the candidates the GPU decoded.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from cudart import memcpy

pytestmark = pytest.mark.gpu


def box_tol(desc) -> float:
    """Bound on |GPU machine - oracle box| in pixels.  Per DFL side, in FP32 with
    u = 2**-24: each weight exp(z - m) is within (|z - m| + 4) u (the
    subtraction's rounding times |z - m| <= 20, expf's 2 ulp), weights below
    e**-20 aside; each of the two R-term sums adds R u; the product w i, the
    division and the multiply by the stride add 3 u.  So the distance, at most
    R - 1 bins, is within (R - 1)(2 R + 51) u bins, times the stride in
    pixels, plus the final rounding of coordinates below 1024 (2 ulp)."""
    u = 2.0 ** -24
    s = max(list(desc.strides)[:desc.nlevels])
    R = desc.reg_max
    return s * (R - 1) * (2 * R + 51) * u + 2 * 2.0 ** -13


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def stream():
    return torch.cuda.current_stream().cuda_stream


def unpack(rows):
    """ws_candidate / ws_detection rows (int32 view [n, 8]) to fields."""
    rows = np.ascontiguousarray(rows)
    return dict(boxes=rows[:, :4].view(np.float32), f4=rows[:, 4].view(np.float32), cls=rows[:, 5].copy(),
                anchor=rows[:, 6].copy())


def gpu_decode(B, desc, head):
    batch, _, A = head.shape
    h = torch.from_numpy(head).cuda()
    cand = torch.zeros((batch, A, 8), dtype=torch.int32, device="cuda")
    count = torch.zeros(batch, dtype=torch.int32, device="cuda")
    B.check(B.ws_detect_decode(desc, h.data_ptr(), batch, cand.data_ptr(), count.data_ptr(), stream()))
    torch.cuda.synchronize()
    c, n = cand.cpu().numpy(), count.cpu().numpy()
    out = []
    for b in range(batch):
        u = unpack(c[b, :n[b]])
        order = np.argsort(u["anchor"], kind="stable")
        out.append({k: v[order] for k, v in u.items()})
    return out


def gpu_nms(B, desc, cands):
    """cands: list per image of dicts (boxes, logits, classes, anchors), any order."""
    batch = len(cands)
    st, A = B.ws_detect_validate(desc, batch)      # the buffer is [batch][A], A the geometry's anchor count
    B.check(st)
    rows = np.zeros((batch, A, 8), np.int32)
    count = np.zeros(batch, np.int32)
    for b, c in enumerate(cands):
        n = len(c["anchors"])
        rows[b, :n, :4] = np.asarray(c["boxes"], np.float32).view(np.int32)
        rows[b, :n, 4] = np.asarray(c["logits"], np.float32).view(np.int32)
        rows[b, :n, 5] = c["classes"]
        rows[b, :n, 6] = c["anchors"]
        count[b] = n
    cand = torch.from_numpy(rows).cuda()
    cnt = torch.from_numpy(count).cuda()
    out = torch.zeros((batch, desc.max_det, 8), dtype=torch.int32, device="cuda")
    oc = torch.zeros(batch, dtype=torch.int32, device="cuda")
    B.check(B.ws_detect_nms(desc, cand.data_ptr(), cnt.data_ptr(), batch, out.data_ptr(), oc.data_ptr(), stream()))
    torch.cuda.synchronize()
    assert np.all(cnt.cpu().numpy() == 0), "candidate counters are reset for the next call"
    o, k = out.cpu().numpy(), oc.cpu().numpy()
    return [unpack(o[b, :k[b]]) for b in range(batch)]


def oracle_cands(oracle, desc, head_b):
    d = oracle.decode(head_b, desc.reg_max, desc.num_classes, desc.in_w, desc.in_h,
                      list(desc.strides)[:desc.nlevels], desc.logit_thr)
    return dict(boxes=d["boxes"], logits=d["logits"], classes=d["classes"], anchors=d["anchors"], total=d["total"])


def check_decode(B, oracle, desc, head):
    got = gpu_decode(B, desc, head)
    for b in range(head.shape[0]):
        want = oracle_cands(oracle, desc, head[b])
        g = got[b]
        assert np.array_equal(g["anchor"], want["anchors"]), b
        assert np.array_equal(g["cls"], want["classes"])
        assert np.array_equal(g["f4"].view(np.uint32), want["logits"].view(np.uint32))
        if len(g["anchor"]):
            assert float(np.max(np.abs(g["boxes"] - want["boxes"]))) <= box_tol(desc)
    return got


def test_decode_parity(B, oracle):
    desc = B.detect_desc()
    head = synth.yolo_head(21, 3)
    got = check_decode(B, oracle, desc, head)
    assert all(50 < len(g["anchor"]) < 1000 for g in got)      # a realistic candidate count


@pytest.mark.parametrize("batch", [16, 17])
def test_decode_split_and_whole_tile_kernels(B, oracle, batch):
    """Up to 1100 tiles in all, four warps split each 128-anchor tile's classes
    and merge; above, one warp scans a whole tile.  A 640x640 head has 66
    tiles: 16 heads take the first form, 17 the second."""
    desc = B.detect_desc()
    head = synth.yolo_head(31, batch)
    got = check_decode(B, oracle, desc, head)
    assert all(50 < len(g["anchor"]) < 1000 for g in got)


def test_decode_whole_tile_kernel_scalar(B, oracle):
    """One 15-anchor tile an image (scalar loads) for 1101 images: the
    whole-tile form's scalar scan."""
    desc = B.detect_desc(in_w=40, in_h=24, strides=(8,), reg_max=4, num_classes=3, conf=0.2)
    desc.nlevels = 1
    head = synth.yolo_head(92, 1101, 40, 24, reg_max=4, num_classes=3, cls_mu=-1.0, strides=(8,))
    got = check_decode(B, oracle, desc, head)
    assert sum(len(g["anchor"]) for g in got) > 1000


@pytest.mark.parametrize("batch", [2, 1101])
@pytest.mark.parametrize("geom", ["64x64", "40x24"])
def test_decode_reg_max_above_16(B, oracle, batch, geom):
    """reg_max 17 .. 32 takes the 32-bin DFL kernels: the split form (2
    images) and the whole-tile form (1101 one-tile images), with 16-byte loads
    (84 anchors) and scalar loads (15 anchors)."""
    if geom == "64x64":
        desc = B.detect_desc(in_w=64, in_h=64, reg_max=20, num_classes=6, conf=0.3)
        head = synth.yolo_head(93, batch, 64, 64, reg_max=20, num_classes=6, cls_mu=-1.0)
    else:
        desc = B.detect_desc(in_w=40, in_h=24, strides=(8,), reg_max=20, num_classes=6, conf=0.3)
        head = synth.yolo_head(94, batch, 40, 24, reg_max=20, num_classes=6, cls_mu=-1.0, strides=(8,))
    got = check_decode(B, oracle, desc, head)
    assert sum(len(g["anchor"]) for g in got) > batch


def test_decode_small_geometry(B, oracle):
    desc = B.detect_desc(in_w=320, in_h=192, reg_max=8, num_classes=3, conf=0.3)
    head = synth.yolo_head(22, 2, 320, 192, reg_max=8, num_classes=3, cls_mu=-2.0)
    check_decode(B, oracle, desc, head)


def test_decode_nan_and_signed_zero(B, oracle):
    desc = B.detect_desc(in_w=64, in_h=64, reg_max=4, num_classes=20, conf=0.3)
    head = synth.yolo_head(25, 2, 64, 64, reg_max=4, num_classes=20, cls_mu=-2.0)
    C0 = 16
    rng = np.random.default_rng(3)
    A = head.shape[2]
    for b in range(2):
        nan_at = rng.random((20, A)) < 0.1                 # scattered NaN class logits
        head[b, C0:][nan_at] = np.nan
        head[b, C0:, :5] = np.nan                           # all-NaN anchors
        head[b, C0:, 5:9] = -3.0                            # -0 / +0 ties above the threshold
        head[b, C0 + 7, 5:9] = -0.0
        head[b, C0 + 2, 5:9] = 0.0
        head[b, C0 + 0, 9] = np.nan                         # NaN in class 0 then a real winner
        head[b, C0 + 19, 9] = 4.0
    got = check_decode(B, oracle, desc, head)
    for g in got:
        assert 9 in g["anchor"] and not any(a < 5 for a in g["anchor"])


@pytest.mark.parametrize("objects,per_object", [(30, 8), (60, 10), (100, 12)])
def test_nms_nan_and_signed_zero(B, oracle, objects, per_object):
    # 240 candidates (one CTA), 600 (cluster, no cap) and 1200 (cluster, cap selection)
    desc = B.detect_desc(iou_thr=0.5)
    c = synth.clustered_candidates(70, objects, per_object)
    lg = np.round(c["logits"])                              # many ties
    lg[::7] = np.nan
    lg[1::5] = np.where(lg[1::5] == 0, -0.0, lg[1::5])
    lg[2::11] = -np.inf
    c["logits"] = lg.astype(np.float32)
    got = gpu_nms(B, desc, [shuffled(c, 1)])[0]
    keep = oracle.nms(c["boxes"], c["logits"], c["classes"], c["anchors"], desc.iou_thr, desc.max_det,
                      desc.max_cand)
    assert list(got["anchor"]) == [int(c["anchors"][i]) for i in keep]


def shuffled(c, seed):
    p = np.random.default_rng(seed).permutation(len(c["anchors"]))
    return {k: np.asarray(v)[p] for k, v in c.items() if k != "total"}


def check_nms(B, oracle, desc, cands_list):
    got = gpu_nms(B, desc, [shuffled(c, i) for i, c in enumerate(cands_list)])
    for b, c in enumerate(cands_list):
        keep = oracle.nms(c["boxes"], c["logits"], c["classes"], c["anchors"], desc.iou_thr, desc.max_det,
                          desc.max_cand)
        assert list(got[b]["anchor"]) == [int(c["anchors"][i]) for i in keep], b
        assert np.array_equal(got[b]["boxes"].view(np.uint32), c["boxes"][keep].view(np.uint32))
        want_score = 1.0 / (1.0 + np.exp(-c["logits"][keep].astype(np.float64)))
        assert np.allclose(got[b]["f4"], want_score, rtol=1e-6, atol=1e-7)
    return got


@pytest.mark.parametrize("iou", [0.45, 0.7, 0.2])
def test_nms_exact(B, oracle, iou):
    desc = B.detect_desc(iou_thr=iou)
    head = synth.yolo_head(23, 2)
    cands = [oracle_cands(oracle, desc, head[b]) for b in range(2)]
    got = check_nms(B, oracle, desc, cands)
    assert all(0 < len(g["anchor"]) <= len(c["anchors"]) for g, c in zip(got, cands))


@pytest.mark.parametrize("iou", [0.2, 0.45, 0.7])
def test_nms_exact_clustered(B, oracle, iou):
    # dense clusters of same-class boxes: most candidates are suppressed
    desc = B.detect_desc(iou_thr=iou)
    cands = [synth.clustered_candidates(50 + b, 40, 20) for b in range(3)]
    got = check_nms(B, oracle, desc, cands)
    assert all(len(g["anchor"]) < len(c["anchors"]) // 2 for g, c in zip(got, cands))


def test_nms_clustered_cap_ties_and_max_det(B, oracle):
    # 3000 candidates > max_cand (radix select), logits on a 0.25 grid (ties), max_det truncation
    cands = [synth.clustered_candidates(60 + b, 100, 30) for b in range(2)]
    for c in cands:
        c["logits"] = np.round(c["logits"] * 4) / 4
    for max_cand, max_det in ((1024, 300), (1024, 25), (257, 257), (1, 1)):
        desc = B.detect_desc(max_cand=max_cand, max_det=max_det)
        check_nms(B, oracle, desc, cands)


def test_nms_caps_and_ties(B, oracle):
    # many candidates (cap by radix select), coarse logits (ties -> lower anchor first), few detections
    desc = B.detect_desc(conf=0.05, max_cand=200, max_det=40)
    head = synth.yolo_head(24, 2, cls_mu=-3.0)
    head[:, 64:] = np.round(head[:, 64:] * 2) / 2
    cands = [oracle_cands(oracle, desc, head[b]) for b in range(2)]
    assert all(len(c["anchors"]) > 1000 for c in cands)
    check_nms(B, oracle, desc, cands)
    desc.max_cand, desc.max_det = 1024, 1024
    check_nms(B, oracle, desc, cands)


def first_n(c, n):
    return {k: np.asarray(v)[:n] for k, v in c.items()}


# Candidate counts across the NMS's paths: none, the one-CTA fast path (at
# most 256), and above it the cluster path (or one CTA when the batch leaves
# no room for clusters), with and without the cap selection.
NMS_COUNTS = [0, 100, 256, 257, 600, 1024, 1025, 3000, 8400]


@pytest.mark.parametrize("batch", [1, 3, 9, 24, 48, 80])
def test_nms_cluster_sizes_and_mixed_counts(B, oracle, batch):
    # the batch sets the CTAs per image (8, 4, 2 or 1 on a 152-SM GPU); images
    # of one launch mix every path
    desc = B.detect_desc(max_cand=1024, max_det=300)
    cands = []
    for b in range(batch):
        n = NMS_COUNTS[(b + batch) % len(NMS_COUNTS)]
        cands.append(first_n(synth.clustered_candidates(400 + b, 280, 30), n))
    check_nms(B, oracle, desc, cands)


@pytest.mark.parametrize("max_cand,max_det", [(1, 1), (5, 5), (9, 3), (200, 40), (257, 257), (1000, 1000)])
def test_nms_cluster_small_caps(B, oracle, max_cand, max_det):
    # caps below the cluster size and around the fast-path limit, on images
    # with more than 256 candidates
    desc = B.detect_desc(max_cand=max_cand, max_det=max_det)
    cands = [first_n(synth.clustered_candidates(500 + b, 280, 30), n) for b, n in enumerate((300, 1500, 8400))]
    check_nms(B, oracle, desc, cands)


@pytest.mark.parametrize("batch", [1, 2])
def test_nms_keys_beyond_registers(B, oracle, batch):
    # a 2560 x 2560 input: 134,400 anchors, every one a candidate, more keys
    # per CTA than its registers hold, so the selection re-reads them
    desc = B.detect_desc(in_w=2560, in_h=2560, max_cand=1024, max_det=300)
    st, A = B.ws_detect_validate(desc, batch)
    B.check(st)
    assert A == 134400
    cands = [synth.clustered_candidates(600 + b, 1344, 100, in_w=2560, in_h=2560, anchors=A) for b in range(batch)]
    for c in cands:
        c["logits"] = np.round(c["logits"] * 8) / 8          # ties resolved by anchor
    check_nms(B, oracle, desc, cands)


def run_detect(B, desc, head, ws=None):
    batch = head.shape[0]
    st, n = B.ws_detect_workspace_bytes(desc, batch)
    B.check(st)
    if ws is None:
        ws = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
    wp = ws.data_ptr() + (-ws.data_ptr()) % 256
    out = torch.zeros((batch, desc.max_det, 8), dtype=torch.int32, device="cuda")
    oc = torch.zeros(batch, dtype=torch.int32, device="cuda")
    return ws, wp, n, out, oc


def test_detect_end_to_end_and_replay(B, oracle):
    desc = B.detect_desc()
    heads = [synth.yolo_head(30 + i, 2) for i in range(3)]
    ws, wp, n, out, oc = run_detect(B, desc, heads[0])
    s = torch.cuda.Stream()
    h = torch.empty((2,) + heads[0].shape[1:], dtype=torch.float32, device="cuda")
    with torch.cuda.stream(s):
        B.check(B.ws_detect_workspace_init(wp, n, s.cuda_stream))
        g = torch.cuda.CUDAGraph()
        for i, head in enumerate(heads):
            h.copy_(torch.from_numpy(head))
            if i < 2:   # plain calls, twice on one workspace
                B.check(B.ws_detect(desc, h.data_ptr(), 2, out.data_ptr(), oc.data_ptr(), wp, n, s.cuda_stream))
            else:       # then captured once and replayed
                with torch.cuda.graph(g, stream=s):
                    B.check(B.ws_detect(desc, h.data_ptr(), 2, out.data_ptr(), oc.data_ptr(), wp, n, s.cuda_stream))
                g.replay()
            s.synchronize()
            dec = gpu_decode(B, desc, head)          # the GPU's own candidates
            o, k = out.cpu().numpy(), oc.cpu().numpy()
            for b in range(2):
                c = dec[b]
                keep = oracle.nms(c["boxes"], c["f4"], c["cls"], c["anchor"], desc.iou_thr, desc.max_det,
                                  desc.max_cand)
                got = unpack(o[b, :k[b]])
                assert list(got["anchor"]) == [int(c["anchor"][j]) for j in keep]
                assert np.array_equal(got["boxes"].view(np.uint32), c["boxes"][keep].view(np.uint32))


def test_detect_no_candidates_and_all_candidates(B, oracle):
    desc = B.detect_desc(max_cand=1024, max_det=300)
    quiet = synth.yolo_head(40, 1, cls_mu=-20.0, cls_sigma=0.1)
    ws, wp, n, out, oc = run_detect(B, desc, quiet)
    B.check(B.ws_detect_workspace_init(wp, n, stream()))
    h = torch.from_numpy(quiet).cuda()
    B.check(B.ws_detect(desc, h.data_ptr(), 1, out.data_ptr(), oc.data_ptr(), wp, n, stream()))
    torch.cuda.synchronize()
    assert int(oc[0]) == 0
    loud = synth.yolo_head(41, 1, cls_mu=5.0)        # every anchor a candidate: 8400 > max_cand
    h = torch.from_numpy(loud).cuda()
    B.check(B.ws_detect(desc, h.data_ptr(), 1, out.data_ptr(), oc.data_ptr(), wp, n, stream()))
    torch.cuda.synchronize()
    dec = gpu_decode(B, desc, loud)[0]
    assert len(dec["anchor"]) == 8400
    keep = oracle.nms(dec["boxes"], dec["f4"], dec["cls"], dec["anchor"], desc.iou_thr, desc.max_det, desc.max_cand)
    got = unpack(out.cpu().numpy()[0, :int(oc[0])])
    assert list(got["anchor"]) == [int(dec["anchor"][j]) for j in keep]


@pytest.mark.parametrize("result_mode,flags", [(0, 0), (1, 0), (2, 2), (0, 1)],
                         ids=["device", "mapped", "copy-stage-timing", "no-graph"])
def test_detection_lane(B, oracle, result_mode, flags):
    """A lane whose graph is letterbox preprocess -> decode -> NMS; the head in
    its logits slot changes between submits."""
    from post_processing_gb300.api import Lane
    desc = B.detect_desc()
    pre = B.preprocess_desc(1280, 720, 640, 640, letterbox=True, norm="scale")
    batch = 2
    d = B.lane_desc(pre, batch, 0, 0, 0, detect=desc, result_mode=result_mode, flags=flags)
    with Lane(d) as lane:
        buf = lane.buffers
        assert buf.result_val_device is None and buf.detections_device
        n_head = buf.logits_bytes // 4
        for rep in range(2):
            head = synth.yolo_head(80 + rep, batch)
            assert head.size == n_head
            hdev = torch.from_numpy(head).cuda()
            memcpy(buf.logits, hdev.data_ptr(), head.nbytes)
            lane.acquire()
            lane.submit()
            t = lane.wait()
            if flags & B.WS_LANE_FLAG_STAGE_TIMING:
                assert t.preprocess_us > 0 and t.post_us > 0
            if result_mode == B.WS_RESULT_DEVICE:
                dets = torch.empty((batch, desc.max_det, 8), dtype=torch.int32, device="cuda")
                cnts = torch.empty(batch, dtype=torch.int32, device="cuda")
                memcpy(dets.data_ptr(), buf.detections_device, dets.numel() * 4)
                memcpy(cnts.data_ptr(), buf.det_count_device, batch * 4)
                o, k = dets.cpu().numpy(), cnts.cpu().numpy()
            else:
                raw = ctypes.string_at(buf.detections_host, batch * desc.max_det * 32)
                o = np.frombuffer(raw, np.int32).reshape(batch, desc.max_det, 8)
                k = np.frombuffer(ctypes.string_at(buf.det_count_host, batch * 4), np.int32)
            dec = gpu_decode(B, desc, head)
            for b in range(batch):
                c = dec[b]
                keep = oracle.nms(c["boxes"], c["f4"], c["cls"], c["anchor"], desc.iou_thr, desc.max_det,
                                  desc.max_cand)
                got = unpack(o[b, :k[b]])
                assert list(got["anchor"]) == [int(c["anchor"][j]) for j in keep]
                assert np.array_equal(got["boxes"].view(np.uint32), c["boxes"][keep].view(np.uint32))


@pytest.mark.parametrize("batch", [1, 3])
def test_detection_lane_all_candidates(B, oracle, batch):
    """The cluster NMS inside a lane's captured graph: every anchor of every
    image a candidate (8400 -> cap 1024 -> 300 kept), alternating with a
    typical head (one CTA), over several replays; each against the oracle's NMS
    of the candidates the GPU decoded."""
    from post_processing_gb300.api import Lane
    desc = B.detect_desc()
    pre = B.preprocess_desc(1280, 720, 640, 640, letterbox=True, norm="scale")
    d = B.lane_desc(pre, batch, 0, 0, 0, detect=desc)
    with Lane(d) as lane:
        buf = lane.buffers
        for rep in range(4):
            head = synth.yolo_head(90 + rep, batch, cls_mu=5.0 if rep % 2 == 0 else -8.0)
            hdev = torch.from_numpy(head).cuda()
            memcpy(buf.logits, hdev.data_ptr(), head.nbytes)
            lane.acquire()
            lane.submit()
            lane.wait()
            dets = torch.empty((batch, desc.max_det, 8), dtype=torch.int32, device="cuda")
            cnts = torch.empty(batch, dtype=torch.int32, device="cuda")
            memcpy(dets.data_ptr(), buf.detections_device, dets.numel() * 4)
            memcpy(cnts.data_ptr(), buf.det_count_device, batch * 4)
            o, k = dets.cpu().numpy(), cnts.cpu().numpy()
            dec = gpu_decode(B, desc, head)
            for b in range(batch):
                c = dec[b]
                if rep % 2 == 0:
                    assert len(c["anchor"]) == 8400
                keep = oracle.nms(c["boxes"], c["f4"], c["cls"], c["anchor"], desc.iou_thr, desc.max_det,
                                  desc.max_cand)
                got = unpack(o[b, :k[b]])
                assert list(got["anchor"]) == [int(c["anchor"][j]) for j in keep], (rep, b)


@pytest.mark.parametrize("geom", [
    dict(in_w=40, in_h=24, strides=(8,), reg_max=4, num_classes=3),          # A = 15: scalar scan
    dict(in_w=64, in_h=64, strides=(8, 16, 32, 64), reg_max=1, num_classes=1),  # one bin, one class, 4 levels
    dict(in_w=96, in_h=32, strides=(32,), reg_max=32, num_classes=130),      # widest DFL, many classes
], ids=["A15-scalar", "R1-C1-L4", "R32-C130"])
def test_decode_edge_geometries(B, oracle, geom):
    strides = geom.pop("strides")
    desc = B.detect_desc(strides=strides, conf=0.2, **geom)
    desc.nlevels = len(strides)
    head = synth.yolo_head(90, 3, geom["in_w"], geom["in_h"], reg_max=geom["reg_max"],
                           num_classes=geom["num_classes"], cls_mu=-1.0, strides=strides)
    got = check_decode(B, oracle, desc, head)
    assert sum(len(g["anchor"]) for g in got) > 0


def test_decode_misaligned_head(B, oracle):
    """A head that is not 16-byte aligned takes the scalar scan."""
    desc = B.detect_desc()
    head = synth.yolo_head(91, 2)
    buf = torch.empty(head.size + 1, dtype=torch.float32, device="cuda")
    buf[1:].copy_(torch.from_numpy(head.reshape(-1)))
    batch, A = 2, head.shape[2]
    cand = torch.zeros((batch, A, 8), dtype=torch.int32, device="cuda")
    count = torch.zeros(batch, dtype=torch.int32, device="cuda")
    B.check(B.ws_detect_decode(desc, buf.data_ptr() + 4, batch, cand.data_ptr(), count.data_ptr(), stream()))
    torch.cuda.synchronize()
    c, n = cand.cpu().numpy(), count.cpu().numpy()
    for b in range(batch):
        u = unpack(c[b, :n[b]])
        order = np.argsort(u["anchor"], kind="stable")
        want = oracle_cands(oracle, desc, head[b])
        assert np.array_equal(u["anchor"][order], want["anchors"])
        assert np.array_equal(u["f4"][order].view(np.uint32), want["logits"].view(np.uint32))
        assert float(np.max(np.abs(u["boxes"][order] - want["boxes"]))) <= box_tol(desc)


def test_python_detect_wrapper(B, oracle):
    from post_processing_gb300 import detect, detection_fields
    desc = B.detect_desc()
    head = synth.yolo_head(95, 2)
    out, cnt = detect(torch.from_numpy(head).cuda(), desc)
    torch.cuda.synchronize()
    f = detection_fields(out)
    dec = gpu_decode(B, desc, head)
    for b in range(2):
        keep = oracle.nms(dec[b]["boxes"], dec[b]["f4"], dec[b]["cls"], dec[b]["anchor"], desc.iou_thr,
                          desc.max_det, desc.max_cand)
        k = int(cnt[b])
        assert f["anchor"][b, :k].cpu().tolist() == [int(dec[b]["anchor"][j]) for j in keep]
        assert np.array_equal(f["boxes"][b, :k].cpu().numpy(), dec[b]["boxes"][keep])
