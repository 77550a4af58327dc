"""The C ABI without a GPU: the library loads, exports every symbol the
header declares, the ctypes structs match the C layout, arguments are
validated on the host before anything is enqueued, and the lane state
machine behaves (host-only lanes)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ws.h")


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def header_functions():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"^\s*[\w\s\*]*?\b(ws_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(B):
    names = header_functions()
    assert len(names) >= 17
    lib = ctypes.CDLL(B.LIBRARY_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in ws.h but not exported"
    assert sorted(B.SIGNATURES) == names, "binding and header disagree"


def test_checked_build_exports_the_same_symbols(B):
    # the checked build (libws_bounds.so, compiled with WS_BOUNDS_CHECK) is a
    # drop-in replacement: same symbols, and it says what it is
    from post_processing_gb300 import build
    lib = ctypes.CDLL(build.BOUNDS_LIBRARY)
    for n in header_functions():
        assert hasattr(lib, n), f"{n} missing from the checked build"
    lib.ws_build_features.restype = ctypes.c_int32
    assert lib.ws_build_features() & B.WS_FEATURE_BOUNDS_CHECK
    expected = B.WS_FEATURE_BOUNDS_CHECK if os.environ.get("WS_BOUNDS_CHECK") == "1" else 0
    assert B.ws_build_features() & B.WS_FEATURE_BOUNDS_CHECK == expected


def test_struct_layout_matches_c(B, tmp_path):
    structs = {"ws_preprocess_desc": B.ws_preprocess_desc, "ws_lane_desc": B.ws_lane_desc,
               "ws_lane_buffers": B.ws_lane_buffers, "ws_lane_timing": B.ws_lane_timing,
               "ws_detect_desc": B.ws_detect_desc, "ws_candidate": B.ws_candidate,
               "ws_detection": B.ws_detection, "ws_debug_counters": B.ws_debug_counters}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "ws.h"', "int main(void) {"]
    for name, cls in structs.items():
        lines.append(f'printf("{name} size %zu\\n", sizeof({name}));')
        for f, _ in cls._fields_:
            lines.append(f'printf("{name} {f} %zu\\n", offsetof({name}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-I" + os.path.join(ROOT, "include"), "-I/usr/local/cuda/include", str(src),
                    "-o", str(exe)], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split("\n")
    for line in filter(None, out):
        name, field, value = line.split()
        cls = structs[name]
        got = ctypes.sizeof(cls) if field == "size" else getattr(cls, field).offset
        assert got == int(value), (name, field, got, value)


def test_status_strings(B):
    assert B.ws_status_string(0) == "WS_OK"
    assert B.ws_status_string(B.WS_ERR_TIMEOUT) == "WS_ERR_TIMEOUT"
    assert B.ws_status_string(12345) == "WS_ERR_UNKNOWN"
    assert B.ws_version() >= 100


@pytest.mark.parametrize("field,value", [
    ("src_w", 0), ("src_h", -1), ("dst_w", 0), ("dst_h", 70000), ("src_row_stride", 5),
    ("src_frame_stride", 10), ("resize", 7), ("pad_value", 256), ("norm", 3), ("channel_order", 2),
    ("dst_type", 3), ("dst_type", -1)])
def test_preprocess_descriptor_rejected(B, field, value):
    d = B.preprocess_desc(32, 16, 8, 8)
    setattr(d, field, value)
    st = B.ws_preprocess_validate(d, 1)
    assert st in (B.WS_ERR_INVALID_ARGUMENT, B.WS_ERR_UNSUPPORTED), field
    assert B.ws_last_error()
    # the entry point rejects it the same way, before touching CUDA
    assert B.ws_preprocess(d, 16, 1, 16, 0) == st


def test_preprocess_validation_accepts_and_rejects(B):
    d = B.preprocess_desc(1920, 1080, 224, 224)
    assert B.ws_preprocess_validate(d, 64) == B.WS_OK
    assert B.ws_preprocess_validate(d, 0) == B.WS_ERR_INVALID_ARGUMENT
    bad = B.preprocess_desc(4, 4, 4, 4)
    bad.std[1] = 0.0
    assert B.ws_preprocess_validate(bad, 1) == B.WS_ERR_INVALID_ARGUMENT
    # NULL pointers are refused before any launch
    assert B.ws_preprocess(d, None, 1, 16, 0) == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_preprocess(d, 16, 1, None, 0) == B.WS_ERR_INVALID_ARGUMENT


@pytest.mark.parametrize("rows,cols,k,ok", [
    (1, 1000, 5, True), (64, 1000, 32, True), (1, 1, 1, True), (1, 1000, 33, False),
    (1, 4, 5, False), (0, 10, 1, False), (1, 0, 1, False), (1, 1 << 31, 1, False), (3, 10, 0, False)])
def test_topk_validation(B, rows, cols, k, ok):
    st = B.ws_topk_validate(rows, cols, k)
    assert (st == B.WS_OK) == ok
    st2, n = B.ws_topk_workspace_bytes(rows, cols, k)
    assert st2 == st
    if not ok:
        assert B.ws_topk(16, rows, cols, k, 16, 16, None, 0, 0) == B.WS_ERR_INVALID_ARGUMENT


def test_topk_workspace_sizes(B):
    assert B.ws_topk_workspace_bytes(64, 1000, 32) == (0, 0)          # one block per row
    st, n = B.ws_topk_workspace_bytes(32, 131072, 32)
    assert st == 0 and n >= 32 * 16 * 32 * 8
    st, n2 = B.ws_topk_workspace_bytes(1, 672000, 32)
    assert st == 0 and n2 > 0
    # a workspace that is too small is refused
    assert B.ws_topk(16, 32, 131072, 32, 16, 16, 256, n - 8, 0) == B.WS_ERR_INVALID_ARGUMENT


def _fake_lane(B, polls=3):
    pre = B.preprocess_desc(64, 48, 32, 32)
    d = B.lane_desc(pre, 1, 1, 100, 5, flags=B.WS_LANE_FLAG_NO_DEVICE, fake_polls=polls)
    st, h = B.ws_lane_create(d)
    assert st == B.WS_OK, B.ws_last_error()
    return h


def test_lane_state_machine_host_only(B):
    h = _fake_lane(B, polls=3)
    assert B.ws_lane_state(h) == B.WS_LANE_FREE
    assert B.ws_lane_submit(h) == B.WS_ERR_LANE_STATE          # submit without acquire
    assert B.ws_lane_wait(h, 0)[0] == B.WS_ERR_LANE_STATE       # nothing in flight
    assert B.ws_lane_release(h) == B.WS_ERR_LANE_STATE
    assert B.ws_lane_acquire(h) == B.WS_OK
    assert B.ws_lane_acquire(h) == B.WS_ERR_LANE_BUSY            # no second owner
    assert B.ws_lane_release(h) == B.WS_OK
    assert B.ws_lane_acquire(h) == B.WS_OK
    assert B.ws_lane_submit(h) == B.WS_OK
    assert B.ws_lane_state(h) == B.WS_LANE_IN_FLIGHT
    assert B.ws_lane_acquire(h) == B.WS_ERR_LANE_BUSY            # no reuse while busy
    assert B.ws_lane_submit(h) == B.WS_ERR_LANE_STATE            # no queue growth
    assert B.ws_lane_destroy(h) == B.WS_ERR_LANE_BUSY
    st, _ = B.ws_lane_wait(h, 0)                                  # not done after one poll
    assert st == B.WS_ERR_TIMEOUT and B.ws_lane_state(h) == B.WS_LANE_IN_FLIGHT
    st, t = B.ws_lane_wait(h, -1)                                 # finishes after its polls
    assert st == B.WS_OK and B.ws_lane_state(h) == B.WS_LANE_FREE and t.host_us >= 0
    assert B.ws_lane_destroy(h) == B.WS_OK


def test_lane_descriptor_rejected(B):
    pre = B.preprocess_desc(64, 48, 32, 32)
    for kw in (dict(k=40), dict(input_mode=9), dict(result_mode=-1), dict(flags=1 << 10)):
        args = dict(batch=1, rows=1, cols=100, k=5)
        args.update(kw)
        d = B.lane_desc(pre, args.pop("batch"), args.pop("rows"), args.pop("cols"), args.pop("k"),
                        flags=B.WS_LANE_FLAG_NO_DEVICE | args.pop("flags", 0), **args)
        st, h = B.ws_lane_create(d)
        assert st == B.WS_ERR_INVALID_ARGUMENT and h is None, kw


def test_preprocess_path_rejected(B):
    d = B.preprocess_desc(64, 48, 32, 32)
    assert B.ws_preprocess_path(d, 4096, 1, 8192, 3, 0) == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_preprocess_path(d, 4096, 1, 8192, -1, 0) == B.WS_ERR_INVALID_ARGUMENT


def test_detection_lane_descriptor(B):
    pre = B.preprocess_desc(1280, 720, 640, 640, letterbox=True, norm="scale")
    fake = dict(flags=B.WS_LANE_FLAG_NO_DEVICE)
    st, h = B.ws_lane_create(B.lane_desc(pre, 2, 0, 0, 0, detect=B.detect_desc(), **fake))
    assert st == B.WS_OK and h is not None
    assert B.ws_lane_destroy(h) == B.WS_OK
    bad = [B.lane_desc(pre, 2, 0, 0, 0, detect=B.detect_desc(max_det=0), **fake),
           B.lane_desc(pre, 2, 0, 0, 0, detect=B.detect_desc(), result_val=64, result_idx=64, **fake),
           B.lane_desc(pre, 2, 0, 0, 0, detect=B.detect_desc(), detections=64, **fake)]
    odd = B.lane_desc(pre, 1, 1, 100, 5, **fake)
    odd.post = 7
    for d in bad + [odd]:
        st, h = B.ws_lane_create(d)
        assert st == B.WS_ERR_INVALID_ARGUMENT and h is None


def test_product_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "post_processing_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "ws_oracle" not in text and "liboracle" not in text, f


def test_detect_validation(B):
    d = B.detect_desc()
    st, A = B.ws_detect_validate(d, 4)
    assert st == B.WS_OK and A == 8400
    st, n = B.ws_detect_workspace_bytes(d, 4)
    assert st == B.WS_OK and n >= 4 * 8400 * 32
    for field, value in (("max_cand", 2000), ("max_det", 0), ("reg_max", 40), ("num_classes", 0),
                         ("nlevels", 5)):
        bad = B.detect_desc()
        setattr(bad, field, value)
        assert B.ws_detect_validate(bad, 1)[0] == B.WS_ERR_INVALID_ARGUMENT, field
        assert B.ws_detect(bad, 16, 1, 16, 16, 256, 1 << 20, 0) == B.WS_ERR_INVALID_ARGUMENT
    bad = B.detect_desc(in_w=650)            # 650 is not a multiple of 32
    assert B.ws_detect_validate(bad, 1)[0] == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_detect_validate(d, 0)[0] == B.WS_ERR_INVALID_ARGUMENT
    # a workspace that is too small is refused before any launch
    assert B.ws_detect(d, 16, 4, 16, 16, 256, n - 32, 0) == B.WS_ERR_INVALID_ARGUMENT


def test_fault_injection_hook_host_only(B):
    """The fault-injection hook arms and disarms without a GPU; host-only
    lanes make no CUDA call, so they reach no fault point and hold nothing."""
    assert B.ws_debug_inject_failure(1, -1) == B.WS_ERR_INVALID_ARGUMENT
    B.check(B.ws_debug_inject_failure(1, 1))
    st, before = B.ws_debug_get_counters()
    assert st == B.WS_OK and before.fault_points == 0
    d = B.lane_desc(B.preprocess_desc(64, 48, 32, 32), 1, 1, 100, 5, flags=B.WS_LANE_FLAG_NO_DEVICE)
    st, h = B.ws_lane_create(d)
    assert st == B.WS_OK
    st, after = B.ws_debug_get_counters()
    assert after.fault_points == 0
    for f in ("device_allocs", "host_allocs", "graphs", "graph_execs", "events", "streams"):
        assert getattr(after, f) == getattr(before, f), f
    assert B.ws_lane_selftest_wait_timeout(h, 1000) == B.WS_ERR_UNSUPPORTED
    assert B.ws_lane_destroy(h) == B.WS_OK
    B.check(B.ws_debug_inject_failure(0, 0))
