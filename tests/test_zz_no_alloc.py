"""ws_topk_noalloc: Top-K for callers that cannot allocate device memory.

Some callers only get their input and output buffers: a plugin or callback
running inside another framework's enqueue has no allocator of its own, and a
latency-critical loop must not call cudaMalloc after start-up because it can
synchronise the device.  ws_topk_noalloc serves them with its scratch in a
fixed array inside the library instead of a caller workspace.  These tests
call it through the C ABI and compare it with ws_topk (the entry point that
takes a workspace) on two calls in a row; Top-K is exact, so they must agree
bit for bit.  The file is collected last so that a stop-at-first-failure run
has already run every other test; it also passes alone in a fresh process.
"""
import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.gpu

LIMIT = 1 << 20   # bytes of scratch the fixed array holds


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def with_workspace(B, x_dev, rows, cols, k, s):
    val = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    st, n = B.ws_topk_workspace_bytes(rows, cols, k)
    B.check(st)
    ws = torch.empty(max(n, 1), dtype=torch.uint8, device="cuda")
    if n:
        B.check(B.ws_topk_workspace_init(ws.data_ptr(), n, s))
    B.check(B.ws_topk(x_dev.data_ptr(), rows, cols, k, val.data_ptr(), idx.data_ptr(),
                      ws.data_ptr() if n else None, n, s))
    return val, idx


def without_allocation(B, x_dev, rows, cols, k, s):
    val = torch.full((rows, k), 3.0, dtype=torch.float32, device="cuda")
    idx = torch.full((rows, k), -1, dtype=torch.int32, device="cuda")
    B.check(B.ws_topk_noalloc(x_dev.data_ptr(), rows, cols, k, val.data_ptr(), idx.data_ptr(), s))
    return val, idx


SHAPES = [
    (32, 131072, 32),   # 4K-batch logits: 16 blocks per row, scratch in use
    (1, 672000, 32),    # one long row of detection scores
    (7, 20001, 5),      # ragged last block
    (64, 1000, 32),     # short rows: no scratch needed
]


@pytest.mark.parametrize("rows,cols,k", SHAPES)
def test_matches_workspace_entry_point_twice(B, rows, cols, k):
    st, need = B.ws_topk_workspace_bytes(rows, cols, k)
    assert st == B.WS_OK and need <= LIMIT
    s = torch.cuda.current_stream().cuda_stream
    for call in range(2):                      # two calls in a row, different data
        x = synth.logits_with_ties(1000 * call + rows + cols, rows, cols)
        if call == 1:
            x[0, ::5] = np.nan
        x_dev = torch.from_numpy(x).cuda()
        want_v, want_i = with_workspace(B, x_dev, rows, cols, k, s)
        got_v, got_i = without_allocation(B, x_dev, rows, cols, k, s)
        torch.cuda.synchronize()
        assert torch.equal(got_i, want_i), f"call {call}: indices differ"
        assert torch.equal(got_v.view(torch.int32), want_v.view(torch.int32)), f"call {call}: values differ"


def test_shape_above_the_limit_is_refused(B):
    rows, cols, k = 512, 131072, 32
    st, need = B.ws_topk_workspace_bytes(rows, cols, k)
    assert st == B.WS_OK and need > LIMIT
    st = B.ws_topk_noalloc(16, rows, cols, k, 16, 16, 0)     # rejected before any launch
    assert st == B.WS_ERR_UNSUPPORTED
    msg = B.ws_last_error()
    assert str(need) in msg and str(LIMIT) in msg
