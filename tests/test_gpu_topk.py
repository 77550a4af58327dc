"""GPU exact Top-K against the oracle: indices and values bit-exact.

Covers the five workloads' logits at full size, row lengths around every
block boundary (8192 per block), K from 1 to 32, ties (including ties at the
cut and +0/-0), NaN and infinities, and adversarial rows that defeat the
threshold (constant rows, sorted rows), which take the radix-select path;
also a misaligned pointer (scalar loads), workspace reuse across calls and
replay inside a captured CUDA Graph.
"""
import numpy as np
import pytest
import torch

import synth
from cudart import memcpy
from pins import check_topk_invariants

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def gpu_topk(B, x, k, offset=0, workspace=None):
    rows, cols = x.shape
    flat = torch.zeros(rows * cols + offset + 8, dtype=torch.float32, device="cuda")
    flat[offset:offset + rows * cols] = torch.from_numpy(x.reshape(-1)).cuda()
    val = torch.full((rows, k), 7.0, dtype=torch.float32, device="cuda")
    idx = torch.full((rows, k), -9, dtype=torch.int32, device="cuda")
    st, n = B.ws_topk_workspace_bytes(rows, cols, k)
    B.check(st)
    s = torch.cuda.current_stream().cuda_stream
    if workspace is None and n:
        workspace = torch.empty(n + 256, dtype=torch.uint8, device="cuda")
    wptr = 0
    if n:
        wptr = workspace.data_ptr() + (-workspace.data_ptr()) % 256
        B.check(B.ws_topk_workspace_init(wptr, n, s))
    B.check(B.ws_topk(flat.data_ptr() + 4 * offset, rows, cols, k, val.data_ptr(), idx.data_ptr(),
                      wptr or None, n, s))
    torch.cuda.synchronize()
    return val.cpu().numpy(), idx.cpu().numpy()


def assert_exact(got, want):
    gv, gi = got
    wv, wi = want
    assert np.array_equal(gi, wi), f"indices differ in rows {np.nonzero((gi != wi).any(1))[0][:8]}"
    assert np.array_equal(gv.view(np.uint32), wv.view(np.uint32)), "values differ"


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_workload_parity(B, oracle, name):
    w = synth.WORKLOADS[name]
    x = synth.make_logits(name)
    assert_exact(gpu_topk(B, x, w["k"]), oracle.topk(x, w["k"]))


@pytest.mark.parametrize("cols", [1, 2, 3, 31, 32, 33, 100, 576, 700, 911, 913, 1000, 4097, 8191, 8192, 8193,
                                  16384, 20001, 65536 + 3])
@pytest.mark.parametrize("k", [1, 5, 32])
def test_lengths(B, oracle, cols, k):
    if k > cols:
        pytest.skip("k > cols is rejected")
    x = synth.logits_with_ties(cols * 31 + k, 3, cols, frac=0.1)
    assert_exact(gpu_topk(B, x, k), oracle.topk(x, k))


def special_rows(cols, rng):
    rows = []
    rows.append(np.zeros(cols, np.float32))                                  # constant
    rows.append(np.full(cols, np.nan, np.float32))                           # all NaN
    z = np.zeros(cols, np.float32); z[::2] = -0.0; rows.append(z)          # +0 / -0 ties
    rows.append(np.arange(cols, dtype=np.float32))                           # ascending
    rows.append(-np.arange(cols, dtype=np.float32))                          # descending
    r = rng.integers(0, 3, cols).astype(np.float32); rows.append(r)         # three values
    r = rng.standard_normal(cols).astype(np.float32)
    r[rng.integers(0, cols, cols // 10)] = np.nan
    r[rng.integers(0, cols, 5)] = np.inf
    r[rng.integers(0, cols, 5)] = -np.inf
    rows.append(r)
    r = rng.standard_normal(cols).astype(np.float32)                        # ties at the cut
    top = np.sort(r)[-20]
    r[rng.integers(0, cols, 40)] = top
    rows.append(r)
    r = np.full(cols, -1.0, np.float32); r[: min(cols, 300)] = 5.0          # one hot region
    rows.append(r)
    r = np.full(cols, 1.0, np.float32); r[-min(cols, 300):] = 2.0           # hot region at the end
    rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("cols", [40, 1000, 8192, 30000])
@pytest.mark.parametrize("k", [1, 17, 32])
def test_special_rows(B, oracle, cols, k):
    x = special_rows(cols, np.random.default_rng(cols + k))
    got = gpu_topk(B, x, k)
    assert_exact(got, oracle.topk(x, k))
    check_topk_invariants(x, got[0], got[1], k)


# The same adversarial rows on long rows cut into 16384-element chunks (10,
# 25, 42 and 49 chunk lists: the merging block's warps fold up to six lists
# each per round, so 49 lists take two rounds).  A constant or all-NaN row
# sends every chunk to the exact radix-select fallback.
@pytest.mark.parametrize("cols", [150000, 393217, 672000, 786433])
@pytest.mark.parametrize("k", [1, 32])
def test_special_long_rows(B, oracle, cols, k):
    x = special_rows(cols, np.random.default_rng(3 * cols + k))
    got = gpu_topk(B, x, k)
    assert_exact(got, oracle.topk(x, k))
    check_topk_invariants(x, got[0], got[1], k)


def test_misaligned_pointer_scalar_path(B, oracle):
    x = synth.logits_normal(5, 4, 10001)
    assert_exact(gpu_topk(B, x, 32, offset=1), oracle.topk(x, 32))
    x = synth.logits_normal(6, 2, 1000)
    assert_exact(gpu_topk(B, x, 5, offset=3), oracle.topk(x, 5))


@pytest.mark.parametrize("rows,cols", [(8, 50000), (32, 40000)], ids=["ticket", "cluster"])
def test_workspace_reuse_and_graph_replay(B, oracle, rows, cols):
    # [8,50000]: 16 chunks a row, the ticket merge; [32,40000]: 5 chunks, the
    # cluster merge, captured as a cluster launch
    k = 32
    xs = [synth.logits_with_ties(40 + i, rows, cols) for i in range(3)]
    st, n = B.ws_topk_workspace_bytes(rows, cols, k)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    x_dev = torch.empty((rows, cols), dtype=torch.float32, device="cuda")
    val = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        B.check(B.ws_topk_workspace_init(ws.data_ptr(), n, s.cuda_stream))
        # plain calls, one after another on one workspace
        for x in xs:
            x_dev.copy_(torch.from_numpy(x))
            B.check(B.ws_topk(x_dev.data_ptr(), rows, cols, k, val.data_ptr(), idx.data_ptr(),
                              ws.data_ptr(), n, s.cuda_stream))
            s.synchronize()
            assert_exact((val.cpu().numpy(), idx.cpu().numpy()), oracle.topk(x, k))
        # captured once, replayed with new inputs in the same buffers
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            B.check(B.ws_topk(x_dev.data_ptr(), rows, cols, k, val.data_ptr(), idx.data_ptr(),
                              ws.data_ptr(), n, s.cuda_stream))
        for x in reversed(xs):
            x_dev.copy_(torch.from_numpy(x))
            g.replay()
            s.synchronize()
            assert_exact((val.cpu().numpy(), idx.cpu().numpy()), oracle.topk(x, k))


def test_torch_sort_agrees(B):
    """Library special case: a stable descending sort after NaN -> -inf."""
    x = synth.logits_with_ties(77, 16, 4096, frac=0.3)
    x[3, ::7] = np.nan
    v, i = gpu_topk(B, x, 32)
    t = torch.from_numpy(np.where(np.isnan(x), -np.inf, x)) + 0.0
    sv, si = torch.sort(t, dim=1, descending=True, stable=True)
    assert np.array_equal(i, si[:, :32].numpy().astype(np.int32))


# Rows of at most 2048 entries take the one-warp-per-row kernel when there
# are at least two rows per SM, or when the rows hold at most 512 entries
# (8, 16, 32 or 64 values per lane); the block kernel takes the rest.  The
# cases below are sized so that they reach the kernel they name: lengths at
# each register-count boundary, aligned and misaligned (16-byte vs scalar
# loads), row counts on both sides of the choice, and rows built to reach the
# warp kernel's exact fallback (more than 256 elements at or above its
# threshold).
def warp_rows(cols):
    """A row count that puts rows of this length on the warp kernel."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return 3 if cols <= 512 else 2 * sms + 3


@pytest.mark.parametrize("cols", [4, 8, 255, 256, 257, 511, 512, 513, 1023, 1024, 1025, 2044, 2047, 2048])
@pytest.mark.parametrize("offset", [0, 1])
def test_warp_rows_lengths(B, oracle, cols, offset):
    for k in (1, 4, 32):
        if k > cols:
            continue
        x = synth.logits_with_ties(cols * 7 + k + offset, warp_rows(cols), cols, frac=0.2)
        assert_exact(gpu_topk(B, x, k, offset=offset), oracle.topk(x, k))


def test_warp_rows_counts(B, oracle):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for rows in (1, 2 * sms - 1, 2 * sms, 2 * sms + 1, 4 * sms + 5):
        x = synth.logits_with_ties(rows + 3, rows, 1000)
        assert_exact(gpu_topk(B, x, 32), oracle.topk(x, 32))
    for rows in (1, 5, 64):
        x = synth.logits_with_ties(rows + 4, rows, 300)
        assert_exact(gpu_topk(B, x, 8), oracle.topk(x, 8))


def warp_fallback_rows(cols, rng):
    rows = []
    r = rng.standard_normal(cols).astype(np.float32)          # 300 copies of the maximum
    r[rng.choice(cols, min(cols, 300), replace=False)] = 9.0
    rows.append(r)
    r = np.full(cols, np.nan, np.float32)                      # too few delegates above -inf
    r[rng.choice(cols, 6, replace=False)] = rng.standard_normal(6)
    rows.append(r)
    r = np.full(cols, -np.inf, np.float32); r[::3] = np.nan    # -inf and NaN only
    rows.append(r)
    r = np.full(cols, np.inf, np.float32)                      # +inf everywhere
    rows.append(r)
    r = rng.standard_normal(cols).astype(np.float32)
    r[rng.choice(cols, min(cols, 40), replace=False)] = np.inf # +inf delegates, search capped
    rows.append(r)
    r = (rng.integers(0, 2, cols) * 2 - 1).astype(np.float32)  # two values: half the row ties
    rows.append(r)
    r = np.ldexp(np.ones(cols, np.float32), rng.integers(-120, 120, cols)).astype(np.float32)
    rows.append(r)                                             # values over 70 binades
    z = np.zeros(cols, np.float32); z[1::2] = -0.0; z[5] = -1e-30
    rows.append(z)
    r = rng.standard_normal(cols).astype(np.float32)          # a plain row between them
    rows.append(r)
    return np.stack(rows)


@pytest.mark.parametrize("cols", [40, 300, 1000, 2048])
@pytest.mark.parametrize("k", [1, 7, 32])
@pytest.mark.parametrize("offset", [0, 1])
def test_warp_rows_fallback(B, oracle, cols, k, offset):
    rng = np.random.default_rng(cols * k + offset)
    base = warp_fallback_rows(cols, rng)
    reps = -(-warp_rows(cols) // len(base))
    x = np.concatenate([base] + [warp_fallback_rows(cols, rng) for _ in range(reps - 1)])
    got = gpu_topk(B, x, k, offset=offset)
    assert_exact(got, oracle.topk(x, k))
    check_topk_invariants(x, got[0], got[1], k)


# Long rows: one block per chunk writes the chunk's K keys, and the row's
# last block merges the lists (its warps fold them into at most eight, then
# every key is ranked by binary searches).  Rows are cut into chunks of up to
# 8192 (cut finer down to 2048 while SMs would idle), or of up to 16384 when
# that would give more than 16 chunks a row or more than two blocks per SM.
# On a 152-SM GB300: [8,131072] 16 lists of 8192, [4,65536] 16 of 4096,
# [2,100000] 16 of 6252, [32,131072] and [64,131072] 8 of 16384 (no fold),
# [200,16384] and [320,9000] one chunk in the 16384-element kernel, [1,150000]
# 10 of 15000, [1,393217] 25, [1,672000] 42, [1,786433] 49 (two fold rounds),
# [1,1000000] 62, [2,2000000] 123.
@pytest.mark.parametrize("rows,cols", [(8, 131072), (4, 65536), (2, 100000), (32, 131072), (64, 131072),
                                       (200, 16384), (320, 9000), (1, 150000), (1, 393217), (1, 672000),
                                       (1, 786433), (1, 1_000_000), (2, 2_000_000)])
@pytest.mark.parametrize("k", [1, 5, 32])
def test_long_row_merge_paths(B, oracle, rows, cols, k):
    x = synth.logits_with_ties(rows * 7 + cols + k, rows, cols, frac=0.05)
    rng = np.random.default_rng(cols + k)
    # ties at the top spread over many chunks, NaN and -0 sprinkled in
    top = x.max(axis=1, keepdims=True)
    for r in range(rows):
        x[r, rng.choice(cols, 40, replace=False)] = top[r, 0]
        x[r, rng.choice(cols, 100, replace=False)] = np.nan
        x[r, rng.choice(cols, 10, replace=False)] = -0.0
    got = gpu_topk(B, x, k)
    assert_exact(got, oracle.topk(x, k))
    check_topk_invariants(x, got[0], got[1], k)



# A row cut into 2 .. 8 chunks merges through a thread-block cluster of its
# blocks when ws_topk is called directly, and through the row ticket inside
# a lane (lanes share the GPU with other lanes' kernels).  Both paths against
# the oracle on the same rows: 8 chunks of 16384, 5 of 8000, 8 of 7500, 2 of
# 8192, and 2 chunks in the 16384-element kernel.  Longer rows take the
# ticket on both paths, checked here inside lanes and replayed: 16 chunks of
# 8192, 16 of 6252, 42 of 16000 and 49 of 16052 (two fold rounds).
@pytest.mark.parametrize("rows,cols", [(32, 131072), (40, 40000), (20, 60000), (64, 16384), (300, 20000),
                                       (8, 131072), (2, 100000), (1, 672000), (1, 786433)])
@pytest.mark.parametrize("k", [1, 7, 32])
def test_cluster_and_ticket_merges(B, oracle, rows, cols, k):
    from post_processing_gb300 import Lane
    x = synth.logits_with_ties(rows * 3 + cols + k, rows, cols, frac=0.05)
    want = oracle.topk(x, k)
    assert_exact(gpu_topk(B, x, k), want)
    pre = B.preprocess_desc(16, 16, 16, 16)
    with Lane(B.lane_desc(pre, 1, rows, cols, k)) as lane:
        b = lane.buffers
        torch.cuda.synchronize()
        memcpy(b.logits, np.ascontiguousarray(x).ctypes.data, x.nbytes)
        for _ in range(2):   # a replay reuses the row tickets
            lane.acquire()
            lane.submit()
            lane.wait()
            v = np.empty((rows, k), np.float32)
            i = np.empty((rows, k), np.int32)
            memcpy(v.ctypes.data, b.result_val_device, v.nbytes)
            memcpy(i.ctypes.data, b.result_idx_device, i.nbytes)
            assert_exact((v, i), want)


# Many ties at the top of a row, or at its cut (the K-th value): a chunk
# then has 385 to 2048 candidates, which take a radix select over the
# candidates before the rank (and above 2048, the select over the chunk).
@pytest.mark.parametrize("rows,cols,ties", [(64, 1000, 600), (4, 1000, 390), (1, 8000, 1500), (3, 16384, 1900),
                                            (2, 50000, 3000), (1, 8000, 2100)])
@pytest.mark.parametrize("k", [1, 5, 32])
@pytest.mark.parametrize("where", ["top", "cut"])
def test_many_tied_candidates(B, oracle, rows, cols, ties, k, where):
    x = synth.logits_normal(rows * 13 + cols + ties + k, rows, cols)
    rng = np.random.default_rng(cols + ties + k)
    for r in range(rows):
        v = x[r].max() + 1.0 if where == "top" else np.sort(x[r])[-k]
        x[r, rng.choice(cols, ties, replace=False)] = v
    got = gpu_topk(B, x, k)
    assert_exact(got, oracle.topk(x, k))
    check_topk_invariants(x, got[0], got[1], k)


# Rows whose chunks all hold the same values (a period of 8192 entries), so
# that every chunk's list holds the same values and only the indices decide
# the ties across lists: 16 chunks of 8192, and 24 of 16384.
@pytest.mark.parametrize("rows,cols", [(2, 16 * 8192), (1, 48 * 8192)])
@pytest.mark.parametrize("k", [1, 5, 32])
def test_merge_of_identical_chunks(B, oracle, rows, cols, k):
    base = synth.logits_normal(cols + k, 1, 8192)[0]
    x = np.ascontiguousarray(np.tile(base, (rows, cols // 8192)))
    got = gpu_topk(B, x, k)
    assert_exact(got, oracle.topk(x, k))
    check_topk_invariants(x, got[0], got[1], k)


@pytest.mark.parametrize("rows,cols", [(3, 150001), (33, 131071), (5, 20003)])
@pytest.mark.parametrize("offset", [1, 2])
def test_long_rows_misaligned(B, oracle, rows, cols, offset):
    """Long rows whose start is not 16-byte aligned (coalesced loads instead of
    the bulk copy), in both chunk sizes, with a ragged last chunk."""
    x = synth.logits_with_ties(rows + cols + offset, rows, cols, frac=0.05)
    got = gpu_topk(B, x, 32, offset=offset)
    assert_exact(got, oracle.topk(x, 32))


def test_long_rows_all_top_in_one_chunk(B, oracle):
    """The whole Top-K inside one chunk (the other lists' keys all rank
    below): the ranks come from one list alone."""
    rows, cols = 4, 200000
    x = synth.logits_normal(91, rows, cols)
    for r in range(rows):
        at = 16384 * (r + 3) + 100
        x[r, at:at + 40] = 50.0 + np.arange(40, dtype=np.float32)
    for k in (1, 32):
        assert_exact(gpu_topk(B, x, k), oracle.topk(x, k))
