"""Lane pool and lane bucket / rebind host logic on host-only lanes (no GPU).

Host-only lanes (WS_LANE_FLAG_NO_DEVICE) run the whole state machine and
finish after `fake_polls` completion queries, so the pool's hand-off, its
ordering, back-pressure and thread safety are tested here on the CPU.
"""
import threading

import pytest


@pytest.fixture(scope="module")
def B():
    import __graft_entry__
    __graft_entry__.build()
    from post_processing_gb300 import binding
    return binding


def fake_desc(B, polls=2, batch=4, flags=0):
    pre = B.preprocess_desc(64, 48, 32, 32)
    return B.lane_desc(pre, batch, batch, 100, 5, flags=B.WS_LANE_FLAG_NO_DEVICE | flags, fake_polls=polls)


def test_pool_order_and_backpressure(B):
    st, P = B.ws_pool_create(fake_desc(B), 3)
    assert st == B.WS_OK
    lanes = []
    for _ in range(3):
        st, L = B.ws_pool_acquire(P, 0)
        assert st == B.WS_OK and L
        lanes.append(L)
    assert len(set(lanes)) == 3
    st, L = B.ws_pool_acquire(P, 0)                     # every lane busy: back-pressure, not a block
    assert st == B.WS_ERR_TIMEOUT and L is None
    st, L = B.ws_pool_acquire(P, 2000)                  # nor after a bounded wait
    assert st == B.WS_ERR_TIMEOUT
    assert B.ws_pool_submit(P, lanes[1], 4) == B.WS_OK
    assert B.ws_pool_submit(P, lanes[0], 2) == B.WS_OK
    assert B.ws_pool_submit(P, lanes[0], 2) == B.WS_ERR_LANE_STATE   # already submitted
    assert B.ws_pool_submit(P, lanes[2], 9) == B.WS_ERR_INVALID_ARGUMENT   # more frames than the batch
    assert B.ws_pool_destroy(P) == B.WS_ERR_LANE_BUSY
    st, L, t = B.ws_pool_complete(P, -1)
    assert st == B.WS_OK and L == lanes[1]              # oldest submission first
    assert B.ws_pool_recycle(P, lanes[0]) == B.WS_ERR_LANE_STATE    # still submitted
    st, L2, _ = B.ws_pool_complete(P, -1)
    assert st == B.WS_OK and L2 == lanes[0]
    st, L3, _ = B.ws_pool_complete(P, 0)
    assert st == B.WS_ERR_TIMEOUT and L3 is None        # nothing submitted
    for L in lanes:                                     # held lanes and the unsubmitted one go back
        assert B.ws_pool_recycle(P, L) == B.WS_OK
    for _ in range(3):
        assert B.ws_pool_acquire(P, 0)[0] == B.WS_OK
    assert B.ws_pool_destroy(P) == B.WS_OK


def test_pool_rejects_borrowed_buffers_and_bad_sizes(B):
    d = fake_desc(B)
    d.input = 4096
    assert B.ws_pool_create(d, 2)[0] == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_pool_create(fake_desc(B), 0)[0] == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_pool_create(fake_desc(B), 65)[0] == B.WS_ERR_INVALID_ARGUMENT
    st, P = B.ws_pool_create(fake_desc(B), 2)
    st2, other = B.ws_lane_create(fake_desc(B))
    assert B.ws_pool_submit(P, other, 1) == B.WS_ERR_INVALID_ARGUMENT   # not a pool lane
    assert B.ws_pool_lane(P, 2)[0] == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_pool_lane(P, 1)[0] == B.WS_OK
    assert B.ws_lane_destroy(other) == B.WS_OK
    assert B.ws_pool_destroy(P) == B.WS_OK


def test_pool_producer_consumer_threads(B):
    """One producer and one consumer thread push 300 jobs through 3 lanes:
    every job completes exactly once, in submission order, and a lane is
    never handed out while its results are still held."""
    st, P = B.ws_pool_create(fake_desc(B, polls=3), 3)
    assert st == B.WS_OK
    jobs = 300
    job_of = {}            # lane -> job id written by the producer
    held = set()
    done, errors = [], []
    lock = threading.Lock()

    def producer():
        for j in range(jobs):
            st, L = B.ws_pool_acquire(P, 5_000_000)
            if st != B.WS_OK:
                errors.append(("acquire", st)); return
            with lock:
                if L in held:
                    errors.append(("handed out while held", j)); return
                job_of[L] = j
            st = B.ws_pool_submit(P, L, 1 + j % 4)
            if st != B.WS_OK:
                errors.append(("submit", st)); return

    def consumer():
        for _ in range(jobs):
            st, L, _ = B.ws_pool_complete(P, 5_000_000)
            if st != B.WS_OK:
                errors.append(("complete", st)); return
            with lock:
                held.add(L)
                done.append(job_of[L])
                held.discard(L)
            if B.ws_pool_recycle(P, L) != B.WS_OK:
                errors.append(("recycle",)); return

    tp, tc = threading.Thread(target=producer), threading.Thread(target=consumer)
    tp.start(); tc.start()
    tp.join(60); tc.join(60)
    assert not tp.is_alive() and not tc.is_alive()
    assert not errors, errors
    assert done == list(range(jobs))
    assert B.ws_pool_destroy(P) == B.WS_OK


def test_submit_n_and_rebind_host_logic(B):
    st, h = B.ws_lane_create(fake_desc(B, polls=0, flags=B.WS_LANE_FLAG_BUCKETS | B.WS_LANE_FLAG_NVTX))
    assert st == B.WS_OK
    assert B.ws_lane_acquire(h) == B.WS_OK
    assert B.ws_lane_submit_n(h, 0) == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_lane_submit_n(h, 5) == B.WS_ERR_INVALID_ARGUMENT
    assert B.ws_lane_submit_n(h, 3) == B.WS_OK
    assert B.ws_lane_rebind(h, 4096, None)[0] == B.WS_ERR_LANE_BUSY     # in flight
    assert B.ws_lane_wait(h, -1)[0] == B.WS_OK
    assert B.ws_lane_rebind(h, 4096, 8192) == (B.WS_OK, 0)
    assert B.ws_lane_destroy(h) == B.WS_OK
    # a bucketed Top-K lane needs per-frame rows
    d = fake_desc(B, flags=B.WS_LANE_FLAG_BUCKETS)
    d.rows = 6
    assert B.ws_lane_create(d)[0] == B.WS_ERR_INVALID_ARGUMENT


def test_python_pool_wrapper(B):
    from post_processing_gb300 import Pool
    with Pool(fake_desc(B, polls=1), 2) as pool:
        a, b = pool.acquire(0), pool.acquire(0)
        assert a and b and pool.acquire(0) is None                 # back-pressure
        pool.submit(a)
        pool.submit(b, 1)
        assert pool.complete()[0] == a and pool.complete()[0] == b
        assert pool.complete(0) == (None, None)
        pool.recycle(a)
        pool.recycle(b)
        assert pool.lane(0) in (a, b)
