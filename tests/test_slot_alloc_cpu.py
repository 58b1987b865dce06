"""Host slot management without a GPU: the allocator over slots 1..P (row 0 the padding row),
the concurrency cap of a pool size, and the track plan of a decode step (ping-pong track
slots, tracked when the length is a multiple of the interval)."""
import json
import os
import threading

import numpy as np
import pytest

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def b():
    from recurrent_state_cache_gb300 import _build, binding
    _build.build()
    return binding


def test_cap_reproduces_the_pages_log(b):
    gold = json.load(open(os.path.join(GOLDEN, "concurrency_cap.json")))
    for c in gold["cases"]:
        assert b.max_running_requests(c["num_slots"], bool(c["overlap"]), bool(c["skip_decode_lock"])) \
            == c["max_running_requests"]
        assert c["num_slots"] // c["slots_per_request"] == c["max_running_requests"]
    # one fewer slot per request with the decode-lock skip, two fewer without overlap
    assert b.max_running_requests(80, True, True) == 80 // 4
    assert b.max_running_requests(80, False, False) == 80 // 3
    assert b.max_running_requests(4, True, False) == 0


def test_acquire_release_and_errors(b):
    a = b.SlotAllocator(6)
    assert a.free_count() == 6
    got = a.acquire(4)
    assert sorted(got.tolist()) == [1, 2, 3, 4] and a.free_count() == 2
    with pytest.raises(b.RscError) as e:
        a.acquire(3)                     # more than is free: nothing taken
    assert e.value.status == b.RSC_ENOSPACE and a.free_count() == 2
    rest = a.acquire(2)
    assert 0 not in set(got.tolist()) | set(rest.tolist()) and a.free_count() == 0
    a.release(got[:2])
    assert a.free_count() == 2
    with pytest.raises(b.RscError) as e:
        a.release(got[:1])               # not held any more: nothing freed
    assert e.value.status == b.RSC_EINVAL and a.free_count() == 2
    with pytest.raises(b.RscError) as e:
        a.release(np.int32([got[2], got[2]]))  # repeated in one call
    assert e.value.status == b.RSC_EINVAL and a.free_count() == 2
    for bad in ([0], [7], [-1]):
        with pytest.raises(b.RscError) as e:
            a.release(np.int32(bad))
        assert e.value.status == b.RSC_ERANGE
    a.release(np.concatenate([got[2:], rest]))
    assert a.free_count() == 6


def test_threads_never_share_a_slot(b):
    P, n_threads, rounds = 64, 8, 300
    a = b.SlotAllocator(P)
    owner = np.full(P + 1, -1, np.int64)
    lock = threading.Lock()
    errors = []

    def work(tid):
        r = np.random.default_rng(tid)
        held = []
        for _ in range(rounds):
            if held and r.random() < 0.5:
                s = held.pop(r.integers(len(held)))
                with lock:
                    if owner[s] != tid:
                        errors.append(("release", s, owner[s], tid))
                    owner[s] = -1
                a.release(np.int32([s]))
            else:
                try:
                    s = int(a.acquire(1)[0])
                except b.RscError:
                    continue
                with lock:
                    if owner[s] != -1:
                        errors.append(("double", s, owner[s], tid))
                    owner[s] = tid
                held.append(s)
        for s in held:
            with lock:
                owner[s] = -1
            a.release(np.int32([s]))

    ts = [threading.Thread(target=work, args=(i,)) for i in range(n_threads)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors and a.free_count() == P


def test_track_plan_interval_and_ping_pong(b):
    """Tracked when the length is a positive multiple of the interval; a request's two track
    slots alternate between the steps it is tracked in (A, B, A, ...); one track slot stays."""
    pairs = np.int32([[11, 12], [21, 22], [31, 32], [41, 42]])
    nxt = np.zeros(4, np.int32)
    mask, ts = b.track_plan([1024, 1000, 1280, 0], 256, pairs, nxt)
    assert mask.tolist() == [1, 0, 1, 0] and ts.tolist() == [11, 0, 31, 0]
    assert nxt.tolist() == [1, 0, 1, 0]
    mask, ts = b.track_plan([1280, 1024, 1281, 256], 256, pairs, nxt)
    assert mask.tolist() == [1, 1, 0, 1] and ts.tolist() == [12, 21, 0, 41]
    assert nxt.tolist() == [0, 1, 1, 1]
    single = np.int32([[7], [8]])
    n1 = np.zeros(2, np.int32)
    for _ in range(3):
        mask, ts = b.track_plan([512, 512], 256, single, n1)
        assert ts.tolist() == [7, 8] and n1.tolist() == [0, 0]
    with pytest.raises(b.RscError) as e:
        b.track_plan([256], 0, np.int32([[1, 2]]), np.zeros(1, np.int32))
    assert e.value.status == b.RSC_ERANGE
