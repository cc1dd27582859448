"""Dynamic offloading of free pages: the three-position state machine (CPU only).

LMCache paper, dynamic offloading mechanism and Figure 7: start (next free page
handed out), current (pages before it are backed up to CPU), end (pages before
it are planned); start <= current <= end always; states #1 init, #2 in
progress, #3 query arrives (end moves forward by the pages taken), #4 steady.
"""
import numpy as np
import pytest

from paged_kv_cache_lmkv_gb300 import build, lmkv


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    lmkv.load()


def test_figure7_states():
    o = lmkv.Offload(num_free=100, window=20)
    s = o.state
    assert (s.start, s.current, s.end) == (0, 0, 20)            # #1: start == current
    first, count = o.plan(8)
    assert (first, count) == (0, 8)
    o.copied(8)
    assert s.start < s.current < s.end                           # #2: current moves toward end
    g, stalled = o.allocate(5)                                   # #3: a query takes 5 pages
    assert (g, stalled) == (5, 0)
    assert (s.start, s.current, s.end) == (5, 8, 25)             #     end moved forward by 5
    while True:
        first, count = o.plan(7)
        if count == 0:
            break
        o.copied(count)
    assert s.current == s.end == 25                              # #4: steady


def test_stall_when_not_backed_up():
    o = lmkv.Offload(num_free=50, window=10)
    o.copied(o.plan(3)[1])
    g, stalled = o.allocate(7)
    assert (g, stalled) == (3, 4)
    assert o.state.start == o.state.current == 3


def test_random_sequences_keep_the_invariant_and_hand_out_backed_up_pages():
    rng = np.random.default_rng(0)
    for trial in range(30):
        window = int(rng.integers(0, 40))
        o = lmkv.Offload(num_free=int(rng.integers(0, 60)), window=window)
        backed_up, handed = set(), []
        for _ in range(200):
            op = rng.integers(0, 4)
            if op == 0:
                first, count = o.plan(int(rng.integers(0, 10)))
                backed_up |= set(range(first, first + count))
                o.copied(count)
            elif op == 1:
                start = o.state.start
                g, stalled = o.allocate(int(rng.integers(0, 12)))
                handed.extend(range(start, start + g))
            elif op == 2:
                o.add_free(int(rng.integers(0, 8)))
            else:
                with pytest.raises(lmkv.LmkvError):
                    o.copied(o.state.end - o.state.current + 1)
            s = o.state
            assert 0 <= s.start <= s.current <= s.end <= s.limit
            assert s.end - s.start <= window
            assert s.current == len(backed_up) or backed_up == set(range(s.current))
        assert set(handed) <= backed_up                          # only backed-up pages go out
        assert handed == list(range(len(handed)))                # in free-list order


def test_larger_window_fewer_stalls_more_copies():
    """The trade-off the mechanism names: a larger window copies more pages and
    makes queries wait less (deterministic arrival pattern, fixed copy rate)."""
    rng = np.random.default_rng(1)
    wants = rng.integers(0, 12, 400)
    frees = rng.integers(0, 12, 400)
    results = []
    for window in (0, 8, 32, 128):
        o = lmkv.Offload(num_free=64, window=window)
        stalled_total, waiting = 0, 0
        for want, freed in zip(wants, frees):
            o.copied(o.plan(4)[1])                              # 4 pages per step of copy bandwidth
            g, stalled = o.allocate(int(want) + waiting)
            waiting = stalled
            stalled_total += stalled
            o.add_free(int(freed))
        results.append((window, stalled_total, o.state.current))
    stalls = [r[1] for r in results]
    copies = [r[2] for r in results]
    assert stalls == sorted(stalls, reverse=True) and stalls[0] > stalls[-1]
    assert copies == sorted(copies)
