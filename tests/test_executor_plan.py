"""The tile executor's plan on the CPU (no GPU needed): dependency inference
from tile accesses in program order, and the stream schedule with its
cross-stream waits.

Hand-built graphs pin the inference rules (read-after-write, write-after-read,
write-after-write) and the stream choices. Seeded random graphs are checked
against brute force: every pair of tasks that touch a common tile, one of them
writing it, must be ordered by the schedule (stream order plus event waits).
"""
import random

import pytest

from tile_task_transformer_gb300 import nnt

R, W, RW = 1, 2, 3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tile_task_transformer_gb300 import build
    build.build()  # host compile only; no GPU needed
    nnt.lib()


def test_chain_stays_on_one_stream():
    s, d, w = nnt.plan_schedule([[(0, W)], [(0, R), (1, W)], [(1, R)]], n_streams=2)
    assert d == [[], [0], [1]]
    assert s == [0, 0, 0]
    assert w == [[], [], []]


def test_war_waw_and_raw_dependencies():
    # 0 writes A; 1 and 2 read A; 3 writes A (after the writer and both readers);
    # 4 reads and writes A (after 3 only: the readers are covered by 3)
    s, d, w = nnt.plan_schedule([[(7, W)], [(7, R)], [(7, R)], [(7, W)], [(7, RW)]], n_streams=1)
    assert d == [[], [0], [0], [0, 1, 2], [3]]
    assert s == [0] * 5 and w == [[]] * 5


def test_independent_chains_use_two_streams_and_one_join():
    uses = [[(0, W)], [(1, W)], [(0, R), (2, W)], [(1, R), (3, W)], [(2, R), (3, R)]]
    s, d, w = nnt.plan_schedule(uses, n_streams=2)
    assert d == [[], [], [0], [1], [2, 3]]
    assert s == [0, 1, 0, 1, 1]  # the join continues the stream of its latest dependency
    assert w == [[], [], [], [], [2]]


def test_copy_tasks_and_stream_hints():
    uses = [[(0, W)], [(0, R), (1, W)], [(5, W)], [(1, R)]]
    s, d, w = nnt.plan_schedule(uses, n_streams=2, copy=[0, 1, 0, 0], hints=[-1, -1, 7, -1])
    assert s[1] == 2  # the copy stream follows the compute streams
    assert s[2] == 1  # hint clamped to the last compute stream
    assert w[1] == [0] and 1 in w[3]


def test_rejects_bad_modes_and_offsets():
    with pytest.raises(nnt.NNTError) as e:
        nnt.plan_schedule([[(0, 4)]], n_streams=1)
    assert e.value.status == nnt.ERR_INVALID_ARG
    with pytest.raises(nnt.NNTError):
        nnt.plan_schedule([[(0, W)]], n_streams=0)
    assert nnt.plan_schedule([], n_streams=3) == ([], [], [])


def _happens_before(streams, waits):
    """For each task, the set of tasks ordered before it by stream order and waits."""
    n = len(streams)
    last = {}
    hb = []
    for i in range(n):
        before = set()
        p = last.get(streams[i])
        if p is not None:
            before |= hb[p] | {p}
        for x in waits[i]:
            before |= hb[x] | {x}
        hb.append(before)
        last[streams[i]] = i
    return hb


@pytest.mark.parametrize("seed", range(40))
def test_random_graphs_order_every_conflict(seed):
    rng = random.Random(seed)
    n = rng.randint(1, 60)
    n_tiles = rng.randint(1, 12)
    n_streams = rng.randint(1, 4)
    uses = [[(rng.randrange(n_tiles), rng.choice((R, R, W, RW))) for _ in range(rng.randint(0, 4))]
            for _ in range(n)]
    copy = [int(rng.random() < 0.15) for _ in range(n)]
    hints = [rng.choice((-1, -1, -1, 0, 1, 5)) for _ in range(n)]
    s, d, w = nnt.plan_schedule(uses, n_streams, copy=copy, hints=hints)

    for i in range(n):
        if copy[i]:
            assert s[i] == n_streams
        elif hints[i] >= 0:
            assert s[i] == min(hints[i], n_streams - 1)
        else:
            assert 0 <= s[i] < n_streams
        assert d[i] == sorted(set(d[i])) and all(0 <= x < i for x in d[i])
        assert set(w[i]) <= set(d[i])

    def modes(i):
        m = {}
        for t, md in uses[i]:
            m[t] = m.get(t, 0) | md
        return m

    # every direct dependency shares a tile with the task, one of them writing it
    for i in range(n):
        mi = modes(i)
        for x in d[i]:
            mx = modes(x)
            assert any(t in mx and ((mi[t] | mx[t]) & W) for t in mi), (i, x)

    # every conflicting pair is ordered by the schedule
    hb = _happens_before(s, w)
    for i in range(n):
        mi = modes(i)
        for x in range(i):
            mx = modes(x)
            if any(t in mx and ((mi[t] | mx[t]) & W) for t in mi):
                assert x in hb[i], (seed, x, i)

    # no wait is implied by the stream order alone
    last = {}
    for i in range(n):
        p = last.get(s[i])
        for x in w[i]:
            assert p is None or x not in (hb[p] | {p}), (seed, i, x)
        last[s[i]] = i
