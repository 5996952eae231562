"""Pins of the oracle's row compiler and label ownership against the pages'
worked fixtures (tests/golden) and against each other."""
import itertools

import numpy as np
import pytest

from conftest import read_golden
from oracle.rows import (depth_states, horizon_counts, label_owned, same_segment_runs,
                         single_sequence_label_counts, states_all_depths)


def ints(vals):
    return [int(v) for v in vals]


def test_two_segment_fixture():
    f, _ = read_golden("rows_two_segments.txt")
    seg = ints(f["segments"])
    n = len(seg)
    valid = [True] * n
    d1 = depth_states(seg, valid, 1, list(range(n)))
    assert [r.base for r in d1] == ints(f["depth1_state_bases"])
    assert [r.base for r in d1 if r.supervised] == ints(f["depth1_supervised_bases"])
    d2 = depth_states(seg, valid, 2, [r.base for r in d1])
    assert [r.base for r in d2] == ints(f["depth2_state_bases"])
    assert [r.parent for r in d2] == ints(f["depth2_previous_physical_rows"])
    assert [r.base for r in d2 if r.supervised] == ints(f["depth2_supervised_bases"])


def test_packed_label_ownership_counts():
    f, _ = read_golden("label_ownership_packed.txt")
    seg_rows = [ints(f["segment_row0"]), ints(f["segment_row1"])]
    act_rows = [[s != -1 for s in row] for row in seg_rows]
    assert horizon_counts(act_rows, seg_rows, 3) == ints(f["owned_counts_h1_h2_h3"])
    assert sum(horizon_counts(act_rows, seg_rows, 3)) == int(f["owned_total"][0])
    S = len(seg_rows[0])
    assert [len(seg_rows) * (S - k) for k in (1, 2, 3)] == ints(f["shape_only_counts_h1_h2_h3"])
    # MTP depth k is supervised at horizon k+1 and has state at horizon k.
    n_state, n_loss = [0, 0], [0, 0]
    for seg, act in zip(seg_rows, act_rows):
        for k, rows in enumerate(states_all_depths(seg, act, 2)):
            n_state[k] += len(rows)
            n_loss[k] += sum(r.supervised for r in rows)
    assert n_state == [9, 6]
    assert n_loss == [6, 3]


def test_single_sequence_counts_and_polynomial():
    f, _ = read_golden("label_counts_single_sequence.txt")
    T, D = int(f["T"][0]), int(f["D"][0])
    assert single_sequence_label_counts(T, D) == ints(f["counts"])
    assert D * (T - 1) - D * (D + 1) // 2 == int(f["unrestricted_polynomial"][0])
    per_depth = states_all_depths([0] * T, [True] * T, D)
    assert [sum(r.supervised for r in rows) for rows in per_depth] == ints(f["counts"])
    for T in range(2, 12):
        for D in range(1, T):
            per_depth = states_all_depths([0] * T, [True] * T, D)
            n = sum(sum(r.supervised for r in rows) for rows in per_depth)
            assert n == D * (T - 1) - D * (D + 1) // 2


def test_depth_two_rows_A_to_F():
    f, _ = read_golden("depth_two_rows_AF.txt")
    names = f["tokens"]
    n = len(names)
    per_depth = states_all_depths([0] * n, [True] * n, 2)
    for k, key in enumerate(("depth1", "depth2")):
        want = [tuple(t.split(",")) for t in f[key]]
        got = [(names[r.base], names[r.input_at], names[r.label_at])
               for r in per_depth[k] if r.supervised]
        assert got == want


def test_tiny_config_counts():
    """Tiny fp32 workload (row 0 active t<=10, row 1 split at t=6): main
    pairs 24, depth-1 state rows 24, depth-1 loss rows 21."""
    seg_rows = [[0] * 11 + [-1] * 5, [0] * 6 + [1] * 10]
    act_rows = [[s != -1 for s in r] for r in seg_rows]
    assert horizon_counts(act_rows, seg_rows, 1) == [24]
    n_state = n_loss = 0
    for seg, act in zip(seg_rows, act_rows):
        rows = depth_states(seg, act, 1, list(range(16)))
        n_state += len(rows)
        n_loss += sum(r.supervised for r in rows)
    assert (n_state, n_loss) == (24, 21)


def brute_force_segments(rng, n):
    seg, sid, t = [], 0, 0
    while t < n:
        L = int(rng.integers(1, 6))
        s = -1 if rng.random() < 0.2 else sid
        seg += [s] * L
        sid += 1
        t += L
    return seg[:n]


@pytest.mark.parametrize("seed", range(30))
def test_compiler_matches_label_ownership(seed):
    """The row compiler (all of base..base+k active and same segment) and the
    label-ownership mask (ends active, same segment) agree on contiguous
    segments: state(k) = owned(k), loss(k) = owned(k+1)."""
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 25))
    seg = brute_force_segments(rng, n)
    act = [s != -1 for s in seg]
    per_depth = states_all_depths(seg, act, 4)
    for k, rows in enumerate(per_depth, start=1):
        state = {r.base for r in rows}
        loss = {r.base for r in rows if r.supervised}
        assert state == {t for t in range(n) if label_owned(act, seg, t, k)}
        assert loss == {t for t in range(n) if label_owned(act, seg, t, k + 1)}
        for r in rows:  # physical row of the same base one depth up
            assert r.input_at == r.base + k
            if r.supervised:
                assert r.label_at == r.base + k + 1


def brute_force_states(seg, act, k):
    """Direct reading of the rule: every input i..i+k real and in i's segment."""
    n = len(seg)
    return [i for i in range(n - k)
            if all(act[j] and seg[j] == seg[i] for j in range(i, i + k + 1))]


@pytest.mark.parametrize("seed", range(20))
def test_runs_match_direct_rule(seed):
    """The run-length evaluation equals the rule read literally (all inputs
    base..base+k present in the base's segment), including streams whose
    segment ids repeat after padding or another segment."""
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 30))
    seg = [int(v) for v in rng.integers(0, 3, n)]
    act = [bool(v) for v in rng.random(n) > 0.15]
    run = same_segment_runs(seg, act)
    for j in range(n):
        want = 0
        while j + want < n and act[j + want] and seg[j + want] == seg[j]:
            want += 1
        assert run[j] == want
    parents = list(range(n))
    for k in range(1, 5):
        rows = depth_states(seg, act, k, parents)
        assert [r.base for r in rows] == brute_force_states(seg, act, k)
        assert [r.base for r in rows if r.supervised] == brute_force_states(seg, act, k + 1)
        assert all(parents[r.parent] == r.base for r in rows)
        parents = [r.base for r in rows]


def test_compiler_errors():
    with pytest.raises(ValueError):
        depth_states([0], [True, True], 1, [0, 1])
    for bad in (0, -1, True, 1.0):
        with pytest.raises(ValueError):
            depth_states([0, 0, 0], [True] * 3, bad, [0, 1, 2])
    with pytest.raises(ValueError):
        depth_states([0, 0, 0], [True] * 3, 1, [0, 0])
    with pytest.raises(ValueError):
        depth_states([0, 0, 0], [True] * 3, 1, [0, 3])
    with pytest.raises(ValueError):  # base 1 has support but no predecessor
        depth_states([0, 0, 0], [True] * 3, 1, [0])
