"""Pins of the oracle's row compiler and label ownership against the pages'
worked fixtures (tests/golden) and against each other."""
import itertools

import numpy as np
import pytest

from conftest import read_golden
from oracle.rows import (compile_all_depths, compile_mtp_rows, horizon_counts,
                         label_owned, single_sequence_label_counts)


def ints(vals):
    return [int(v) for v in vals]


def test_two_segment_fixture():
    f, _ = read_golden("rows_two_segments.txt")
    seg = ints(f["segments"])
    n = len(seg)
    tokens = list(range(100, 100 + n))
    valid = [True] * n
    d1 = compile_mtp_rows(tokens, seg, valid, 1, list(range(n)))
    assert [r.base for r in d1] == ints(f["depth1_state_bases"])
    assert [r.base for r in d1 if r.loss_valid] == ints(f["depth1_supervised_bases"])
    d2 = compile_mtp_rows(tokens, seg, valid, 2, [r.base for r in d1])
    assert [r.base for r in d2] == ints(f["depth2_state_bases"])
    assert [r.previous_depth_row for r in d2] == ints(f["depth2_previous_physical_rows"])
    assert [r.base for r in d2 if r.loss_valid] == ints(f["depth2_supervised_bases"])


def test_packed_label_ownership_counts():
    f, _ = read_golden("label_ownership_packed.txt")
    seg_rows = [ints(f["segment_row0"]), ints(f["segment_row1"])]
    act_rows = [[s != -1 for s in row] for row in seg_rows]
    assert horizon_counts(act_rows, seg_rows, 3) == ints(f["owned_counts_h1_h2_h3"])
    assert sum(horizon_counts(act_rows, seg_rows, 3)) == int(f["owned_total"][0])
    S = len(seg_rows[0])
    assert [len(seg_rows) * (S - k) for k in (1, 2, 3)] == ints(f["shape_only_counts_h1_h2_h3"])
    # MTP depth k is supervised at horizon k+1 and has state at horizon k.
    toks = [ints(f["tokens_row0"]), ints(f["tokens_row1"])]
    n_state, n_loss = [0, 0], [0, 0]
    for tok, seg, act in zip(toks, seg_rows, act_rows):
        for k, rows in enumerate(compile_all_depths(tok, seg, act, 2)):
            n_state[k] += len(rows)
            n_loss[k] += sum(r.loss_valid for r in rows)
    assert n_state == [9, 6]
    assert n_loss == [6, 3]


def test_single_sequence_counts_and_polynomial():
    f, _ = read_golden("label_counts_single_sequence.txt")
    T, D = int(f["T"][0]), int(f["D"][0])
    assert single_sequence_label_counts(T, D) == ints(f["counts"])
    assert D * (T - 1) - D * (D + 1) // 2 == int(f["unrestricted_polynomial"][0])
    per_depth = compile_all_depths(list(range(T)), [0] * T, [True] * T, D)
    assert [sum(r.loss_valid for r in rows) for rows in per_depth] == ints(f["counts"])
    for T in range(2, 12):
        for D in range(1, T):
            per_depth = compile_all_depths(list(range(T)), [0] * T, [True] * T, D)
            n = sum(sum(r.loss_valid for r in rows) for rows in per_depth)
            assert n == D * (T - 1) - D * (D + 1) // 2


def test_depth_two_rows_A_to_F():
    f, _ = read_golden("depth_two_rows_AF.txt")
    names = f["tokens"]
    n = len(names)
    per_depth = compile_all_depths(list(range(n)), [0] * n, [True] * n, 2)
    for k, key in enumerate(("depth1", "depth2")):
        want = [tuple(t.split(",")) for t in f[key]]
        got = [(names[r.base], names[r.shifted_token_index], names[r.label_index])
               for r in per_depth[k] if r.loss_valid]
        assert got == want


def test_tiny_config_counts():
    """Tiny fp32 workload (row 0 active t<=10, row 1 split at t=6): main
    pairs 24, depth-1 state rows 24, depth-1 loss rows 21."""
    seg_rows = [[0] * 11 + [-1] * 5, [0] * 6 + [1] * 10]
    act_rows = [[s != -1 for s in r] for r in seg_rows]
    assert horizon_counts(act_rows, seg_rows, 1) == [24]
    n_state = n_loss = 0
    for seg, act in zip(seg_rows, act_rows):
        rows = compile_mtp_rows([0] * 16, seg, act, 1, list(range(16)))
        n_state += len(rows)
        n_loss += sum(r.loss_valid for r in rows)
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
    per_depth = compile_all_depths([0] * n, seg, act, 4)
    for k, rows in enumerate(per_depth, start=1):
        state = {r.base for r in rows}
        loss = {r.base for r in rows if r.loss_valid}
        assert state == {t for t in range(n) if label_owned(act, seg, t, k)}
        assert loss == {t for t in range(n) if label_owned(act, seg, t, k + 1)}
        for r in rows:  # physical row of the same base one depth up
            assert r.shifted_token_index == r.base + k
            if r.loss_valid:
                assert r.label_index == r.base + k + 1


def test_compiler_errors():
    with pytest.raises(ValueError):
        compile_mtp_rows([1, 2], [0], [True, True], 1, [0, 1])
    for bad in (0, -1, True, 1.0):
        with pytest.raises(ValueError):
            compile_mtp_rows([1, 2, 3], [0, 0, 0], [True] * 3, bad, [0, 1, 2])
    with pytest.raises(ValueError):
        compile_mtp_rows([1, 2, 3], [0, 0, 0], [True] * 3, 1, [0, 0])
    with pytest.raises(ValueError):
        compile_mtp_rows([1, 2, 3], [0, 0, 0], [True] * 3, 1, [0, 3])
    with pytest.raises(ValueError):  # base 1 has support but no predecessor
        compile_mtp_rows([1, 2, 3], [0, 0, 0], [True] * 3, 1, [0])
