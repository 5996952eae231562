"""Semantic state rows and label ownership -- oracle, test infrastructure only.

Written from the rule stated in prose by "M7.6 - DeepSeek MTP: Sequential
Modules, Teacher Forcing, and Speculative Runtime" §0x04C (compile the rows
of a depth before gathering any tensor), with the counts of §0x05A and the
label ownership of "M7.4 - Multi-Token Prediction Foundations" §0x01A /
§0x03A (padded, packed batches).

The rule, restated.  Depth k gives a packed position i (its *base*) a state
when the k+1 teacher-forced inputs x_i, ..., x_{i+k} are all real tokens of
the segment that holds i.  The state is *supervised* when x_{i+k+1} is a real
token of that same segment as well; a state without a label is still kept,
because the next depth may need it.  The state of depth k is built from the
state of the same base at depth k-1, which must exist: it is looked up by
base and never replaced by a neighbouring row.

This module evaluates the rule through run lengths: for every position j,
``run[j]`` counts the consecutive real tokens j, j+1, ... that share j's
segment.  Base i then has a depth-k state iff run[i] >= k+1 and a label iff
run[i] >= k+2.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence


@dataclass(frozen=True)
class StateRow:
    """A depth-k state (M7.6 §0x04C).

    ``base``: packed position i the state belongs to; ``parent``: index of
    the same base in the previous depth's list of states (the physical row
    gathered as h^{k-1}); ``input_at``: i+k, the position whose token the
    depth embeds; ``label_at``: i+k+1 when that token supervises the state,
    else None; ``segment``: the segment id of i."""

    base: int
    parent: int
    input_at: int
    label_at: Optional[int]
    segment: int

    @property
    def supervised(self) -> bool:
        return self.label_at is not None


def _whole_number(v) -> bool:
    return isinstance(v, int) and not isinstance(v, bool)


def same_segment_runs(segment: Sequence[int], active: Sequence[bool]) -> list[int]:
    """run[j] = length of the stretch j, j+1, ... of real tokens that share
    the segment of j (0 when j itself is padding), computed right to left."""
    n = len(segment)
    run = [0] * n
    for j in reversed(range(n)):
        if not active[j]:
            continue
        joins_next = j + 1 < n and active[j + 1] and segment[j + 1] == segment[j]
        run[j] = run[j + 1] + 1 if joins_next else 1
    return run


def depth_states(segment: Sequence[int], active: Sequence[bool], depth: int,
                 parent_bases: Sequence[int]) -> list[StateRow]:
    """States of one packed stream at ``depth``, in base order (M7.6 §0x04C).

    ``parent_bases`` lists, in row order, the bases that hold a state at
    depth-1 (every position for depth 1, where h^0 covers the stream).
    Raises ValueError when the two per-position lists differ in length, when
    the depth is not an integer >= 1, when a parent base lies outside the
    stream or is listed twice, and when a base with support at this depth has
    no parent state (the page's rule forbids substituting another row)."""
    n = len(segment)
    if len(active) != n:
        raise ValueError("segment ids and activity flags must cover the same positions")
    if not _whole_number(depth) or depth < 1:
        raise ValueError(f"depth must be an integer >= 1, got {depth!r}")
    row_of_base: dict[int, int] = {}
    for row, b in enumerate(parent_bases):
        if not _whole_number(b) or not 0 <= b < n:
            raise ValueError(f"parent base {b!r} is not a position of the stream")
        if b in row_of_base:
            raise ValueError(f"parent base {b} appears more than once")
        row_of_base[b] = row

    run = same_segment_runs(segment, active)
    states = []
    for i, length in enumerate(run):
        if length <= depth:  # x_i..x_{i+depth} are not all in i's segment
            continue
        if i not in row_of_base:
            raise ValueError(f"base {i} has support at depth {depth} but no state at depth {depth - 1}")
        label = i + depth + 1 if length >= depth + 2 else None
        states.append(StateRow(base=i, parent=row_of_base[i], input_at=i + depth,
                               label_at=label, segment=int(segment[i])))
    return states


def states_all_depths(segment: Sequence[int], active: Sequence[bool], D: int) -> list[list[StateRow]]:
    """States of depths 1..D; each depth's bases are the next depth's parents
    (M7.6 §0x04C, §0x06A: compile, gather, run, repeat)."""
    parents = list(range(len(segment)))
    out = []
    for k in range(1, D + 1):
        states = depth_states(segment, active, k, parents)
        out.append(states)
        parents = [s.base for s in states]
    return out


def label_owned(active: Sequence[bool], segment: Sequence[int], t: int, k: int) -> bool:
    """Label ownership m^{(k)}_{t} = M_t * M_{t+k} * 1[G_t = G_{t+k}]
    (M7.4 §0x01A): source t owns the label k steps ahead."""
    if t + k >= len(active):
        return False
    return bool(active[t]) and bool(active[t + k]) and segment[t] == segment[t + k]


def horizon_counts(active_rows, segment_rows, K: int) -> list[int]:
    """Number of owned labels per horizon 1..K over a batch (M7.4 §0x01A)."""
    counts = []
    for k in range(1, K + 1):
        c = 0
        for act, seg in zip(active_rows, segment_rows):
            for t in range(len(act)):
                c += label_owned(act, seg, t, k)
        counts.append(c)
    return counts


def single_sequence_label_counts(T: int, D: int) -> list[int]:
    """|V_k| = max(T - k - 1, 0) for one unpadded length-T stream (M7.6 §0x05A)."""
    return [max(T - k - 1, 0) for k in range(1, D + 1)]
