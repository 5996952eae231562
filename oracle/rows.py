"""Semantic rows and label ownership -- oracle, test infrastructure only.

Follows "M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and
Speculative Runtime" §0x04C (compile semantic rows before gathering tensors),
§0x05A (label counts) and "M7.4 - Multi-Token Prediction Foundations" §0x01A /
§0x03A (label ownership on padded, packed batches).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence


@dataclass(frozen=True)
class MTPRow:
    """One state row of depth k (M7.6 §0x04C).

    ``base`` is the semantic address i of the row in the packed stream;
    ``previous_depth_row`` is the physical row of the same base in the
    previous depth's tensor; the row reads token x_{i+k}
    (``shifted_token_index``) and, when ``loss_valid``, is supervised by
    x_{i+k+1} (``label_index``)."""

    base: int
    previous_depth_row: int
    shifted_token_index: int
    label_index: Optional[int]
    loss_valid: bool
    position: int
    segment: int


def _is_int(v) -> bool:
    return isinstance(v, int) and not isinstance(v, bool)


def compile_mtp_rows(tokens: Sequence[int], segment_ids: Sequence[int],
                     valid: Sequence[bool], depth: int,
                     previous_bases: Sequence[int]) -> list[MTPRow]:
    """State rows of one packed stream at ``depth`` (M7.6 §0x04C).

    A base i has state support at depth k when every teacher-forced input
    i, i+1, ..., i+k is active and lies in the segment of i.  Such a row keeps
    its state even without a label; it is supervised only if x_{i+k+1} exists,
    is active and belongs to the same segment.  The predecessor state must be
    present among ``previous_bases``; a missing one is an error, never a
    fallback to another row.  Raises ``ValueError`` on misaligned inputs, a
    non-positive depth, out-of-range or duplicate previous bases.
    """
    n = len(tokens)
    if len(segment_ids) != n or len(valid) != n:
        raise ValueError("unaligned packed inputs")
    if not _is_int(depth) or depth < 1:
        raise ValueError("depth must be positive")
    for b in previous_bases:
        if not _is_int(b) or b < 0 or b >= n:
            raise ValueError("invalid previous base")
    physical_row_of = {}
    for row, b in enumerate(previous_bases):
        if b in physical_row_of:
            raise ValueError("duplicate previous base")
        physical_row_of[b] = row

    out: list[MTPRow] = []
    for base in range(n):
        shifted = base + depth
        if shifted >= n:
            continue
        own_segment = segment_ids[base]
        supported = True
        for j in range(base, shifted + 1):
            if not valid[j] or segment_ids[j] != own_segment:
                supported = False
                break
        if not supported:
            continue
        if base not in physical_row_of:
            raise ValueError("required predecessor state is missing")
        label = shifted + 1
        has_label = label < n and bool(valid[label]) and segment_ids[label] == own_segment
        out.append(MTPRow(base=base, previous_depth_row=physical_row_of[base],
                          shifted_token_index=shifted,
                          label_index=label if has_label else None,
                          loss_valid=has_label, position=base, segment=own_segment))
    return out


def compile_all_depths(tokens, segment_ids, valid, D: int) -> list[list[MTPRow]]:
    """Rows of depths 1..D, carrying each depth's bases forward as the next
    depth's ``previous_bases`` (M7.6 §0x04C, §0x06A)."""
    bases = list(range(len(tokens)))
    per_depth = []
    for k in range(1, D + 1):
        rows = compile_mtp_rows(tokens, segment_ids, valid, k, bases)
        per_depth.append(rows)
        bases = [r.base for r in rows]
    return per_depth


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
