"""Exact speculative verification -- oracle, test infrastructure only.

Restates the one-proposal selector of "M7.6 - DeepSeek MTP: Sequential
Modules, Teacher Forcing, and Speculative Runtime" §0x09 (accept y with
probability min(1, p[y]/q[y]); on rejection emit a correction drawn from the
normalised positive residual (p - q)+; on acceptance a bonus drawn from the
next target row; EOS and the output budget truncate before any bonus),
generalised to γ drafts by the left-to-right rule of the speculative-decoding
page (ailearn "投机解码", one round of standard speculative sampling: accept a
prefix, correct at the first rejection and drop the rest, or draw one extra
token from the target when all γ pass).

Uniforms come from Philox4x32-10 as published by Salmon, Moraes, Dror and
Shaw, "Parallel random numbers: as easy as 1, 2, 3" (SC'11): multipliers
0xD2511F53 / 0xCD9E8D57, Weyl key increments 0x9E3779B9 / 0xBB67AE85, ten
rounds.  Stream layout of this library: key = (seed_lo, seed_hi), counter =
(j, r, offset_lo, offset_hi) for draft position j of request r; word 0 is the
accept uniform of position j, word 1 the resample (or, at j = γ, bonus)
uniform; u = (w >> 8) * 2^-24.

Sampling a normalised distribution r / Σr with uniform u' picks the smallest
index v whose running sum exceeds u' * Σr (zero-mass entries are never
picked).  Everything here is fp64 from the fp32 inputs.
"""
from __future__ import annotations

import numpy as np

MASK32 = np.uint64(0xFFFFFFFF)
PHILOX_M0 = np.uint64(0xD2511F53)
PHILOX_M1 = np.uint64(0xCD9E8D57)
PHILOX_W0 = np.uint64(0x9E3779B9)
PHILOX_W1 = np.uint64(0xBB67AE85)

STATUS_OK = 0
STATUS_INVALID_DRAFT = 1
STATUS_ZERO_RESIDUAL = 2
STATUS_INVALID_PROBS = 3
STATUS_INVALID_BUDGET = 4


def philox4x32_10(ctr, key):
    """Philox4x32-10 on numpy arrays of 32-bit words held in uint64.

    ctr: 4 arrays (c0..c3), key: 2 arrays (k0, k1), broadcastable.  Each round
    multiplies c0 and c2 by the two constants (full 64-bit products), and
    forms (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2), hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)); the
    key is bumped by the Weyl constants between rounds."""
    c0, c1, c2, c3 = (np.asarray(c, dtype=np.uint64) & MASK32 for c in ctr)
    k0, k1 = (np.asarray(k, dtype=np.uint64) & MASK32 for k in key)
    for _ in range(10):
        prod0 = PHILOX_M0 * c0
        prod1 = PHILOX_M1 * c2
        hi0, lo0 = prod0 >> np.uint64(32), prod0 & MASK32
        hi1, lo1 = prod1 >> np.uint64(32), prod1 & MASK32
        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0
        k0 = (k0 + PHILOX_W0) & MASK32
        k1 = (k1 + PHILOX_W1) & MASK32
    return c0, c1, c2, c3


def uniform24(word):
    """u = (w >> 8) * 2^-24 in [0, 1)."""
    return (np.asarray(word, dtype=np.uint64) >> np.uint64(8)).astype(np.float64) * 2.0 ** -24


def verify_uniforms(seed: int, offset: int, r, j):
    """(accept uniform, resample/bonus uniform) of request r, position j."""
    seed = int(seed)
    offset = int(offset)
    key = (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)
    ctr = (j, r, offset & 0xFFFFFFFF, (offset >> 32) & 0xFFFFFFFF)
    w = philox4x32_10(ctr, key)
    return uniform24(w[0]), uniform24(w[1])


def inverse_cdf(weights, u):
    """Smallest v with Σ_{i<=v} w_i > u * Σ w (running sum in index order,
    fp64).  Returns (index, margin) where margin is the distance, relative to
    the total, from u * Σ w to the nearer running sum bounding the chosen
    index -- a draw with a tiny margin may legitimately flip under another
    summation order.  If rounding leaves no running sum above the target, the
    last index with positive weight is returned."""
    w = np.asarray(weights, dtype=np.float64)
    cs = np.cumsum(w)
    mass = cs[-1]
    target = u * mass
    v = int(np.searchsorted(cs, target, side="right"))
    if v >= len(w):
        v = int(np.nonzero(w > 0)[0][-1])
    lo = cs[v - 1] if v > 0 else 0.0
    margin = min(cs[v] - target, target - lo) / mass
    return v, margin


def _row_ok(row) -> bool:
    return bool(np.all(np.isfinite(row)) and np.all(row >= 0))


def verify_one(p, q, y, u_acc, u_res, eos=-1, remaining=None):
    """One request: p [γ+1, V], q [γ, V], y [γ]; uniforms u_acc[j], u_res[j].

    Returns dict(accepted=A, token=correction or bonus or -1, n_emit, status,
    margin) where the emitted tokens are y[0:A] followed by ``token`` when it
    is not -1.  ``margin`` is the smallest relative distance of a decision to
    its threshold (accept ratio or CDF boundary), for excluding knife-edge draws
    from bit-exact comparisons."""
    gamma, V = q.shape
    if remaining is None:
        remaining = gamma + 1
    res = {"accepted": 0, "token": -1, "n_emit": 0, "status": STATUS_OK, "margin": np.inf}
    if remaining < 1:
        res["status"] = STATUS_INVALID_BUDGET
        return res
    n_out = 0
    for j in range(gamma):
        yj = int(y[j])
        if yj < 0 or yj >= V:
            res["status"] = STATUS_INVALID_DRAFT
            return res
        pj, qj = float(p[j, yj]), float(q[j, yj])
        if not (np.isfinite(pj) and np.isfinite(qj) and pj >= 0 and qj >= 0):
            res["status"] = STATUS_INVALID_PROBS
            return res
        if qj <= 0:
            res["status"] = STATUS_INVALID_DRAFT
            return res
        ratio = min(1.0, pj / qj)
        res["margin"] = min(res["margin"], abs(u_acc[j] - ratio))
        if u_acc[j] < ratio:
            n_out += 1
            res["accepted"] = n_out
            res["n_emit"] = n_out
            if n_out == remaining or yj == eos:
                return res
            continue
        prow = np.asarray(p[j], dtype=np.float64)
        qrow = np.asarray(q[j], dtype=np.float64)
        if not (_row_ok(prow) and _row_ok(qrow)):
            res["status"] = STATUS_INVALID_PROBS
            return res
        residual = np.maximum(prow - qrow, 0.0)
        if not residual.sum() > 0:
            res["status"] = STATUS_ZERO_RESIDUAL
            return res
        c, m = inverse_cdf(residual, u_res[j])
        res["margin"] = min(res["margin"], m)
        res["token"] = c
        res["n_emit"] = n_out + 1
        return res
    bonus_row = np.asarray(p[gamma], dtype=np.float64)
    if not _row_ok(bonus_row):
        res["status"] = STATUS_INVALID_PROBS
        return res
    if not bonus_row.sum() > 0:
        res["status"] = STATUS_ZERO_RESIDUAL
        return res
    b, m = inverse_cdf(bonus_row, u_res[gamma])
    res["margin"] = min(res["margin"], m)
    res["token"] = b
    res["n_emit"] = n_out + 1
    return res


def spec_verify(p, q, draft, seed, offset, eos=None, remaining=None):
    """Batched verification: p [R, γ+1, V], q [R, γ, V], draft [R, γ].
    Uniforms from Philox4x32-10 with this library's stream layout.  Returns
    arrays accepted, token, n_emit, status and margin of length R."""
    p = np.asarray(p)
    q = np.asarray(q)
    draft = np.asarray(draft)
    R, gamma = draft.shape
    js = np.arange(gamma + 1)
    out = {k: np.zeros(R, dtype=np.int64) for k in ("accepted", "token", "n_emit", "status")}
    out["margin"] = np.zeros(R)
    for r in range(R):
        ua, ur = verify_uniforms(seed, offset, r, js)
        res = verify_one(p[r], q[r], draft[r], ua, ur,
                         eos=-1 if eos is None else int(eos[r]),
                         remaining=None if remaining is None else int(remaining[r]))
        for k in out:
            out[k][r] = res[k]
    return out
