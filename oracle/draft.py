"""Decode-shaped MTP draft step -- oracle, test infrastructure only.

"M7.6 - DeepSeek MTP: Sequential Modules, Teacher Forcing, and Speculative
Runtime" §0x09: a carried-frontier round proposes one token from the saved
parent hidden state and the embedding of the pending frontier token, keeping
the draft distribution q for exact verification; §0x09A: the MTP block's
attention reads its own K/V cache.  Per request r the module of depth 1
(``oracle.chain``'s fusion and block pieces) runs on one new row whose
attention covers the cached keys/values [0, ctx_len_r) -- used as stored -- and
the new row itself at position pos_r; then q_r = softmax(W_U Norm_out(h)) and
the draw is the inverse CDF of q_r at u = word 2 of Philox4x32-10 with key
(seed) and counter (0, r, offset) (the verifier's stream uses words 0 and 1).

Multi-step drafting (recurrent reuse of the module, γ proposals) feeds each
step's output state and draw into the next step, with the step's key/value
row staged for the later steps' attention.

Parity status: pinned by the chain oracle -- with the cache holding a
segment's own rotated keys and values the draft state equals the chain's
depth-1 state of the next row and -log q of its label equals that row's loss
(tests/test_oracle_draft.py); q sums to one; the draw follows the verifier's
pinned inverse-CDF rule.  A round of gamma steps is pinned to the single step:
step s equals one draft step from the previous step's state and draw over the
cache extended by the staged rows.
"""
from __future__ import annotations

import math

import numpy as np

from .bf16 import round_bf16
from .chain import Dims, _f64, block_qkv, block_tail, fusion, rmsnorm
from .verify import inverse_cdf, philox4x32_10, uniform24


def draft_uniform(seed: int, offset: int, r: int, step: int = 0) -> float:
    """Uniform of the draw of request r at draft step `step`: word 2 of
    Philox4x32-10 at counter (step, r, offset lo, offset hi), key = seed."""
    seed, offset = int(seed), int(offset)
    w = philox4x32_10((int(step), r, offset & 0xFFFFFFFF, (offset >> 32) & 0xFFFFFFFF),
                      (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    return float(uniform24(w[2]))


def cached_attention(q, k_all, v_all, n_heads, head_dim):
    """softmax(q K^T / sqrt(hd)) V per head for one query row over all given keys."""
    out = np.empty(n_heads * head_dim)
    for hh in range(n_heads):
        sl = slice(hh * head_dim, (hh + 1) * head_dim)
        s = (k_all[:, sl] @ q[sl]) / math.sqrt(head_dim)
        s = np.exp(s - s.max())
        out[sl] = (s / s.sum()) @ v_all[:, sl]
    return out


def _module_row(parent, frontier, position, k_prev, v_prev, W, dims: Dims, rnd):
    """One new row of the depth-1 module: fusion of (parent, E[frontier]), the
    block with attention over the given earlier keys/values plus the row itself
    at `position`, the normalised head.  Returns (h, k, v, q distribution)."""
    WU = W["head"]
    u = fusion(_f64(parent)[None], [int(frontier)], W, 0, dims, rnd)
    q, k, v = block_qkv(u, W, 0, [int(position)], dims, rnd)
    k_all = np.concatenate([k_prev, k], axis=0)
    v_all = np.concatenate([v_prev, v], axis=0)
    o = rnd(cached_attention(q[0], k_all, v_all, dims.n_heads, dims.head_dim))[None]
    h = block_tail(u, o, W, 0, dims, rnd)
    x = rnd(rmsnorm(h, W["out_norm"], dims.eps))
    z = np.concatenate([x @ _f64(WU[v0:v0 + 16384]).T for v0 in range(0, WU.shape[0], 16384)], axis=1)[0]
    p = np.exp(z - z.max())
    p /= p.sum()
    return h[0], k[0], v[0], p


def draft_round(parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, W, dims: Dims, gamma, seed, offset,
                precision="bf16", requests=None, forced_y=None, forced_h=None):
    """gamma recurrent draft steps per request by reuse of one module (M7.6
    §0x09: the retained depth proposes the next token from its own output
    state).  Step s (0-based) runs on parent h_{s-1} and frontier y_{s-1}
    (h_{-1} = parent_hidden, y_{-1} = frontier) at position pos + s; its
    attention covers the cached rows [0, ctx_len), the rows staged by steps
    0..s-1 (their post-RoPE keys and values) and the row itself.  The draw y_s
    is the inverse CDF of q_s at draft_uniform(seed, offset, r, s).  With
    ``forced_y`` [R, gamma] the next step's frontier is forced_y[r][s] instead
    of the own draw (the draw and its margin are still reported); with
    ``forced_h`` [R, gamma, d] the next step's parent state is forced_h[r][s]
    instead of the own state (so each step can be compared on its own).

    Returns h [R', gamma, d], q [R', gamma, V], y and margin [R', gamma]."""
    rnd = round_bf16 if precision == "bf16" else (lambda a: a)
    R = len(frontier)
    requests = list(range(R)) if requests is None else list(requests)
    out = {"h": [], "q": [], "y": [], "margin": []}
    for r in requests:
        L = int(ctx_len[r])
        k_prev, v_prev = _f64(kv_k[r][:L]), _f64(kv_v[r][:L])
        parent, f = parent_hidden[r], int(frontier[r])
        hs, qs, ys, ms = [], [], [], []
        for step in range(int(gamma)):
            h, k, v, p = _module_row(parent, f, int(pos[r]) + step, k_prev, v_prev, W, dims, rnd)
            y, m = inverse_cdf(p, draft_uniform(seed, offset, r, step))
            hs.append(h)
            qs.append(p)
            ys.append(y)
            ms.append(m)
            k_prev = np.concatenate([k_prev, k[None]], axis=0)
            v_prev = np.concatenate([v_prev, v[None]], axis=0)
            parent = forced_h[r][step] if forced_h is not None else h
            f = int(forced_y[r][step]) if forced_y is not None else y
        out["h"].append(hs)
        out["q"].append(qs)
        out["y"].append(ys)
        out["margin"].append(ms)
    return {k: np.array(v) for k, v in out.items()}


def draft_step(parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, W, dims: Dims, seed, offset,
               precision="bf16", requests=None):
    """One draft step (a round of one): returns h [R', d], q [R', V] (fp64),
    y [R'] and the draw's CDF margin for the requested subset of requests."""
    r = draft_round(parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, W, dims, 1, seed, offset,
                    precision=precision, requests=requests)
    return {k: v[:, 0] for k, v in r.items()}
