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

Parity status: pinned by the chain oracle -- with the cache holding a
segment's own rotated keys and values the draft state equals the chain's
depth-1 state of the next row and -log q of its label equals that row's loss
(tests/test_oracle_draft.py); q sums to one; the draw follows the verifier's
pinned inverse-CDF rule.
"""
from __future__ import annotations

import math

import numpy as np

from .bf16 import round_bf16
from .chain import Dims, _f64, block_qkv, block_tail, fusion, rmsnorm
from .verify import inverse_cdf, philox4x32_10, uniform24


def draft_uniform(seed: int, offset: int, r: int) -> float:
    seed, offset = int(seed), int(offset)
    w = philox4x32_10((0, r, offset & 0xFFFFFFFF, (offset >> 32) & 0xFFFFFFFF),
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


def draft_step(parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, W, dims: Dims, seed, offset,
               precision="bf16", requests=None):
    """Returns h [R', d], q [R', V] (fp64), y [R'] and the draw's CDF margin for
    the requested subset of requests (all by default)."""
    rnd = round_bf16 if precision == "bf16" else (lambda a: a)
    R = len(frontier)
    requests = list(range(R)) if requests is None else list(requests)
    WU = W["head"]
    out = {"h": [], "q": [], "y": [], "margin": []}
    for r in requests:
        u = fusion(_f64(parent_hidden[r])[None], [int(frontier[r])], W, 0, dims, rnd)
        q, k, v = block_qkv(u, W, 0, [int(pos[r])], dims, rnd)
        L = int(ctx_len[r])
        k_all = np.concatenate([_f64(kv_k[r][:L]), k], axis=0)
        v_all = np.concatenate([_f64(kv_v[r][:L]), v], axis=0)
        o = rnd(cached_attention(q[0], k_all, v_all, dims.n_heads, dims.head_dim))[None]
        h = block_tail(u, o, W, 0, dims, rnd)
        x = rnd(rmsnorm(h, W["out_norm"], dims.eps))
        z = np.concatenate([x @ _f64(WU[v0:v0 + 16384]).T for v0 in range(0, WU.shape[0], 16384)], axis=1)[0]
        p = np.exp(z - z.max())
        p /= p.sum()
        y, m = inverse_cdf(p, draft_uniform(seed, offset, r))
        out["h"].append(h[0])
        out["q"].append(p)
        out["y"].append(y)
        out["margin"].append(m)
    return {k: np.array(v) for k, v in out.items()}
