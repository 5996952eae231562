"""Gradients of the MTP chain loss -- oracle, test infrastructure only.

The chain oracle's forward ("M7.6 - DeepSeek MTP: Sequential Modules, Teacher
Forcing, and Speculative Runtime" §0x03-§0x05, as restated in
``oracle.chain``) written a second time in float64 PyTorch CPU operations over
the same compiled compact rows, so that autograd returns the exact derivative
of the assembled loss L = L_main + Σ_k w_k L^(k) with respect to the main
model's hidden states h^0 and every weight: the shared embedding E and head
W_U (which receive the main term's and every depth's gradient, §0x05), the
final norm's gain, and each depth's fusion, block and norm weights.

Every step follows ``oracle.chain`` one to one (RMSNorm, rotate-half RoPE,
segment-causal attention, SwiGLU, "he" concatenation, normalised head,
log-sum-exp cross entropy, the reductions of ``oracle.chain.assemble_loss``);
there is no bf16 rounding (the derivative of the fp64 definition).

Pins (tests/test_oracle_grad.py): the loss equals ``oracle.chain``'s fp64
loss; central finite differences of ``oracle.chain``'s numpy forward agree
with the autograd gradient on sampled coordinates of every tensor; a depth's
weights get no gradient from the terms of shallower depths.
"""
from __future__ import annotations

import math

import numpy as np
import torch

from .chain import Dims, assemble_loss
from .rows import label_owned, states_all_depths

_F = torch.float64
PER_DEPTH = ("hnorm", "enorm", "eh_proj", "attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up",
             "w_down")
SHARED = ("embed", "head", "out_norm")


def _rmsnorm(z, g, eps):
    return g * z / torch.sqrt((z * z).mean(dim=-1, keepdim=True) + eps)


def _rope(x, positions, n_heads, head_dim, base):
    if base == 0:
        return x
    n = x.shape[0]
    half = head_dim // 2
    inv_freq = base ** (-2.0 * torch.arange(half, dtype=_F) / head_dim)
    ang = torch.as_tensor(np.asarray(positions), dtype=_F)[:, None] * inv_freq[None, :]
    cos, sin = torch.cos(ang)[:, None, :], torch.sin(ang)[:, None, :]
    xh = x.reshape(n, n_heads, head_dim)
    x1, x2 = xh[..., :half], xh[..., half:]
    return torch.cat([x1 * cos - x2 * sin, x2 * cos + x1 * sin], dim=-1).reshape(n, n_heads * head_dim)


def _attention(q, k, v, segments, bases, n_heads, head_dim):
    segments = torch.as_tensor(np.asarray(segments))
    bases = torch.as_tensor(np.asarray(bases))
    visible = (segments[None, :] == segments[:, None]) & (bases[None, :] <= bases[:, None])
    scale = 1.0 / math.sqrt(head_dim)
    outs = []
    for hh in range(n_heads):
        sl = slice(hh * head_dim, (hh + 1) * head_dim)
        s = (q[:, sl] @ k[:, sl].T) * scale
        s = s.masked_fill(~visible, -math.inf)
        outs.append(torch.softmax(s, dim=1) @ v[:, sl])
    return torch.cat(outs, dim=1)


def _module(prev, shifted, P, k, positions, segments, bases, dims: Dims):
    e = P["embed"][torch.as_tensor(np.asarray(shifted, dtype=np.int64))]
    c = torch.cat([_rmsnorm(prev, P["hnorm"][k], dims.eps), _rmsnorm(e, P["enorm"][k], dims.eps)], dim=1)
    u = c @ P["eh_proj"][k].T
    x = _rmsnorm(u, P["attn_norm"][k], dims.eps)
    q = _rope(x @ P["wq"][k].T, positions, dims.n_heads, dims.head_dim, dims.rope_base)
    kk = _rope(x @ P["wk"][k].T, positions, dims.n_heads, dims.head_dim, dims.rope_base)
    v = x @ P["wv"][k].T
    a = u + _attention(q, kk, v, segments, bases, dims.n_heads, dims.head_dim) @ P["wo"][k].T
    y = _rmsnorm(a, P["ffn_norm"][k], dims.eps)
    g = torch.nn.functional.silu(y @ P["w_gate"][k].T) * (y @ P["w_up"][k].T)
    return a + g @ P["w_down"][k].T


def _row_ce(h, labels, P, dims: Dims):
    z = _rmsnorm(h, P["out_norm"], dims.eps) @ P["head"].T
    return torch.logsumexp(z, dim=1) - z[torch.arange(len(labels)), torch.as_tensor(np.asarray(labels))]


def chain_loss_grads(tokens, seg, pos, h0, W, dims: Dims, lam=0.3, den="fixed", with_main=True,
                     depth_weights=None):
    """Loss and gradients of the chain (fp64).  W: numpy weight dict as for
    ``oracle.chain`` (per-depth lists).  Returns the assembled losses, the
    per-term sums and counts, ``dh0`` [B, T, d] and ``grads`` (same structure
    as W)."""
    tokens, seg, pos = np.asarray(tokens), np.asarray(seg), np.asarray(pos)
    B, T = tokens.shape
    D = dims.D
    P = {}
    for name in SHARED:
        P[name] = torch.tensor(np.asarray(W[name], dtype=np.float64), requires_grad=True)
    for name in PER_DEPTH:
        P[name] = [torch.tensor(np.asarray(W[name][k], dtype=np.float64), requires_grad=True) for k in range(D)]
    h0_t = torch.tensor(np.asarray(h0, dtype=np.float64), requires_grad=True)

    sums = [torch.zeros((), dtype=_F) for _ in range(D + 1)]
    counts = [0] * (D + 1)
    for b in range(B):
        tok = [int(v) for v in tokens[b]]
        sg = [int(v) for v in seg[b]]
        active = [s != -1 for s in sg]
        if with_main:
            main_rows = [t for t in range(T) if label_owned(active, sg, t, 1)]
            if main_rows:
                ell = _row_ce(h0_t[b][main_rows], [tok[t + 1] for t in main_rows], P, dims)
                sums[0] = sums[0] + ell.sum()
                counts[0] += len(main_rows)
        state = h0_t[b]
        for k, rows in enumerate(states_all_depths(sg, active, D)):
            if not rows:
                state = state[:0]
                continue
            prev = state[[r.parent for r in rows]]
            h = _module(prev, [tok[r.input_at] for r in rows], P, k,
                        pos[b][[r.base for r in rows]], [r.segment for r in rows], [r.base for r in rows], dims)
            state = h
            sup = [j for j, r in enumerate(rows) if r.supervised]
            if sup:
                ell = _row_ce(h[sup], [tok[rows[j].label_at] for j in sup], P, dims)
                sums[k + 1] = sums[k + 1] + ell.sum()
                counts[k + 1] += len(sup)

    out = assemble_loss(sums, counts, B * T, D, lam, den, with_main, depth_weights=depth_weights)
    total = out["loss_total"]
    total.backward()
    grads = {name: P[name].grad.numpy().copy() for name in SHARED}
    for name in PER_DEPTH:
        grads[name] = [p.grad.numpy().copy() if p.grad is not None else np.zeros(tuple(p.shape)) for p in P[name]]
    val = lambda t: float(t.detach()) if torch.is_tensor(t) else float(t)  # noqa: E731
    return {"loss_total": val(total), "loss_main": val(out["loss_main"]),
            "loss_mtp": [val(x) for x in out["loss_mtp"]], "sums": np.array([val(s) for s in sums]),
            "counts": np.array(counts), "dh0": h0_t.grad.numpy().copy(), "grads": grads}
