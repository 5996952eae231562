"""Teacher-forced sequential MTP chain and its loss -- oracle, test
infrastructure only.

A plain fp64 restatement of "M7.6 - DeepSeek MTP: Sequential Modules, Teacher
Forcing, and Speculative Runtime":

* §0x03 / §0x03C: h̄ = RMSNorm_h(h^{k-1}), ē = RMSNorm_e(E(x_{i+k})),
  c = [h̄; ē], u = M_k c, then one pre-norm block
  a = u + Attn(Norm_a u; causal), h^k = a + FFN(Norm_f a);
* §0x03 / §0x04B: shared head p = softmax(W_U Norm_out(h^k)), the state handed
  to the next depth being the pre-final-norm h^k;
* §0x04C / §0x06A: the rows of each depth are compiled first
  (``oracle.rows.depth_states``), previous states are gathered by
  physical row, attention is restricted to the same segment and to earlier
  bases;
* §0x05: per-depth loss with the fixed denominator or the masked mean, and
  L = L_main + (λ/D) Σ_k L^(k);
* "M7.4 - Multi-Token Prediction Foundations" §0x06F: row cross-entropy as
  -z_target + max + log Σ exp(z - max).

Readings where the pages leave the step open (the pages defer the block's
MLA/MoE internals): the block is dense multi-head causal attention with RoPE
(rotate-half, base ``rope_base``, position = index within the segment) and a
SwiGLU FFN silu(y W_g^T) * (y W_u^T) W_d^T; no biases; RMSNorm epsilon 1e-6.

``precision="bf16"`` rounds to the bf16 grid at exactly the points where a
bf16 program stores a tensor (c, u, the normalised block inputs, q/k/v after
RoPE, the attention output, a, the SwiGLU product, h^k and the normalised head
input); everything between those points is fp64.  ``precision="f64"`` rounds
nowhere.

Parity status: components pinned (tests/test_oracle_chain.py); the composed
chain has no printed numeric output on the pages -- parity unpinned beyond the
component pins, the packing invariance and the causal-dependency checks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np

from .bf16 import round_bf16
from .rows import label_owned, states_all_depths


@dataclass(frozen=True)
class Dims:
    n_heads: int
    head_dim: int
    D: int
    eps: float = 1e-6
    rope_base: float = 10000.0


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def rmsnorm(z, g, eps):
    """g ⊙ z / sqrt(mean(z²) + ε) over the last axis (M7.6 §0x03C)."""
    z = _f64(z)
    return _f64(g) * z / np.sqrt(np.mean(z * z, axis=-1, keepdims=True) + eps)


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(x, positions, n_heads, head_dim, base):
    """Rotate-half rotary embedding of each head: pair (j, j + hd/2) rotated by
    angle position * base^(-2j/hd).  ``base == 0`` disables it."""
    x = _f64(x)
    if base == 0:
        return x
    n = x.shape[0]
    half = head_dim // 2
    inv_freq = base ** (-2.0 * np.arange(half, dtype=np.float64) / head_dim)
    ang = _f64(positions)[:, None] * inv_freq[None, :]
    cos, sin = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    xh = x.reshape(n, n_heads, head_dim)
    x1, x2 = xh[..., :half], xh[..., half:]
    out = np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)
    return out.reshape(n, n_heads * head_dim)


def segment_causal_attention(q, k, v, segments, bases, n_heads, head_dim):
    """softmax(q k^T / sqrt(hd)) v per head, where row i sees row j only when
    both lie in the same segment and base_j <= base_i (M7.6 §0x04C: the
    segment rule restricts the attention graph as well as the rows)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    segments = np.asarray(segments)
    bases = np.asarray(bases)
    visible = (segments[None, :] == segments[:, None]) & (bases[None, :] <= bases[:, None])
    n = q.shape[0]
    out = np.empty((n, n_heads * head_dim))
    scale = 1.0 / math.sqrt(head_dim)
    for hh in range(n_heads):
        sl = slice(hh * head_dim, (hh + 1) * head_dim)
        s = (q[:, sl] @ k[:, sl].T) * scale
        s = np.where(visible, s, -np.inf)
        s = s - s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        out[:, sl] = p @ v[:, sl]
    return out


def block_qkv(u, W, k, positions, dims: Dims, rnd):
    """Attention inputs of the block: x = Norm_a(u); q, k after RoPE, v."""
    x = rnd(rmsnorm(u, W["attn_norm"][k], dims.eps))
    q = rnd(rope(x @ _f64(W["wq"][k]).T, positions, dims.n_heads, dims.head_dim, dims.rope_base))
    kk = rnd(rope(x @ _f64(W["wk"][k]).T, positions, dims.n_heads, dims.head_dim, dims.rope_base))
    v = rnd(x @ _f64(W["wv"][k]).T)
    return q, kk, v


def block_tail(u, o, W, k, dims: Dims, rnd):
    """a = u + o W_o^T; h = a + SwiGLU(Norm_f(a)) (M7.6 §0x03C)."""
    a = rnd(u + _f64(o) @ _f64(W["wo"][k]).T)
    y = rnd(rmsnorm(a, W["ffn_norm"][k], dims.eps))
    g = rnd(silu(y @ _f64(W["w_gate"][k]).T) * (y @ _f64(W["w_up"][k]).T))
    return rnd(a + g @ _f64(W["w_down"][k]).T)


def transformer_block(u, W, k, positions, segments, bases, dims: Dims, rnd, return_kv=False):
    """Pre-norm block of depth k (M7.6 §0x03C):
    a = u + Attention(Norm_a(u)); h = a + FFN(Norm_f(a)).  With
    ``return_kv`` the rotated keys and the values are returned as well."""
    q, kk, v = block_qkv(u, W, k, positions, dims, rnd)
    o = rnd(segment_causal_attention(q, kk, v, segments, bases, dims.n_heads, dims.head_dim))
    h = block_tail(u, o, W, k, dims, rnd)
    return (h, kk, v) if return_kv else h


def fusion(prev_hidden, shifted_tokens, W, k, dims, rnd):
    """u = M_k [RMSNorm_h(h^{k-1}); RMSNorm_e(E(x))] (M7.6 §0x03)."""
    e = _f64(W["embed"][np.asarray(shifted_tokens)])
    h_bar = rmsnorm(prev_hidden, W["hnorm"][k], dims.eps)
    e_bar = rmsnorm(e, W["enorm"][k], dims.eps)
    c = rnd(np.concatenate([h_bar, e_bar], axis=1))
    return rnd(c @ _f64(W["eh_proj"][k]).T)


def mtp_module(prev_hidden, shifted_tokens, W, k, positions, segments, bases, dims, rnd, return_kv=False):
    """One MTP module (M7.6 §0x03): normalise both paths, concatenate in
    hidden-then-embedding order, project 2d -> d, run the block."""
    u = fusion(prev_hidden, shifted_tokens, W, k, dims, rnd)
    return transformer_block(u, W, k, positions, segments, bases, dims, rnd, return_kv=return_kv)


def row_cross_entropy(h, labels, W, dims, rnd, vocab_chunk=16384):
    """ℓ = -z_label + max z + log Σ_v exp(z_v - max z) with
    z = W_U Norm_out(h) (M7.6 §0x03; M7.4 §0x06F).  The vocabulary is visited
    in chunks only to bound memory; every logit is one dot product."""
    x = rnd(rmsnorm(h, W["out_norm"], dims.eps))
    WU = W["head"]
    V = WU.shape[0]
    z = np.empty((x.shape[0], V))
    for v0 in range(0, V, vocab_chunk):
        z[:, v0:v0 + vocab_chunk] = x @ _f64(WU[v0:v0 + vocab_chunk]).T
    zmax = z.max(axis=1)
    lse = zmax + np.log(np.exp(z - zmax[:, None]).sum(axis=1))
    return lse - z[np.arange(len(labels)), np.asarray(labels)]


def chain_forward_loss(tokens, seg, pos, h0, W, dims: Dims, precision="f64",
                       lam=0.3, den="fixed", with_main=True, with_loss=True):
    """Run depths 1..D over every packed row and assemble the loss.

    tokens, seg (-1 = padding), pos: int [B, T]; h0: [B, T, d] main-model
    hidden states.  Returns ``h`` [D, B, T, d] (NaN where a base has no state
    at that depth), ``row_loss`` [D+1, B, T] (index 0 = main next-token loss
    on h0, index k = depth k; NaN where no label is owned), ``sums`` and
    ``counts`` [D+1] and the assembled losses.

    ``den="fixed"`` divides every term by B*T (the fixed 1/T denominator of
    M7.6 §0x05 for a batch of B rows of T); ``den="masked_mean"`` divides by
    the term's own row count, an empty term contributing 0 to the D-depth mean
    (M7.6 §0x05, §0x06A).
    """
    rnd = round_bf16 if precision == "bf16" else (lambda a: a)
    tokens = np.asarray(tokens)
    seg = np.asarray(seg)
    pos = np.asarray(pos)
    B, T = tokens.shape
    d = np.asarray(h0).shape[-1]
    D = dims.D
    h_out = np.full((D, B, T, d), np.nan)
    row_loss = np.full((D + 1, B, T), np.nan)

    for b in range(B):
        tok = [int(v) for v in tokens[b]]
        sg = [int(v) for v in seg[b]]
        active = [s != -1 for s in sg]
        if with_main and with_loss:
            main_rows = [t for t in range(T) if label_owned(active, sg, t, 1)]
            if main_rows:
                x0 = _f64(h0[b][main_rows])
                row_loss[0, b, main_rows] = row_cross_entropy(
                    x0, [tok[t + 1] for t in main_rows], W, dims, rnd)
        state = _f64(h0[b])
        for k, rows in enumerate(states_all_depths(sg, active, D)):
            if not rows:
                state = state[:0]
                continue
            prev = state[[r.parent for r in rows]]
            shifted = [tok[r.input_at] for r in rows]
            bases = [r.base for r in rows]
            h = mtp_module(prev, shifted, W, k, pos[b][bases],
                           [r.segment for r in rows], bases, dims, rnd)
            state = h
            h_out[k, b, bases] = h
            if with_loss:
                sup = [j for j, r in enumerate(rows) if r.supervised]
                if sup:
                    row_loss[k + 1, b, [rows[j].base for j in sup]] = row_cross_entropy(
                        h[sup], [tok[rows[j].label_at] for j in sup], W, dims, rnd)

    out = {"h": h_out, "row_loss": row_loss}
    if not with_loss:
        return out
    finite = np.isfinite(row_loss)
    sums = np.where(finite, row_loss, 0.0).sum(axis=(1, 2))
    counts = finite.sum(axis=(1, 2)).astype(np.int64)
    out.update(assemble_loss(sums, counts, B * T, D, lam, den, with_main))
    out["sums"] = sums
    out["counts"] = counts
    return out


REDUCTIONS = ("fixed", "masked_mean", "sum", "global", "weighted_pair")


def assemble_loss(sums, counts, n_positions, D, lam, den, with_main=True, depth_weights=None):
    """L = L_main + Σ_k w_k L^(k) with per-depth weights w_k (default λ/D,
    M7.6 §0x05: L_main + (λ/D) Σ_k L^(k)) and the depth reduction ``den``
    (the four reductions of "M7.4 - Multi-Token Prediction Foundations"
    §0x02C, plus the fixed denominator):
      fixed          L^(k) = S_k / n_positions (the paper's 1/T for a batch)
      masked_mean    L^(k) = S_k / N_k          (head mean; empty term -> 0)
      sum            L^(k) = S_k
      global         L^(k) = S_k / Σ_j N_j      (so Σ_k w_k L^(k) = Σ w S / Σ N)
      weighted_pair  L^(k) = S_k / Σ_j w_j N_j  (so Σ_k w_k L^(k) = Σ w S / Σ w N)
    with S_k, N_k the loss sum and supervised-row count of depth k.  The main
    term is S_0 / n_positions (fixed), S_0 (sum) or S_0 / N_0 (the others);
    an empty denominator gives 0."""
    if den not in REDUCTIONS:
        raise ValueError(den)
    w = [lam / D] * D if depth_weights is None else [float(x) for x in depth_weights]
    n_all = sum(counts[1:D + 1])
    wn_all = sum(w[k - 1] * counts[k] for k in range(1, D + 1))

    def div(a, b):
        return a / b if b > 0 else 0.0

    def term(i):
        if den == "fixed":
            return sums[i] / n_positions
        if den == "sum":
            return sums[i]
        if den == "masked_mean" or i == 0:
            return div(sums[i], counts[i])
        if den == "global":
            return div(sums[i], n_all)
        return div(sums[i], wn_all)

    L_main = term(0) if with_main else 0.0
    L_k = [term(i) for i in range(1, D + 1)]
    return {"loss_main": L_main, "loss_mtp": L_k,
            "loss_total": L_main + sum(w[k] * L_k[k] for k in range(D))}


def deepseek_v3_lambda(tokens_seen: float) -> float:
    """MTP weight of the DeepSeek-V3 schedule quoted by M7.6 §0x05: 0.3 for the
    first 10T training tokens, 0.1 for the rest."""
    return 0.3 if tokens_seen < 10e12 else 0.1


def weights_to_numpy(weights) -> dict:
    """Host copies (float32 holds every bf16 value exactly) of a weight dict
    whose leaves are torch tensors or lists of them."""
    out = {}
    for key, val in weights.items():
        if isinstance(val, (list, tuple)):
            out[key] = [t.float().cpu().numpy() for t in val]
        else:
            out[key] = val.float().cpu().numpy()
    return out
