"""Seeded synthetic inputs for the sequential-MTP hot path.

This module only *draws data*: packed token batches with segment ids and
positions, random-init weights of the MTP module shapes, main-model hidden
states, and probability rows for speculative verification.  It contains none
of the method's arithmetic (no normalisation, projection, attention, loss or
accept/resample step).  Both the CUDA path (through the binding) and the CPU
oracle consume what it returns, so it is the one module they share.

Shapes and distributions follow the workloads of "M7.6 - DeepSeek MTP:
Sequential Modules, Teacher Forcing, and Speculative Runtime" (§0x02-§0x06A:
packed rows, segment ids, -1 padding) and of the speculative-decoding page
(γ drafts scored against target rows).  Every generator takes an explicit
seed; weights are drawn with a ``torch.Generator`` on the requested device so
the benchmark can create multi-GB weights on the GPU, while tests draw them on
the CPU and copy them over.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch

PAD_SEGMENT = -1


# --------------------------------------------------------------------------
# Configurations
# --------------------------------------------------------------------------
@dataclass(frozen=True)
class ChainConfig:
    """One teacher-forced MTP-chain workload.

    ``layout`` selects how packed rows are cut into documents:
      * ``"tiny"``      -- row 0 active for t <= pad_after, padded after;
                           row 1 split into two segments at ``split_at``.
      * ``"split"``     -- every row split into segments at ``split_at``.
      * ``"geometric"`` -- documents with Geometric(1/doc_mean) lengths packed
                           in order, the last one truncated at T; when
                           ``pad_rows`` > 0 the first ``pad_rows`` rows end with
                           ``pad_len`` padding positions.
    """

    name: str
    B: int
    T: int
    d: int
    n_heads: int
    head_dim: int
    ffn: int
    V: int
    D: int
    dtype: str  # "f32" or "bf16"
    lam: float = 0.3
    w_std: float = 0.02
    gain_std: float = 0.0  # gains = 1 + gain_std * N(0, 1)
    tokens: str = "uniform"  # "uniform" or "zipf"
    zipf_s: float = 1.1
    layout: str = "geometric"
    doc_mean: int = 256
    split_at: int = 0
    pad_after: int = -1
    pad_rows: int = 0
    pad_len: int = 0
    eps: float = 1e-6
    rope_base: float = 10000.0

    @property
    def M(self) -> int:
        return self.B * self.T

    def with_(self, **kw) -> "ChainConfig":
        return replace(self, **kw)


# The five workloads of the build, plus small parity shapes that span several
# GEMM tiles with ragged tails.
TINY_F32 = ChainConfig(
    name="tiny_f32", B=2, T=16, d=64, n_heads=4, head_dim=16, ffn=172, V=512, D=1,
    dtype="f32", lam=0.3, w_std=0.02, gain_std=0.0, tokens="uniform",
    layout="tiny", split_at=6, pad_after=10)

MID_BF16 = ChainConfig(
    name="mid_bf16_D3", B=8, T=1024, d=1024, n_heads=16, head_dim=64, ffn=2816,
    V=32000, D=3, dtype="bf16", lam=0.3, w_std=0.02, gain_std=0.05, tokens="zipf",
    layout="geometric", doc_mean=256)

DSV3_BF16 = ChainConfig(
    name="dsv3_width_bf16_D1", B=1, T=4096, d=7168, n_heads=56, head_dim=128,
    ffn=18432, V=129280, D=1, dtype="bf16", lam=0.3, w_std=0.006, gain_std=0.05,
    tokens="zipf", layout="split", split_at=2048)

# Parity shapes (not benchmark lines): several tiles in every GEMM dimension,
# ragged M (B*T), ragged vocab and ragged ffn tiles, padding and packing.
SMALL_BF16 = ChainConfig(
    name="small_bf16_D2", B=2, T=300, d=256, n_heads=4, head_dim=64, ffn=576,
    V=1000, D=2, dtype="bf16", lam=0.3, w_std=0.05, gain_std=0.1, tokens="zipf",
    layout="geometric", doc_mean=64, pad_rows=1, pad_len=37)

SMALL_BF16_HD128 = ChainConfig(
    name="small_bf16_hd128", B=1, T=520, d=384, n_heads=3, head_dim=128, ffn=704,
    V=2100, D=2, dtype="bf16", lam=0.3, w_std=0.04, gain_std=0.1, tokens="zipf",
    layout="geometric", doc_mean=150)

SMALL_F32 = ChainConfig(
    name="small_f32_D3", B=3, T=40, d=96, n_heads=3, head_dim=32, ffn=100, V=300,
    D=3, dtype="f32", lam=0.3, w_std=0.05, gain_std=0.1, tokens="uniform",
    layout="geometric", doc_mean=12, pad_rows=1, pad_len=5)

CHAIN_CONFIGS = {c.name: c for c in
                 (TINY_F32, MID_BF16, DSV3_BF16, SMALL_BF16, SMALL_BF16_HD128, SMALL_F32)}


@dataclass(frozen=True)
class VerifyConfig:
    """Speculative verification workload: R requests, γ drafts each.

    Target logits are N(0, logit_std) plus a Zipf-rank bias -zipf_bias*ln(v+1);
    draft logits are the target logits of the γ draft positions plus
    N(0, draft_sigma) noise.  ``draft_sigma`` was calibrated once so that the
    mean overlap sum_v min(p, q) is about 0.70 at V=129280.
    """

    name: str
    R: int
    gamma: int
    V: int
    logit_std: float = 2.0
    zipf_bias: float = 1.1
    draft_sigma: float = 0.818


VERIFY_C4 = VerifyConfig(name="verify_R64_g4_V129280", R=64, gamma=4, V=129280)
VERIFY_SMALL = VerifyConfig(name="verify_R9_g3_V3000", R=9, gamma=3, V=3000)


@dataclass(frozen=True)
class DraftConfig:
    """Self-speculative decode round: one depth-1 MTP draft step per request
    over a module-local K/V cache of ``ctx`` prior positions, then γ=1
    verification against target rows built like ``VerifyConfig``."""

    name: str
    R: int
    ctx: int
    d: int
    n_heads: int
    head_dim: int
    ffn: int
    V: int
    w_std: float = 0.006
    gain_std: float = 0.05
    eps: float = 1e-6
    rope_base: float = 10000.0


DRAFT_C5 = DraftConfig(name="draft_R32_ctx8192_d7168", R=32, ctx=8192, d=7168,
                       n_heads=56, head_dim=128, ffn=18432, V=129280)
DRAFT_SMALL = DraftConfig(name="draft_small", R=5, ctx=300, d=256, n_heads=4,
                          head_dim=64, ffn=576, V=1000, w_std=0.05, gain_std=0.1)
# 128-wide heads, two key splits of 576 keys, ragged last tiles
DRAFT_SMALL_HD128 = DraftConfig(name="draft_small_hd128", R=4, ctx=1100, d=256, n_heads=2,
                                head_dim=128, ffn=512, V=777, w_std=0.05, gain_std=0.1)


# --------------------------------------------------------------------------
# Packed token batches
# --------------------------------------------------------------------------
def _segments_for_row(cfg: ChainConfig, b: int, rng: np.random.Generator) -> np.ndarray:
    T = cfg.T
    seg = np.empty(T, dtype=np.int32)
    if cfg.layout == "tiny":
        if b == 0:
            seg[:] = 0
            seg[cfg.pad_after + 1:] = PAD_SEGMENT
        else:
            seg[:cfg.split_at] = 0
            seg[cfg.split_at:] = 1
        return seg
    if cfg.layout == "split":
        seg[:cfg.split_at] = 0
        seg[cfg.split_at:] = 1
        return seg
    if cfg.layout == "geometric":
        n_active = T - (cfg.pad_len if b < cfg.pad_rows else 0)
        t, sid = 0, 0
        while t < n_active:
            length = int(rng.geometric(1.0 / cfg.doc_mean))
            seg[t:min(n_active, t + length)] = sid
            t += length
            sid += 1
        seg[n_active:] = PAD_SEGMENT
        return seg
    raise ValueError(f"unknown layout {cfg.layout!r}")


def _draw_tokens(cfg: ChainConfig, n: int, rng: np.random.Generator) -> np.ndarray:
    if cfg.tokens == "uniform":
        return rng.integers(0, cfg.V, size=n, dtype=np.int64).astype(np.int32)
    if cfg.tokens == "zipf":
        # P(id = v) proportional to (v + 1)^-s over [0, V), by inverse CDF.
        w = np.arange(1, cfg.V + 1, dtype=np.float64) ** (-cfg.zipf_s)
        cdf = np.cumsum(w)
        cdf /= cdf[-1]
        ids = np.searchsorted(cdf, rng.random(n), side="right")
        return np.minimum(ids, cfg.V - 1).astype(np.int32)
    raise ValueError(f"unknown token distribution {cfg.tokens!r}")


def make_batch(cfg: ChainConfig, seed: int) -> dict:
    """tokens, seg (-1 = pad) and pos (position within the segment) as int32 [B, T]."""
    rng = np.random.default_rng(seed)
    seg = np.stack([_segments_for_row(cfg, b, rng) for b in range(cfg.B)])
    tokens = _draw_tokens(cfg, cfg.B * cfg.T, rng).reshape(cfg.B, cfg.T)
    pos = np.zeros_like(seg)
    for b in range(cfg.B):
        start = 0
        for t in range(cfg.T):
            if t == 0 or seg[b, t] != seg[b, t - 1]:
                start = t
            pos[b, t] = t - start if seg[b, t] != PAD_SEGMENT else 0
    return {"tokens": tokens, "seg": seg, "pos": pos}


# --------------------------------------------------------------------------
# Weights and hidden states
# --------------------------------------------------------------------------
def torch_dtype(cfg_dtype: str) -> torch.dtype:
    return {"f32": torch.float32, "bf16": torch.bfloat16}[cfg_dtype]


def _normal(gen, shape, std, mean, dtype, device):
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(mean=mean, std=std, generator=gen)
    return x.to(dtype)


def make_weights(cfg: ChainConfig, seed: int, device="cpu") -> dict:
    """Random-init weights of the MTP chain.

    Shared: ``embed`` [V, d], ``head`` [V, d], ``out_norm`` [d].
    Per depth k (lists of length D): ``hnorm``, ``enorm``, ``attn_norm``,
    ``ffn_norm`` [d]; ``eh_proj`` [d, 2d] with columns in hidden-then-embedding
    order; ``wq``, ``wk``, ``wv``, ``wo`` [d, d]; ``w_gate``, ``w_up`` [ffn, d];
    ``w_down`` [d, ffn].  Matrices ~ N(0, w_std); gains = 1 + gain_std*N(0,1).
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = torch_dtype(cfg.dtype)
    d, f, V = cfg.d, cfg.ffn, cfg.V

    def mat(*shape):
        return _normal(gen, shape, cfg.w_std, 0.0, dt, device)

    def gain():
        if cfg.gain_std == 0.0:
            return torch.ones(d, dtype=dt, device=device)
        return _normal(gen, (d,), cfg.gain_std, 1.0, dt, device)

    w = {"embed": mat(V, d), "head": mat(V, d), "out_norm": gain()}
    for key in ("hnorm", "enorm", "eh_proj", "attn_norm", "wq", "wk", "wv", "wo",
                "ffn_norm", "w_gate", "w_up", "w_down"):
        w[key] = []
    for _ in range(cfg.D):
        w["hnorm"].append(gain())
        w["enorm"].append(gain())
        w["eh_proj"].append(mat(d, 2 * d))
        w["attn_norm"].append(gain())
        w["wq"].append(mat(d, d))
        w["wk"].append(mat(d, d))
        w["wv"].append(mat(d, d))
        w["wo"].append(mat(d, d))
        w["ffn_norm"].append(gain())
        w["w_gate"].append(mat(f, d))
        w["w_up"].append(mat(f, d))
        w["w_down"].append(mat(d, f))
    return w


def make_h0(cfg: ChainConfig, seed: int, device="cpu") -> torch.Tensor:
    """Synthetic main-model hidden states h^0 ~ N(0, 1), [B, T, d]."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed + 7919)
    return _normal(gen, (cfg.B, cfg.T, cfg.d), 1.0, 0.0, torch_dtype(cfg.dtype), device)


def make_chain_inputs(cfg: ChainConfig, seed: int, device="cpu") -> dict:
    batch = make_batch(cfg, seed)
    out = {k: torch.from_numpy(v).to(device) for k, v in batch.items()}
    out["h0"] = make_h0(cfg, seed, device)
    out["weights"] = make_weights(cfg, seed + 1, device)
    return out


# --------------------------------------------------------------------------
# Speculative verification inputs
# --------------------------------------------------------------------------
def _softmax64(z: torch.Tensor) -> torch.Tensor:
    # Input construction only: the verifier receives probability rows.
    z = z - z.max(dim=-1, keepdim=True).values
    e = torch.exp(z)
    return e / e.sum(dim=-1, keepdim=True)


def make_verify_inputs(cfg: VerifyConfig, seed: int, device="cpu") -> dict:
    """p [R, γ+1, V] f32, q [R, γ, V] f32 and draft tokens y [R, γ] int32, y_j ~ q_j."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    R, g, V = cfg.R, cfg.gamma, cfg.V
    bias = -cfg.zipf_bias * torch.log(torch.arange(1, V + 1, dtype=torch.float64, device=device))
    zt = torch.empty((R, g + 1, V), dtype=torch.float64, device=device)
    zt.normal_(0.0, cfg.logit_std, generator=gen)
    zt += bias
    noise = torch.empty((R, g, V), dtype=torch.float64, device=device)
    noise.normal_(0.0, cfg.draft_sigma, generator=gen)
    zd = zt[:, :g] + noise
    p = _softmax64(zt).to(torch.float32)
    q = _softmax64(zd).to(torch.float32)
    y = torch.multinomial(q.reshape(R * g, V).double(), 1, generator=gen).reshape(R, g)
    return {"p": p.contiguous(), "q": q.contiguous(), "draft": y.to(torch.int32).contiguous()}


def make_small_verify_case(seed: int, R: int, gamma: int, V: int, device="cpu",
                           overlap: str = "mixed") -> dict:
    """Small verification cases with hand-shaped supports for edge coverage:
    zero-probability entries, p == q rows, disjoint supports."""
    rng = np.random.default_rng(seed)
    p = rng.gamma(0.3, size=(R, gamma + 1, V))
    q = rng.gamma(0.3, size=(R, gamma, V))
    if overlap in ("mixed", "zeros"):
        p[rng.random(p.shape) < 0.3] = 0.0
        q[rng.random(q.shape) < 0.3] = 0.0
    if overlap == "mixed":
        same = rng.random(R) < 0.25
        q[same] = p[same, :gamma]
    p[..., 0] += 1e-3  # keep every row non-empty
    q[..., 0] += 1e-3
    p /= p.sum(-1, keepdims=True)
    q /= q.sum(-1, keepdims=True)
    p32 = p.astype(np.float32)
    q32 = q.astype(np.float32)
    y = np.empty((R, gamma), dtype=np.int32)
    for r in range(R):
        for j in range(gamma):
            w = q32[r, j].astype(np.float64)
            y[r, j] = rng.choice(V, p=w / w.sum())
    return {"p": torch.from_numpy(p32).to(device), "q": torch.from_numpy(q32).to(device),
            "draft": torch.from_numpy(y).to(device)}


# --------------------------------------------------------------------------
# Draft-step inputs (decode-shaped)
# --------------------------------------------------------------------------
FP8_LINEAR_MAPS = ("eh_proj", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


def quantize_fp8_blocks(w: torch.Tensor):
    """Synthetic FP8 checkpoint form of one [n, K] weight matrix, the format
    DeepSeek-V3 releases: per 128 x 128 block a float32 scale = max|w| / 448
    and the E4M3 codes of w / scale (torch's float8_e4m3fn conversion).
    Returns (q uint8 [n, K], scale float32 [ceil(n/128), ceil(K/128)]) on w's
    device.  Input generation only: the hot path reads q and scale as given."""
    w32 = w.float()
    n, k = w32.shape
    nb, kb = -(-n // 128), -(-k // 128)
    pad = torch.zeros((nb * 128, kb * 128), dtype=torch.float32, device=w.device)
    pad[:n, :k] = w32.abs()
    amax = pad.view(nb, 128, kb, 128).amax(dim=(1, 3))
    scale = torch.clamp(amax, min=1e-30) / 448.0
    expanded = scale.repeat_interleave(128, 0)[:n].repeat_interleave(128, 1)[:, :k]
    q = torch.clamp(w32 / expanded, -448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.contiguous(), scale.contiguous()


def make_fp8_block(weights: dict) -> dict:
    """FP8 forms of the depth-1 module's eight linear maps of a weight dict."""
    return {name: quantize_fp8_blocks(weights[name][0]) for name in FP8_LINEAR_MAPS}


def make_draft_inputs(cfg: DraftConfig, seed: int, device="cpu") -> dict:
    """parent_hidden [R, d], frontier tokens [R], position [R], the module's own
    K/V cache [R, ctx, d] (bf16, N(0,1)) with ctx_len [R], and depth-1 weights."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    rng = np.random.default_rng(seed)
    R, d = cfg.R, cfg.d
    chain_cfg = ChainConfig(name=cfg.name + "_weights", B=1, T=1, d=d, n_heads=cfg.n_heads,
                            head_dim=cfg.head_dim, ffn=cfg.ffn, V=cfg.V, D=1, dtype="bf16",
                            w_std=cfg.w_std, gain_std=cfg.gain_std, eps=cfg.eps,
                            rope_base=cfg.rope_base)
    out = {
        "parent_hidden": _normal(gen, (R, d), 1.0, 0.0, torch.bfloat16, device),
        "frontier": torch.from_numpy(rng.integers(0, cfg.V, R).astype(np.int32)).to(device),
        "ctx_len": torch.full((R,), cfg.ctx, dtype=torch.int32, device=device),
        "kv_k": _normal(gen, (R, cfg.ctx, d), 1.0, 0.0, torch.bfloat16, device),
        "kv_v": _normal(gen, (R, cfg.ctx, d), 1.0, 0.0, torch.bfloat16, device),
        "weights": make_weights(chain_cfg, seed + 3, device),
    }
    out["pos"] = out["ctx_len"].clone()
    return out
