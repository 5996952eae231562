"""FP8 block-scaled weights on the GPU, through the C ABI, against the FP8
oracle (exact dequantisation W = e4m3(q) * scale per 128 x 128 block).

GEMM (mtp_gemm_fp8w): out += x~ W^T, x~ the two-term e4m3 form of x (the
oracle's split, bit for bit), within 2e-5 of Σ_k |x~||W| per entry, and
against the unsplit x W^T within that plus the split's exactness bound -- the
kernel sums exact e4m3 x e4m3 products in fp32 per 128-wide k-block and adds
the scaled partials in fp32, so its error is a few hundred fp32 roundings of
that sum at most; any layout, split or scale-index mistake is O(1).  Shapes
cover one and several 256-row tiles, ragged rows (N % 256, N % 128), ragged
k-blocks (K % 128), 1..32 tokens and work ranges that cut row tiles between
CTAs; activations span many binades so both split terms and the subnormal
range are exercised.

Draft step and round with FP8 linear maps (mtp_draft_round_fp8): the draft
oracle run on the exactly dequantised weights (its activations are not split:
the split moves an element by at most 2^-17.8 of its k-tile's largest, far
below these bars), with the bf16 draft bars except
the per-entry q bar, 5e-3 max(q) (Q_BAR): one bf16 rounding flip of an element
x_j of the normalised head input moves every logit z_v by W_U[v, j] ulp(x_j),
up to ~0.17 * 2^-6 = 2.7e-3 with these weights (|W_U| <= ~0.17, |x_j| < 4), and
q_v by that fraction; a probe over ten seeds saw 1.6e-3 with bf16 weights and
3.0e-3 with FP8 weights, each from such flips (h off by one bf16 ulp)."""
import numpy as np
import pytest
import torch

from deepseek_sequential_mtp_gb300 import lib, synth
from oracle import chain as oc
from oracle import draft as od
from oracle import fp8 as of
from oracle import verify as ov

from test_gpu_draft import _check_round, check

pytestmark = pytest.mark.gpu
Q_BAR = 5e-3


def _codes(rng, shape):
    q = rng.integers(0, 256, size=shape).astype(np.uint8)
    q[(q & 0x7F) == 0x7F] = 0x3A  # no NaN codes
    return q


@pytest.mark.parametrize("R,N,K", [(1, 128, 128), (5, 200, 144), (32, 384, 1040), (17, 1000, 2064),
                                   (32, 7168, 7168), (3, 130, 18432), (32, 18432, 7168)])
def test_gemm_parity(R, N, K):
    rng = np.random.default_rng(R * 7 + N + K)
    q = _codes(rng, (N, K))
    s = rng.uniform(1e-3, 1e-2, size=(-(-N // 128), -(-K // 128))).astype(np.float32)
    mag = np.exp(rng.uniform(-6, 3, size=(R, K)))
    x = torch.from_numpy((rng.standard_normal((R, K)) * mag).astype(np.float32)).to(torch.bfloat16)
    out0 = torch.randn(R, N, generator=torch.Generator().manual_seed(N))
    out = out0.clone().cuda()
    lib.gemm_fp8w(x.cuda(), torch.from_numpy(q).cuda(), torch.from_numpy(s).cuda(), out)
    lib.check_errors()
    xs = of.represented_activations(x.double().numpy())
    W = of.dequantize(q, s)
    ref = out0.double().numpy() + xs @ W.T
    bound = np.abs(xs) @ np.abs(W).T
    got = out.cpu().double().numpy()
    err = np.abs(got - ref)
    assert np.all(err <= 2e-5 * bound + 1e-6 * np.abs(out0.double().numpy())), err.max()
    # against the unsplit product x W^T as well: the two-term form moves an element by at most
    # 2^-17 of its 128-wide k-tile's largest (the split's exactness bound, from the e4m3
    # mantissas alone), so the difference is bounded without reference to the split itself
    xd = x.double().numpy()
    nkb = -(-K // 128)
    tile_max = np.stack([np.abs(xd[:, i * 128:(i + 1) * 128]).max(axis=1) for i in range(nkb)], axis=1)
    absW = np.abs(W)
    wsum = np.stack([absW[:, i * 128:(i + 1) * 128].sum(axis=1) for i in range(nkb)], axis=1)  # [N, nkb]
    split_bound = 2.0 ** -17 * tile_max @ wsum.T
    err_u = np.abs(got - (out0.double().numpy() + xd @ W.T))
    assert np.all(err_u <= 2e-5 * (np.abs(xd) @ absW.T) + split_bound + 1e-6 * np.abs(out0.double().numpy()))


def test_gemm_argument_errors():
    x = torch.zeros(4, 120, dtype=torch.bfloat16, device="cuda")  # K % 16 != 0
    q = torch.zeros(128, 120, dtype=torch.uint8, device="cuda")
    s = torch.ones(1, 1, dtype=torch.float32, device="cuda")
    out = torch.zeros(4, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(lib.MtpError):
        lib.gemm_fp8w(x, q, s, out)
    x = torch.zeros(33, 128, dtype=torch.bfloat16, device="cuda")  # more than 32 tokens
    with pytest.raises(lib.MtpError):
        lib.gemm_fp8w(x, torch.zeros(128, 128, dtype=torch.uint8, device="cuda"), s,
                      torch.zeros(33, 128, dtype=torch.float32, device="cuda"))


def _np(t):
    return t.float().cpu().numpy() if t.dtype.is_floating_point else t.cpu().numpy()


def _fp8(inp):
    f8 = synth.make_fp8_block(inp["weights"])
    W = oc.weights_to_numpy(inp["weights"])
    W8 = of.draft_weights(W, {k: (_np(q), _np(s)) for k, (q, s) in f8.items()})
    f8dev = {k: (q.cuda(), s.cuda()) for k, (q, s) in f8.items()}
    return f8dev, W8


def _step(cfg, inp, seed, offset, requests=None):
    f8dev, W8 = _fp8(inp)
    dev = {k: v.cuda() for k, v in inp.items() if k != "weights"}
    wdev = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    step = lib.DraftStep(cfg, wdev, fp8=f8dev)
    h = torch.empty((cfg.R, cfg.d), dtype=torch.bfloat16, device="cuda")
    g = step(dev["parent_hidden"], dev["frontier"], dev["pos"], dev["kv_k"], dev["kv_v"], dev["ctx_len"],
             seed, offset, h_out=h)
    lib.check_errors()
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1, eps=cfg.eps, rope_base=cfg.rope_base)
    requests = list(range(cfg.R)) if requests is None else requests
    sel = lambda t: _np(t[requests])  # noqa: E731  (select on the device first)
    r = od.draft_step(sel(inp["parent_hidden"]), sel(inp["frontier"]), sel(inp["pos"]), sel(inp["kv_k"]),
                      sel(inp["kv_v"]), sel(inp["ctx_len"]), W8, dims, seed, offset, requests=range(len(requests)))
    r["y"], r["margin"] = [], []
    for i, rid in enumerate(requests):
        y, m = ov.inverse_cdf(r["q"][i], od.draft_uniform(seed, offset, rid))
        r["y"].append(y)
        r["margin"].append(m)
    return {k: _np(v) for k, v in g.items()}, r, requests


def _draws(g, r, req, seed, offset):
    for i, rid in enumerate(req):
        y_own, m_own = ov.inverse_cdf(g["q"][rid].astype(np.float64), od.draft_uniform(seed, offset, rid))
        if m_own > 1e-6:
            assert g["y"][rid] == y_own
        if r["margin"][i] > 5e-3:
            assert g["y"][rid] == r["y"][i]


def test_fp8_step_small_hd64():
    """head_dim 64, empty, one-key and ragged caches."""
    cfg = synth.DRAFT_SMALL
    inp = synth.make_draft_inputs(cfg, 4)
    inp["ctx_len"] = torch.tensor([0, 1, 100, 299, 300][:cfg.R], dtype=torch.int32)
    inp["pos"] = inp["ctx_len"].clone()
    g, r, req = _step(cfg, inp, seed=13, offset=3)
    check(g, r, req, qbar=Q_BAR)
    _draws(g, r, req, 13, 3)


def test_fp8_step_small_hd128():
    cfg = synth.DRAFT_SMALL_HD128
    inp = synth.make_draft_inputs(cfg, 6)
    inp["ctx_len"] = torch.tensor([0, 63, 577, 1100], dtype=torch.int32)
    inp["pos"] = inp["ctx_len"].clone()
    g, r, req = _step(cfg, inp, seed=8, offset=1)
    check(g, r, req, qbar=Q_BAR)
    _draws(g, r, req, 8, 1)


def test_fp8_round_hd64():
    """Recurrent drafting with FP8 linear maps, gamma = 3."""
    cfg = synth.DRAFT_SMALL
    gamma = 3
    inp = synth.make_draft_inputs(cfg, 9)
    inp["ctx_len"] = torch.tensor([0, 1, 100, 299, 300][:cfg.R], dtype=torch.int32)
    inp["pos"] = inp["ctx_len"].clone()
    f8dev, W8 = _fp8(inp)
    dev = {k: v.cuda() for k, v in inp.items() if k != "weights"}
    wdev = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    rnd = lib.DraftRound(cfg, wdev, gamma, fp8=f8dev)
    h = torch.empty((cfg.R, gamma, cfg.d), dtype=torch.bfloat16, device="cuda")
    g = rnd(dev["parent_hidden"], dev["frontier"], dev["pos"], dev["kv_k"], dev["kv_v"], dev["ctx_len"], 31, 7,
            h_out=h)
    lib.check_errors()
    g = {k: _np(v) for k, v in g.items()}
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1, eps=cfg.eps, rope_base=cfg.rope_base)
    r = od.draft_round(*[_np(inp[k]) for k in ("parent_hidden", "frontier", "pos", "kv_k", "kv_v", "ctx_len")],
                       W8, dims, gamma, 31, 7, forced_y=g["y"], forced_h=g["h"])
    _check_round(cfg, g, r, 31, 7, bar0=Q_BAR)


def test_fp8_step_full_size_sampled_requests():
    """32 requests, cache 8192 x d=7168 (56 x 128 heads), ffn 18432,
    V=129280 with FP8 linear maps; oracle on two requests, draws on all."""
    cfg = synth.DRAFT_C5
    inp = synth.make_draft_inputs(cfg, 3, device="cuda")
    g, r, req = _step(cfg, inp, seed=5, offset=4, requests=[1, 30])
    check(g, r, req, qbar=Q_BAR)
    for rid in range(cfg.R):
        y_own, m_own = ov.inverse_cdf(g["q"][rid].astype(np.float64), od.draft_uniform(5, 4, rid))
        if m_own > 1e-6:
            assert g["y"][rid] == y_own
