"""Gradients of the chain loss on the GPU (mtp_chain_loss_grad) against the
gradient oracle (fp64 autograd of the chain oracle's forward, pinned by finite
differences).  The GPU's forward rounds at the bf16 points and its head
backward runs on bf16 operands, while the oracle differentiates the unrounded
fp64 forward.  Bars per tensor: normwise relative error <= 2e-2, and every
element within 5e-2 of its own magnitude plus 0.1 of the rms of its row (a
wrong or missing row, column, tile or scattered embedding row moves its
elements by their full size and fails the element bar even when the norm
hides it)."""
import numpy as np
import pytest
import torch

from deepseek_sequential_mtp_gb300 import lib, synth
from oracle import chain as oc
from oracle import grad as og

pytestmark = pytest.mark.gpu


def _rel(g, r):
    return float(np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30))


def _run(cfg, seed, lam, den, with_main, want_h0, depth_weights=None):
    inp = synth.make_chain_inputs(cfg, seed=seed)
    w = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    chain = lib.Chain(cfg, w)
    grads = {"head": torch.zeros((cfg.V, cfg.d), dtype=torch.float32, device="cuda"),
             "out_norm": torch.zeros(cfg.d, dtype=torch.float32, device="cuda")}
    if want_h0:
        grads["h0"] = torch.zeros((cfg.B, cfg.T, cfg.d), dtype=torch.float32, device="cuda")
    out = chain.loss_grad(inp["tokens"].cuda(), inp["seg"].cuda(), inp["pos"].cuda(), inp["h0"].cuda(), grads,
                          lam=lam, den=den, with_main=with_main, depth_weights=depth_weights)
    lib.check_errors()
    W = oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=cfg.D, eps=cfg.eps, rope_base=cfg.rope_base)
    r = og.chain_loss_grads(inp["tokens"].numpy(), inp["seg"].numpy(), inp["pos"].numpy(),
                            inp["h0"].float().numpy(), W, dims, lam=lam, den=den, with_main=with_main,
                            depth_weights=depth_weights)
    return out, {k: v.cpu().numpy() for k, v in grads.items()}, r


def test_main_term_gradients():
    """lam = 0: the head, final norm and h^0 gradients of the main term."""
    cfg = synth.SMALL_BF16
    out, g, r = _run(cfg, 5, 0.0, "fixed", True, True)
    assert np.isclose(out["losses"][0].item(), r["loss_total"], rtol=2e-3)
    assert _rel(g["head"], r["grads"]["head"]) < 2e-2
    assert _rel(g["out_norm"], r["grads"]["out_norm"]) < 2e-2
    assert _rel(g["h0"], r["dh0"]) < 2e-2


@pytest.mark.parametrize("den", ["fixed", "masked_mean", "weighted_pair"])
def test_shared_head_gradient_all_terms(den):
    """The shared head and final norm collect the main term's and both
    depths' gradients (M7.6 §0x05)."""
    cfg = synth.SMALL_BF16
    out, g, r = _run(cfg, 6, 0.3, den, True, False)
    assert _rel(g["head"], r["grads"]["head"]) < 2e-2
    assert _rel(g["out_norm"], r["grads"]["out_norm"]) < 2e-2


def test_hd128_depth_weights_and_accumulation():
    cfg = synth.SMALL_BF16_HD128
    out, g, r = _run(cfg, 7, 0.3, "global", False, False, depth_weights=[0.7, 0.2])
    assert _rel(g["head"], r["grads"]["head"]) < 2e-2
    assert _rel(g["out_norm"], r["grads"]["out_norm"]) < 2e-2


PER_DEPTH = ("hnorm", "enorm", "eh_proj", "attn_norm", "wq", "wk", "wv", "wo", "ffn_norm", "w_gate", "w_up",
             "w_down")


def _run_all(cfg, seed, lam, den, with_main=True, depth_weights=None):
    inp = synth.make_chain_inputs(cfg, seed=seed)
    w = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    chain = lib.Chain(cfg, w)
    z = lambda t: torch.zeros(tuple(t.shape), dtype=torch.float32, device="cuda")  # noqa: E731
    grads = {k: z(w[k]) for k in ("embed", "head", "out_norm")}
    grads["h0"] = torch.zeros((cfg.B, cfg.T, cfg.d), dtype=torch.float32, device="cuda")
    for k in PER_DEPTH:
        grads[k] = [z(t) for t in w[k]]
    out = chain.loss_grad(inp["tokens"].cuda(), inp["seg"].cuda(), inp["pos"].cuda(), inp["h0"].cuda(), grads,
                          lam=lam, den=den, with_main=with_main, depth_weights=depth_weights)
    lib.check_errors()
    W = oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=cfg.D, eps=cfg.eps, rope_base=cfg.rope_base)
    r = og.chain_loss_grads(inp["tokens"].numpy(), inp["seg"].numpy(), inp["pos"].numpy(),
                            inp["h0"].float().numpy(), W, dims, lam=lam, den=den, with_main=with_main,
                            depth_weights=depth_weights)
    return out, grads, r


def _elementwise(g, r, rtol=5e-2, rms_tol=0.1):
    """Largest |g - r| / (rtol |r| + rms_tol rms(r's row)) over the tensor
    (<= 1 passes).  An element of a gradient is a sum of many products; its
    rounding error follows the size of those terms, which the rms of its row
    (an output feature of a weight, one token's scattered embedding rows,
    one position's hidden state) measures, not its own possibly cancelled
    value."""
    g = np.asarray(g, dtype=np.float64).reshape(-1, np.shape(g)[-1])
    r = np.asarray(r, dtype=np.float64).reshape(-1, np.shape(r)[-1])
    row_rms = np.sqrt(np.mean(r * r, axis=1, keepdims=True))
    scale = rtol * np.abs(r) + rms_tol * np.maximum(row_rms, 1e-30)
    return float(np.max(np.abs(g - r) / scale))


def _check_all(cfg, grads, r, bar=2e-2):
    pairs = {k: (grads[k].cpu().numpy(), r["grads"][k]) for k in ("embed", "head", "out_norm")}
    pairs["h0"] = (grads["h0"].cpu().numpy(), r["dh0"])
    for k in PER_DEPTH:
        for i in range(cfg.D):
            pairs[f"{k}[{i}]"] = (grads[k][i].cpu().numpy(), r["grads"][k][i])
    errs = {k: _rel(g, w) for k, (g, w) in pairs.items()}
    bad = {k: v for k, v in errs.items() if not v < bar}
    assert not bad, bad
    elem = {k: _elementwise(g, w) for k, (g, w) in pairs.items()}
    bad = {k: v for k, v in elem.items() if not v <= 1.0}
    assert not bad, bad
    return errs


@pytest.mark.parametrize("den", ["fixed", "masked_mean", "global"])
def test_full_chain_gradients(den):
    """Every gradient of the two-depth chain: shared embedding/head/final norm,
    h^0, and each depth's fusion, block and norm weights."""
    cfg = synth.SMALL_BF16
    out, grads, r = _run_all(cfg, 8, 0.3, den)
    assert np.isclose(out["losses"][0].item(), r["loss_total"], rtol=2e-3)
    _check_all(cfg, grads, r)


def test_full_chain_gradients_hd128_weights():
    cfg = synth.SMALL_BF16_HD128
    out, grads, r = _run_all(cfg, 9, 0.3, "weighted_pair", with_main=False, depth_weights=[0.6, 0.4])
    _check_all(cfg, grads, r)


def test_full_chain_gradients_mid_width():
    """Mid width (d=1024, 16x64 heads, ffn 2816, V=32000) at T=1024 with
    D=2: full-size tiles in every GEMM of the backward, 16 heads of
    attention backward over ~256-token documents."""
    cfg = synth.MID_BF16.with_(name="mid_grad", B=1, T=1024, D=2)
    out, grads, r = _run_all(cfg, 10, 0.3, "fixed")
    assert np.isclose(out["losses"][0].item(), r["loss_total"], rtol=2e-3)
    _check_all(cfg, grads, r)


LONG_GRAD = [
    synth.ChainConfig(name="long_grad_hd64", B=1, T=2048, d=256, n_heads=4, head_dim=64, ffn=512, V=1000, D=1,
                      dtype="bf16", w_std=0.05, gain_std=0.1, tokens="zipf", layout="split", split_at=1024),
    synth.ChainConfig(name="long_grad_hd128", B=1, T=2048, d=256, n_heads=2, head_dim=128, ffn=512, V=1000, D=1,
                      dtype="bf16", w_std=0.05, gain_std=0.1, tokens="zipf", layout="split", split_at=1024),
]


@pytest.mark.parametrize("cfg", LONG_GRAD, ids=lambda c: c.name)
def test_long_segment_gradients(cfg):
    """Two 1024-token segments at both head widths: the attention backward of
    a 128-key block streams up to eight query blocks (every ring phase and
    the dq reductions of many key blocks into the same rows)."""
    out, grads, r = _run_all(cfg, 12, 0.3, "fixed")
    assert np.isclose(out["losses"][0].item(), r["loss_total"], rtol=2e-3)
    _check_all(cfg, grads, r)


def test_gradients_accumulate():
    """Two calls add their gradients into the same buffers."""
    cfg = synth.SMALL_BF16
    inp = synth.make_chain_inputs(cfg, seed=4)
    w = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    chain = lib.Chain(cfg, w)
    g1 = {"head": torch.zeros((cfg.V, cfg.d), device="cuda"), "wq": [torch.zeros_like(t, dtype=torch.float32)
                                                                      for t in w["wq"]]}
    args = (inp["tokens"].cuda(), inp["seg"].cuda(), inp["pos"].cuda(), inp["h0"].cuda())
    chain.loss_grad(*args, g1)
    once = {"head": g1["head"].clone(), "wq": [t.clone() for t in g1["wq"]]}
    chain.loss_grad(*args, g1)
    lib.check_errors()
    torch.testing.assert_close(g1["head"], 2 * once["head"], rtol=1e-5, atol=1e-7)
    torch.testing.assert_close(g1["wq"][1], 2 * once["wq"][1], rtol=1e-5, atol=1e-7)
