"""Gradients of the chain loss on the GPU (mtp_chain_loss_grad) against the
gradient oracle (fp64 autograd of the chain oracle's forward, pinned by finite
differences).  The GPU's forward rounds at the bf16 points and its head
backward runs on bf16 operands, while the oracle differentiates the unrounded
fp64 forward: bar = normwise relative error <= 2e-2 per tensor."""
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


def test_unsupported_requests_are_refused():
    cfg = synth.SMALL_BF16
    inp = synth.make_chain_inputs(cfg, seed=1)
    w = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    chain = lib.Chain(cfg, w)
    grads = {"head": torch.zeros((cfg.V, cfg.d), device="cuda"), "out_norm": torch.zeros(cfg.d, device="cuda"),
             "h0": torch.zeros((cfg.B, cfg.T, cfg.d), device="cuda")}
    with pytest.raises(lib.MtpError):
        chain.loss_grad(inp["tokens"].cuda(), inp["seg"].cuda(), inp["pos"].cuda(), inp["h0"].cuda(), grads, lam=0.3)
