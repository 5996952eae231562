"""Depth reductions and per-depth weights on the GPU (mtp_loss_assemble_weighted
and mtp_chain_loss) against the oracle's assembly.  The assembly is fp64 on
both sides with fp32 outputs: relative agreement 1e-6."""
import numpy as np
import pytest
import torch

from deepseek_sequential_mtp_gb300 import lib, synth
from oracle import chain as oc

pytestmark = pytest.mark.gpu

DENS = ["fixed", "masked_mean", "sum", "global", "weighted_pair"]


@pytest.mark.parametrize("den", DENS)
@pytest.mark.parametrize("weights", [None, [0.5, 0.25, 0.125]])
@pytest.mark.parametrize("with_main", [True, False])
def test_assemble_matches_oracle(den, weights, with_main):
    rng = np.random.default_rng(hash((den, with_main)) % 2**32)
    D = 3
    counts = np.array([4000.0, 3000.0, 0.0, 1000.0])  # depth 2 empty
    sums = rng.random(D + 1) * counts * 3
    sc = torch.tensor(np.stack([sums, counts], 1).reshape(-1), dtype=torch.float64, device="cuda")
    g = lib.loss_assemble(sc, D, 8192.0, 0.3, den=den, with_main=with_main, depth_weights=weights)
    lib.check_errors()
    r = oc.assemble_loss(sums, counts, 8192.0, D, 0.3, den, with_main=with_main, depth_weights=weights)
    want = np.array([r["loss_total"], r["loss_main"], *r["loss_mtp"]])
    np.testing.assert_allclose(g.cpu().numpy(), want, rtol=1e-6, atol=0)


@pytest.mark.parametrize("den", ["sum", "global", "weighted_pair"])
def test_chain_loss_reductions(den):
    cfg = synth.SMALL_BF16
    inp = synth.make_chain_inputs(cfg, seed=5)
    w = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    chain = lib.Chain(cfg, w)
    out = chain.loss(inp["tokens"].cuda(), inp["seg"].cuda(), inp["pos"].cuda(), inp["h0"].cuda(), den=den,
                     with_main=True)
    lib.check_errors()
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=cfg.D, eps=cfg.eps, rope_base=cfg.rope_base)
    r = oc.chain_forward_loss(inp["tokens"].numpy(), inp["seg"].numpy(), inp["pos"].numpy(),
                              inp["h0"].float().numpy(), oc.weights_to_numpy(inp["weights"]), dims,
                              precision="bf16", lam=cfg.lam, den=den)
    want = np.array([r["loss_total"], r["loss_main"], *r["loss_mtp"]])
    np.testing.assert_allclose(out["losses"].cpu().numpy(), want, rtol=2e-3)
    # the reported (sum, count) pairs reassemble under every other reduction
    sc = out["sums_counts"]
    for other in DENS:
        g = lib.loss_assemble(sc, cfg.D, cfg.B * cfg.T, cfg.lam, den=other).cpu().numpy()
        s, c = sc.cpu().numpy()[0::2], sc.cpu().numpy()[1::2]
        ro = oc.assemble_loss(s, c, cfg.B * cfg.T, cfg.D, cfg.lam, other)
        np.testing.assert_allclose(g, [ro["loss_total"], ro["loss_main"], *ro["loss_mtp"]], rtol=1e-6)
