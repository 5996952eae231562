"""Pins of the draft-step oracle: with the module's cache holding a segment's
own rotated keys and values, one draft step reproduces the chain oracle's
depth-1 state of the next row and its loss; q is a distribution; the draw is
the inverse CDF at the Philox word-2 uniform."""
import math

import numpy as np

from deepseek_sequential_mtp_gb300 import synth
from oracle import chain as oc
from oracle import draft as od
from oracle import verify as ov


def test_draft_step_equals_chain_row_with_matching_cache():
    cfg = synth.ChainConfig(name="d", B=1, T=9, d=32, n_heads=2, head_dim=16, ffn=40, V=60, D=1,
                            dtype="f32", w_std=0.2, gain_std=0.2, layout="split", split_at=0)
    rng = np.random.default_rng(3)
    W = oc.weights_to_numpy(synth.make_weights(cfg, 5))
    dims = oc.Dims(n_heads=2, head_dim=16, D=1)
    T = cfg.T
    tok = rng.integers(0, cfg.V, T)
    h0 = rng.standard_normal((T, cfg.d))
    pos = np.arange(T)
    seg = np.zeros(T, int)
    # chain oracle on the whole segment: states of depth 1 for bases 0..T-2
    full = oc.chain_forward_loss(tok[None], seg[None], pos[None], h0[None], W, dims, precision="f64")
    rows = list(range(T - 1))
    u = oc.fusion(h0[rows], tok[[t + 1 for t in rows]], W, 0, dims, lambda a: a)
    _, kk, vv = oc.transformer_block(u, W, 0, pos[rows], seg[rows], rows, dims, lambda a: a, return_kv=True)
    for t in (0, 3, T - 2):  # draft for base t with the cache holding bases < t
        kv_k = kk[None, :t] if t else np.zeros((1, 0, cfg.d))
        kv_v = vv[None, :t] if t else np.zeros((1, 0, cfg.d))
        out = od.draft_step(h0[t][None], [tok[t + 1]], [t], kv_k, kv_v, [t], W, dims, 7, 1, precision="f64")
        np.testing.assert_allclose(out["h"][0], full["h"][0, 0, t], rtol=1e-10, atol=1e-12)
        if t + 2 < T:  # -log q(label) is the chain's depth-1 row loss
            assert math.isclose(-math.log(out["q"][0][tok[t + 2]]), full["row_loss"][1, 0, t], rel_tol=1e-9)


def test_draft_distribution_and_draw():
    cfg = synth.DRAFT_SMALL
    inp = synth.make_draft_inputs(cfg, 1)
    W = oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1)
    f = lambda t: t.float().numpy() if t.dtype.is_floating_point else t.numpy()
    out = od.draft_step(f(inp["parent_hidden"]), f(inp["frontier"]), f(inp["pos"]), f(inp["kv_k"]),
                        f(inp["kv_v"]), f(inp["ctx_len"]), W, dims, seed=11, offset=4, requests=[0, 3])
    for i, r in enumerate((0, 3)):
        q = out["q"][i]
        assert np.all(q >= 0) and math.isclose(q.sum(), 1.0, rel_tol=1e-12)
        u = od.draft_uniform(11, 4, r)
        assert out["y"][i] == ov.inverse_cdf(q, u)[0]
    # the draft stream is independent of the verifier's words 0 and 1
    ua, ur = ov.verify_uniforms(11, 4, 0, 0)
    assert od.draft_uniform(11, 4, 0) not in (float(ua), float(ur))
