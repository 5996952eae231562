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


def _np(t):
    return t.float().numpy() if t.dtype.is_floating_point else t.numpy()


def test_round_of_one_is_the_draft_step():
    cfg = synth.DRAFT_SMALL
    inp = synth.make_draft_inputs(cfg, 2)
    W = oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1)
    args = [_np(inp[k]) for k in ("parent_hidden", "frontier", "pos", "kv_k", "kv_v", "ctx_len")]
    one = od.draft_step(*args, W, dims, 5, 9, requests=[1, 4])
    rnd = od.draft_round(*args, W, dims, 1, 5, 9, requests=[1, 4])
    for k in ("h", "q", "y", "margin"):
        np.testing.assert_array_equal(rnd[k][:, 0], one[k])


def test_round_steps_are_draft_steps_over_the_extended_cache():
    """Step s of a round = one draft step from step s-1's state and draw, at
    position pos + s, over the cache extended by the rows staged by steps
    0..s-1 (keys rotated at their own positions)."""
    cfg = synth.DRAFT_SMALL
    inp = synth.make_draft_inputs(cfg, 4)
    W = oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1)
    ph, fr, pos, kk, vv, L = (_np(inp[k]) for k in ("parent_hidden", "frontier", "pos", "kv_k", "kv_v", "ctx_len"))
    L = np.array([0, 7, 120, 299, 300])[:cfg.R].astype(np.int32)
    pos = L.copy()
    gamma = 3
    rnd = od.draft_round(ph, fr, pos, kk, vv, L, W, dims, gamma, 3, 1, precision="f64")
    for r in range(cfg.R):
        parent, f = ph[r], int(fr[r])
        k_ext, v_ext = kk[r][:L[r]].astype(np.float64), vv[r][:L[r]].astype(np.float64)
        for s in range(gamma):
            one = od.draft_step(parent[None], [f], [pos[r] + s], k_ext[None], v_ext[None], [L[r] + s], W, dims, 3, 1,
                                precision="f64")
            np.testing.assert_allclose(rnd["h"][r, s], one["h"][0], rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(rnd["q"][r, s], one["q"][0], rtol=1e-10, atol=1e-15)
            # the staged row of step s: the new row's rotated key and value
            u = oc.fusion(parent[None].astype(np.float64), [f], W, 0, dims, lambda a: a)
            _, k_new, v_new = oc.block_qkv(u, W, 0, [pos[r] + s], dims, lambda a: a)
            k_ext = np.concatenate([k_ext, k_new], axis=0)
            v_ext = np.concatenate([v_ext, v_new], axis=0)
            parent, f = rnd["h"][r, s], int(rnd["y"][r, s])
        # each step draws with its own counter
        for s in range(gamma):
            assert rnd["y"][r, s] == ov.inverse_cdf(rnd["q"][r, s], od.draft_uniform(3, 1, r, s))[0]


def test_forced_frontier_tokens():
    cfg = synth.DRAFT_SMALL
    inp = synth.make_draft_inputs(cfg, 6)
    W = oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1)
    args = [_np(inp[k]) for k in ("parent_hidden", "frontier", "pos", "kv_k", "kv_v", "ctx_len")]
    free = od.draft_round(*args, W, dims, 3, 8, 2, requests=[2])
    forced = od.draft_round(*args, W, dims, 3, 8, 2, requests=[2], forced_y=np.tile(free["y"][0], (cfg.R, 1)))
    for k in ("h", "q", "y"):
        np.testing.assert_array_equal(forced[k], free[k])
    other = (free["y"][0] + 1) % cfg.V
    moved = od.draft_round(*args, W, dims, 3, 8, 2, requests=[2], forced_y=np.tile(other, (cfg.R, 1)))
    np.testing.assert_array_equal(moved["q"][0, 0], free["q"][0, 0])  # step 0 does not see the forcing
    assert not np.allclose(moved["q"][0, 1], free["q"][0, 1])
    # the draft streams of different steps differ
    assert len({od.draft_uniform(8, 2, 2, s) for s in range(3)}) == 3
    # forcing the own states changes nothing; forcing other states moves later steps only
    same = od.draft_round(*args, W, dims, 3, 8, 2, requests=[2], forced_h=np.tile(free["h"][0], (cfg.R, 1, 1)))
    np.testing.assert_array_equal(same["q"], free["q"])
    noise = np.random.default_rng(0).standard_normal(free["h"][0].shape)  # RMSNorm ignores a pure rescale
    bumped = od.draft_round(*args, W, dims, 3, 8, 2, requests=[2],
                            forced_h=np.tile(free["h"][0] + noise, (cfg.R, 1, 1)))
    np.testing.assert_array_equal(bumped["q"][0, 0], free["q"][0, 0])
    assert not np.allclose(bumped["q"][0, 1], free["q"][0, 1])
