"""Pins of the oracle's MTP chain: closed forms and special cases of each
component, the coordinate expansion of the fusion projection, packing
invariance, the causal dependency structure of the depth chain and the loss
relations the pages state."""
import math

import numpy as np
import pytest
import scipy.special
import torch

from deepseek_sequential_mtp_gb300 import synth
from oracle import chain as oc
from oracle.bf16 import round_bf16


def test_round_bf16_matches_library_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(20000) * 10 ** rng.uniform(-6, 6, 20000),
                        [1.0, 1 + 2**-8, 1 + 3 * 2**-8, -2.5, 0.0, 65504.0]])
    x32 = x.astype(np.float32)
    lib = torch.from_numpy(x32).to(torch.bfloat16).float().numpy().astype(np.float64)
    assert np.array_equal(round_bf16(x32.astype(np.float64)), lib)
    assert round_bf16(1 + 2**-8) == 1.0        # tie -> even
    assert round_bf16(1 + 3 * 2**-8) == 1 + 2**-6


def test_rmsnorm_closed_forms():
    g = np.array([0.5, 2.0, -1.0, 3.0])
    for c in (2.0, -0.3, 7.0):
        z = np.full(4, c)
        want = g * np.sign(c) * abs(c) / math.sqrt(c * c + 1e-6)
        assert np.allclose(oc.rmsnorm(z, g, 1e-6), want, rtol=1e-14)
    z = np.array([3.0, -4.0, 0.0, 12.0])   # mean square = 169/4
    assert np.allclose(oc.rmsnorm(z, np.ones(4), 0.0), z / 6.5, rtol=1e-14)


def test_rope_properties():
    rng = np.random.default_rng(1)
    H, hd = 2, 8
    x = rng.standard_normal((5, H * hd))
    assert np.allclose(oc.rope(x, np.zeros(5), H, hd, 10000.0), x)
    y = oc.rope(x, np.arange(5) * 7, H, hd, 10000.0)
    xp = x.reshape(5, H, 2, hd // 2)
    yp = y.reshape(5, H, 2, hd // 2)
    assert np.allclose((xp ** 2).sum(2), (yp ** 2).sum(2))  # each pair rotates
    q, k = rng.standard_normal((1, H * hd)), rng.standard_normal((1, H * hd))
    dots = [(oc.rope(q, [a + 5], H, hd, 500.0) @ oc.rope(k, [a], H, hd, 500.0).T).item()
            for a in (0, 3, 11)]
    assert np.allclose(dots, dots[0])  # relative-position property
    assert np.array_equal(oc.rope(x, np.arange(5), H, hd, 0.0), x)


def test_rope_unit_vectors():
    """Rotate-half RoPE at head_dim 4, base 10000: coordinate i pairs with
    i + 2 and turns by pos * 10000^(-2i/4), i.e. by pos rad for i = 0 and by
    pos / 100 rad for i = 1; a unit vector on coordinate i lands on
    (cos, sin) of that angle in coordinates (i, i + 2) and nowhere else.  A
    wrong frequency exponent, pairing (adjacent instead of halves) or sign of
    the sine fails here."""
    p = 3.0
    e = np.eye(4)
    y = oc.rope(e, np.full(4, p), 1, 4, 10000.0)
    want = np.zeros((4, 4))
    want[0, 0], want[0, 2] = np.cos(p), np.sin(p)            # x0 -> (x0, x2), angle p
    want[2, 2], want[2, 0] = np.cos(p), -np.sin(p)           # x2 -> rotated by the same angle
    want[1, 1], want[1, 3] = np.cos(p / 100), np.sin(p / 100)
    want[3, 3], want[3, 1] = np.cos(p / 100), -np.sin(p / 100)
    np.testing.assert_allclose(y, want, atol=1e-12)
    # two heads rotate independently with the same per-head frequencies
    y2 = oc.rope(np.tile(e[0], (1, 2)), [p], 2, 4, 10000.0)
    np.testing.assert_allclose(y2[0], np.tile(want[0], 2), atol=1e-12)


def test_attention_special_cases():
    rng = np.random.default_rng(2)
    n, H, hd = 6, 2, 4
    q, k, v = (rng.standard_normal((n, H * hd)) for _ in range(3))
    seg = [0, 0, 0, 1, 2, 2]
    bases = list(range(n))
    o = oc.segment_causal_attention(q, k, v, seg, bases, H, hd)
    assert np.allclose(o[0], v[0]) and np.allclose(o[3], v[3]) and np.allclose(o[4], v[4])
    o0 = oc.segment_causal_attention(np.zeros_like(q), k, v, seg, bases, H, hd)
    assert np.allclose(o0[2], v[:3].mean(0)) and np.allclose(o0[5], v[4:6].mean(0))
    # explicit softmax for row 2 head 1
    s = np.array([q[2, 4:] @ k[j, 4:] for j in range(3)]) / 2.0
    w = np.exp(s - s.max())
    w /= w.sum()
    assert np.allclose(o[2, 4:], w @ v[:3, 4:])


def test_cross_entropy_special_cases():
    rng = np.random.default_rng(3)
    d, V, n = 8, 50, 4
    dims = oc.Dims(n_heads=1, head_dim=d, D=1)
    h = rng.standard_normal((n, d))
    W = {"out_norm": np.ones(d), "head": np.zeros((V, d))}
    labels = [0, 7, 49, 3]
    assert np.allclose(oc.row_cross_entropy(h, labels, W, dims, lambda a: a), math.log(V))
    W["head"] = rng.standard_normal((V, d))
    x = oc.rmsnorm(h, np.ones(d), 1e-6)
    z = x @ W["head"].T
    want = scipy.special.logsumexp(z, axis=1) - z[np.arange(n), labels]
    got = oc.row_cross_entropy(h, labels, W, dims, lambda a: a, vocab_chunk=7)
    assert np.allclose(got, want, rtol=1e-12)
    W["head"] = np.zeros((V, d))
    W["head"][5] = 100.0 * x[0] / np.dot(x[0], x[0])  # logit 100 at label 5
    assert oc.row_cross_entropy(h[:1], [5], W, dims, lambda a: a)[0] < 1e-30 + V * math.exp(-100)


def _tiny_weights(cfg, seed):
    return oc.weights_to_numpy(synth.make_weights(cfg, seed))


def test_projection_coordinate_expansion():
    """u_r = Σ_j M_{r,j} h̄_j + Σ_j M_{r,d+j} ē_j (M7.6 §0x03C): with W_o = 0
    and W_down = 0 the block is the identity, so the module returns u."""
    cfg = synth.ChainConfig(name="t", B=1, T=3, d=4, n_heads=1, head_dim=4, ffn=4, V=9,
                            D=1, dtype="f32", w_std=0.5, gain_std=0.3)
    W = _tiny_weights(cfg, 4)
    W["wo"][0][:] = 0.0
    W["w_down"][0][:] = 0.0
    dims = oc.Dims(n_heads=1, head_dim=4, D=1)
    rng = np.random.default_rng(4)
    prev = rng.standard_normal((3, 4)) * 3.0
    toks = [2, 8, 5]
    got = oc.mtp_module(prev, toks, W, 0, [0, 1, 2], [0, 0, 0], [0, 1, 2], dims, lambda a: a)
    M = W["eh_proj"][0].astype(np.float64)
    for i in range(3):
        hb = W["hnorm"][0].astype(np.float64) * prev[i] / math.sqrt(np.mean(prev[i] ** 2) + 1e-6)
        e = W["embed"][toks[i]].astype(np.float64)
        eb = W["enorm"][0].astype(np.float64) * e / math.sqrt(np.mean(e ** 2) + 1e-6)
        for r in range(4):
            u_r = sum(M[r, j] * hb[j] for j in range(4)) + sum(M[r, 4 + j] * eb[j] for j in range(4))
            assert math.isclose(got[i, r], u_r, rel_tol=1e-9, abs_tol=1e-12)


def test_block_tail_swiglu_coordinates():
    """FFN of the block (M7.6 §0x03C with the dense stand-in
    h = a + (silu(y W_g^T) * (y W_u^T)) W_d^T, y = Norm_f(a)): with one-hot
    rows in W_g and W_u and W_d an injection of the ffn coordinates into the
    d outputs, h - a is silu(y_i) * y_j at the coordinate W_d sends the pair
    to and zero elsewhere.  The pairs are asymmetric and W_d is not square,
    so a swapped gate/up, a silu on the up branch or a transposed W_d fails.
    The output projection is checked the same way: with W_d = 0 and W_o a
    cyclic permutation, h = u + o W_o^T picks o at the permuted coordinate."""
    d, ffn = 6, 4
    cfg = synth.ChainConfig(name="t", B=1, T=3, d=d, n_heads=1, head_dim=d, ffn=ffn, V=9,
                            D=1, dtype="f32", w_std=0.5, gain_std=0.3)
    W = _tiny_weights(cfg, 7)
    dims = oc.Dims(n_heads=1, head_dim=d, D=1)
    rng = np.random.default_rng(8)
    u = rng.standard_normal((3, d)) * 2.0
    o = rng.standard_normal((3, d))
    gate_src, up_src, dest = [1, 4, 0, 5], [3, 2, 5, 1], [3, 0, 5, 1]
    W["wo"][0][:] = 0.0
    W["w_gate"][0][:] = 0.0
    W["w_up"][0][:] = 0.0
    W["w_down"][0][:] = 0.0
    for m in range(ffn):
        W["w_gate"][0][m, gate_src[m]] = 1.0
        W["w_up"][0][m, up_src[m]] = 1.0
        W["w_down"][0][dest[m], m] = 1.0
    h = oc.block_tail(u, o, W, 0, dims, lambda a: a)
    g = W["ffn_norm"][0].astype(np.float64)
    for i in range(3):
        y = g * u[i] / math.sqrt(np.mean(u[i] ** 2) + 1e-6)
        want = np.zeros(d)
        for m in range(ffn):
            want[dest[m]] = y[gate_src[m]] * scipy.special.expit(y[gate_src[m]]) * y[up_src[m]]
        np.testing.assert_allclose(h[i] - u[i], want, rtol=1e-12, atol=1e-14)
    # the output projection's orientation: W_o[r, perm[r]] = 1
    perm = [2, 0, 4, 1, 5, 3]
    W["w_down"][0][:] = 0.0
    for r in range(d):
        W["wo"][0][r, perm[r]] = 1.0
    h = oc.block_tail(u, o, W, 0, dims, lambda a: a)
    np.testing.assert_allclose(h, u + o[:, perm], rtol=1e-14)


def _run(cfg, batch, h0, W, **kw):
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=cfg.D)
    return oc.chain_forward_loss(batch["tokens"], batch["seg"], batch["pos"], h0, W, dims, **kw)


SMALL = synth.ChainConfig(name="s", B=1, T=14, d=16, n_heads=2, head_dim=8, ffn=24, V=40,
                          D=3, dtype="f32", w_std=0.3, gain_std=0.2)


def test_packing_invariance():
    """A packed row [doc A | doc B] equals each document run alone: the
    segment rule restricts rows and the attention graph (M7.6 §0x04C)."""
    rng = np.random.default_rng(5)
    W = _tiny_weights(SMALL, 6)
    la, lb = 6, 8
    toks = rng.integers(0, SMALL.V, la + lb)
    h0 = rng.standard_normal((la + lb, SMALL.d))
    packed = {"tokens": toks[None], "seg": np.array([[0] * la + [1] * lb]),
              "pos": np.array([list(range(la)) + list(range(lb))])}
    alone = {"tokens": np.stack([np.r_[toks[:la], np.zeros(lb, int)],
                                 np.r_[toks[la:], np.zeros(la, int)]]),
             "seg": np.array([[0] * la + [-1] * lb, [0] * lb + [-1] * la]),
             "pos": np.array([list(range(la)) + [0] * lb, list(range(lb)) + [0] * la])}
    h0_alone = np.stack([np.r_[h0[:la], np.zeros((lb, SMALL.d))],
                         np.r_[h0[la:], np.zeros((la, SMALL.d))]])
    P = _run(SMALL, packed, h0[None], W)
    A = _run(SMALL.with_(B=2), alone, h0_alone, W)
    for k in range(SMALL.D):
        np.testing.assert_allclose(P["h"][k, 0, :la], A["h"][k, 0, :la], rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(P["h"][k, 0, la:], A["h"][k, 1, :lb], rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(P["row_loss"][:, 0, :la], A["row_loss"][:, 0, :la], rtol=1e-12)
    np.testing.assert_allclose(P["row_loss"][:, 0, la:], A["row_loss"][:, 1, :lb], rtol=1e-12)
    assert np.array_equal(P["counts"], A["counts"])


def test_causal_dependency_on_tokens():
    """h^k_i reads x_{i'+k'} for i' <= i, k' <= k only: perturbing token x_j
    leaves every h^k_i with i + k < j unchanged and changes those at i + k = j;
    the depth-k loss of row i additionally reads its label x_{i+k+1}."""
    rng = np.random.default_rng(7)
    W = _tiny_weights(SMALL, 8)
    T = SMALL.T
    batch = {"tokens": rng.integers(0, SMALL.V, (1, T)), "seg": np.zeros((1, T), int),
             "pos": np.arange(T)[None]}
    h0 = rng.standard_normal((1, T, SMALL.d))
    base = _run(SMALL, batch, h0, W)
    j = 8
    b2 = dict(batch, tokens=batch["tokens"].copy())
    b2["tokens"][0, j] = (b2["tokens"][0, j] + 1) % SMALL.V
    pert = _run(SMALL, b2, h0, W)
    for k in range(1, SMALL.D + 1):
        for i in range(T - k):
            same = np.array_equal(base["h"][k - 1, 0, i], pert["h"][k - 1, 0, i])
            if i + k < j:
                assert same, (k, i)
            elif i + k == j:
                assert not same, (k, i)
        i = j - k - 1  # its label is x_j, its state is unchanged
        if i >= 0 and np.isfinite(base["row_loss"][k, 0, i]):
            assert np.array_equal(base["h"][k - 1, 0, i], pert["h"][k - 1, 0, i])
            assert base["row_loss"][k, 0, i] != pert["row_loss"][k, 0, i]
    # h^0 perturbation only moves rows at or after its base (causal attention)
    h0b = h0.copy()
    h0b[0, 5] += 0.5
    pert = _run(SMALL, batch, h0b, W)
    for k in range(SMALL.D):
        assert np.array_equal(base["h"][k, 0, :5], pert["h"][k, 0, :5], equal_nan=True)
        assert not np.array_equal(base["h"][k, 0, 5], pert["h"][k, 0, 5])


def test_depth_ownership_by_finite_differences():
    """∂L^(k)/∂θ_j vanishes for j > k and not for j <= k: a depth-j module
    receives its own loss and every deeper loss that traverses it, and no
    shallower one (M7.6 §0x05, gradient ledger)."""
    rng = np.random.default_rng(9)
    W = _tiny_weights(SMALL, 10)
    T = SMALL.T
    batch = {"tokens": rng.integers(0, SMALL.V, (1, T)), "seg": np.zeros((1, T), int),
             "pos": np.arange(T)[None]}
    h0 = rng.standard_normal((1, T, SMALL.d))
    base = _run(SMALL, batch, h0, W, den="masked_mean")
    eps = 1e-6
    for j in range(SMALL.D):
        W2 = {k: ([a.copy() for a in v] if isinstance(v, list) else v) for k, v in W.items()}
        W2["eh_proj"][j] = W2["eh_proj"][j] + eps * rng.standard_normal(W2["eh_proj"][j].shape)
        pert = _run(SMALL, batch, h0, W2, den="masked_mean")
        fd = (np.array(pert["loss_mtp"]) - np.array(base["loss_mtp"])) / eps
        assert pert["loss_main"] == base["loss_main"]
        for k in range(SMALL.D):
            if k < j:
                assert fd[k] == 0.0
            else:
                assert abs(fd[k]) > 1e-6


def test_loss_relations_and_policies():
    rng = np.random.default_rng(11)
    cfg = SMALL.with_(B=2, T=9, D=3)
    W = _tiny_weights(cfg, 12)
    batch = synth.make_batch(cfg.with_(layout="geometric", doc_mean=4), 3)
    h0 = rng.standard_normal((2, 9, cfg.d))
    fixed = _run(cfg, batch, h0, W, den="fixed")
    mean = _run(cfg, batch, h0, W, den="masked_mean")
    BT = cfg.B * cfg.T
    for k in range(cfg.D):  # L_paper = (|V_k| / T) L_valid  (M7.6 §0x05)
        if mean["counts"][k + 1] > 0:
            assert math.isclose(fixed["loss_mtp"][k], mean["counts"][k + 1] / BT * mean["loss_mtp"][k])
    lam0 = _run(cfg, batch, h0, W, lam=0.0)
    assert lam0["loss_total"] == lam0["loss_main"]
    assert math.isclose(fixed["loss_total"], fixed["loss_main"] + 0.3 / 3 * sum(fixed["loss_mtp"]))
    # an exhausted depth contributes a 0 term that stays in the D-way mean
    short = {"tokens": batch["tokens"][:, :3], "seg": np.zeros((2, 3), int),
             "pos": np.tile(np.arange(3), (2, 1))}
    out = _run(cfg.with_(T=3), short, h0[:, :3], W, den="masked_mean")
    assert list(out["counts"][1:]) == [2, 0, 0]
    assert out["loss_mtp"][1] == 0.0 and out["loss_mtp"][2] == 0.0
    assert math.isclose(out["loss_total"], out["loss_main"] + 0.3 / 3 * out["loss_mtp"][0])


def test_bf16_mode_stays_on_grid():
    cfg = synth.SMALL_BF16.with_(B=1, T=40, D=2)
    inp = synth.make_chain_inputs(cfg, 13)
    W = oc.weights_to_numpy(inp["weights"])
    batch = {k: inp[k].numpy() for k in ("tokens", "seg", "pos")}
    out = _run(cfg, batch, inp["h0"].float().numpy(), W, precision="bf16")
    h = out["h"][np.isfinite(out["h"])]
    assert h.size > 0 and np.array_equal(round_bf16(h), h)
    ref = _run(cfg, batch, inp["h0"].float().numpy(), W, precision="f64")
    m = np.isfinite(ref["h"])
    assert np.max(np.abs(ref["h"][m] - out["h"][m])) < 0.1
