"""Pins of the gradient oracle (oracle/grad.py): its loss equals the chain
oracle's fp64 loss, central finite differences of the chain oracle's numpy
forward match the autograd gradient on sampled coordinates of h^0 and of
every weight, and a depth's weights get no gradient from terms it cannot
reach (M7.6 §0x05: depth k's module affects terms k..D only)."""
import numpy as np
import pytest

from deepseek_sequential_mtp_gb300 import synth
from oracle import chain as oc
from oracle import grad as og

CFG = synth.ChainConfig(name="grad_tiny", B=2, T=12, d=32, n_heads=2, head_dim=16, ffn=40, V=50, D=2,
                        dtype="f32", lam=0.3, w_std=0.2, gain_std=0.2, tokens="uniform", layout="geometric",
                        doc_mean=5)


def _case(seed=3):
    inp = synth.make_chain_inputs(CFG, seed=seed)
    W = oc.weights_to_numpy(inp["weights"])
    W = {k: ([x.astype(np.float64) for x in v] if isinstance(v, list) else v.astype(np.float64)) for k, v in W.items()}
    args = (inp["tokens"].numpy(), inp["seg"].numpy(), inp["pos"].numpy(), inp["h0"].float().numpy().astype(np.float64))
    dims = oc.Dims(n_heads=CFG.n_heads, head_dim=CFG.head_dim, D=CFG.D, eps=CFG.eps, rope_base=CFG.rope_base)
    return args, W, dims


@pytest.mark.parametrize("den", ["fixed", "masked_mean", "global"])
def test_loss_equals_chain_oracle(den):
    args, W, dims = _case()
    g = og.chain_loss_grads(*args, W, dims, lam=0.3, den=den)
    r = oc.chain_forward_loss(*args, W, dims, precision="f64", lam=0.3, den=den)
    assert np.isclose(g["loss_total"], r["loss_total"], rtol=1e-12, atol=0)
    np.testing.assert_allclose(g["sums"], r["sums"], rtol=1e-12)
    np.testing.assert_array_equal(g["counts"], r["counts"])


def test_finite_differences():
    args, W, dims = _case(5)
    g = og.chain_loss_grads(*args, W, dims, lam=0.3, den="fixed")
    rng = np.random.default_rng(0)

    def loss(Wx, h0x):
        return oc.chain_forward_loss(args[0], args[1], args[2], h0x, Wx, dims, precision="f64",
                                     lam=0.3, den="fixed")["loss_total"]

    def check(get, grad, n=3):
        arr = get()
        for _ in range(n):
            idx = tuple(int(rng.integers(0, s)) for s in arr.shape)
            x0 = arr[idx]
            eps = 1e-5 * max(1.0, abs(x0))
            arr[idx] = x0 + eps
            lp = loss(W, args[3])
            arr[idx] = x0 - eps
            lm = loss(W, args[3])
            arr[idx] = x0
            fd = (lp - lm) / (2 * eps)
            assert abs(fd - grad[idx]) <= 1e-6 * max(1e-3, abs(grad[idx])) + 1e-9, (idx, fd, grad[idx])

    check(lambda: args[3], g["dh0"], n=6)
    for name in og.SHARED:
        check(lambda name=name: W[name], g["grads"][name], n=4)
    # embedding rows that are gathered (rows of unused tokens must get exactly zero)
    used = set(int(t) for t in args[0].reshape(-1))
    unused = [v for v in range(CFG.V) if v not in used]
    if unused:
        assert np.all(g["grads"]["embed"][unused] == 0.0)
    for name in og.PER_DEPTH:
        for k in range(CFG.D):
            check(lambda name=name, k=k: W[name][k], g["grads"][name][k], n=2)


def test_depth_ownership_of_gradients():
    args, W, dims = _case(7)
    g = og.chain_loss_grads(*args, W, dims, lam=0.3, den="fixed", with_main=False, depth_weights=[1.0, 0.0])
    for name in og.PER_DEPTH:
        assert np.all(g["grads"][name][1] == 0.0), name  # depth 2 only reaches term 2, whose weight is 0
        assert np.any(g["grads"][name][0] != 0.0), name
    # the shared head: main-only gradient plus depth-only gradient = gradient of the sum
    gm = og.chain_loss_grads(*args, W, dims, lam=0.0, den="fixed", with_main=True)
    gd = og.chain_loss_grads(*args, W, dims, lam=0.3, den="fixed", with_main=False)
    ga = og.chain_loss_grads(*args, W, dims, lam=0.3, den="fixed", with_main=True)
    np.testing.assert_allclose(ga["grads"]["head"], gm["grads"]["head"] + gd["grads"]["head"], rtol=1e-10,
                               atol=1e-14)
