"""mtp_draft_step on the GPU against the draft-step oracle, through the C ABI.

Bars: the new row's state h within the bf16 chain bars (2e-2 + 2e-2|h|); the
draft distribution q within total variation 5e-3 and 2e-3 of max(q) per
entry; the draw y bit-exact against the inverse CDF of the kernel's own q at
the Philox word-2 uniform (excluding draws within 1e-6 of a CDF boundary),
and equal to the oracle's draw when the oracle's margin exceeds the q
tolerance."""
import numpy as np
import pytest
import torch

from deepseek_sequential_mtp_gb300 import lib, synth
from oracle import chain as oc
from oracle import draft as od
from oracle import verify as ov

pytestmark = pytest.mark.gpu


def _np(t):
    return t.float().cpu().numpy() if t.dtype.is_floating_point else t.cpu().numpy()


def run(cfg, inp, seed, offset, requests=None, W=None):
    dev = {k: v.cuda() for k, v in inp.items() if k != "weights"}
    wdev = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    step = lib.DraftStep(cfg, wdev)
    h = torch.empty((cfg.R, cfg.d), dtype=torch.bfloat16, device="cuda")
    g = step(dev["parent_hidden"], dev["frontier"], dev["pos"], dev["kv_k"], dev["kv_v"], dev["ctx_len"],
             seed, offset, h_out=h)
    lib.check_errors()
    W = W if W is not None else oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1, eps=cfg.eps, rope_base=cfg.rope_base)
    requests = list(range(cfg.R)) if requests is None else requests
    kvk = _np(inp["kv_k"][requests])
    kvv = _np(inp["kv_v"][requests])
    sel = lambda t: _np(t)[requests]
    r = od.draft_step(sel(inp["parent_hidden"]), sel(inp["frontier"]), sel(inp["pos"]), kvk, kvv,
                      sel(inp["ctx_len"]), W, dims, seed, offset, requests=range(len(requests)))
    # the oracle saw the subset renumbered; redo the draws with the true request ids
    r["y"], r["margin"] = [], []
    for i, rid in enumerate(requests):
        y, m = ov.inverse_cdf(r["q"][i], od.draft_uniform(seed, offset, rid))
        r["y"].append(y)
        r["margin"].append(m)
    return {k: _np(v) for k, v in g.items()}, r, requests


def check(g, r, requests, qbar=2e-3):
    gh, gq, gy = g["h"][requests], g["q"][requests], g["y"][requests]
    err = np.abs(gh - r["h"])
    assert np.all(err <= 2e-2 + 2e-2 * np.abs(r["h"])), err.max()
    assert np.all(np.isfinite(gq)) and np.allclose(gq.sum(1), 1.0, atol=1e-4)
    tv = 0.5 * np.abs(gq - r["q"]).sum(1)
    assert tv.max() < 5e-3, tv
    assert np.all(np.abs(gq - r["q"]).max(1) <= qbar * r["q"].max(1))
    return gy


@pytest.mark.parametrize("seed", [0, 1])
def test_small_full_parity(seed):
    cfg = synth.DRAFT_SMALL
    inp = synth.make_draft_inputs(cfg, seed)
    inp["ctx_len"] = torch.tensor([0, 1, 100, 299, 300][:cfg.R], dtype=torch.int32)  # empty and ragged caches
    inp["pos"] = inp["ctx_len"].clone()
    for offset in (0, 5):
        g, r, req = run(cfg, inp, seed=21, offset=offset)
        gy = check(g, r, req)
        for i, rid in enumerate(req):
            u = od.draft_uniform(21, offset, rid)
            y_own, m_own = ov.inverse_cdf(g["q"][rid].astype(np.float64), u)
            if m_own > 1e-6:
                assert gy[i] == y_own
            if r["margin"][i] > 5e-3:
                assert gy[i] == r["y"][i]


def test_hd128_split_keys_parity():
    """head_dim 128 with the cache split into two 576-key units: empty, one
    ragged tile, a split boundary crossed by one key, and a full cache."""
    cfg = synth.DRAFT_SMALL_HD128
    inp = synth.make_draft_inputs(cfg, 7)
    inp["ctx_len"] = torch.tensor([0, 63, 577, 1100], dtype=torch.int32)
    inp["pos"] = inp["ctx_len"].clone()
    g, r, req = run(cfg, inp, seed=9, offset=1)
    check(g, r, req)


def test_full_size_sampled_requests():
    """32 requests, module cache 8192 x d=7168 (56 x 128 heads), ffn 18432,
    V=129280; oracle on two requests, draw consistency on all 32."""
    cfg = synth.DRAFT_C5
    inp = synth.make_draft_inputs(cfg, 3, device="cuda")
    W = oc.weights_to_numpy(inp["weights"])
    g, r, req = run(cfg, {k: v for k, v in inp.items()}, seed=5, offset=2, requests=[0, 17], W=W)
    check(g, r, req)
    for rid in range(cfg.R):
        y_own, m_own = ov.inverse_cdf(g["q"][rid].astype(np.float64), od.draft_uniform(5, 2, rid))
        if m_own > 1e-6:
            assert g["y"][rid] == y_own


def _round_case(cfg, seed, ctx, gamma, dseed, offset):
    inp = synth.make_draft_inputs(cfg, seed)
    inp["ctx_len"] = torch.tensor(ctx, dtype=torch.int32)
    inp["pos"] = inp["ctx_len"].clone()
    dev = {k: v.cuda() for k, v in inp.items() if k != "weights"}
    wdev = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    rnd = lib.DraftRound(cfg, wdev, gamma)
    h = torch.empty((cfg.R, gamma, cfg.d), dtype=torch.bfloat16, device="cuda")
    g = rnd(dev["parent_hidden"], dev["frontier"], dev["pos"], dev["kv_k"], dev["kv_v"], dev["ctx_len"],
            dseed, offset, h_out=h)
    lib.check_errors()
    g = {k: _np(v) for k, v in g.items()}
    W = oc.weights_to_numpy(inp["weights"])
    dims = oc.Dims(n_heads=cfg.n_heads, head_dim=cfg.head_dim, D=1, eps=cfg.eps, rope_base=cfg.rope_base)
    # each step is compared on its own: the oracle continues from the GPU's state and draw of the
    # previous step (a wrong parent or frontier on the GPU would show as a mismatch of the next step)
    r = od.draft_round(*[_np(inp[k]) for k in ("parent_hidden", "frontier", "pos", "kv_k", "kv_v", "ctx_len")],
                       W, dims, gamma, dseed, offset, forced_y=g["y"], forced_h=g["h"])
    return g, r


def _check_round(cfg, g, r, dseed, offset, bar0=2e-3):
    """Per-step bars as for one draft step, except the per-entry q bar of
    steps >= 1: 5e-3 max(q).  The oracle continues from the GPU's state and
    draw, but its staged rows of earlier steps are its own (equal to the GPU's
    up to bf16 rounding flips), and with a small cache each staged row carries
    a large share of the attention weight (one flip moved q by ~0.2%)."""
    gamma = g["y"].shape[1]
    for s in range(gamma):
        err = np.abs(g["h"][:, s] - r["h"][:, s])
        assert np.all(err <= 2e-2 + 2e-2 * np.abs(r["h"][:, s])), (s, err.max())
        gq = g["q"][:, s]
        assert np.all(np.isfinite(gq)) and np.allclose(gq.sum(1), 1.0, atol=1e-4)
        assert (0.5 * np.abs(gq - r["q"][:, s]).sum(1)).max() < 5e-3, s
        bar = bar0 if s == 0 else 5e-3
        assert np.all(np.abs(gq - r["q"][:, s]).max(1) <= bar * r["q"][:, s].max(1)), s
        for rid in range(cfg.R):
            y_own, m_own = ov.inverse_cdf(gq[rid].astype(np.float64), od.draft_uniform(dseed, offset, rid, s))
            if m_own > 1e-6:
                assert g["y"][rid, s] == y_own, (rid, s)
            if r["margin"][rid, s] > 5e-3:
                assert g["y"][rid, s] == r["y"][rid, s], (rid, s)


@pytest.mark.parametrize("gamma", [2, 4])
def test_round_parity_hd64(gamma):
    """Recurrent drafting, head_dim 64: empty, one-key and ragged caches."""
    cfg = synth.DRAFT_SMALL
    g, r = _round_case(cfg, 3, [0, 1, 100, 299, 300][:cfg.R], gamma, dseed=31, offset=7)
    _check_round(cfg, g, r, 31, 7)


def test_round_parity_hd128():
    cfg = synth.DRAFT_SMALL_HD128
    g, r = _round_case(cfg, 8, [0, 63, 577, 1100], 3, dseed=2, offset=2**33 + 1)
    _check_round(cfg, g, r, 2, 2**33 + 1)


def test_round_of_one_is_the_step_and_feeds_verify():
    """mtp_draft_round with gamma = 1 equals mtp_draft_step bit for bit; a
    gamma = 3 round's q and draws drive spec_verify as its draft distributions
    and tokens, matching the verify oracle on the same inputs."""
    cfg = synth.DRAFT_SMALL
    inp = synth.make_draft_inputs(cfg, 5)
    dev = {k: v.cuda() for k, v in inp.items() if k != "weights"}
    wdev = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda()) for k, v in inp["weights"].items()}
    args = (dev["parent_hidden"], dev["frontier"], dev["pos"], dev["kv_k"], dev["kv_v"], dev["ctx_len"])
    one = lib.DraftRound(cfg, wdev, 1)(*args, 4, 9)
    step = lib.DraftStep(cfg, wdev)(*args, 4, 9)
    assert torch.equal(one["q"][:, 0], step["q"]) and torch.equal(one["y"][:, 0], step["y"])
    gamma = 3
    rnd = lib.DraftRound(cfg, wdev, gamma)(*args, 4, 9)
    vcase = synth.make_small_verify_case(2, R=cfg.R, gamma=gamma, V=cfg.V)
    p = vcase["p"].cuda()
    vout = lib.spec_verify(p, rnd["q"], rnd["y"], seed=17, offset=3)
    lib.check_errors()
    ref = ov.spec_verify(vcase["p"].numpy(), rnd["q"].cpu().numpy(), rnd["y"].cpu().numpy(), 17, 3)
    keep = ref["margin"] > 1e-7
    for kg, kr in (("accepted", "accepted"), ("next_token", "token"), ("n_emit", "n_emit"), ("status", "status")):
        np.testing.assert_array_equal(vout[kg].cpu().numpy()[keep], ref[kr][keep])
