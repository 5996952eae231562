"""Pins of the oracle's speculative verifier and Philox generator against the
pages' worked example, the closed form for the expected emitted length,
published known-answer vectors and exact distributional identities."""
import math

import numpy as np
import pytest

from conftest import read_golden
from oracle import verify as ov


def test_philox_known_answers():
    _, rows = read_golden("philox4x32_10_kat.txt")
    assert len(rows) == 3
    for row in rows:
        w = [int(x, 16) for x in row]
        out = ov.philox4x32_10(w[0:4], w[4:6])
        assert [int(o) for o in out] == w[6:10]


def test_uniforms_are_uniform():
    r = np.arange(200)[:, None]
    j = np.arange(50)[None, :]
    ua, ur = ov.verify_uniforms(12345, 77, r, j)
    for u in (ua, ur):
        assert u.min() >= 0 and u.max() < 1
        assert abs(u.mean() - 0.5) < 0.01
        assert abs(u.var() - 1 / 12) < 0.005
        assert np.all(u * 2**24 == np.floor(u * 2**24))  # 24-bit grid
    assert np.corrcoef(ua.ravel(), ur.ravel())[0, 1] < 0.05


def _emitted_distribution_single(p, q):
    """Exact distribution of the token emitted at position 0 by the oracle's
    selector, integrating over y ~ q and over the two uniforms on fine grids
    (every decision of the selector is a threshold on one uniform)."""
    V = len(p)
    grid = (np.arange(4096) + 0.5) / 4096
    out = np.zeros(V)
    P = np.stack([p, p])  # γ = 1: row 0 verifies y, row 1 is the bonus row
    Q = q[None, :]
    for y in range(V):
        if q[y] <= 0:
            continue
        # accept probability = measure of {u : u < min(1, p/q)}
        acc = np.mean([ov.verify_one(P, Q, [y], [u], [0.5, 0.5])["n_emit"] == 2 for u in grid[::16]])
        res = ov.verify_one(P, Q, [y], [min(1.0, p[y] / q[y]) + 1e-9 if p[y] < q[y] else 0.0], [0.5, 0.5])
        out[y] += q[y] * min(1.0, p[y] / q[y])
        assert abs(acc - min(1.0, p[y] / q[y])) <= 16 / 4096 + 1e-12
        if p[y] < q[y]:
            counts = np.zeros(V)
            for u2 in grid:
                c = ov.verify_one(P, Q, [y], [0.999999], [u2, 0.5])
                assert c["status"] == ov.STATUS_OK and c["n_emit"] == 1
                counts[c["token"]] += 1
            out += q[y] * (1.0 - p[y] / q[y]) * counts / len(grid)
            assert res["accepted"] == 0
    return out


def test_single_token_identity_worked_example():
    f, _ = read_golden("spec_pq_example.txt")
    p = np.array([float(v) for v in f["p"]])
    q = np.array([float(v) for v in f["q"]])
    assert np.allclose(np.minimum(p, q), [float(v) for v in f["min_pq"]])
    assert math.isclose(np.minimum(p, q).sum(), float(f["accepted_mass"][0]))
    assert math.isclose(1 - np.minimum(p, q).sum(), float(f["reject_probability"][0]))
    # the oracle's correction on every rejection is index 0 (residual [1,0,0])
    P = np.stack([p, p])
    for y in (1, 2):
        for u2 in np.linspace(0, 0.999, 50):
            r = ov.verify_one(P, q[None, :], [y], [0.9999], [u2, 0.5])
            assert r["token"] == 0
    resid = np.maximum(p - q, 0)
    assert np.allclose(resid / resid.sum(), [float(v) for v in f["residual_normalised"]])
    dist = _emitted_distribution_single(p, q)
    assert np.allclose(dist, p, atol=1e-3)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_first_emitted_token_is_target_distributed_exactly(seed):
    rng = np.random.default_rng(seed)
    V = 6
    p = rng.dirichlet(np.ones(V) * 0.7)
    q = rng.dirichlet(np.ones(V) * 0.7)
    dist = _emitted_distribution_single(p, q)
    assert np.allclose(dist, p, atol=2e-3)


def test_expected_emitted_closed_form_monte_carlo():
    """E[N_emit] = (1 - α^{γ+1}) / (1 - α) (speculative-decoding page), by
    Monte Carlo over the oracle with Philox uniforms; α = Σ min(p, q)."""
    f, _ = read_golden("expected_emitted.txt")
    alpha, gamma = float(f["alpha"][0]), int(f["gamma"][0])
    closed = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(closed - float(f["expected_emitted"][0])) < 5e-4
    p_row = np.array([0.7, 0.3, 0.0])
    q_row = np.array([0.7, 0.0, 0.3])
    assert math.isclose(np.minimum(p_row, q_row).sum(), alpha)
    for g, want in ((gamma, closed), (4, (1 - alpha ** 5) / (1 - alpha))):
        R = 6000
        rng = np.random.default_rng(g)
        p = np.broadcast_to(p_row, (R, g + 1, 3))
        q = np.broadcast_to(q_row, (R, g, 3))
        y = rng.choice(3, size=(R, g), p=q_row)
        out = ov.spec_verify(p, q, y, seed=2024 + g, offset=0)
        assert np.all(out["status"] == ov.STATUS_OK)
        n = out["n_emit"]
        se = n.std() / math.sqrt(R)
        assert abs(n.mean() - want) < 4 * se, (n.mean(), want, se)
        assert np.all(n == out["accepted"] + 1)


def test_chi_square_first_token():
    rng = np.random.default_rng(5)
    V, R, g = 8, 20000, 2
    p_row = rng.dirichlet(np.ones(V))
    q_row = rng.dirichlet(np.ones(V))
    p = np.broadcast_to(p_row, (R, g + 1, V))
    q = np.broadcast_to(q_row, (R, g, V))
    y = rng.choice(V, size=(R, g), p=q_row)
    out = ov.spec_verify(p, q, y, seed=99, offset=3)
    first = np.where(out["accepted"] > 0, y[:, 0], out["token"])
    obs = np.bincount(first, minlength=V)
    exp = p_row * R
    chi2 = ((obs - exp) ** 2 / exp).sum()
    assert chi2 < 30.0  # 7 dof: P(chi2 > 30) ~ 1e-4


def test_deterministic_cases():
    V, g = 5, 3
    p = np.tile(np.array([0.1, 0.2, 0.3, 0.25, 0.15]), (g + 1, 1))
    q = p[:g].copy()
    ua, ur = ov.verify_uniforms(1, 0, 0, np.arange(g + 1))
    r = ov.verify_one(p, q, [2, 3, 4], ua, ur)  # p == q: always accept + bonus
    assert (r["accepted"], r["n_emit"]) == (3, 4) and 0 <= r["token"] < V
    q1 = np.zeros((g, V))
    q1[:, 2] = 1.0
    p1 = p.copy()
    p1[:, 2] = 0.0
    p1 /= p1.sum(1, keepdims=True)
    r = ov.verify_one(p1, q1, [2, 2, 2], ua, ur)  # p[y] = 0: always reject
    assert r["accepted"] == 0 and r["n_emit"] == 1 and r["token"] != 2


def test_budget_eos_and_error_statuses():
    V, g = 4, 2
    p = np.full((g + 1, V), 0.25)
    q = np.full((g, V), 0.25)
    u_acc, u_res = [0.1, 0.1, 0.1], [0.5, 0.5, 0.5]
    assert ov.verify_one(p, q, [1, 2], u_acc, u_res, remaining=1)["n_emit"] == 1
    r = ov.verify_one(p, q, [1, 2], u_acc, u_res, remaining=2)
    assert (r["n_emit"], r["token"]) == (2, -1)
    r = ov.verify_one(p, q, [3, 2], u_acc, u_res, eos=3)
    assert (r["accepted"], r["n_emit"], r["token"]) == (1, 1, -1)
    assert ov.verify_one(p, q, [1, 2], u_acc, u_res, remaining=0)["status"] == ov.STATUS_INVALID_BUDGET
    q0 = q.copy()
    q0[0, 1] = 0.0
    assert ov.verify_one(p, q0, [1, 2], u_acc, u_res)["status"] == ov.STATUS_INVALID_DRAFT
    assert ov.verify_one(p, q, [4, 2], u_acc, u_res)["status"] == ov.STATUS_INVALID_DRAFT
    pn = p.copy()
    pn[0] = [0.1, 0.1, 0.4, np.nan]  # p[y]/q[y] = 0.4: u = 0.99 rejects and reads row 0
    r = ov.verify_one(pn, q, [1, 2], [0.99, 0.1, 0.1], u_res)
    assert r["status"] == ov.STATUS_INVALID_PROBS
    ph = 0.5 * p  # unnormalised: p <= q everywhere, a rejection has no residual
    r = ov.verify_one(ph, q, [1, 2], [0.9, 0.1, 0.1], u_res)
    assert r["status"] == ov.STATUS_ZERO_RESIDUAL


def test_inverse_cdf_picks_smallest_crossing_index():
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    assert ov.inverse_cdf(w, 0.0)[0] == 1  # zero-mass index 0 never picked
    assert ov.inverse_cdf(w, 0.2499)[0] == 1
    assert ov.inverse_cdf(w, 0.25)[0] == 3  # strict '>' moves past the boundary
    assert ov.inverse_cdf(w, 0.7499)[0] == 3
    assert ov.inverse_cdf(w, 0.75)[0] == 4
    assert ov.inverse_cdf(w, 1 - 2**-24)[0] == 4
