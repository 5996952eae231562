"""Pins of the depth reductions ("M7.4 - Multi-Token Prediction Foundations"
§0x02C) and the DeepSeek-V3 lambda schedule (M7.6 §0x05): closed forms on the
page's worked counts (segment lengths [5] and [3, 4] give 9, 6, 3 supervised
pairs for horizons 1..3) with unit per-row losses."""
import math

import numpy as np
import pytest

from oracle import chain as oc

COUNTS = [20.0, 9.0, 6.0, 3.0]  # main term, then the page's horizons 1..3
W = [0.5, 0.3, 0.2]


def test_unit_losses_closed_forms():
    sums = list(COUNTS)  # every supervised row has loss 1
    n_pos = 40.0
    r = {den: oc.assemble_loss(sums, COUNTS, n_pos, 3, 0.3, den, depth_weights=W)["loss_total"] - 1.0
         for den in ("sum", "global", "weighted_pair", "masked_mean")}
    assert math.isclose(r["sum"], 0.5 * 9 + 0.3 * 6 + 0.2 * 3 + 20.0 - 1.0)  # main term is S_0 under sum
    assert math.isclose(r["global"], (0.5 * 9 + 0.3 * 6 + 0.2 * 3) / 18.0)
    assert math.isclose(r["weighted_pair"], 1.0)  # a weighted average of unit losses
    assert math.isclose(r["masked_mean"], sum(W))  # every horizon counts fully, whatever its size
    fixed = oc.assemble_loss(sums, COUNTS, n_pos, 3, 0.3, "fixed", depth_weights=W)
    assert math.isclose(fixed["loss_total"], 20 / 40 + (0.5 * 9 + 0.3 * 6 + 0.2 * 3) / 40)


def test_head_mean_vs_global_horizon_weights():
    """head mean: the 3-row horizon moves the aggregate as much as the 9-row one; global: in
    proportion to its rows (the page's comparison)."""
    base = [0.0, 9.0, 6.0, 3.0]
    def bump(k, den):
        s = list(base)
        s[k] += COUNTS[k]  # raise horizon k's mean loss by 1
        a = oc.assemble_loss(s, COUNTS, 1.0, 3, 0.3, den, with_main=False, depth_weights=[1, 1, 1])["loss_total"]
        b = oc.assemble_loss(base, COUNTS, 1.0, 3, 0.3, den, with_main=False, depth_weights=[1, 1, 1])["loss_total"]
        return a - b
    assert math.isclose(bump(1, "masked_mean"), bump(3, "masked_mean"))
    assert math.isclose(bump(1, "global") / bump(3, "global"), 9.0 / 3.0)


def test_uniform_weights_are_the_paper_objective():
    rng = np.random.default_rng(0)
    sums = rng.random(4) * 10
    for den in ("fixed", "masked_mean"):
        a = oc.assemble_loss(sums, COUNTS, 50.0, 3, 0.3, den)
        b = oc.assemble_loss(sums, COUNTS, 50.0, 3, 0.3, den, depth_weights=[0.1, 0.1, 0.1])
        assert math.isclose(a["loss_total"], b["loss_total"])
        assert math.isclose(a["loss_total"], a["loss_main"] + 0.3 / 3 * sum(a["loss_mtp"]))


def test_weighted_pair_ignores_weight_scale_and_empty_terms():
    sums = [1.0, 4.0, 0.0, 2.0]
    counts = [2.0, 4.0, 0.0, 2.0]
    a = oc.assemble_loss(sums, counts, 1.0, 3, 0.3, "weighted_pair", depth_weights=[1, 2, 3])
    b = oc.assemble_loss(sums, counts, 1.0, 3, 0.3, "weighted_pair", depth_weights=[10, 20, 30])
    assert math.isclose(a["loss_total"], b["loss_total"])
    assert math.isclose(a["loss_total"] - a["loss_main"], (1 * 4 + 3 * 2) / (1 * 4 + 3 * 2))
    empty = oc.assemble_loss([1.0, 0, 0, 0], [2.0, 0, 0, 0], 1.0, 3, 0.3, "global")
    assert empty["loss_mtp"] == [0.0, 0.0, 0.0] and empty["loss_total"] == 0.5
    with pytest.raises(ValueError):
        oc.assemble_loss(sums, counts, 1.0, 3, 0.3, "median")


def test_deepseek_v3_lambda_schedule():
    assert oc.deepseek_v3_lambda(0) == 0.3
    assert oc.deepseek_v3_lambda(9.999e12) == 0.3
    assert oc.deepseek_v3_lambda(10e12) == 0.1
    assert oc.deepseek_v3_lambda(14.8e12) == 0.1
