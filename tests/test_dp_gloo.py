"""Data-parallel loss reduction across two CPU ranks (gloo): each rank owns
half of the packed rows; reducing (sum, count) pairs and then assembling
gives exactly the single-process loss under both denominator policies, while
averaging per-rank normalised losses does not (M7.6 §0x06A)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from deepseek_sequential_mtp_gb300 import dp, synth
from oracle import chain as oc


CFG = synth.SMALL_F32.with_(name="dp", B=4, T=24, D=2, doc_mean=7, pad_rows=1, pad_len=6)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_sums(rank, world):
    inp = synth.make_chain_inputs(CFG, seed=4)
    W = oc.weights_to_numpy(inp["weights"])
    rows = slice(rank * CFG.B // world, (rank + 1) * CFG.B // world)
    dims = oc.Dims(n_heads=CFG.n_heads, head_dim=CFG.head_dim, D=CFG.D)
    out = oc.chain_forward_loss(inp["tokens"].numpy()[rows], inp["seg"].numpy()[rows],
                                inp["pos"].numpy()[rows], inp["h0"].numpy()[rows], W, dims, lam=CFG.lam)
    sc = np.empty(2 * (CFG.D + 1))
    sc[0::2], sc[1::2] = out["sums"], out["counts"]
    return sc


def _worker(rank, world, port, results):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sc = torch.from_numpy(_rank_sums(rank, world))
        local = sc.clone()
        dp.allreduce_sums_counts(sc)
        n_pos = dp.global_positions(CFG.B // world, CFG.T)
        results[rank] = (sc.numpy().tolist(), local.numpy().tolist(), n_pos)
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(300)
def test_two_rank_reduction_matches_single_process():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        procs = [ctx.Process(target=_worker, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(240)
            assert p.exitcode == 0
        res = dict(results)
    reduced = np.array(res[0][0])
    assert np.array_equal(reduced, np.array(res[1][0]))  # every rank holds the same totals
    single = _rank_sums(0, 1)
    np.testing.assert_allclose(reduced, single, rtol=1e-12)
    assert res[0][2] == CFG.B * CFG.T
    for den in ("fixed", "masked_mean"):
        glob = oc.assemble_loss(reduced[0::2], reduced[1::2], CFG.B * CFG.T, CFG.D, CFG.lam, den)
        ref = oc.assemble_loss(single[0::2], single[1::2], CFG.B * CFG.T, CFG.D, CFG.lam, den)
        assert glob["loss_total"] == pytest.approx(ref["loss_total"], rel=1e-12)
    # averaging per-rank masked means is a different (wrong) objective when counts differ
    l0 = np.array(res[0][1])
    l1 = np.array(res[1][1])
    per_rank = [oc.assemble_loss(l[0::2], l[1::2], CFG.B * CFG.T // 2, CFG.D, CFG.lam, "masked_mean")["loss_total"]
                for l in (l0, l1)]
    ref = oc.assemble_loss(single[0::2], single[1::2], CFG.B * CFG.T, CFG.D, CFG.lam, "masked_mean")["loss_total"]
    assert not np.isclose(np.mean(per_rank), ref, rtol=1e-9)


def test_lambda_schedule_matches_the_oracle():
    from deepseek_sequential_mtp_gb300 import dp
    from oracle import chain as oc
    for t in (0, 1e12, 9.99e12, 10e12, 12e12, 14.8e12):
        assert dp.deepseek_v3_lambda(t) == oc.deepseek_v3_lambda(t)
