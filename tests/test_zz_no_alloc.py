"""The allocation-free chain-loss entry point (mtp_chain_loss_noalloc), called
through the C ABI, against the workspace entry point (mtp_chain_loss).

It serves callers that cannot allocate device memory: its workspace is a
fixed array inside the library.  Two calls in a row, on different inputs,
must each match the workspace entry point within the chain parity
tolerances; a shape whose workspace exceeds the array is refused before any
device work.  This file is collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from deepseek_sequential_mtp_gb300 import lib, synth

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    fn = lib.load().mtp_chain_loss_noalloc
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    fn.restype = i32
    fn.argtypes = [ctypes.POINTER(lib.Dims), ctypes.POINTER(lib.Weights), vp, vp, vp, vp, ctypes.c_float,
                   i32, i32, vp, vp, vp, vp, vp]
    return fn


def _dev(inp):
    out = {k: v.cuda() for k, v in inp.items() if k != "weights"}
    out["weights"] = {k: ([t.cuda() for t in v] if isinstance(v, list) else v.cuda())
                      for k, v in inp["weights"].items()}
    return out


def _noalloc_call(cfg, x, den):
    D = cfg.D
    dims = lib.make_dims(cfg)
    w = lib.ChainWeights(x["weights"], D)
    res = {"sums_counts": torch.empty(2 * (D + 1), dtype=torch.float64, device="cuda"),
           "losses": torch.empty(D + 2, dtype=torch.float32, device="cuda"),
           "row_loss": torch.empty((D + 1, cfg.B, cfg.T), dtype=torch.float32, device="cuda"),
           "h": torch.empty((D, cfg.B, cfg.T, cfg.d), dtype=synth.torch_dtype(cfg.dtype), device="cuda")}
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = _noalloc_fn()(ctypes.byref(dims), ctypes.byref(w.struct), p(x["tokens"]), p(x["seg"]), p(x["pos"]),
                       p(x["h0"]), cfg.lam, lib.DEN[den], 1, p(res["sums_counts"]), p(res["losses"]),
                       p(res["row_loss"]), p(res["h"]),
                       ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, lib.load().mtp_status_string(st)
    return res


@pytest.mark.parametrize("name", ["small_bf16_D2", "small_f32_D3"])
def test_noalloc_matches_workspace_entry_point_twice(name):
    cfg = synth.CHAIN_CONFIGS[name]
    bf16 = cfg.dtype == "bf16"
    for seed, den in ((21, "fixed"), (22, "masked_mean")):  # two calls in a row, different inputs
        x = _dev(synth.make_chain_inputs(cfg, seed=seed))
        got = _noalloc_call(cfg, x, den)
        ref_h = torch.empty_like(got["h"])
        ref = lib.Chain(cfg, x["weights"]).loss(x["tokens"], x["seg"], x["pos"], x["h0"], den=den,
                                                 row_loss=True, h_out=ref_h)
        lib.check_errors()
        g = {k: v.double().cpu().numpy() for k, v in got.items()}
        r = {k: v.double().cpu().numpy() for k, v in ref.items()}
        ltol = 1e-3 if bf16 else 1e-5
        np.testing.assert_array_equal(g["sums_counts"][1::2], r["sums_counts"][1::2])
        np.testing.assert_allclose(g["losses"], r["losses"], rtol=ltol)
        np.testing.assert_allclose(g["sums_counts"][0::2], r["sums_counts"][0::2], rtol=ltol)
        assert np.array_equal(np.isnan(g["row_loss"]), np.isnan(r["row_loss"]))
        m = ~np.isnan(r["row_loss"])
        np.testing.assert_allclose(g["row_loss"][m], r["row_loss"][m], rtol=ltol)
        valid = np.isfinite(r["h"])
        atol, rtol = (2e-2, 2e-2) if bf16 else (1e-4, 0.0)
        np.testing.assert_allclose(g["h"][valid], r["h"][valid], atol=atol, rtol=rtol)


def test_noalloc_refuses_shapes_beyond_its_array():
    cfg = synth.MID_BF16
    dims = lib.make_dims(cfg)
    assert lib.load().mtp_chain_workspace_bytes(ctypes.byref(dims)) > 32 * 1024 * 1024
    fake = ctypes.c_void_p(1 << 20)
    w = lib.Weights()
    st = _noalloc_fn()(ctypes.byref(dims), ctypes.byref(w), fake, fake, fake, fake, 0.3, 0, 1,
                       fake, fake, None, None, None)
    assert st == 4  # MTP_ERR_WORKSPACE
