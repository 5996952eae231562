"""The C-ABI library builds, loads and exports every entry point that
include/mtp.h declares (no compute calls: runs without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mtp.h"), encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([a-z_][a-z0-9_]*)\s*\(",
                       src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def lib():
    from deepseek_sequential_mtp_gb300 import build, lib as binding
    build.build()
    return binding.load()


def test_header_declares_the_hot_path():
    names = declared_functions()
    for required in ("mtp_chain_forward", "mtp_chain_loss", "spec_verify",
                     "mtp_chain_workspace_bytes", "mtp_check_errors", "mtp_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_host_only_calls(lib):
    assert lib.mtp_abi_version() == 1
    assert lib.mtp_status_string(0) == b"ok"
    assert lib.mtp_status_string(7) == b"unsupported shape or dtype"


def test_argument_errors_return_without_launching(lib):
    # null pointers and bad sizes are rejected on the host
    assert lib.spec_verify(4, 2, 10, None, None, None, 0, 0, None, None,
                           None, None, None, None, None) == 1
    assert lib.spec_verify(4, 40, 10, None, None, None, 0, 0, None, None,
                           None, None, None, None, None) == 7
    assert lib.spec_verify(0, 2, 10, None, None, None, 0, 0, None, None,
                           None, None, None, None, None) == 0
    # one past the largest draft count (31) and vocabulary (512 chunks of 1024)
    assert lib.spec_verify(4, 32, 10, None, None, None, 0, 0, None, None,
                           None, None, None, None, None) == 7
    assert lib.spec_verify(4, 2, 512 * 1024 + 1, None, None, None, 0, 0, None, None,
                           None, None, None, None, None) == 7


def _dims(binding, **kw):
    from deepseek_sequential_mtp_gb300 import synth
    cfg = synth.SMALL_BF16.with_(**kw)
    return binding.make_dims(cfg)


def test_chain_host_validation(lib):
    import ctypes
    from deepseek_sequential_mtp_gb300 import lib as binding
    good = _dims(binding)
    assert lib.mtp_chain_workspace_bytes(ctypes.byref(good)) > 0
    for bad in (dict(B=0), dict(n_heads=3), dict(D=0), dict(V=0)):
        d = _dims(binding, **bad)
        assert lib.mtp_chain_workspace_bytes(ctypes.byref(d)) == 0
    unsup = _dims(binding, d=192, n_heads=3, head_dim=64)  # bf16 needs d % 128 == 0
    assert lib.mtp_chain_workspace_bytes(ctypes.byref(unsup)) == 0
    # host-side errors return before any device work (fake, aligned pointers)
    fake = ctypes.c_void_p(1 << 20)
    arr = (ctypes.c_void_p * good.D)(*([1 << 20] * good.D))
    w = binding.Weights()
    w.embed = w.head = w.out_norm = 1 << 20
    for k in binding._WEIGHT_LISTS:
        setattr(w, k, ctypes.cast(arr, binding._PP))
    sc = fake
    st = lib.mtp_chain_loss(ctypes.byref(good), ctypes.byref(w), fake, fake, fake, fake, 0.3, 0, 1,
                            sc, sc, None, None, fake, 16, None)
    assert st == 4  # workspace too small
    st = lib.mtp_chain_loss(ctypes.byref(good), ctypes.byref(w), fake, fake, fake, fake, 0.3, 7, 1,
                            sc, sc, None, None, fake, 1 << 40, None)
    assert st == 1  # bad denominator policy
    bad = _dims(binding, B=0)
    st = lib.mtp_chain_forward(ctypes.byref(bad), ctypes.byref(w), fake, fake, fake, fake, fake,
                               fake, 1 << 40, None)
    assert st == 2
    mis = ctypes.c_void_p((1 << 20) + 4)
    st = lib.mtp_chain_forward(ctypes.byref(good), ctypes.byref(w), mis, fake, fake, fake, fake,
                               fake, 1 << 40, None)
    assert st == 3


def test_fp8_host_validation(lib):
    """FP8 entry points reject bad arguments on the host, before any launch."""
    fake = ctypes.c_void_p(1 << 20)
    assert lib.mtp_gemm_fp8w(4, 128, 128, None, fake, fake, fake, fake, 1 << 20, None) == 1
    assert lib.mtp_gemm_fp8w(4, 128, 120, fake, fake, fake, fake, fake, 1 << 20, None) == 3   # K % 16 != 0
    assert lib.mtp_gemm_fp8w(33, 128, 128, fake, fake, fake, fake, fake, 1 << 20, None) == 2  # > 32 tokens
    assert lib.mtp_gemm_fp8w(4, 128, 128, fake, fake, fake, fake, fake, 16, None) == 4         # workspace
    assert lib.mtp_gemm_fp8w_workspace_bytes(7168) >= 64 * 7168
    from deepseek_sequential_mtp_gb300 import lib as binding, synth
    cfg = synth.DRAFT_SMALL
    dims = binding.Dims(cfg.R, cfg.ctx, cfg.d, cfg.n_heads, cfg.head_dim, cfg.ffn, cfg.V, 1, cfg.eps,
                        cfg.rope_base, binding.MTP_BF16)
    w = binding.Weights()
    st = lib.mtp_draft_round_fp8(ctypes.byref(dims), ctypes.byref(w), None, fake, fake, fake, fake, fake, fake, 1,
                                 0, 0, fake, fake, None, fake, 1 << 30, None)
    assert st == 1
