"""Thin ctypes binding of libmtp (include/mtp.h).

Argument marshalling only: every step of the hot path runs in the library's
CUDA kernels.  PyTorch supplies device memory and the current stream.  The
binding raises if the library is missing or a call returns an error; there
is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmtp.so")

MTP_F32, MTP_BF16 = 0, 1
DEN = {"fixed": 0, "masked_mean": 1, "sum": 2, "global": 3, "weighted_pair": 4}
VERIFY_STATUS = {0: "ok", 1: "invalid_draft", 2: "zero_residual", 3: "invalid_probs",
                 4: "invalid_budget"}


class MtpError(RuntimeError):
    pass


class Dims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("T", ctypes.c_int), ("d", ctypes.c_int),
                ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int), ("ffn", ctypes.c_int),
                ("V", ctypes.c_int), ("D", ctypes.c_int), ("eps", ctypes.c_float),
                ("rope_base", ctypes.c_float), ("dtype", ctypes.c_int)]


_PP = ctypes.POINTER(ctypes.c_void_p)
_WEIGHT_LISTS = ("hnorm", "enorm", "eh_proj", "attn_norm", "wq", "wk", "wv", "wo",
                 "ffn_norm", "w_gate", "w_up", "w_down")


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("head", ctypes.c_void_p),
                ("out_norm", ctypes.c_void_p)] + [(k, _PP) for k in _WEIGHT_LISTS]


class Grads(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("head", ctypes.c_void_p), ("out_norm", ctypes.c_void_p),
                ("h0", ctypes.c_void_p)] + [(k, _PP) for k in _WEIGHT_LISTS]


FP8_LINEAR_MAPS = ("eh_proj", "wq", "wk", "wv", "wo", "w_gate", "w_up", "w_down")


class Fp8Matrix(ctypes.Structure):
    _fields_ = [("q", ctypes.c_void_p), ("scale", ctypes.c_void_p)]


class BlockFp8(ctypes.Structure):
    _fields_ = [(k, Fp8Matrix) for k in FP8_LINEAR_MAPS]


_lib = None


def load() -> ctypes.CDLL:
    """Load libmtp.so (built by ``__graft_entry__.build()``); raises if absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise MtpError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, u64, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    lib.mtp_status_string.restype = ctypes.c_char_p
    lib.mtp_status_string.argtypes = [i32]
    lib.mtp_abi_version.restype = i32
    lib.mtp_check_errors.restype = i32
    lib.mtp_check_errors.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    lib.spec_verify.restype = i32
    lib.spec_verify.argtypes = [i32, i32, i32, vp, vp, vp, u64, u64, vp, vp, vp, vp, vp, vp, vp]
    lib.mtp_gemm_bf16.restype = i32
    lib.mtp_gemm_bf16.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    lib.mtp_chain_workspace_bytes.restype = sz
    lib.mtp_chain_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
    lib.mtp_chain_forward.restype = i32
    lib.mtp_chain_forward.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Weights),
                                      vp, vp, vp, vp, vp, vp, sz, vp]
    lib.mtp_chain_loss.restype = i32
    lib.mtp_chain_loss.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Weights),
                                   vp, vp, vp, vp, ctypes.c_float, i32, i32,
                                   vp, vp, vp, vp, vp, sz, vp]
    lib.mtp_loss_assemble_weighted.restype = i32
    lib.mtp_loss_assemble_weighted.argtypes = [i32, vp, ctypes.c_double, ctypes.POINTER(ctypes.c_float),
                                               ctypes.c_float, i32, i32, vp, vp]
    lib.mtp_loss_assemble.restype = i32
    lib.mtp_loss_assemble.argtypes = [i32, vp, ctypes.c_double, ctypes.c_float, i32, i32, vp, vp]
    lib.mtp_profile_kernel.restype = i32
    lib.mtp_profile_kernel.argtypes = [i32, vp, i32, ctypes.POINTER(ctypes.c_int)]
    lib.mtp_draft_workspace_bytes.restype = sz
    lib.mtp_draft_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
    lib.mtp_draft_round_workspace_bytes.restype = sz
    lib.mtp_draft_round_workspace_bytes.argtypes = [ctypes.POINTER(Dims), i32]
    lib.mtp_draft_round.restype = i32
    lib.mtp_draft_round.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Weights), vp, vp, vp, vp, vp, vp, i32,
                                    ctypes.c_uint64, ctypes.c_uint64, vp, vp, vp, vp, sz, vp]
    lib.mtp_draft_step.restype = i32
    lib.mtp_draft_step.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Weights), vp, vp, vp, vp, vp, vp,
                                   u64, u64, vp, vp, vp, vp, sz, vp]
    lib.mtp_draft_round_fp8.restype = i32
    lib.mtp_draft_round_fp8.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Weights), ctypes.POINTER(BlockFp8),
                                        vp, vp, vp, vp, vp, vp, i32, ctypes.c_uint64, ctypes.c_uint64, vp, vp, vp,
                                        vp, sz, vp]
    lib.mtp_gemm_decode_bf16.restype = i32
    lib.mtp_gemm_decode_bf16.argtypes = [i32, i32, i32, vp, vp, vp, vp]
    lib.mtp_gemm_f32acc.restype = i32
    lib.mtp_gemm_f32acc.argtypes = [i32, i32, i32, vp, i32, i32, vp, i32, i32, vp, i32, i32, vp]
    lib.mtp_gemm_fp8w_workspace_bytes.restype = sz
    lib.mtp_gemm_fp8w_workspace_bytes.argtypes = [i32]
    lib.mtp_gemm_fp8w.restype = i32
    lib.mtp_gemm_fp8w.argtypes = [i32, i32, i32, vp, vp, vp, vp, vp, sz, vp]
    lib.mtp_chain_grad_workspace_bytes.restype = sz
    lib.mtp_chain_grad_workspace_bytes.argtypes = [ctypes.POINTER(Dims)]
    lib.mtp_chain_loss_grad.restype = i32
    lib.mtp_chain_loss_grad.argtypes = [ctypes.POINTER(Dims), ctypes.POINTER(Weights), vp, vp, vp, vp,
                                        ctypes.c_float, i32, i32, ctypes.POINTER(ctypes.c_float), vp, vp,
                                        ctypes.POINTER(Grads), vp, sz, vp]
    lib.mtp_diag_verify_starved.restype = i32
    lib.mtp_diag_verify_starved.argtypes = [i32, i32, i32, vp, vp, vp, u64, u64, vp, vp, vp, vp,
                                            ctypes.c_longlong, vp]
    lib.mtp_kernel_launches.restype = ctypes.c_ulonglong
    lib.mtp_kernel_launches.argtypes = []
    _lib = lib
    return lib


def _check(status: int, what: str):
    if status != 0:
        msg = load().mtp_status_string(status).decode()
        raise MtpError(f"{what}: {msg} (status {status})")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype: torch.dtype):
    if not t.is_cuda:
        raise MtpError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise MtpError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise MtpError(f"{name} must be contiguous")


def check_errors(stream=None) -> int:
    """Synchronise and return the device error bits (raises if any is set)."""
    flags = ctypes.c_uint(0)
    st = load().mtp_check_errors(_stream(stream), ctypes.byref(flags))
    if st != 0:
        raise MtpError(f"device error word 0x{flags.value:x} ({load().mtp_status_string(st).decode()})")
    return flags.value


# --------------------------------------------------------------------------
# spec_verify
# --------------------------------------------------------------------------
def spec_verify(p: torch.Tensor, q: torch.Tensor, draft: torch.Tensor, seed: int, offset: int,
                eos: Optional[torch.Tensor] = None, remaining: Optional[torch.Tensor] = None,
                out: Optional[dict] = None, stream=None) -> dict:
    """Exact speculative verification (include/mtp.h: spec_verify)."""
    R, gamma = draft.shape
    V = p.shape[-1]
    _need(p, "p", torch.float32)
    _need(q, "q", torch.float32)
    _need(draft, "draft", torch.int32)
    if p.shape != (R, gamma + 1, V) or q.shape != (R, gamma, V):
        raise MtpError("p must be [R, gamma+1, V] and q [R, gamma, V]")
    for name, t in (("eos", eos), ("remaining", remaining)):
        if t is not None:
            _need(t, name, torch.int32)
    if out is None:
        out = {k: torch.empty(R, dtype=torch.int32, device=p.device)
               for k in ("accepted", "next_token", "n_emit", "status")}
    st = load().spec_verify(R, gamma, V, _ptr(p), _ptr(q), _ptr(draft),
                            int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                            _ptr(eos), _ptr(remaining), _ptr(out["accepted"]),
                            _ptr(out["next_token"]), _ptr(out["n_emit"]), _ptr(out["status"]),
                            _stream(stream))
    _check(st, "spec_verify")
    return out


def verify_starved(p: torch.Tensor, q: torch.Tensor, draft: torch.Tensor, seed: int, offset: int,
                   wait_limit_cycles: int, stream=None) -> dict:
    """spec_verify with a producer that issues no copy, so every row sweep's
    bounded wait runs out (include/mtp.h: mtp_diag_verify_starved)."""
    R, gamma = draft.shape
    V = p.shape[-1]
    _need(p, "p", torch.float32)
    _need(q, "q", torch.float32)
    _need(draft, "draft", torch.int32)
    out = {k: torch.empty(R, dtype=torch.int32, device=p.device)
           for k in ("accepted", "next_token", "n_emit", "status")}
    st = load().mtp_diag_verify_starved(R, gamma, V, _ptr(p), _ptr(q), _ptr(draft),
                                        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1),
                                        _ptr(out["accepted"]), _ptr(out["next_token"]), _ptr(out["n_emit"]),
                                        _ptr(out["status"]), int(wait_limit_cycles), _stream(stream))
    _check(st, "mtp_diag_verify_starved")
    return out


# --------------------------------------------------------------------------
# GEMM diagnostic
# --------------------------------------------------------------------------
def gemm_bf16(A: torch.Tensor, B: torch.Tensor, C: Optional[torch.Tensor] = None, stream=None):
    """C = A · B^T on the library's tcgen05 GEMM core (bf16 in/out, fp32 accumulate)."""
    _need(A, "A", torch.bfloat16)
    _need(B, "B", torch.bfloat16)
    M, K = A.shape
    N = B.shape[0]
    if B.shape[1] != K:
        raise MtpError("A and B must share K")
    if C is None:
        C = torch.empty((M, N), dtype=torch.bfloat16, device=A.device)
    _check(load().mtp_gemm_bf16(M, N, K, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "mtp_gemm_bf16")
    return C


# --------------------------------------------------------------------------
# Chain
# --------------------------------------------------------------------------
def make_dims(cfg) -> Dims:
    return Dims(cfg.B, cfg.T, cfg.d, cfg.n_heads, cfg.head_dim, cfg.ffn, cfg.V, cfg.D,
                cfg.eps, cfg.rope_base, MTP_BF16 if cfg.dtype == "bf16" else MTP_F32)


class ChainWeights:
    """Holds the ctypes views of a weight dict (see synth.make_weights)."""

    def __init__(self, weights: dict, D: int):
        self._keep = []
        self.struct = Weights()
        self.struct.embed = weights["embed"].data_ptr()
        self.struct.head = weights["head"].data_ptr()
        self.struct.out_norm = weights["out_norm"].data_ptr()
        for k in _WEIGHT_LISTS:
            lst = weights[k]
            if len(lst) != D:
                raise MtpError(f"weights[{k!r}] must have D={D} entries")
            arr = (ctypes.c_void_p * D)(*[t.data_ptr() for t in lst])
            self._keep.append(arr)
            setattr(self.struct, k, ctypes.cast(arr, _PP))


class Fp8Block:
    """ctypes view of the FP8 linear maps of one module: fp8[name] = (q, scale)
    with q uint8 [n, K] e4m3 codes and scale float32 [ceil(n/128), ceil(K/128)]."""

    def __init__(self, fp8: dict):
        self.fp8 = fp8
        self.struct = BlockFp8()
        for name in FP8_LINEAR_MAPS:
            q, sc = fp8[name]
            _need(q, name + ".q", torch.uint8)
            _need(sc, name + ".scale", torch.float32)
            nb, kb = -(-q.shape[0] // 128), -(-q.shape[1] // 128)
            if tuple(sc.shape) != (nb, kb):
                raise MtpError(f"{name}.scale must be [{nb}, {kb}]")
            m = getattr(self.struct, name)
            m.q = q.data_ptr()
            m.scale = sc.data_ptr()


def gemm_decode_bf16(x: torch.Tensor, w: torch.Tensor, out: torch.Tensor, stream=None):
    """out[R, N] += x[R, K] @ w[N, K]^T for R <= 32 tokens (mtp_gemm_decode_bf16)."""
    _need(x, "x", torch.bfloat16)
    _need(w, "w", torch.bfloat16)
    _need(out, "out", torch.float32)
    R, K = x.shape
    N = w.shape[0]
    if w.shape[1] != K or tuple(out.shape) != (R, N):
        raise MtpError("gemm_decode_bf16: x [R, K], w [N, K], out [R, N]")
    _check(load().mtp_gemm_decode_bf16(R, N, K, _ptr(x), _ptr(w), _ptr(out), _stream(stream)), "mtp_gemm_decode_bf16")
    return out


def gemm_f32acc(A: torch.Tensor, B: torch.Tensor, out: torch.Tensor, a_mn=False, b_mn=False, splits=1, stream=None):
    """out += A' B'^T (mtp_gemm_f32acc): A' = A ([M, K]) or, with a_mn, A^T of a
    [K, M] tensor; B' = B ([N, K]) or, with b_mn, B^T of a [K, N] tensor."""
    _need(A, "A", torch.bfloat16)
    _need(B, "B", torch.bfloat16)
    _need(out, "out", torch.float32)
    M = A.shape[1] if a_mn else A.shape[0]
    K = A.shape[0] if a_mn else A.shape[1]
    N = B.shape[1] if b_mn else B.shape[0]
    if (B.shape[0] if b_mn else B.shape[1]) != K or tuple(out.shape) != (M, N):
        raise MtpError("gemm_f32acc: inconsistent shapes")
    _check(load().mtp_gemm_f32acc(M, N, K, _ptr(A), A.shape[1], int(a_mn), _ptr(B), B.shape[1], int(b_mn), _ptr(out),
                                  out.shape[1], int(splits), _stream(stream)), "mtp_gemm_f32acc")
    return out


def gemm_fp8w(x: torch.Tensor, q: torch.Tensor, scale: torch.Tensor, out: torch.Tensor, stream=None, ws=None):
    """out[R, N] += x~[R, K] @ W^T, W = e4m3(q) * block scales, x~ the two-term
    e4m3 form of x (mtp_gemm_fp8w)."""
    _need(x, "x", torch.bfloat16)
    _need(q, "q", torch.uint8)
    _need(scale, "scale", torch.float32)
    _need(out, "out", torch.float32)
    R, K = x.shape
    N = q.shape[0]
    if q.shape[1] != K or tuple(out.shape) != (R, N):
        raise MtpError("gemm_fp8w: x [R, K], q [N, K], out [R, N]")
    if ws is None:
        ws = torch.empty(max(16, int(load().mtp_gemm_fp8w_workspace_bytes(K))), dtype=torch.uint8, device=x.device)
    _check(load().mtp_gemm_fp8w(R, N, K, _ptr(x), _ptr(q), _ptr(scale), _ptr(out), _ptr(ws), ws.numel(),
                                _stream(stream)), "mtp_gemm_fp8w")
    return out


def _check_chain_inputs(cfg, tokens, seg, pos, h0, weights):
    dt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float32
    for name, t in (("tokens", tokens), ("seg", seg), ("pos", pos)):
        _need(t, name, torch.int32)
        if tuple(t.shape) != (cfg.B, cfg.T):
            raise MtpError(f"{name} must be [B, T]")
    _need(h0, "h0", dt)
    for k, v in weights.items():
        for t in (v if isinstance(v, (list, tuple)) else [v]):
            _need(t, k, dt)
    return dt


def chain_workspace_bytes(cfg) -> int:
    dims = make_dims(cfg)
    return int(load().mtp_chain_workspace_bytes(ctypes.byref(dims)))


class Chain:
    """Reusable call state (dims, weight views, workspace) for one shape."""

    def __init__(self, cfg, weights: dict, device="cuda"):
        self.cfg = cfg
        self.dims = make_dims(cfg)
        self.w = ChainWeights(weights, cfg.D)
        self.weights = weights
        nbytes = chain_workspace_bytes(cfg)
        if nbytes == 0:
            raise MtpError("invalid chain dimensions")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def loss_grad(self, tokens, seg, pos, h0, grads: dict, lam=None, den="fixed", with_main=True,
                  depth_weights=None, out=None, stream=None):
        """Training step (include/mtp.h: mtp_chain_loss_grad): losses as
        ``loss`` and the gradients added into ``grads`` (fp32 tensors keyed as
        the weights, plus "h0"; per-depth entries are lists; missing keys are
        not computed)."""
        cfg = self.cfg
        _check_chain_inputs(cfg, tokens, seg, pos, h0, self.weights)
        if not hasattr(self, "gws"):
            nbytes = int(load().mtp_chain_grad_workspace_bytes(ctypes.byref(self.dims)))
            if nbytes == 0:
                raise MtpError("the training step does not support these dimensions")
            self.gws = torch.empty(nbytes, dtype=torch.uint8, device=h0.device)
        dev = h0.device
        if out is None:
            out = {"sums_counts": torch.empty(2 * (cfg.D + 1), dtype=torch.float64, device=dev),
                   "losses": torch.empty(cfg.D + 2, dtype=torch.float32, device=dev)}
        g = Grads()
        keep = []
        for k in ("embed", "head", "out_norm", "h0"):
            t = grads.get(k)
            if t is not None:
                _need(t, f"grads[{k!r}]", torch.float32)
                setattr(g, k, t.data_ptr())
        for k in _WEIGHT_LISTS:
            lst = grads.get(k)
            if lst is not None:
                arr = (ctypes.c_void_p * cfg.D)(*[t.data_ptr() for t in lst])
                keep.append(arr)
                setattr(g, k, ctypes.cast(arr, _PP))
        w = None
        if depth_weights is not None:
            w = (ctypes.c_float * cfg.D)(*[float(x) for x in depth_weights])
        st = load().mtp_chain_loss_grad(ctypes.byref(self.dims), ctypes.byref(self.w.struct),
                                        _ptr(tokens), _ptr(seg), _ptr(pos), _ptr(h0),
                                        float(cfg.lam if lam is None else lam), DEN[den], int(with_main), w,
                                        _ptr(out["sums_counts"]), _ptr(out["losses"]), ctypes.byref(g),
                                        _ptr(self.gws), self.gws.numel(), _stream(stream))
        _check(st, "mtp_chain_loss_grad")
        return out

    def forward(self, tokens, seg, pos, h0, h_out=None, stream=None):
        cfg = self.cfg
        dt = _check_chain_inputs(cfg, tokens, seg, pos, h0, self.weights)
        if h_out is None:
            h_out = torch.empty((cfg.D, cfg.B, cfg.T, cfg.d), dtype=dt, device=h0.device)
        st = load().mtp_chain_forward(ctypes.byref(self.dims), ctypes.byref(self.w.struct),
                                      _ptr(tokens), _ptr(seg), _ptr(pos), _ptr(h0), _ptr(h_out),
                                      _ptr(self.ws), self.ws.numel(), _stream(stream))
        _check(st, "mtp_chain_forward")
        return h_out

    def loss(self, tokens, seg, pos, h0, lam=None, den="fixed", with_main=True,
             row_loss=False, h_out=None, out=None, stream=None):
        cfg = self.cfg
        _check_chain_inputs(cfg, tokens, seg, pos, h0, self.weights)
        dev = h0.device
        if out is None:
            out = {"sums_counts": torch.empty(2 * (cfg.D + 1), dtype=torch.float64, device=dev),
                   "losses": torch.empty(cfg.D + 2, dtype=torch.float32, device=dev)}
            if row_loss:
                out["row_loss"] = torch.empty((cfg.D + 1, cfg.B, cfg.T), dtype=torch.float32, device=dev)
        st = load().mtp_chain_loss(ctypes.byref(self.dims), ctypes.byref(self.w.struct),
                                   _ptr(tokens), _ptr(seg), _ptr(pos), _ptr(h0),
                                   float(cfg.lam if lam is None else lam), DEN[den], int(with_main),
                                   _ptr(out["sums_counts"]), _ptr(out["losses"]),
                                   _ptr(out.get("row_loss")), _ptr(h_out),
                                   _ptr(self.ws), self.ws.numel(), _stream(stream))
        _check(st, "mtp_chain_loss")
        if h_out is not None:
            out["h"] = h_out
        return out


# --------------------------------------------------------------------------
# Loss assembly (data-parallel callers) and measurement hooks
# --------------------------------------------------------------------------
def loss_assemble(sums_counts: torch.Tensor, D: int, n_positions: float, lam: float, den="fixed",
                  with_main=True, losses: Optional[torch.Tensor] = None, stream=None,
                  depth_weights=None) -> torch.Tensor:
    """L, L_main, L^(1..D) from (already all-reduced) per-term sums and counts
    under reduction ``den`` (include/mtp.h: mtp_den) with per-depth weights
    (a sequence of D floats; None = lam / D each)."""
    _need(sums_counts, "sums_counts", torch.float64)
    if losses is None:
        losses = torch.empty(D + 2, dtype=torch.float32, device=sums_counts.device)
    w = None
    if depth_weights is not None:
        if len(depth_weights) != D:
            raise MtpError("depth_weights must hold D values")
        w = (ctypes.c_float * D)(*[float(x) for x in depth_weights])
    _check(load().mtp_loss_assemble_weighted(D, _ptr(sums_counts), float(n_positions), w, float(lam), DEN[den],
                                             int(with_main), _ptr(losses), _stream(stream)),
           "mtp_loss_assemble_weighted")
    return losses


KERNEL_CLASSES = {"head_ce_gemm": 0, "gate_up_gemm": 1, "down_gemm": 2, "qkv_gemm": 3, "o_gemm": 4,
                  "proj_gemm": 5, "attention": 6, "spec_verify": 7, "prologue": 8}


class KernelTimer:
    """Arms the library's event hook for one kernel class: CUDA events are
    recorded on the launching stream around each launch of that class."""

    def __init__(self, kernel_class: str, max_launches: int):
        self.cls = KERNEL_CLASSES[kernel_class]
        self.events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * max_launches)]
        for e in self.events:  # CUDA creates the events on first record
            e.record()
        self._handles = (ctypes.c_void_p * (2 * max_launches))(*[e.cuda_event for e in self.events])
        self.recorded = ctypes.c_int(0)
        self.max = max_launches

    def arm(self):
        _check(load().mtp_profile_kernel(self.cls, self._handles, self.max, ctypes.byref(self.recorded)),
               "mtp_profile_kernel")

    @staticmethod
    def disarm_all():
        for c in KERNEL_CLASSES.values():
            load().mtp_profile_kernel(c, None, 0, None)

    def durations_ms(self):
        n = self.recorded.value
        return [self.events[2 * i].elapsed_time(self.events[2 * i + 1]) for i in range(n)]


def kernel_launches() -> int:
    return int(load().mtp_kernel_launches())


# --------------------------------------------------------------------------
# Draft step (decode-shaped MTP proposal)
# --------------------------------------------------------------------------
class DraftStep:
    """Reusable call state of mtp_draft_step for one shape (see synth.DraftConfig)."""

    def __init__(self, cfg, weights: dict, device="cuda", fp8: Optional[dict] = None):
        self.cfg = cfg
        self.dims = Dims(cfg.R, cfg.ctx, cfg.d, cfg.n_heads, cfg.head_dim, cfg.ffn, cfg.V, 1, cfg.eps,
                         cfg.rope_base, MTP_BF16)
        self.weights = weights
        self.w = ChainWeights(weights, 1)
        self.f8 = Fp8Block(fp8) if fp8 is not None else None
        nbytes = int(load().mtp_draft_workspace_bytes(ctypes.byref(self.dims)))
        if nbytes == 0:
            raise MtpError("invalid draft-step dimensions")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, seed, offset,
                 out=None, h_out=None, stream=None):
        cfg = self.cfg
        _need(parent_hidden, "parent_hidden", torch.bfloat16)
        for name, t in (("kv_k", kv_k), ("kv_v", kv_v)):
            _need(t, name, torch.bfloat16)
            if tuple(t.shape) != (cfg.R, cfg.ctx, cfg.d):
                raise MtpError(f"{name} must be [R, ctx, d]")
        for name, t in (("frontier", frontier), ("pos", pos), ("ctx_len", ctx_len)):
            _need(t, name, torch.int32)
        dev = parent_hidden.device
        if out is None:
            out = {"q": torch.empty((cfg.R, cfg.V), dtype=torch.float32, device=dev),
                   "y": torch.empty(cfg.R, dtype=torch.int32, device=dev)}
        if self.f8 is not None:  # one step of the FP8 round
            st = load().mtp_draft_round_fp8(ctypes.byref(self.dims), ctypes.byref(self.w.struct),
                                            ctypes.byref(self.f8.struct), _ptr(parent_hidden), _ptr(frontier),
                                            _ptr(pos), _ptr(kv_k), _ptr(kv_v), _ptr(ctx_len), 1,
                                            int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(out["q"]),
                                            _ptr(out["y"]), _ptr(h_out), _ptr(self.ws), self.ws.numel(),
                                            _stream(stream))
            _check(st, "mtp_draft_round_fp8")
        else:
            st = load().mtp_draft_step(ctypes.byref(self.dims), ctypes.byref(self.w.struct), _ptr(parent_hidden),
                                       _ptr(frontier), _ptr(pos), _ptr(kv_k), _ptr(kv_v), _ptr(ctx_len),
                                       int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(out["q"]),
                                       _ptr(out["y"]), _ptr(h_out), _ptr(self.ws), self.ws.numel(),
                                       _stream(stream))
            _check(st, "mtp_draft_step")
        if h_out is not None:
            out["h"] = h_out
        return out


class DraftRound:
    """Reusable call state of mtp_draft_round: gamma recurrent draft steps of
    one module for one shape (see synth.DraftConfig)."""

    def __init__(self, cfg, weights: dict, gamma: int, device="cuda", fp8: Optional[dict] = None):
        self.cfg = cfg
        self.gamma = int(gamma)
        self.dims = Dims(cfg.R, cfg.ctx, cfg.d, cfg.n_heads, cfg.head_dim, cfg.ffn, cfg.V, 1, cfg.eps,
                         cfg.rope_base, MTP_BF16)
        self.weights = weights
        self.w = ChainWeights(weights, 1)
        self.f8 = Fp8Block(fp8) if fp8 is not None else None
        nbytes = int(load().mtp_draft_round_workspace_bytes(ctypes.byref(self.dims), self.gamma))
        if nbytes == 0:
            raise MtpError("invalid draft-round dimensions or gamma")
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=device)

    def __call__(self, parent_hidden, frontier, pos, kv_k, kv_v, ctx_len, seed, offset,
                 out=None, h_out=None, stream=None):
        cfg, g = self.cfg, self.gamma
        _need(parent_hidden, "parent_hidden", torch.bfloat16)
        for name, t in (("kv_k", kv_k), ("kv_v", kv_v)):
            _need(t, name, torch.bfloat16)
            if tuple(t.shape) != (cfg.R, cfg.ctx, cfg.d):
                raise MtpError(f"{name} must be [R, ctx, d]")
        for name, t in (("frontier", frontier), ("pos", pos), ("ctx_len", ctx_len)):
            _need(t, name, torch.int32)
        if h_out is not None:
            _need(h_out, "h_out", torch.bfloat16)
            if tuple(h_out.shape) != (cfg.R, g, cfg.d):
                raise MtpError("h_out must be [R, gamma, d]")
        dev = parent_hidden.device
        if out is None:
            out = {"q": torch.empty((cfg.R, g, cfg.V), dtype=torch.float32, device=dev),
                   "y": torch.empty((cfg.R, g), dtype=torch.int32, device=dev)}
        if self.f8 is not None:
            st = load().mtp_draft_round_fp8(ctypes.byref(self.dims), ctypes.byref(self.w.struct),
                                            ctypes.byref(self.f8.struct), _ptr(parent_hidden), _ptr(frontier),
                                            _ptr(pos), _ptr(kv_k), _ptr(kv_v), _ptr(ctx_len), g,
                                            int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(out["q"]),
                                            _ptr(out["y"]), _ptr(h_out), _ptr(self.ws), self.ws.numel(),
                                            _stream(stream))
            _check(st, "mtp_draft_round_fp8")
        else:
            st = load().mtp_draft_round(ctypes.byref(self.dims), ctypes.byref(self.w.struct), _ptr(parent_hidden),
                                        _ptr(frontier), _ptr(pos), _ptr(kv_k), _ptr(kv_v), _ptr(ctx_len), g,
                                        int(seed) & (2**64 - 1), int(offset) & (2**64 - 1), _ptr(out["q"]),
                                        _ptr(out["y"]), _ptr(h_out), _ptr(self.ws), self.ws.numel(),
                                        _stream(stream))
            _check(st, "mtp_draft_round")
        if h_out is not None:
            out["h"] = h_out
        return out
