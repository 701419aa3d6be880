"""Python binding of the GDN verify C ABI (include/gdn.h).

Argument marshalling only: each function checks the torch tensors' device,
dtype, contiguity and element counts, and passes raw pointers and the CUDA
stream to the library, where every step runs in sm_103a kernels.  There is no
fallback: if ``libgdn_sm103a.so`` is missing the first call raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

EXPORTED = ("gdn_conv_step", "gdn_verify_step", "gdn_verify_resume", "gdn_verify_tree", "gdn_verify_gated",
            "gdn_verify_workspace_size", "gdn_verify_step_static_scratch", "gdn_prefill", "gdn_prefill_workspace_size",
            "gdn_rollback", "gdn_device_status", "gdn_last_error")

GDN_OK, GDN_ERR_INVALID_ARG, GDN_ERR_UNSUPPORTED, GDN_ERR_ALIAS, GDN_ERR_NO_SNAPSHOT, GDN_ERR_CUDA = range(6)
STATUS_NAMES = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_ALIAS",
                4: "GDN_ERR_NO_SNAPSHOT", 5: "GDN_ERR_CUDA"}
DEVERR_TIMEOUT, DEVERR_ACCEPT_RANGE, DEVERR_NO_SNAPSHOT, DEVERR_TREE_PARENT, DEVERR_SEQLENS = 1, 2, 4, 8, 16


class GdnDims(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("K", ctypes.c_int32), ("Hk", ctypes.c_int32), ("Hv", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("conv_w", ctypes.c_int32),
                ("q_scale", ctypes.c_float), ("l2_eps", ctypes.c_float), ("out_f32", ctypes.c_int32)]

    @property
    def C(self) -> int:
        return 2 * self.Hk * self.dk + self.Hv * self.dv


def make_dims(B, K, Hk, Hv, dk, dv, W=4, q_scale=1.0, l2_eps=1e-6, out_f32=1) -> GdnDims:
    return GdnDims(B, K, Hk, Hv, dk, dv, W, q_scale, l2_eps, out_f32)


class GdnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libgdn_sm103a.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with __graft_entry__.build() "
                           "or python -m speculative_decode_verify_gdn_gb300.build")
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    D = ctypes.POINTER(GdnDims)
    lib.gdn_conv_step.argtypes = [D, P, P, P, P, P, P]
    lib.gdn_verify_step.argtypes = [D] + [P] * 14 + [ctypes.c_uint64, P]
    lib.gdn_verify_resume.argtypes = [D] + [P] * 19 + [ctypes.c_uint64, P]
    lib.gdn_verify_tree.argtypes = [D] + [P] * 15 + [ctypes.c_uint64, P]
    lib.gdn_verify_gated.argtypes = [D] + [P] * 14 + [ctypes.c_float, P, P, ctypes.c_uint64, P]
    lib.gdn_verify_workspace_size.argtypes = [D, ctypes.POINTER(ctypes.c_uint64)]
    lib.gdn_prefill.argtypes = [D, ctypes.c_int64] + [P] * 13 + [ctypes.c_uint64, P]
    lib.gdn_prefill_workspace_size.argtypes = [D, ctypes.c_int64, ctypes.POINTER(ctypes.c_uint64)]
    lib.gdn_verify_step_static_scratch.argtypes = [D] + [P] * 14
    lib.gdn_rollback.argtypes = [D] + [P] * 8
    lib.gdn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int32, P]
    lib.gdn_last_error.argtypes = []
    lib.gdn_last_error.restype = ctypes.c_char_p
    for f in ("gdn_conv_step", "gdn_verify_step", "gdn_verify_resume", "gdn_verify_tree", "gdn_verify_gated",
              "gdn_verify_workspace_size", "gdn_verify_step_static_scratch", "gdn_prefill",
              "gdn_prefill_workspace_size", "gdn_rollback", "gdn_device_status"):
        getattr(lib, f).restype = ctypes.c_int
    _lib = lib
    return lib


def last_error() -> str:
    return load_library().gdn_last_error().decode()


def _check(status: int) -> None:
    if status != GDN_OK:
        raise GdnError(status, last_error())


def _ptr(t, name, dtype, numel, allow_none=False):
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{name} has {t.numel()} elements, expected {numel}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def gdn_conv_step(dims: GdnDims, x, conv_w, conv_state, conv_inter, y, stream=None) -> None:
    """a1: conv + SiLU over a K-token window; conv_state updated in place."""
    d = dims
    C, BK = d.C, d.B * d.K
    ydt = torch.float32 if d.out_f32 else torch.bfloat16
    _check(load_library().gdn_conv_step(
        ctypes.byref(d), _ptr(x, "x", torch.bfloat16, BK * C), _ptr(conv_w, "conv_w", torch.float32, C * d.conv_w),
        _ptr(conv_state, "conv_state", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_inter, "conv_inter", torch.float32, BK * (d.conv_w - 1) * C, allow_none=True),
        _ptr(y, "y", ydt, BK * C), _stream(stream)))


def gdn_verify_workspace_size(dims: GdnDims) -> int:
    """Bytes of device scratch gdn_verify_step needs for these dims."""
    n = ctypes.c_uint64(0)
    _check(load_library().gdn_verify_workspace_size(ctypes.byref(dims), ctypes.byref(n)))
    return n.value


def alloc_workspace(dims: GdnDims, device="cuda") -> torch.Tensor:
    """A uint8 device tensor large enough to serve as gdn_verify_step's workspace."""
    return torch.empty(max(16, gdn_verify_workspace_size(dims)), dtype=torch.uint8, device=device)


def gdn_prefill_workspace_size(dims: GdnDims, n_tokens: int) -> int:
    """Bytes of device scratch gdn_prefill needs for B prompts holding n_tokens tokens."""
    n = ctypes.c_uint64(0)
    _check(load_library().gdn_prefill_workspace_size(ctypes.byref(dims), ctypes.c_int64(n_tokens), ctypes.byref(n)))
    return n.value


def alloc_prefill_workspace(dims: GdnDims, n_tokens: int, device="cuda") -> torch.Tensor:
    return torch.empty(max(16, gdn_prefill_workspace_size(dims, n_tokens)), dtype=torch.uint8, device=device)


def gdn_prefill(dims: GdnDims, cu_seqlens, x, a, b, A_log, dt_bias, conv_w, conv_state_in, conv_state_out,
                state_in, state_out, out, workspace, stream=None) -> None:
    """a1..a4 over whole prompts packed token-major: cu_seqlens [B + 1] int32 (device),
    x [N, C], a, b [N, Hv] bf16, out [N, Hv, dv]; states and histories per prompt."""
    d = dims
    N = int(x.shape[0]) if x is not None else 0
    C = d.C
    S = d.Hv * d.dv * d.dk
    H = d.B * (d.conv_w - 1) * C
    odt = torch.float32 if d.out_f32 else torch.bfloat16
    empty = N == 0

    def tok(t, name, dtype, numel):
        if empty and (t is None or t.numel() == 0):
            return None
        return _ptr(t, name, dtype, numel)

    _check(load_library().gdn_prefill(
        ctypes.byref(d), ctypes.c_int64(N), _ptr(cu_seqlens, "cu_seqlens", torch.int32, d.B + 1),
        tok(x, "x", torch.bfloat16, N * C), tok(a, "a", torch.bfloat16, N * d.Hv),
        tok(b, "b", torch.bfloat16, N * d.Hv), _ptr(A_log, "A_log", torch.float32, d.Hv),
        _ptr(dt_bias, "dt_bias", torch.float32, d.Hv), _ptr(conv_w, "conv_w", torch.float32, C * d.conv_w),
        _ptr(conv_state_in, "conv_state_in", torch.float32, H), _ptr(conv_state_out, "conv_state_out", torch.float32, H),
        _ptr(state_in, "state_in", torch.float32, d.B * S), _ptr(state_out, "state_out", torch.float32, d.B * S),
        tok(out, "out", odt, N * d.Hv * d.dv), _ws_ptr(workspace), ctypes.c_uint64(_ws_bytes(workspace)),
        _stream(stream)))


def gdn_verify_step(dims: GdnDims, x, a, b, A_log, dt_bias, conv_w, conv_state_in, conv_state_out, conv_inter,
                    state_in, state_out, state_inter, out, workspace, stream=None) -> None:
    """a1..a4 fused over one verify window (see include/gdn.h for layouts and aliasing)."""
    d = dims
    C, BK = d.C, d.B * d.K
    S = d.Hv * d.dv * d.dk
    odt = torch.float32 if d.out_f32 else torch.bfloat16
    _check(load_library().gdn_verify_step(
        ctypes.byref(d), _ptr(x, "x", torch.bfloat16, BK * C), _ptr(a, "a", torch.bfloat16, BK * d.Hv),
        _ptr(b, "b", torch.bfloat16, BK * d.Hv), _ptr(A_log, "A_log", torch.float32, d.Hv),
        _ptr(dt_bias, "dt_bias", torch.float32, d.Hv), _ptr(conv_w, "conv_w", torch.float32, C * d.conv_w),
        _ptr(conv_state_in, "conv_state_in", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_state_out, "conv_state_out", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_inter, "conv_inter", torch.float32, BK * (d.conv_w - 1) * C, allow_none=True),
        _ptr(state_in, "state_in", torch.float32, d.B * S), _ptr(state_out, "state_out", torch.float32, d.B * S),
        _ptr(state_inter, "state_inter", torch.float32, d.B * (d.K - 1) * S, allow_none=(d.K == 1)),
        _ptr(out, "out", odt, BK * d.Hv * d.dv), _ws_ptr(workspace), ctypes.c_uint64(_ws_bytes(workspace)),
        _stream(stream)))


def gdn_verify_tree(dims: GdnDims, parent, x, a, b, A_log, dt_bias, conv_w, conv_state_in, conv_state_out, conv_inter,
                    state_in, state_out, state_inter, out, workspace, stream=None) -> None:
    """a1..a4 over a token tree: parent [B, K] int32 (device), parent[b][t] in -1..t-1."""
    d = dims
    C, BK = d.C, d.B * d.K
    S = d.Hv * d.dv * d.dk
    odt = torch.float32 if d.out_f32 else torch.bfloat16
    _check(load_library().gdn_verify_tree(
        ctypes.byref(d), _ptr(parent, "parent", torch.int32, BK),
        _ptr(x, "x", torch.bfloat16, BK * C), _ptr(a, "a", torch.bfloat16, BK * d.Hv),
        _ptr(b, "b", torch.bfloat16, BK * d.Hv), _ptr(A_log, "A_log", torch.float32, d.Hv),
        _ptr(dt_bias, "dt_bias", torch.float32, d.Hv), _ptr(conv_w, "conv_w", torch.float32, C * d.conv_w),
        _ptr(conv_state_in, "conv_state_in", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_state_out, "conv_state_out", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_inter, "conv_inter", torch.float32, BK * (d.conv_w - 1) * C, allow_none=True),
        _ptr(state_in, "state_in", torch.float32, d.B * S), _ptr(state_out, "state_out", torch.float32, d.B * S),
        _ptr(state_inter, "state_inter", torch.float32, d.B * (d.K - 1) * S, allow_none=(d.K == 1)),
        _ptr(out, "out", odt, BK * d.Hv * d.dv), _ws_ptr(workspace), ctypes.c_uint64(_ws_bytes(workspace)),
        _stream(stream)))


def gdn_verify_gated(dims: GdnDims, x, a, b, A_log, dt_bias, conv_w, conv_state_in, conv_state_out, conv_inter,
                     state_in, state_out, state_inter, z, norm_w, norm_eps, out, workspace, stream=None) -> None:
    """a1..a4 with the gated RMS norm fused into the output: z [B, K, Hv, dv] bf16, norm_w [dv] f32."""
    d = dims
    C, BK = d.C, d.B * d.K
    S = d.Hv * d.dv * d.dk
    odt = torch.float32 if d.out_f32 else torch.bfloat16
    _check(load_library().gdn_verify_gated(
        ctypes.byref(d), _ptr(x, "x", torch.bfloat16, BK * C), _ptr(a, "a", torch.bfloat16, BK * d.Hv),
        _ptr(b, "b", torch.bfloat16, BK * d.Hv), _ptr(A_log, "A_log", torch.float32, d.Hv),
        _ptr(dt_bias, "dt_bias", torch.float32, d.Hv), _ptr(conv_w, "conv_w", torch.float32, C * d.conv_w),
        _ptr(conv_state_in, "conv_state_in", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_state_out, "conv_state_out", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_inter, "conv_inter", torch.float32, BK * (d.conv_w - 1) * C, allow_none=True),
        _ptr(state_in, "state_in", torch.float32, d.B * S), _ptr(state_out, "state_out", torch.float32, d.B * S),
        _ptr(state_inter, "state_inter", torch.float32, d.B * (d.K - 1) * S, allow_none=(d.K == 1)),
        _ptr(z, "z", torch.bfloat16, BK * d.Hv * d.dv), _ptr(norm_w, "norm_w", torch.float32, d.dv),
        ctypes.c_float(norm_eps), _ptr(out, "out", odt, BK * d.Hv * d.dv), _ws_ptr(workspace),
        ctypes.c_uint64(_ws_bytes(workspace)), _stream(stream)))


def gdn_verify_resume(dims: GdnDims, accept_len_prev, x, a, b, A_log, dt_bias, conv_w, conv_state_in,
                      conv_inter_prev, conv_state_snapshot_prev, conv_state_out, conv_inter, state_in,
                      state_inter_prev, state_snapshot_prev, state_out, state_inter, out, workspace,
                      stream=None) -> None:
    """Rollback of the previous window (accept_len_prev) applied on read, then a1..a4 of this window."""
    d = dims
    C, BK = d.C, d.B * d.K
    S = d.Hv * d.dv * d.dk
    k1 = d.K == 1
    H = d.B * (d.conv_w - 1) * C
    odt = torch.float32 if d.out_f32 else torch.bfloat16
    _check(load_library().gdn_verify_resume(
        ctypes.byref(d), _ptr(accept_len_prev, "accept_len_prev", torch.int32, d.B),
        _ptr(x, "x", torch.bfloat16, BK * C), _ptr(a, "a", torch.bfloat16, BK * d.Hv),
        _ptr(b, "b", torch.bfloat16, BK * d.Hv), _ptr(A_log, "A_log", torch.float32, d.Hv),
        _ptr(dt_bias, "dt_bias", torch.float32, d.Hv), _ptr(conv_w, "conv_w", torch.float32, C * d.conv_w),
        _ptr(conv_state_in, "conv_state_in", torch.float32, H),
        _ptr(conv_inter_prev, "conv_inter_prev", torch.float32, BK * (d.conv_w - 1) * C, allow_none=k1),
        _ptr(conv_state_snapshot_prev, "conv_state_snapshot_prev", torch.float32, H, allow_none=True),
        _ptr(conv_state_out, "conv_state_out", torch.float32, H),
        _ptr(conv_inter, "conv_inter", torch.float32, BK * (d.conv_w - 1) * C, allow_none=True),
        _ptr(state_in, "state_in", torch.float32, d.B * S),
        _ptr(state_inter_prev, "state_inter_prev", torch.float32, d.B * (d.K - 1) * S, allow_none=k1),
        _ptr(state_snapshot_prev, "state_snapshot_prev", torch.float32, d.B * S, allow_none=True),
        _ptr(state_out, "state_out", torch.float32, d.B * S),
        _ptr(state_inter, "state_inter", torch.float32, d.B * (d.K - 1) * S, allow_none=k1),
        _ptr(out, "out", odt, BK * d.Hv * d.dv), _ws_ptr(workspace), ctypes.c_uint64(_ws_bytes(workspace)),
        _stream(stream)))


def gdn_verify_step_static_scratch(dims: GdnDims, x, a, b, A_log, dt_bias, conv_w, conv_state_in, conv_state_out,
                                   conv_inter, state_in, state_out, state_inter, out, stream=None) -> None:
    """gdn_verify_step without a workspace argument, for callers that must not allocate device memory:
    a fixed array inside the library stands in for the workspace (the verify kernels need none).  The
    first call on a device looks the array up; make it before any stream capture."""
    d = dims
    C, BK = d.C, d.B * d.K
    S = d.Hv * d.dv * d.dk
    odt = torch.float32 if d.out_f32 else torch.bfloat16
    _check(load_library().gdn_verify_step_static_scratch(
        ctypes.byref(d), _ptr(x, "x", torch.bfloat16, BK * C), _ptr(a, "a", torch.bfloat16, BK * d.Hv),
        _ptr(b, "b", torch.bfloat16, BK * d.Hv), _ptr(A_log, "A_log", torch.float32, d.Hv),
        _ptr(dt_bias, "dt_bias", torch.float32, d.Hv), _ptr(conv_w, "conv_w", torch.float32, C * d.conv_w),
        _ptr(conv_state_in, "conv_state_in", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_state_out, "conv_state_out", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_inter, "conv_inter", torch.float32, BK * (d.conv_w - 1) * C, allow_none=True),
        _ptr(state_in, "state_in", torch.float32, d.B * S), _ptr(state_out, "state_out", torch.float32, d.B * S),
        _ptr(state_inter, "state_inter", torch.float32, d.B * (d.K - 1) * S, allow_none=(d.K == 1)),
        _ptr(out, "out", odt, BK * d.Hv * d.dv), _stream(stream)))


def _ws_ptr(ws):
    if ws is None:
        return None
    if not isinstance(ws, torch.Tensor) or not ws.is_cuda or not ws.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    return ctypes.c_void_p(ws.data_ptr())


def _ws_bytes(ws) -> int:
    return 0 if ws is None else ws.numel() * ws.element_size()


def gdn_rollback(dims: GdnDims, accept_len, state_in_snapshot, state, state_inter, conv_state_in_snapshot,
                 conv_state, conv_inter, stream=None) -> None:
    """a5: restore state and conv history to the accepted length of each sequence."""
    d = dims
    C = d.C
    S = d.Hv * d.dv * d.dk
    k1 = d.K == 1
    _check(load_library().gdn_rollback(
        ctypes.byref(d), _ptr(accept_len, "accept_len", torch.int32, d.B),
        _ptr(state_in_snapshot, "state_in_snapshot", torch.float32, d.B * S, allow_none=True),
        _ptr(state, "state", torch.float32, d.B * S),
        _ptr(state_inter, "state_inter", torch.float32, d.B * (d.K - 1) * S, allow_none=k1),
        _ptr(conv_state_in_snapshot, "conv_state_in_snapshot", torch.float32, d.B * (d.conv_w - 1) * C,
             allow_none=True),
        _ptr(conv_state, "conv_state", torch.float32, d.B * (d.conv_w - 1) * C),
        _ptr(conv_inter, "conv_inter", torch.float32, d.B * d.K * (d.conv_w - 1) * C, allow_none=k1),
        _stream(stream)))


def gdn_device_status(clear: bool = True, stream=None) -> int:
    """OR of the device error bits (DEVERR_*) set since the last clear; synchronises `stream`."""
    flags = ctypes.c_uint32(0)
    _check(load_library().gdn_device_status(ctypes.byref(flags), int(bool(clear)), _stream(stream)))
    return flags.value
