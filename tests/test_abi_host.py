"""Host side of the C ABI: the library loads, exports every declared entry point, and
rejects bad arguments before anything is enqueued.

Every call here with made-up pointers is built to fail validation (bad shape, NULL,
misalignment or overlap), which happens before the library touches CUDA, so these tests
run without a GPU and never launch a kernel.
"""
import ctypes
import os
import re

import pytest

from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import LIB_PATH, build_library

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "gdn.h")


@pytest.fixture(scope="module")
def lib():
    build_library()
    return gdn.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(gdn_\w+)\s*\(", text, flags=re.M)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared_functions()
    assert set(names) == set(gdn.EXPORTED)
    for n in names:
        assert hasattr(lib, n), n


BASE = dict(B=2, K=4, Hk=2, Hv=4, dk=64, dv=64)
P = 1 << 32          # fake, never dereferenced: every call below fails validation first
MB = 1 << 24


def _ptrs(n, step=MB):
    return [ctypes.c_void_p(P + i * step) for i in range(n)]


NV = 14              # pointer arguments of gdn_verify_step (the 14th is the workspace, which is unused)


def _verify(lib, dims, ptrs, ws_bytes=1 << 40):
    return lib.gdn_verify_step(ctypes.byref(dims), *ptrs, ctypes.c_uint64(ws_bytes), None)


def test_last_error_and_bad_dims(lib):
    assert lib.gdn_verify_step(None, *_ptrs(NV), ctypes.c_uint64(1 << 40), None) == gdn.GDN_ERR_INVALID_ARG
    assert "dims" in gdn.last_error()
    cases = [
        (dict(K=0), gdn.GDN_ERR_UNSUPPORTED), (dict(K=17), gdn.GDN_ERR_UNSUPPORTED),
        (dict(dk=96), gdn.GDN_ERR_UNSUPPORTED), (dict(dv=256), gdn.GDN_ERR_UNSUPPORTED),
        (dict(Hv=5), gdn.GDN_ERR_UNSUPPORTED), (dict(Hk=0), gdn.GDN_ERR_INVALID_ARG),
        (dict(B=-1), gdn.GDN_ERR_INVALID_ARG), (dict(W=3), gdn.GDN_ERR_UNSUPPORTED),
        (dict(out_f32=2), gdn.GDN_ERR_INVALID_ARG), (dict(l2_eps=-1.0), gdn.GDN_ERR_INVALID_ARG),
        (dict(q_scale=float("nan")), gdn.GDN_ERR_INVALID_ARG),
    ]
    for over, status in cases:
        kw = dict(BASE)
        kw.update(over)
        dims = gdn.make_dims(**kw)
        assert _verify(lib, dims, _ptrs(NV)) == status, over
        assert gdn.last_error() != ""


def test_empty_batch_is_a_noop(lib):
    dims = gdn.make_dims(**dict(BASE, B=0))
    assert _verify(lib, dims, [None] * NV) == gdn.GDN_OK
    assert gdn.last_error() == ""
    assert lib.gdn_conv_step(ctypes.byref(dims), None, None, None, None, None, None) == gdn.GDN_OK
    assert lib.gdn_rollback(ctypes.byref(dims), None, None, None, None, None, None, None, None) == gdn.GDN_OK


def test_null_and_misaligned_pointers(lib):
    dims = gdn.make_dims(**BASE)
    for i in range(NV - 1):   # (every call here must fail validation: the pointers are not real)
        if i in (8,):          # conv_inter is optional
            continue
        ptrs = _ptrs(NV)
        ptrs[i] = None
        assert _verify(lib, dims, ptrs) == gdn.GDN_ERR_INVALID_ARG, i
        ptrs = _ptrs(NV)
        ptrs[i] = ctypes.c_void_p(P + i * MB + 4)
        assert _verify(lib, dims, ptrs) == gdn.GDN_ERR_INVALID_ARG, i
        assert "aligned" in gdn.last_error()


def test_aliasing_rules(lib):
    dims = gdn.make_dims(**BASE)
    # out overlapping x
    ptrs = _ptrs(NV)
    ptrs[12] = ptrs[0]
    assert _verify(lib, dims, ptrs) == gdn.GDN_ERR_ALIAS
    # state_out partially overlapping state_in (shifted by 16 bytes)
    ptrs = _ptrs(NV)
    ptrs[10] = ctypes.c_void_p(ptrs[9].value + 16)
    assert _verify(lib, dims, ptrs) == gdn.GDN_ERR_ALIAS
    # state_inter overlapping state_out
    ptrs = _ptrs(NV)
    ptrs[11] = ctypes.c_void_p(ptrs[10].value + 64)
    assert _verify(lib, dims, ptrs) == gdn.GDN_ERR_ALIAS
    # conv_inter overlapping conv_state_in
    ptrs = _ptrs(NV)
    ptrs[8] = ptrs[6]
    assert _verify(lib, dims, ptrs) == gdn.GDN_ERR_ALIAS
    # K > 1 needs state_inter
    ptrs = _ptrs(NV)
    ptrs[11] = None
    assert _verify(lib, dims, ptrs) == gdn.GDN_ERR_INVALID_ARG


def test_workspace_size_formula(lib):
    dims = gdn.make_dims(B=32, K=16, Hk=16, Hv=32, dk=128, dv=128)
    assert gdn.gdn_verify_workspace_size(dims) == 0   # the verify kernels share nothing through global scratch
    with pytest.raises(gdn.GdnError):
        gdn.gdn_verify_workspace_size(gdn.make_dims(B=1, K=0, Hk=1, Hv=1, dk=64, dv=64))


def test_rollback_validation(lib):
    dims = gdn.make_dims(**BASE)
    pt = _ptrs(7)   # accept_len, state_snap, state, state_inter, conv_snap, conv_state, conv_inter
    # only one of the two snapshots
    args = list(pt)
    args[4] = None
    assert lib.gdn_rollback(ctypes.byref(dims), *args, None) == gdn.GDN_ERR_NO_SNAPSHOT
    # state overlapping state_inter
    args = list(pt)
    args[2] = args[3]
    assert lib.gdn_rollback(ctypes.byref(dims), *args, None) == gdn.GDN_ERR_ALIAS
    # K > 1 without intermediates
    args = list(pt)
    args[3] = None
    assert lib.gdn_rollback(ctypes.byref(dims), *args, None) == gdn.GDN_ERR_INVALID_ARG
    args = list(pt)
    args[0] = ctypes.c_void_p(P + 2)
    assert lib.gdn_rollback(ctypes.byref(dims), *args, None) == gdn.GDN_ERR_INVALID_ARG


def test_tree_validation(lib):
    dims = gdn.make_dims(**BASE)
    ptrs = _ptrs(NV)
    assert lib.gdn_verify_tree(ctypes.byref(dims), None, *ptrs, ctypes.c_uint64(1 << 40), None) == gdn.GDN_ERR_INVALID_ARG
    assert lib.gdn_verify_tree(ctypes.byref(dims), ctypes.c_void_p(P - 2), *ptrs, ctypes.c_uint64(1 << 40),
                               None) == gdn.GDN_ERR_INVALID_ARG
    # parent overlapping an output
    assert lib.gdn_verify_tree(ctypes.byref(dims), ptrs[12], *ptrs, ctypes.c_uint64(1 << 40), None) == gdn.GDN_ERR_ALIAS


def test_gated_validation(lib):
    dims = gdn.make_dims(**BASE)

    def call(z_null=False, w_null=False, eps=1e-6, z=None):
        pt = _ptrs(16)
        zp = None if z_null else (z if z is not None else pt[12])
        wp = None if w_null else pt[13]
        return lib.gdn_verify_gated(ctypes.byref(dims), *pt[:12], zp, wp, ctypes.c_float(eps), pt[14], pt[15],
                                    ctypes.c_uint64(1 << 40), None)

    assert call(z_null=True) == gdn.GDN_ERR_INVALID_ARG and "z" in gdn.last_error()
    assert call(w_null=True) == gdn.GDN_ERR_INVALID_ARG and "norm_w" in gdn.last_error()
    assert call(eps=float("nan")) == gdn.GDN_ERR_INVALID_ARG
    assert call(eps=-1.0) == gdn.GDN_ERR_INVALID_ARG
    assert call(z=ctypes.c_void_p(P + 12 * MB + 8)) == gdn.GDN_ERR_INVALID_ARG   # misaligned
    assert call(z=ctypes.c_void_p(P + 14 * MB)) == gdn.GDN_ERR_ALIAS            # z overlapping out
    assert "z" in gdn.last_error()


def test_prefill_validation(lib):
    dims = gdn.make_dims(**BASE)
    N = 100

    def call(n=N, cu="ok", ws=1 << 40, dims=dims, **swap):
        pt = _ptrs(13)
        names = ["cu", "x", "a", "b", "A_log", "dt_bias", "conv_w", "conv_state_in", "conv_state_out", "state_in",
                 "state_out", "out", "workspace"]
        args = dict(zip(names, pt))
        if cu is None:
            args["cu"] = None
        elif cu == "odd":
            args["cu"] = ctypes.c_void_p(P + 2)
        args.update(swap)
        return lib.gdn_prefill(ctypes.byref(dims), ctypes.c_int64(n), *[args[k] for k in names],
                               ctypes.c_uint64(ws), None)

    assert call(cu=None) == gdn.GDN_ERR_INVALID_ARG and "cu_seqlens" in gdn.last_error()
    assert call(cu="odd") == gdn.GDN_ERR_INVALID_ARG
    assert call(n=-1) == gdn.GDN_ERR_INVALID_ARG
    assert call(n=1 << 31) == gdn.GDN_ERR_INVALID_ARG
    assert call(ws=16) == gdn.GDN_ERR_INVALID_ARG and "workspace" in gdn.last_error()
    assert call(x=None) == gdn.GDN_ERR_INVALID_ARG
    assert call(state_out=ctypes.c_void_p(P + MB + 16)) == gdn.GDN_ERR_ALIAS        # state_out inside x
    assert call(conv_state_out=ctypes.c_void_p(P + 11 * MB)) == gdn.GDN_ERR_ALIAS  # conv_state_out == out
    assert call(dims=gdn.make_dims(**dict(BASE, dk=96))) == gdn.GDN_ERR_UNSUPPORTED
    assert call(dims=gdn.make_dims(**dict(BASE, B=0))) == gdn.GDN_ERR_INVALID_ARG   # tokens without prompts
    assert lib.gdn_prefill(ctypes.byref(gdn.make_dims(**dict(BASE, B=0))), ctypes.c_int64(0), *([None] * 13),
                           ctypes.c_uint64(0), None) == gdn.GDN_OK                   # nothing to do
    need = ctypes.c_uint64(0)
    assert lib.gdn_prefill_workspace_size(ctypes.byref(dims), ctypes.c_int64(N), ctypes.byref(need)) == gdn.GDN_OK
    cap = (N + 63) // 64 + dims.B
    expect = 16 * ((dims.B + 5 + 3) // 4) + cap * (16 + dims.Hk * 512 * dims.dk + dims.Hv * 33280)
    assert need.value == expect


def test_conv_step_validation(lib):
    dims = gdn.make_dims(**BASE)
    pt = _ptrs(5)
    args = list(pt)
    args[4] = args[0]                    # y overlapping x
    assert lib.gdn_conv_step(ctypes.byref(dims), *args, None) == gdn.GDN_ERR_ALIAS
    args = list(pt)
    args[2] = None
    assert lib.gdn_conv_step(ctypes.byref(dims), *args, None) == gdn.GDN_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors():
    import torch
    dims = gdn.make_dims(**BASE)
    t = torch.zeros(4)
    with pytest.raises(ValueError):
        gdn.gdn_conv_step(dims, t, t, t, None, t)


def test_library_path_in_tree():
    assert os.path.dirname(LIB_PATH).endswith("speculative_decode_verify_gdn_gb300")
