"""gdn_verify_gated (verify step with the gated RMS output norm fused into its epilogue)
against the oracle's verify step followed by its gated_rms_norm, and its states against
the plain verify step.

Output tolerance: the verify outputs' own, per (b, t, v-head) vector
max_i |y_i - y_ref_i| / max_i |y_ref_i| <= 2e-3 (f32 outputs; bf16 outputs add 2^-8), with
y_ref = the oracle's gated norm of the oracle's verify output.
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from parity_util import OUT_TOL, OUT_TOL_BF16, STATE_TOL, oracle_round, out_rel_err, state_rel_err
from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import (WORKLOADS, Dims, Dists, Gen, Round, bf16_bits_to_f32,
                                                        make_layer, make_output_gate, make_round)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    gdn.gdn_device_status(clear=True)
    yield
    assert gdn.gdn_device_status(clear=True) == 0


def _gated_err(y, o_ref, z_bits, w, eps):
    """Per (b, t, v-head) vector: max |y - y_ref| / max |y_ref|, the plain outputs' metric."""
    y_ref = O.gated_rms_norm(np.asarray(o_ref, np.float64), bf16_bits_to_f32(z_bits).astype(np.float64), w, eps)
    return out_rel_err(y, y_ref)


def _run_gated(d, lay, rnd, z_bits, w, eps, out_f32=True, q_scale=1.0):
    st = GdnLayerState.create(d, lay, out_f32=out_f32, q_scale=q_scale)
    st.load_round(rnd)
    z = torch.from_numpy(z_bits.view(np.int16)).cuda().view(torch.bfloat16)
    st.verify_gated(z, torch.from_numpy(w).cuda(), eps)
    torch.cuda.synchronize()
    return st


@pytest.mark.parametrize("shape,out_f32", [((2, 16, 2, 4, 128, 128), True), ((3, 7, 1, 3, 64, 64), True),
                                           ((2, 5, 2, 4, 128, 64), False), ((1, 1, 2, 2, 64, 128), True),
                                           ((4, 16, 16, 32, 128, 128), False)])
def test_shapes_against_oracle(shape, out_f32):
    B, K, Hk, Hv, dk, dv = shape
    d = Dims(B=B, K=K, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(900 + sum(shape))
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    z, w = make_output_gate(g, d)
    eps = 1e-6
    st = _run_gated(d, lay, rnd, z, w, eps, out_f32=out_f32, q_scale=0.8)
    ref = oracle_round(d, lay, lay.state.astype(np.float64), lay.conv_state.astype(np.float64), rnd, q_scale=0.8)
    assert _gated_err(st.out.float().cpu().numpy(), ref["out"], z, w, eps) <= (OUT_TOL if out_f32 else OUT_TOL_BF16)
    assert state_rel_err(st.states[0].cpu().numpy(), ref["state_out"]) <= STATE_TOL
    if K > 1:
        assert state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"]) <= STATE_TOL
    np.testing.assert_array_equal(st.conv_inter.cpu().numpy(), ref["conv_inter"])


def test_large_eps_and_zero_weight_rows():
    """A large eps shrinks every output (the norm stops dividing by the rms); zero weights
    give exact zeros."""
    d = Dims(B=2, K=8, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(931)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    z, w = make_output_gate(g, d)
    w[::3] = 0.0
    eps = 10.0
    st = _run_gated(d, lay, rnd, z, w, eps)
    ref = oracle_round(d, lay, lay.state.astype(np.float64), lay.conv_state.astype(np.float64), rnd)
    y = st.out.cpu().numpy()
    assert _gated_err(y, ref["out"], z, w, eps) <= OUT_TOL
    assert np.all(y[..., ::3] == 0.0)


def test_states_and_history_equal_plain_verify_bitwise():
    """The fused norm changes only the output: states, intermediates and conv history are the
    plain verify step's, bit for bit."""
    d = Dims(B=3, K=12, Hk=2, Hv=8, dk=128, dv=128)
    g = Gen(947)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    z, w = make_output_gate(g, d)
    ga = _run_gated(d, lay, rnd, z, w, 1e-6)
    pl = GdnLayerState.create(d, lay)
    pl.load_round(rnd)
    pl.verify()
    torch.cuda.synchronize()
    for a, b in [(ga.states[0], pl.states[0]), (ga.state_inter, pl.state_inter),
                 (ga.conv_inter, pl.conv_inter), (ga.conv_states[0], pl.conv_states[0])]:
        assert torch.equal(a, b)


def test_decode_step_equals_first_token_of_a_window():
    """The one-token instantiation of the gated variant against a two-token window's first
    token, bit for bit (outputs after the norm, state and conv history)."""
    d2 = Dims(B=3, K=2, Hk=2, Hv=8, dk=128, dv=128)
    d1 = Dims(B=3, K=1, Hk=2, Hv=8, dk=128, dv=128)
    g = Gen(4200)
    lay = make_layer(g, d2, Dists())
    rnd = make_round(g, d2, Dists())
    one = Round(x=rnd.x[:, :1].copy(), a=rnd.a[:, :1].copy(), b=rnd.b[:, :1].copy(),
                accept_len=np.ones(d1.B, np.int32))
    z_bits, w = make_output_gate(g, d2)
    win = _run_gated(d2, lay, rnd, z_bits, w, 1e-6)
    dec = _run_gated(d1, lay, one, np.ascontiguousarray(z_bits[:, :1]), w, 1e-6)
    assert torch.equal(dec.out[:, 0], win.out[:, 0])
    assert torch.equal(dec.states[0], win.state_inter[:, 0])
    assert torch.equal(dec.conv_states[0], win.conv_inter[:, 0])


def test_serving_shape_sampled_sequences():
    """B=32, K=16, Hv=32 (the K=16 serving shape, cluster of 4 row tiles per head): sampled
    sequences against the oracle run on those sequences alone."""
    w0 = WORKLOADS["serve16"]
    d = w0.dims
    g = Gen(w0.seed + 50)
    lay = make_layer(g, d, w0.dists)
    rnd = make_round(g, d, w0.dists)
    z, w = make_output_gate(g, d)
    st = _run_gated(d, lay, rnd, z, w, 1e-6, out_f32=False)
    d1 = Dims(B=1, K=d.K, Hk=d.Hk, Hv=d.Hv, dk=d.dk, dv=d.dv)
    for bi in (0, 17, 31):
        sl = slice(bi, bi + 1)
        r1 = Round(rnd.x[sl], rnd.a[sl], rnd.b[sl], rnd.accept_len[sl])
        ref = oracle_round(d1, lay, lay.state[sl].astype(np.float64), lay.conv_state[sl].astype(np.float64), r1)
        assert _gated_err(st.out[sl].float().cpu().numpy(), ref["out"], z[sl], w, 1e-6) <= OUT_TOL_BF16
        assert state_rel_err(st.states[0][sl].cpu().numpy(), ref["state_out"]) <= STATE_TOL
