"""gdn_verify_resume: the previous window's rollback applied on read, checked bit for bit against
gdn_rollback + gdn_verify_step, and against the oracle over many rounds."""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from parity_util import OUT_TOL, STATE_TOL, oracle_round, out_rel_err, state_rel_err
from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Dims, Dists, Gen, make_layer, make_round

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    gdn.gdn_device_status(clear=True)
    yield
    assert gdn.gdn_device_status(clear=True) == 0


@pytest.mark.parametrize("shape", [(3, 7, 2, 4, 128, 128), (2, 16, 1, 3, 64, 128), (4, 5, 2, 2, 64, 64)])
def test_resume_equals_rollback_then_verify_bitwise(shape):
    B, K, Hk, Hv, dk, dv = shape
    d = Dims(B=B, K=K, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(300 + sum(shape))
    lay = make_layer(g, d, Dists())
    a = GdnLayerState.create(d, lay)       # verify + rollback copy
    r = GdnLayerState.create(d, lay)       # rollback applied on the next verify's read
    prev = None
    for rd in range(6):
        rnd = make_round(g, d, Dists())
        a.load_round(rnd)
        r.load_round(rnd)
        a.verify()
        if prev is None:
            r.verify()
        else:
            r.verify_resume(prev)
        torch.cuda.synchronize()
        assert torch.equal(a.out, r.out), rd
        assert torch.equal(a.state, r.state), rd
        assert torch.equal(a.state_inter, r.state_inter), rd
        assert torch.equal(a.conv_inter, r.conv_inter), rd
        assert torch.equal(a.conv_state, r.conv_state), rd
        a.rollback()
        prev = r.accept_len.clone()
    # materialise the last rollback on the resume side too
    r.rollback()
    torch.cuda.synchronize()
    assert torch.equal(a.state, r.state) and torch.equal(a.conv_state, r.conv_state)


def test_resume_against_oracle_dflash_rounds():
    """B=1, K=16 DFlash-width workload, 60 rounds chained through gdn_verify_resume only."""
    w = WORKLOADS["dflash"]
    d = w.dims
    g = Gen(w.seed)
    lay = make_layer(g, d, w.dists)
    st = GdnLayerState.create(d, lay)
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    prev = None
    for rd in range(60):
        rnd = make_round(g, d, w.dists)
        st.load_round(rnd)
        if prev is None:
            st.verify()
        else:
            st.verify_resume(prev)
        ref = oracle_round(d, lay, S, H, rnd)
        assert out_rel_err(st.out.cpu().numpy(), ref["out"]) <= OUT_TOL
        if rd % 10 == 0:
            assert state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"]) <= STATE_TOL
            np.testing.assert_array_equal(st.conv_inter.cpu().numpy(), ref["conv_inter"])
        S, H = O.rollback(rnd.accept_len, S, ref["states"], H, ref["conv_inter"])
        prev = st.accept_len.clone()


def test_resume_serving_shape_against_oracle():
    w = WORKLOADS["serve16"]
    d = w.dims
    g = Gen(w.seed + 7)
    lay = make_layer(g, d, w.dists)
    st = GdnLayerState.create(d, lay, out_f32=True)
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    prev = None
    for rd in range(2):
        rnd = make_round(g, d, w.dists)
        st.load_round(rnd)
        st.verify() if prev is None else st.verify_resume(prev)
        ref = oracle_round(d, lay, S, H, rnd)
        assert out_rel_err(st.out.cpu().numpy(), ref["out"]) <= OUT_TOL
        assert state_rel_err(st.state.cpu().numpy(), ref["state_out"]) <= STATE_TOL
        assert state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"]) <= STATE_TOL
        S, H = O.rollback(rnd.accept_len, S, ref["states"], H, ref["conv_inter"])
        prev = st.accept_len.clone()
        del ref


def test_resume_zero_accept_with_snapshots_and_bad_lengths():
    """L = 0 reads the snapshots; out-of-range lengths read the final state and set a status bit."""
    d = Dims(B=5, K=4, Hk=1, Hv=2, dk=64, dv=64)
    g = Gen(61)
    lay = make_layer(g, d, Dists())
    r1, r2 = make_round(g, d, Dists()), make_round(g, d, Dists())
    st = GdnLayerState.create(d, lay, keep_snapshot=True)   # window 1: states[0] -> states[1]
    st.load_round(r1)
    st.verify()
    snap, csnap = st.states[0], st.conv_states[0]
    fin, cfin = st.states[1], st.conv_states[1]
    acc = torch.tensor([0, 2, 4, -1, 9], dtype=torch.int32, device="cuda")
    st.load_round(r2)
    gdn.gdn_verify_resume(st.dims, acc, st.x, st.a, st.b, st.A_log, st.dt_bias, st.conv_w, cfin, st.conv_inter,
                          csnap, cfin, st.conv_inter, fin, st.state_inter, snap, fin, st.state_inter, st.out,
                          st.workspace)
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(clear=True) == gdn.DEVERR_ACCEPT_RANGE
    ref1 = oracle_round(d, lay, lay.state, lay.conv_state, r1)
    eff = np.array([0, 2, 4, 4, 4])                                   # bad lengths read as K
    S, H = O.rollback(eff, lay.state, ref1["states"], lay.conv_state, ref1["conv_inter"])
    ref2 = oracle_round(d, lay, S, H, r2)
    assert out_rel_err(st.out.cpu().numpy(), ref2["out"]) <= OUT_TOL
    assert state_rel_err(fin.cpu().numpy(), ref2["state_out"]) <= STATE_TOL
    np.testing.assert_array_equal(cfin.cpu().numpy(), ref2["conv_state_out"])
