"""The verify calls with their optional outputs left out: no per-token conv snapshots
(conv_inter NULL) and no workspace (the verify kernels need none).  The second kernel of a call
then writes only the q|k channels' new history; everything else must be the full call's, bit
for bit, and the oracle's."""
import numpy as np
import pytest
import torch

from parity_util import OUT_TOL, STATE_TOL, oracle_round, out_rel_err, state_rel_err
from oracle import gdn_oracle as O
from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import (WORKLOADS, Dims, Dists, Gen, bf16_bits_to_f32, make_layer,
                                                        make_round, make_tree)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    gdn.gdn_device_status(clear=True)
    yield
    assert gdn.gdn_device_status(clear=True) == 0


def _bare(st):
    """The same window through gdn_verify_step without snapshots or workspace, in place."""
    gdn.gdn_verify_step(st.dims, st.x, st.a, st.b, st.A_log, st.dt_bias, st.conv_w, st.conv_states[0],
                        st.conv_states[0], None, st.states[0], st.states[0], st.state_inter, st.out, None)


@pytest.mark.parametrize("shape", [(3, 9, 2, 4, 128, 128), (2, 5, 1, 3, 64, 128), (1, 1, 2, 4, 128, 64)])
def test_verify_without_snapshots_or_workspace(shape):
    B, K, Hk, Hv, dk, dv = shape
    d = Dims(B=B, K=K, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(1300 + sum(shape))
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    full = GdnLayerState.create(d, lay)
    full.load_round(rnd)
    full.verify()
    bare = GdnLayerState.create(d, lay)
    bare.load_round(rnd)
    _bare(bare)
    torch.cuda.synchronize()
    pairs = [(bare.out, full.out), (bare.states[0], full.states[0]), (bare.conv_states[0], full.conv_states[0])]
    if K > 1:
        pairs.append((bare.state_inter, full.state_inter))
    for a, b in pairs:
        assert torch.equal(a, b)
    ref = oracle_round(d, lay, lay.state.astype(np.float64), lay.conv_state.astype(np.float64), rnd)
    assert out_rel_err(bare.out.cpu().numpy(), ref["out"]) <= OUT_TOL
    assert state_rel_err(bare.states[0].cpu().numpy(), ref["state_out"]) <= STATE_TOL
    np.testing.assert_array_equal(bare.conv_states[0].cpu().numpy(), ref["conv_state_out"])


def test_serving_shape_without_snapshots_two_windows():
    """B=32, K=16 at the serving head shape, two windows carried in place: the bare call's history
    and states stay the full call's, bit for bit."""
    w = WORKLOADS["serve16"]
    d = w.dims
    g = Gen(1351)
    lay = make_layer(g, d, w.dists)
    full = GdnLayerState.create(d, lay, out_f32=False)
    bare = GdnLayerState.create(d, lay, out_f32=False)
    for _ in range(2):
        rnd = make_round(g, d, w.dists)
        full.load_round(rnd)
        full.verify()
        bare.load_round(rnd)
        _bare(bare)
    torch.cuda.synchronize()
    for a, b in [(bare.out, full.out), (bare.states[0], full.states[0]), (bare.state_inter, full.state_inter),
                 (bare.conv_states[0], full.conv_states[0])]:
        assert torch.equal(a, b)


def test_tree_without_snapshots():
    d = Dims(B=3, K=12, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(1377)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    parent = make_tree(g, d.B, d.K, 0.5)
    par = torch.from_numpy(parent.astype(np.int32)).cuda()
    full = GdnLayerState.create(d, lay)
    full.load_round(rnd)
    full.verify_tree(par)
    bare = GdnLayerState.create(d, lay)
    bare.load_round(rnd)
    gdn.gdn_verify_tree(bare.dims, par, bare.x, bare.a, bare.b, bare.A_log, bare.dt_bias, bare.conv_w,
                        bare.conv_states[0], bare.conv_states[0], None, bare.states[0], bare.states[0],
                        bare.state_inter, bare.out, None)
    torch.cuda.synchronize()
    for a, b in [(bare.out, full.out), (bare.states[0], full.states[0]), (bare.state_inter, full.state_inter),
                 (bare.conv_states[0], full.conv_states[0])]:
        assert torch.equal(a, b)
    ref = O.tree_verify_step(d, parent, bf16_bits_to_f32(rnd.x), bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b),
                             lay.A_log, lay.dt_bias, lay.conv_w, lay.conv_state, lay.state)
    np.testing.assert_array_equal(bare.conv_states[0].cpu().numpy(), ref["conv_state_out"])
