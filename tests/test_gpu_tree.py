"""gdn_verify_tree (token-tree verify) against the tree oracle, and its consistency with the
chain verify and with gdn_rollback to an accepted node."""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from parity_util import OUT_TOL, STATE_TOL, out_rel_err, state_rel_err
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


def _oracle_tree(d, lay, rnd, parent, q_scale=1.0):
    return O.tree_verify_step(d, parent, bf16_bits_to_f32(rnd.x), bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b),
                              lay.A_log, lay.dt_bias, lay.conv_w, lay.conv_state, lay.state, q_scale=q_scale)


def _run(d, lay, rnd, parent, out_f32=True, q_scale=1.0):
    st = GdnLayerState.create(d, lay, out_f32=out_f32, q_scale=q_scale)
    st.load_round(rnd)
    par = torch.from_numpy(parent.astype(np.int32)).cuda()
    st.verify_tree(par)
    torch.cuda.synchronize()
    return st


def _check(st, ref, d):
    assert out_rel_err(st.out.float().cpu().numpy(), ref["out"]) <= OUT_TOL
    assert state_rel_err(st.states[0].cpu().numpy(), ref["state_out"]) <= STATE_TOL
    if d.K > 1:
        assert state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"]) <= STATE_TOL
    np.testing.assert_array_equal(st.conv_inter.cpu().numpy(), ref["conv_inter"])
    np.testing.assert_array_equal(st.conv_states[0].cpu().numpy(), ref["conv_state_out"])


@pytest.mark.parametrize("shape,p_chain", [((3, 9, 2, 4, 128, 128), 0.5), ((2, 16, 1, 3, 64, 128), 0.3),
                                           ((4, 6, 2, 2, 64, 64), 0.0), ((2, 16, 16, 32, 128, 128), 0.6),
                                           ((1, 1, 2, 4, 128, 64), 0.5)])
def test_random_trees_against_oracle(shape, p_chain):
    B, K, Hk, Hv, dk, dv = shape
    d = Dims(B=B, K=K, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(700 + sum(shape))
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    parent = make_tree(g, B, K, p_chain)
    st = _run(d, lay, rnd, parent, q_scale=0.9)
    _check(st, _oracle_tree(d, lay, rnd, parent, q_scale=0.9), d)


def test_chain_tree_equals_verify_step():
    """A chain-shaped tree is the chain window: the histories bit for bit (the same conv code), the
    states and outputs up to f32 rounding order (the tree kernel sums a row's dot products over the
    whole warp, the chain kernel over the row's eight lanes), and both against the oracle."""
    d = Dims(B=3, K=12, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(711)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    parent = np.tile(np.arange(-1, d.K - 1, dtype=np.int32), (d.B, 1))
    tr = _run(d, lay, rnd, parent)
    ch = GdnLayerState.create(d, lay, out_f32=True)
    ch.load_round(rnd)
    ch.verify()
    torch.cuda.synchronize()
    for a, b in [(tr.conv_inter, ch.conv_inter), (tr.conv_states[0], ch.conv_states[0])]:
        assert torch.equal(a, b)
    assert out_rel_err(tr.out.cpu().numpy(), ch.out.cpu().numpy().astype(np.float64)) <= OUT_TOL
    assert state_rel_err(tr.states[0].cpu().numpy(), ch.states[0].cpu().numpy().astype(np.float64)) <= STATE_TOL
    assert state_rel_err(tr.state_inter.cpu().numpy(), ch.state_inter.cpu().numpy().astype(np.float64)) <= STATE_TOL
    _check(tr, _oracle_tree(d, lay, rnd, parent), d)


def test_star_and_deep_branching_trees():
    d = Dims(B=2, K=16, Hk=2, Hv=4, dk=64, dv=128)
    g = Gen(712)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    star = np.full((1, d.K), -1, np.int32)
    comb = np.array([[-1, 0, 1, 2, 1, 4, 0, 6, 7, 3, 9, 10, 5, 12, 8, 14]], np.int32)   # restores mid-chain
    parent = np.concatenate([star, comb])
    st = _run(d, lay, rnd, parent, out_f32=False)
    ref = _oracle_tree(d, lay, rnd, parent)
    assert out_rel_err(st.out.float().cpu().numpy(), ref["out"]) <= OUT_TOL + 2.0 ** -8
    assert state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"]) <= STATE_TOL
    np.testing.assert_array_equal(st.conv_inter.cpu().numpy(), ref["conv_inter"])


def test_tree_rollback_to_accepted_node():
    """gdn_rollback with accept_len = n + 1 restores the state and history after node n."""
    w = WORKLOADS["serve16"]
    d = Dims(B=4, K=16, Hk=16, Hv=32, dk=128, dv=128)
    g = Gen(713)
    lay = make_layer(g, d, w.dists)
    rnd = make_round(g, d, w.dists)
    parent = make_tree(g, d.B, d.K, 0.5)
    st = GdnLayerState.create(d, lay, keep_snapshot=True)
    st.load_round(rnd)
    st.verify_tree(torch.from_numpy(parent).cuda())
    accepted = np.array([-1, 3, 15, 7], np.int32)                 # the last accepted node per sequence
    st.accept_len.copy_(torch.from_numpy(accepted + 1))
    st.rollback()
    torch.cuda.synchronize()
    ref = _oracle_tree(d, lay, rnd, parent)
    for bi, n in enumerate(accepted):
        S = lay.state[bi] if n < 0 else ref["states"][bi, n]
        H = lay.conv_state[bi] if n < 0 else ref["conv_inter"][bi, n]
        assert state_rel_err(st.state[bi].cpu().numpy(), S) <= STATE_TOL
        np.testing.assert_array_equal(st.conv_state[bi].cpu().numpy(), H)


def test_bad_parent_is_flagged_and_read_as_root():
    d = Dims(B=1, K=4, Hk=1, Hv=2, dk=64, dv=64)
    g = Gen(714)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    bad = np.array([[-1, 0, 5, 1]], np.int32)
    st = _run(d, lay, rnd, bad)
    assert gdn.gdn_device_status(clear=True) == gdn.DEVERR_TREE_PARENT
    ref = _oracle_tree(d, lay, rnd, np.array([[-1, 0, -1, 1]]))
    _check(st, ref, d)
