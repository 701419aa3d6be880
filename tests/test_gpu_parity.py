"""Parity of the sm_103a path (through the C ABI) with the CPU oracle.

Inputs come from the seeded generator; expected values only from oracle/.  Sizes span
several row tiles and head groups with ragged windows (odd K, odd B), every supported head
shape, both output types, in place and ping-pong states, and the named workloads at their
full sizes (all outputs, or sampled sequences / layers where the oracle would be slow).
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from parity_util import (OUT_TOL, OUT_TOL_BF16, STATE_TOL, bf16_tensor_to_f32, oracle_round, out_rel_err,
                         state_rel_err)
from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import (WORKLOADS, Dims, Dists, Gen, Round, bf16_bits_to_f32,
                                                        make_layer, make_round)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    gdn.gdn_device_status(clear=True)
    yield
    assert gdn.gdn_device_status(clear=True) == 0


def _check_round(st, ref, d, out_f32=True, verified_state=None):
    """Compare the verify outputs on the device with an oracle round."""
    out = bf16_tensor_to_f32(st.out)
    tol = OUT_TOL if out_f32 else OUT_TOL_BF16
    e_out = out_rel_err(out, ref["out"])
    assert e_out <= tol, f"out rel err {e_out}"
    S = (verified_state if verified_state is not None else st.states[0]).cpu().numpy()
    e_s = state_rel_err(S, ref["state_out"])
    assert e_s <= STATE_TOL, f"final state rel err {e_s}"
    if d.K > 1:
        e_i = state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"])
        assert e_i <= STATE_TOL, f"intermediate state rel err {e_i}"
    np.testing.assert_array_equal(st.conv_inter.cpu().numpy(), ref["conv_inter"])
    return e_out, e_s


SHAPES = [
    # B, K, Hk, Hv, dk, dv   (head groups r = 1..5, dk and dv 64 or 128)
    (3, 5, 2, 4, 128, 128),
    (2, 16, 1, 3, 128, 128),
    (2, 7, 2, 2, 64, 128),
    (1, 3, 4, 8, 128, 64),
    (2, 9, 1, 5, 64, 64),
    (2, 11, 2, 2, 64, 64),
    (1, 1, 2, 4, 128, 128),
    (5, 2, 1, 2, 128, 64),
]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("out_f32", [1, 0])
def test_shapes_against_oracle(shape, out_f32):
    B, K, Hk, Hv, dk, dv = shape
    d = Dims(B=B, K=K, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(1000 + sum(shape) + out_f32)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    q_scale = 0.75 if out_f32 else 1.0
    st = GdnLayerState.create(d, lay, out_f32=bool(out_f32), q_scale=q_scale)
    st.load_round(rnd)
    st.verify()
    torch.cuda.synchronize()
    ref = oracle_round(d, lay, lay.state, lay.conv_state, rnd, q_scale=q_scale)
    _check_round(st, ref, d, out_f32=bool(out_f32))
    np.testing.assert_array_equal(st.conv_state.cpu().numpy(), ref["conv_state_out"])


def test_many_vheads_per_qk_head():
    """Hv/Hk = 8: one q/k head feeds eight v-heads (32 verify CTAs convolve and normalise its q|k)."""
    d = Dims(B=2, K=6, Hk=1, Hv=8, dk=128, dv=128)
    g = Gen(77)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    st = GdnLayerState.create(d, lay)
    st.load_round(rnd)
    st.verify()
    torch.cuda.synchronize()
    _check_round(st, oracle_round(d, lay, lay.state, lay.conv_state, rnd), d)


def test_tiny_rounds_with_rollback_and_zero_accept():
    """Tiny workload: 50 verify + rollback rounds, accept lengths U{0..4} (0 needs the snapshot)."""
    w = WORKLOADS["tiny"]
    d = w.dims
    g = Gen(w.seed)
    lay = make_layer(g, d, w.dists)
    st = GdnLayerState.create(d, lay, keep_snapshot=True)
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    seen = set()
    for _ in range(w.rounds):
        rnd = make_round(g, d, w.dists)
        st.load_round(rnd)
        st.verify()
        ref = oracle_round(d, lay, S, H, rnd)
        _check_round(st, ref, d, verified_state=st.states[1 - st.cur])
        st.rollback()
        S, H = O.rollback(rnd.accept_len, S, ref["states"], H, ref["conv_inter"])
        assert state_rel_err(st.state.cpu().numpy(), S) <= STATE_TOL
        np.testing.assert_array_equal(st.conv_state.cpu().numpy(), H)
        seen.update(int(v) for v in rnd.accept_len)
    assert 0 in seen and 4 in seen


def test_in_place_equals_ping_pong_and_is_deterministic():
    d = Dims(B=3, K=7, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(5)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    outs = []
    for keep in (False, True, False):
        st = GdnLayerState.create(d, lay, keep_snapshot=keep)
        st.load_round(rnd)
        st.verify()
        torch.cuda.synchronize()
        fin = st.states[1 - st.cur] if keep else st.states[0]
        outs.append((st.out.cpu(), fin.cpu(), st.state_inter.cpu(), st.conv_inter.cpu(),
                     st.conv_states[1 - st.cur if keep else 0].cpu()))
    for a, b in zip(outs[0], outs[1]):
        assert torch.equal(a, b)
    for a, b in zip(outs[0], outs[2]):
        assert torch.equal(a, b)


def test_window_equals_serial_one_token_steps_on_gpu():
    """Batched verify stays aligned with serial decode (the drift the pages call a bug)."""
    d = Dims(B=2, K=16, Hk=2, Hv=4, dk=128, dv=128)
    d1 = Dims(B=2, K=1, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(9)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    win = GdnLayerState.create(d, lay)
    win.load_round(rnd)
    win.verify()
    one = GdnLayerState.create(d1, lay)
    outs, states = [], []
    for t in range(d.K):
        one.x.copy_(win.x[:, t:t + 1])
        one.a.copy_(win.a[:, t:t + 1])
        one.b.copy_(win.b[:, t:t + 1])
        one.verify()
        outs.append(one.out[:, 0].cpu().numpy())
        states.append(one.state.cpu().numpy())
    torch.cuda.synchronize()
    assert out_rel_err(win.out.cpu().numpy(), np.stack(outs, axis=1)) <= OUT_TOL
    assert state_rel_err(win.state_inter.cpu().numpy(), np.stack(states[:-1], axis=1)) <= STATE_TOL
    assert state_rel_err(win.state.cpu().numpy(), states[-1]) <= STATE_TOL


@pytest.mark.parametrize("out_f32", [1, 0])
def test_conv_step_against_oracle(out_f32):
    d = Dims(B=3, K=9, Hk=2, Hv=6, dk=64, dv=128)
    g = Gen(31)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    dims = gdn.make_dims(d.B, d.K, d.Hk, d.Hv, d.dk, d.dv, out_f32=out_f32)
    x = torch.from_numpy(rnd.x.view(np.int16)).cuda().view(torch.bfloat16)
    w = torch.from_numpy(lay.conv_w).cuda()
    hist = torch.from_numpy(lay.conv_state).cuda()
    inter = torch.empty((d.B, d.K, 3, d.C), dtype=torch.float32, device="cuda")
    y = torch.empty((d.B, d.K, d.C), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    gdn.gdn_conv_step(dims, x, w, hist, inter, y)
    torch.cuda.synchronize()
    y_ref, inter_ref, hist_ref = O.conv_step(bf16_bits_to_f32(rnd.x), lay.conv_w, lay.conv_state)
    yv = bf16_tensor_to_f32(y)
    rel = np.max(np.abs(yv - y_ref)) / np.max(np.abs(y_ref))
    assert rel <= (1e-5 if out_f32 else 2.0 ** -8)
    np.testing.assert_array_equal(inter.cpu().numpy(), inter_ref)
    np.testing.assert_array_equal(hist.cpu().numpy(), hist_ref)


def test_rollback_edge_cases_and_device_flags():
    d = Dims(B=6, K=5, Hk=1, Hv=2, dk=64, dv=64)
    g = Gen(41)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    st = GdnLayerState.create(d, lay, keep_snapshot=True)
    st.load_round(rnd)
    st.verify()
    torch.cuda.synchronize()
    o = 1 - st.cur
    fin, inter = st.states[o].clone(), st.state_inter.clone()
    cfin, cinter = st.conv_states[o].clone(), st.conv_inter.clone()
    S0, H0 = st.states[st.cur].clone(), st.conv_states[st.cur].clone()
    st.accept_len.copy_(torch.tensor([0, 1, 3, 5, -1, 6], dtype=torch.int32))
    st.rollback()
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(clear=True) == gdn.DEVERR_ACCEPT_RANGE
    got, cgot = st.state, st.conv_state
    assert torch.equal(got[0], S0[0]) and torch.equal(cgot[0], H0[0])          # L = 0: snapshot
    assert torch.equal(got[1], inter[1, 0]) and torch.equal(cgot[1], cinter[1, 0])
    assert torch.equal(got[2], inter[2, 2]) and torch.equal(cgot[2], cinter[2, 2])
    assert torch.equal(got[3], fin[3]) and torch.equal(cgot[3], cfin[3])      # L = K: untouched
    assert torch.equal(got[4], fin[4]) and torch.equal(got[5], fin[5])        # out of range: untouched
    # in place with no snapshot: L = 0 cannot be served
    st2 = GdnLayerState.create(d, lay)
    st2.load_round(rnd)
    st2.verify()
    before = st2.state.clone()
    st2.accept_len.copy_(torch.tensor([0, 5, 5, 5, 5, 5], dtype=torch.int32))
    st2.rollback()
    torch.cuda.synchronize()
    assert gdn.gdn_device_status(clear=True) == gdn.DEVERR_NO_SNAPSHOT
    assert torch.equal(st2.state, before)


def test_empty_batch_through_binding():
    d = Dims(B=0, K=4, Hk=2, Hv=4, dk=64, dv=64)
    dims = gdn.make_dims(0, 4, 2, 4, 64, 64)
    e = torch.empty(0, device="cuda")
    eb = torch.empty(0, device="cuda", dtype=torch.bfloat16)
    gdn.gdn_verify_step(dims, eb, eb, eb, torch.zeros(4, device="cuda"), torch.zeros(4, device="cuda"),
                        torch.zeros(d.C * 4, device="cuda"), e, e, e, e, e, e, e, None)


def test_decode_workload_1000_carried_steps():
    """Plain decode K=1, B=1, 16/32 heads of 128: 1000 successive steps with carried state."""
    w = WORKLOADS["decode"]
    d = w.dims
    g = Gen(w.seed)
    lay = make_layer(g, d, w.dists)
    st = GdnLayerState.create(d, lay)
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    worst = 0.0
    for step in range(w.rounds):
        rnd = make_round(g, d, w.dists)
        st.load_round(rnd)
        st.verify()
        ref = oracle_round(d, lay, S, H, rnd)
        S, H = ref["state_out"], ref["conv_state_out"]
        worst = max(worst, out_rel_err(st.out.cpu().numpy(), ref["out"]))
        if step % 100 == 99:
            assert state_rel_err(st.state.cpu().numpy(), S) <= STATE_TOL
            np.testing.assert_array_equal(st.conv_state.cpu().numpy(), H)
    assert worst <= OUT_TOL


def test_dflash_workload_200_rounds_rollback_resume():
    """B=1, K=16: accept U{1..16}, rollback and resume for 200 rounds."""
    w = WORKLOADS["dflash"]
    d = w.dims
    g = Gen(w.seed)
    lay = make_layer(g, d, w.dists)
    st = GdnLayerState.create(d, lay)
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    for rd in range(w.rounds):
        rnd = make_round(g, d, w.dists)
        st.load_round(rnd)
        st.verify()
        ref = oracle_round(d, lay, S, H, rnd)
        if rd % 20 == 0:
            _check_round(st, ref, d)
        else:
            assert out_rel_err(st.out.cpu().numpy(), ref["out"]) <= OUT_TOL
        st.rollback()
        S, H = O.rollback(rnd.accept_len, S, ref["states"], H, ref["conv_inter"])
        if rd % 10 == 9:
            assert state_rel_err(st.state.cpu().numpy(), S) <= STATE_TOL
            np.testing.assert_array_equal(st.conv_state.cpu().numpy(), H)


@pytest.mark.parametrize("name,rounds", [("decode", 4), ("dspark", 3), ("serve16", 2)])
def test_batched_workloads_full_outputs(name, rounds):
    """Plain decode (B=1, K=1) and B=32 (K=8 and K=16), per-sequence rollback, every output
    compared."""
    w = WORKLOADS[name]
    d = w.dims
    g = Gen(w.seed)
    lay = make_layer(g, d, w.dists)
    st = GdnLayerState.create(d, lay)
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    for _ in range(rounds):
        rnd = make_round(g, d, w.dists)
        st.load_round(rnd)
        st.verify()
        ref = oracle_round(d, lay, S, H, rnd)
        _check_round(st, ref, d)
        st.rollback()
        S, H = O.rollback(rnd.accept_len, S, ref["states"], H, ref["conv_inter"])
        assert state_rel_err(st.state.cpu().numpy(), S) <= STATE_TOL
        np.testing.assert_array_equal(st.conv_state.cpu().numpy(), H)
        del ref


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128), (128, 64), (64, 64)])
def test_decode_step_equals_first_token_of_a_window(dk, dv):
    """A one-token call runs its own kernel instantiation (the window length fixed at compile
    time); the recurrence is the same, so it gives, bit for bit, what a two-token window gives
    for its first token: the output, the state after the token and the conv history after it."""
    d2 = Dims(B=5, K=2, Hk=4, Hv=8, dk=dk, dv=dv)
    d1 = Dims(B=5, K=1, Hk=4, Hv=8, dk=dk, dv=dv)
    g = Gen(4100 + dk + dv)
    lay = make_layer(g, d2, Dists())
    rnd = make_round(g, d2, Dists())
    one = Round(x=rnd.x[:, :1].copy(), a=rnd.a[:, :1].copy(), b=rnd.b[:, :1].copy(),
                accept_len=np.ones(d1.B, np.int32))
    win = GdnLayerState.create(d2, lay)
    win.load_round(rnd)
    win.verify()
    dec = GdnLayerState.create(d1, lay)
    dec.load_round(one)
    dec.verify()
    torch.cuda.synchronize()
    assert torch.equal(dec.out[:, 0], win.out[:, 0])
    assert torch.equal(dec.states[0], win.state_inter[:, 0])
    assert torch.equal(dec.conv_states[0], win.conv_inter[:, 0])
    assert torch.equal(dec.conv_inter[:, 0], win.conv_inter[:, 0])
    ref = oracle_round(d1, lay, lay.state.astype(np.float64), lay.conv_state.astype(np.float64), one)
    _check_round(dec, ref, d1)


def test_stack48_workload_sampled_layers():
    """48 layers with distinct weights and states, B=8, K=16: every layer runs on the GPU,
    sampled layers are checked against the oracle over two rounds."""
    w = WORKLOADS["stack48"]
    d = w.dims
    g = Gen(w.seed)
    layers = [make_layer(g, d, w.dists) for _ in range(w.layers)]
    states = [GdnLayerState.create(d, lay) for lay in layers]
    sample = (0, 23, 47)
    carried = {i: (layers[i].state.astype(np.float64), layers[i].conv_state.astype(np.float64)) for i in sample}
    for _ in range(2):
        rnds = [make_round(g, d, w.dists) for _ in range(w.layers)]
        for st, rnd in zip(states, rnds):
            st.load_round(rnd)
            st.step()
        torch.cuda.synchronize()
        for i in sample:
            S, H = carried[i]
            ref = oracle_round(d, layers[i], S, H, rnds[i])
            S, H = O.rollback(rnds[i].accept_len, S, ref["states"], H, ref["conv_inter"])
            carried[i] = (S, H)
            assert state_rel_err(states[i].state.cpu().numpy(), S) <= STATE_TOL
            np.testing.assert_array_equal(states[i].conv_state.cpu().numpy(), H)
    assert gdn.gdn_device_status(clear=False) == 0


def test_large_batch_sampled_sequences():
    """B=128 at the K=16 serving shape (a 128-row grid, 4 GB of intermediates):
    sampled sequences against the oracle run on those sequences alone."""
    d = Dims(B=128, K=16, Hk=16, Hv=32, dk=128, dv=128)
    dists = WORKLOADS["serve16"].dists
    g = Gen(99)
    lay = make_layer(g, d, dists)
    rnd = make_round(g, d, dists)
    st = GdnLayerState.create(d, lay)
    st.load_round(rnd)
    st.verify()
    torch.cuda.synchronize()
    for bi in (0, 77, 127):
        d1 = Dims(B=1, K=16, Hk=16, Hv=32, dk=128, dv=128)
        sl = slice(bi, bi + 1)
        from speculative_decode_verify_gdn_gb300.synth import Round
        r1 = Round(rnd.x[sl], rnd.a[sl], rnd.b[sl], rnd.accept_len[sl])
        ref = oracle_round(d1, lay, lay.state[sl], lay.conv_state[sl], r1)
        assert out_rel_err(st.out[sl].cpu().numpy(), ref["out"]) <= OUT_TOL
        assert state_rel_err(st.states[0][sl].cpu().numpy(), ref["state_out"]) <= STATE_TOL
        assert state_rel_err(st.state_inter[sl].cpu().numpy(), ref["state_inter"]) <= STATE_TOL
        np.testing.assert_array_equal(st.conv_inter[sl].cpu().numpy(), ref["conv_inter"])
    del st
    torch.cuda.empty_cache()
