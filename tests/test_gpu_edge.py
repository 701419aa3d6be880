"""The CUDA path through the method's degenerate and extreme cases, against the oracle.

The seeded workloads (a, b ~ N(0,1), A_log ~ U(-1,1)) almost never reach the corners of the
gate formula or of the L2 norm, so these tests build inputs that do, per v-head:

  head 0  b = -inf and A_log = -inf: beta = 0 and g = 1, so the state must come through the
          window unchanged (bit for bit: every update term is an exact zero) and o_t = S0 q^_t;
  head 1  A_log = +inf: g = 0 (full forget), S_t = beta_t v_t k^_t^T;
  head 2  a + dt_bias around the softplus clip at 20 and far above it (90, 150, 250, where
          e^z no longer fits in f32, so a missing clip would give g = 0), with a mild decay;
  head 3  A_log = 2 with a near +4 (log g ~ -30 per token: the decay products underflow f32
          within a few tokens) or spread wide (strong and weak decays mixed);

and, on top, q/k slabs that are zero over their whole conv window (x and history), where only
eps keeps the norm finite: a zero q^ must give o = 0, a zero k^ a pure decay of the state.
(Raw gates: lucebox #637, review of ggml-cuda/gated_delta_net.cu, raw-gate mode with the
softplus clipped at 20; one L2 norm over the q|k slab and the head broadcast: lucebox #637,
commit list.)  Tolerances are those of every other parity test.
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from parity_util import OUT_TOL, STATE_TOL, oracle_round, out_rel_err, state_rel_err
from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import (Dims, Dists, Gen, bf16_bits_to_f32, f32_to_bf16_bits,
                                                        make_layer, make_output_gate, make_prompts, make_round,
                                                        make_tree)

pytestmark = pytest.mark.gpu

NEG_INF_BF16 = np.uint16(0xFF80)
CLIP_PATTERN = [19.5, 20.5, 90.0, 150.0, 18.0, 21.0, 250.0, 20.0]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    gdn.gdn_device_status(clear=True)
    yield
    assert gdn.gdn_device_status(clear=True) == 0


def _bf16(values) -> np.ndarray:
    return f32_to_bf16_bits(np.asarray(values, np.float32))


def _extreme_params(lay, g: Gen):
    """Gate parameters of heads 0..3 as in the module docstring (per-token inputs set apart)."""
    lay.A_log[0] = -np.inf
    lay.A_log[1] = np.inf
    lay.A_log[2], lay.dt_bias[2] = -6.0, 0.0
    lay.A_log[3], lay.dt_bias[3] = 2.0, 0.0


def _extreme_gate_inputs(a, b, g: Gen, lead_shape):
    """a, b [..., Hv] bf16 bits: b = -inf on head 0, the clip pattern on head 2, a near +4 (first
    sequence / prompt) or wide (the rest) on head 3."""
    b[..., 0] = NEG_INF_BF16
    a[..., 2] = _bf16(np.resize(CLIP_PATTERN, lead_shape))
    wide = g.normal(lead_shape, 4.0)
    wide[0] = 4.0 + 0.05 * wide[0]
    a[..., 3] = _bf16(wide)


def _zero_slab(x, hist, d, kh, which, rows=slice(None)):
    """Zero the q (which=0) or k (which=1) channels of q/k head kh in x [.., T, C] over `rows`
    and, when given, in the history [W-1, C]."""
    c0 = which * d.Hk * d.dk + kh * d.dk
    x[..., rows, c0:c0 + d.dk] = 0
    if hist is not None:
        hist[..., c0:c0 + d.dk] = 0.0


def _verify_problem(dk=128, dv=128, seed=3100):
    d = Dims(B=2, K=16, Hk=2, Hv=4, dk=dk, dv=dv)
    g = Gen(seed)
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    _extreme_params(lay, g)
    _extreme_gate_inputs(rnd.a, rnd.b, g, (d.B, d.K))
    _zero_slab(rnd.x[1], lay.conv_state[1], d, kh=0, which=0)   # sequence 1: q of q/k head 0 is zero
    _zero_slab(rnd.x[0], lay.conv_state[0], d, kh=1, which=1)   # sequence 0: k of q/k head 1 is zero
    return d, lay, rnd, g


def _check_head0_unchanged(S0, fin, inter):
    """beta = 0, g = 1: the state after every token is the state before the window, exactly."""
    s0 = torch.from_numpy(np.ascontiguousarray(S0[:, 0])).cuda()
    assert torch.equal(fin[:, 0], s0)
    for t in range(inter.shape[1]):
        assert torch.equal(inter[:, t, 0], s0)


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 64)])
def test_verify_step_gate_and_norm_extremes(dk, dv):
    d, lay, rnd, _ = _verify_problem(dk, dv)
    st = GdnLayerState.create(d, lay)
    st.load_round(rnd)
    st.verify()
    torch.cuda.synchronize()
    ref = oracle_round(d, lay, lay.state, lay.conv_state, rnd)
    assert np.all(np.isfinite(ref["out"])) and np.all(np.isfinite(ref["states"]))
    out = st.out.cpu().numpy()
    assert np.all(np.isfinite(out))
    assert out_rel_err(out, ref["out"]) <= OUT_TOL
    assert state_rel_err(st.state.cpu().numpy(), ref["state_out"]) <= STATE_TOL
    assert state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"]) <= STATE_TOL
    np.testing.assert_array_equal(st.conv_inter.cpu().numpy(), ref["conv_inter"])
    np.testing.assert_array_equal(st.conv_state.cpu().numpy(), ref["conv_state_out"])
    _check_head0_unchanged(lay.state, st.state, st.state_inter)
    # the cases reached what they were built for
    assert np.array_equal(out[1, :, 0:2], np.zeros_like(out[1, :, 0:2]))          # zero q^: o = 0
    g_ref = O.raw_gates(bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b), lay.A_log, lay.dt_bias)[1]
    assert np.all(g_ref[..., 1] == 0.0) and np.all(g_ref[..., 0] == 1.0)
    assert np.all(g_ref[..., 2] > 0.5)                                               # the clip held
    assert np.prod(g_ref[0, :4, 3]) < 1e-45                                          # below f32's range
    # o_t = S0 q^_t on head 0 (a plain matrix-vector product of the oracle's normalised q)
    q = O.split_qkv(ref["y"], d.Hk, d.Hv, d.dk, d.dv)[0]
    qn = O.l2_normalize(q, 1e-6)
    o_mv = np.einsum("bij,btj->bti", lay.state[:, 0].astype(np.float64), qn[:, :, 0])
    assert out_rel_err(out[:, :, 0], o_mv) <= OUT_TOL


def test_tree_verify_gate_and_norm_extremes():
    d, lay, rnd, g = _verify_problem(seed=3200)
    parent = make_tree(g, d.B, d.K, 0.5)
    st = GdnLayerState.create(d, lay)
    st.load_round(rnd)
    st.verify_tree(torch.from_numpy(parent).cuda())
    torch.cuda.synchronize()
    ref = O.tree_verify_step(d, parent, bf16_bits_to_f32(rnd.x), bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b),
                             lay.A_log, lay.dt_bias, lay.conv_w, lay.conv_state, lay.state)
    assert out_rel_err(st.out.cpu().numpy(), ref["out"]) <= OUT_TOL
    assert state_rel_err(st.state.cpu().numpy(), ref["state_out"]) <= STATE_TOL
    assert state_rel_err(st.state_inter.cpu().numpy(), ref["state_inter"]) <= STATE_TOL
    np.testing.assert_array_equal(st.conv_inter.cpu().numpy(), ref["conv_inter"])
    _check_head0_unchanged(lay.state, st.state, st.state_inter)


def test_gated_verify_gate_and_norm_extremes():
    d, lay, rnd, g = _verify_problem(seed=3300)
    z, w = make_output_gate(g, d)
    st = GdnLayerState.create(d, lay)
    st.load_round(rnd)
    st.verify_gated(torch.from_numpy(z.view(np.int16)).cuda().view(torch.bfloat16), torch.from_numpy(w).cuda(), 1e-6)
    torch.cuda.synchronize()
    ref = oracle_round(d, lay, lay.state, lay.conv_state, rnd)
    y_ref = O.gated_rms_norm(ref["out"], bf16_bits_to_f32(z), w, 1e-6)
    y = st.out.cpu().numpy()
    assert out_rel_err(y, y_ref) <= OUT_TOL
    assert np.array_equal(y[1, :, 0:2], np.zeros_like(y[1, :, 0:2]))
    assert state_rel_err(st.state.cpu().numpy(), ref["state_out"]) <= STATE_TOL
    _check_head0_unchanged(lay.state, st.state, st.state_inter)


def _prefill_run(d, lay, pr):
    dims = gdn.make_dims(d.B, 1, d.Hk, d.Hv, d.dk, d.dv, d.W, 1.0, 1e-6, 1)
    N = int(pr.x.shape[0])

    def bf(bits):
        return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)

    def f32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()

    S, CS = f32(lay.state), f32(lay.conv_state)
    out = torch.empty((N, d.Hv, d.dv), dtype=torch.float32, device="cuda")
    gdn.gdn_prefill(dims, torch.from_numpy(pr.cu).cuda(), bf(pr.x), bf(pr.a), bf(pr.b), f32(lay.A_log),
                    f32(lay.dt_bias), f32(lay.conv_w), CS, CS, S, S, out, gdn.alloc_prefill_workspace(dims, N))
    torch.cuda.synchronize()
    return out.cpu().numpy(), S, CS.cpu().numpy()


@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 128)])
def test_prefill_gate_and_norm_extremes(dk, dv):
    """The same extremes through gdn_prefill, over 64-token chunks with ragged tails: the chunk
    kernel's decay products, its triangular inverse and the tensor-core state pass."""
    d = Dims(B=3, K=1, Hk=2, Hv=4, dk=dk, dv=dv)
    g = Gen(3400 + dk + dv)
    lay = make_layer(g, d, Dists())
    lens = [200, 77, 130]
    pr = make_prompts(g, d, lens, Dists())
    _extreme_params(lay, g)
    _extreme_gate_inputs(pr.a, pr.b, g, (pr.a.shape[0],))
    a3 = bf16_bits_to_f32(pr.a[:, 3]).copy()
    a3[:lens[0]] = 4.0                                             # prompt 0: log g ~ -30 per token
    pr.a[:, 3] = _bf16(a3)
    _zero_slab(pr.x, None, d, kh=0, which=0, rows=slice(70, 141))  # prompt 0: q of head 0 zero in 2 chunks
    _zero_slab(pr.x[lens[0]:lens[0] + lens[1]], lay.conv_state[1], d, kh=1, which=1)  # prompt 1: k of head 1 zero
    out, S, cs = _prefill_run(d, lay, pr)
    ref = O.prefill(d, pr.cu, bf16_bits_to_f32(pr.x), bf16_bits_to_f32(pr.a), bf16_bits_to_f32(pr.b), lay.A_log,
                    lay.dt_bias, lay.conv_w, lay.conv_state, lay.state)
    assert np.all(np.isfinite(out))
    assert out_rel_err(out, ref["out"]) <= OUT_TOL
    assert state_rel_err(S.cpu().numpy(), ref["state_out"]) <= STATE_TOL
    np.testing.assert_array_equal(cs, ref["conv_state_out"])
    assert torch.equal(S[:, 0], torch.from_numpy(lay.state[:, 0]).cuda())    # beta = 0, g = 1: unchanged
    assert np.array_equal(out[73:141, 0:2], np.zeros_like(out[73:141, 0:2]))  # q^ = 0 once the window is zero


def test_prefill_single_token_and_exact_chunk_prompts_with_extremes():
    """Prompts of 1, 64 and 128 tokens (a chunk with one token, whole chunks only) with the gate
    extremes: padding rows of a ragged chunk must stay exact zeros next to g = 0 and beta = 0."""
    d = Dims(B=3, K=1, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(3500)
    lay = make_layer(g, d, Dists())
    pr = make_prompts(g, d, [1, 64, 128], Dists())
    _extreme_params(lay, g)
    _extreme_gate_inputs(pr.a, pr.b, g, (pr.a.shape[0],))
    out, S, cs = _prefill_run(d, lay, pr)
    ref = O.prefill(d, pr.cu, bf16_bits_to_f32(pr.x), bf16_bits_to_f32(pr.a), bf16_bits_to_f32(pr.b), lay.A_log,
                    lay.dt_bias, lay.conv_w, lay.conv_state, lay.state)
    assert out_rel_err(out, ref["out"]) <= OUT_TOL
    assert state_rel_err(S.cpu().numpy(), ref["state_out"]) <= STATE_TOL
    np.testing.assert_array_equal(cs, ref["conv_state_out"])


def test_verify_extremes_carried_over_rounds_with_rollback():
    """Ten verify + rollback rounds with the extremes in every window: errors do not build up
    in the carried state, and head 0 never moves."""
    d, lay, _, g = _verify_problem(seed=3600)
    st = GdnLayerState.create(d, lay)
    S, H = lay.state.astype(np.float64), lay.conv_state.astype(np.float64)
    for _ in range(10):
        rnd = make_round(g, d, Dists())
        _extreme_gate_inputs(rnd.a, rnd.b, g, (d.B, d.K))
        st.load_round(rnd)
        st.step()
        ref = oracle_round(d, lay, S, H, rnd)
        S, H = O.rollback(rnd.accept_len, S, ref["states"], H, ref["conv_inter"])
        assert out_rel_err(st.out.cpu().numpy(), ref["out"]) <= OUT_TOL
    torch.cuda.synchronize()
    assert state_rel_err(st.state.cpu().numpy(), S) <= STATE_TOL
    np.testing.assert_array_equal(st.conv_state.cpu().numpy(), H)
    assert torch.equal(st.state[:, 0], torch.from_numpy(lay.state[:, 0]).cuda())
