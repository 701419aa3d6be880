"""gdn_prefill (whole prompts, packed token-major, chunks of 64 in the WY form) against the
oracle's per-token prefill, and against the verify step over the same tokens.

Tolerances are those of the verify step: outputs per (token, v-head) vector max abs error /
max abs reference <= 2e-3 (f32 outputs; bf16 adds 2^-8), states per (prompt, v-head)
Frobenius relative error <= 1e-4, conv histories bit-exact (they are copies of inputs).
"""
import numpy as np
import pytest
import torch

from oracle import gdn_oracle as O
from parity_util import OUT_TOL, OUT_TOL_BF16, STATE_TOL, out_rel_err, state_rel_err
from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import (WORKLOADS, Dims, Dists, Gen, Layer, Prompts, Round,
                                                        bf16_bits_to_f32, make_layer, make_prompts)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    gdn.gdn_device_status(clear=True)
    yield
    assert gdn.gdn_device_status(clear=True) == 0


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def _f32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _problem(seed, lens, Hk=2, Hv=4, dk=128, dv=128, dists=Dists()):
    d = Dims(B=len(lens), K=1, Hk=Hk, Hv=Hv, dk=dk, dv=dv)
    g = Gen(seed)
    lay = make_layer(g, d, dists)
    pr = make_prompts(g, d, lens, dists)
    return d, lay, pr


def _run(d, lay, pr, out_f32=True, q_scale=1.0, in_place=False, state=None, conv=None):
    dims = gdn.make_dims(d.B, 1, d.Hk, d.Hv, d.dk, d.dv, d.W, q_scale, 1e-6, int(out_f32))
    N = int(pr.x.shape[0])
    st_in = _f32(lay.state if state is None else state)
    cs_in = _f32(lay.conv_state if conv is None else conv)
    st_out = st_in if in_place else torch.full_like(st_in, 7.0)
    cs_out = cs_in if in_place else torch.full_like(cs_in, 7.0)
    out = torch.empty((N, d.Hv, d.dv), dtype=torch.float32 if out_f32 else torch.bfloat16, device="cuda")
    ws = gdn.alloc_prefill_workspace(dims, N)
    gdn.gdn_prefill(dims, torch.from_numpy(pr.cu).cuda(), _bf16(pr.x), _bf16(pr.a), _bf16(pr.b), _f32(lay.A_log),
                    _f32(lay.dt_bias), _f32(lay.conv_w), cs_in, cs_out, st_in, st_out, out, ws)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), st_out.cpu().numpy(), cs_out.cpu().numpy()


def _oracle(d, lay, pr, q_scale=1.0, state=None, conv=None):
    return O.prefill(d, pr.cu, bf16_bits_to_f32(pr.x), bf16_bits_to_f32(pr.a), bf16_bits_to_f32(pr.b), lay.A_log,
                     lay.dt_bias, lay.conv_w, lay.conv_state if conv is None else conv,
                     lay.state if state is None else state, q_scale=q_scale)


def _check(res, ref, out_tol=OUT_TOL):
    out, st, cs = res
    if out.size:
        assert out_rel_err(out, ref["out"]) <= out_tol
    assert state_rel_err(st, ref["state_out"]) <= STATE_TOL
    np.testing.assert_array_equal(cs, ref["conv_state_out"])


@pytest.mark.parametrize("lens,dk,dv,out_f32", [([200, 64, 1, 0, 130], 128, 128, True),
                                                ([5, 70, 2], 64, 64, True),
                                                ([129, 63], 128, 64, False),
                                                ([65, 3, 128], 64, 128, True)])
def test_ragged_prompts_against_oracle(lens, dk, dv, out_f32):
    d, lay, pr = _problem(1100 + sum(lens) + dk + dv, lens, dk=dk, dv=dv)
    res = _run(d, lay, pr, out_f32=out_f32, q_scale=0.8)
    _check(res, _oracle(d, lay, pr, q_scale=0.8), OUT_TOL if out_f32 else OUT_TOL_BF16)


def test_many_vheads_per_qk_head_and_long_prompt():
    d, lay, pr = _problem(1201, [700, 45], Hk=1, Hv=3)
    _check(_run(d, lay, pr), _oracle(d, lay, pr))


def test_in_place_equals_out_of_place_bitwise():
    d, lay, pr = _problem(1202, [150, 0, 77])
    a = _run(d, lay, pr)
    b = _run(d, lay, pr, in_place=True)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_all_prompts_empty_passes_state_through():
    d, lay, pr = _problem(1203, [0, 0, 0])
    out, st, cs = _run(d, lay, pr)
    np.testing.assert_array_equal(st, lay.state)
    np.testing.assert_array_equal(cs, lay.conv_state)


def test_split_prompt_equals_one_prefill():
    """Two calls over the halves of a prompt, the second from the first's state and history,
    against the oracle over the whole prompt."""
    d, lay, pr = _problem(1204, [300])
    ref = _oracle(d, lay, pr)
    cut = 130
    from speculative_decode_verify_gdn_gb300.synth import Prompts
    p1 = Prompts(np.array([0, cut], np.int32), pr.x[:cut], pr.a[:cut], pr.b[:cut])
    p2 = Prompts(np.array([0, 300 - cut], np.int32), pr.x[cut:], pr.a[cut:], pr.b[cut:])
    o1, s1, c1 = _run(d, lay, p1)
    o2, s2, c2 = _run(d, lay, p2, state=s1, conv=c1)
    _check((np.concatenate([o1, o2]), s2, c2), ref)


def test_prefill_matches_verify_windows():
    """The prefill of a 48-token prompt and three 16-token verify windows over the same tokens
    (carried state) agree within the tolerances."""
    d, lay, pr = _problem(1205, [48], Hk=2, Hv=4)
    out_p, st_p, cs_p = _run(d, lay, pr)
    dv = Dims(B=1, K=16, Hk=d.Hk, Hv=d.Hv, dk=d.dk, dv=d.dv)
    st = GdnLayerState.create(dv, lay)
    outs = []
    for w in range(3):
        rows = slice(16 * w, 16 * w + 16)
        st.load_round(Round(pr.x[None, rows], pr.a[None, rows], pr.b[None, rows], np.array([16], np.int32)))
        st.verify()
        torch.cuda.synchronize()
        outs.append(st.out.cpu().numpy()[0])
    out_v = np.concatenate(outs)
    assert out_rel_err(out_p, out_v) <= 2 * OUT_TOL
    assert state_rel_err(st_p, st.state.cpu().numpy()) <= 2 * STATE_TOL
    np.testing.assert_array_equal(cs_p, st.conv_state.cpu().numpy())


@pytest.mark.parametrize("cu,N", [([0, 5, 3, 8], 8), ([0, 4, 6], 8), ([1, 4, 8], 8)])
def test_bad_seqlens_set_the_flag_and_write_nothing(cu, N):
    B = len(cu) - 1
    lens = [2] * B
    d, lay, pr = _problem(1206, lens)
    g = Gen(1207)
    from speculative_decode_verify_gdn_gb300.synth import Prompts, f32_to_bf16_bits
    x = f32_to_bf16_bits(g.normal((N, d.C)).astype(np.float32))
    a = f32_to_bf16_bits(g.normal((N, d.Hv)).astype(np.float32))
    bad = Prompts(np.array(cu, np.int32), x, a, a)
    gdn.gdn_device_status(clear=True)
    out, st, cs = _run(d, lay, bad)
    assert gdn.gdn_device_status(clear=True) == gdn.DEVERR_SEQLENS
    assert np.all(st == 7.0) and np.all(cs == 7.0)


def test_serving_shape_prompts_against_oracle():
    """Hk=16, Hv=32, dk=dv=128 (the serving layer): ragged prompts, bf16 outputs."""
    dims = WORKLOADS["serve16"].dims
    d, lay, pr = _problem(1208, [1000, 333, 64, 0], Hk=dims.Hk, Hv=dims.Hv, dk=dims.dk, dv=dims.dv,
                          dists=WORKLOADS["serve16"].dists)
    _check(_run(d, lay, pr, out_f32=False), _oracle(d, lay, pr), OUT_TOL_BF16)


def test_many_short_prompts():
    """1500 prompts of 0..5 tokens: the offset check and chunk numbering take several prompts per
    thread, most prompts are shorter than the conv history, and many are empty."""
    g0 = Gen(1209)
    lens = [int(v) for v in g0.integers((1500,), 0, 5)]
    d, lay, pr = _problem(1210, lens, Hk=1, Hv=2, dk=64, dv=64)
    _check(_run(d, lay, pr), _oracle(d, lay, pr))


def _head_group(d, lay, pr, i, kh):
    """q/k head kh of prompt i as a problem of its own (Hk = 1 and the kh-th group of r v-heads):
    the channels, taps, gates, history and state that those outputs depend on, nothing else."""
    r = d.Hv // d.Hk
    heads = np.arange(kh * r, kh * r + r)
    ch = np.concatenate([kh * d.dk + np.arange(d.dk), d.Hk * d.dk + kh * d.dk + np.arange(d.dk),
                         2 * d.Hk * d.dk + (heads[:, None] * d.dv + np.arange(d.dv)).ravel()])
    s, e = int(pr.cu[i]), int(pr.cu[i + 1])
    d1 = Dims(B=1, K=1, Hk=1, Hv=r, dk=d.dk, dv=d.dv)
    lay1 = Layer(conv_w=lay.conv_w[ch], A_log=lay.A_log[heads], dt_bias=lay.dt_bias[heads],
                 conv_state=lay.conv_state[i:i + 1][:, :, ch], state=lay.state[i:i + 1, heads])
    pr1 = Prompts(np.array([0, e - s], np.int32), pr.x[s:e][:, ch], pr.a[s:e][:, heads], pr.b[s:e][:, heads])
    return d1, lay1, pr1, heads, ch, slice(s, e)


def test_8192_token_prompt_at_the_serving_shape_sampled_heads():
    """A prompt of 8192 tokens (128 chunks, the benchmark's prompt length) and a short one at
    Hk=16, Hv=32, dk=dv=128, every head on the GPU; sampled q/k head groups against the oracle
    run on those heads alone: every output token of the group, its final state after 128
    chunks and its conv history."""
    w = WORKLOADS["serve16"]
    d, lay, pr = _problem(1212, [8192, 100], Hk=w.dims.Hk, Hv=w.dims.Hv, dk=w.dims.dk, dv=w.dims.dv,
                          dists=w.dists)
    out, st, cs = _run(d, lay, pr, out_f32=True)
    for i, kh in [(0, 0), (0, 9), (0, 15), (1, 4)]:
        d1, lay1, pr1, heads, ch, rows = _head_group(d, lay, pr, i, kh)
        ref = _oracle(d1, lay1, pr1)
        assert out_rel_err(out[rows][:, heads], ref["out"]) <= OUT_TOL
        assert state_rel_err(st[i, heads], ref["state_out"][0]) <= STATE_TOL
        np.testing.assert_array_equal(cs[i][:, ch], ref["conv_state_out"][0])
