"""Stream order around the verify kernels.  The verify kernel is launched with programmatic
dependent launch: its CTAs may be scheduled while the kernel ahead of it on the stream still
runs, and wait for it before reading anything.  These tests let ordinary torch kernels produce
every input right before a call, and read every output right after it, with no
synchronisation in between; all results must be those of the fully synchronised call, bit for
bit."""
import numpy as np
import pytest
import torch

from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import Dims, Dists, Gen, make_layer, make_round, make_tree

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    gdn.gdn_device_status(clear=True)
    yield
    assert gdn.gdn_device_status(clear=True) == 0


def _produce(dst, src):
    """dst <- src by an elementwise kernel on the current stream (not a copy engine transfer)."""
    torch.mul(src, 1, out=dst)


@pytest.mark.parametrize("tree", [False, True])
def test_inputs_from_the_kernel_just_ahead_and_outputs_to_the_kernel_just_after(tree):
    d = Dims(B=4, K=16, Hk=4, Hv=8, dk=128, dv=128)
    g = Gen(4300 + int(tree))
    lay = make_layer(g, d, Dists())
    rnd = make_round(g, d, Dists())
    parent = torch.from_numpy(make_tree(g, d.B, d.K, 0.5).astype(np.int32)).cuda()

    def call(st, par):
        if tree:
            st.verify_tree(par)
        else:
            st.verify()

    ref = GdnLayerState.create(d, lay)
    ref.load_round(rnd)
    torch.cuda.synchronize()
    call(ref, parent)
    torch.cuda.synchronize()

    st = GdnLayerState.create(d, lay)
    st.load_round(rnd)
    # the same inputs, parked in other buffers; the call's own buffers hold garbage until the
    # kernels just ahead of the call write them
    srcs = [(st.x, st.x.clone()), (st.a, st.a.clone()), (st.b, st.b.clone()),
            (st.states[0], st.states[0].clone()), (st.conv_states[0], st.conv_states[0].clone())]
    par_src = parent.clone()
    par = torch.full_like(parent, -7)
    for dst, _ in srcs:
        dst.fill_(float("nan"))
    torch.cuda.synchronize()
    for dst, src in srcs:
        _produce(dst, src)
    _produce(par, par_src)
    call(st, par)
    # read by the kernels just after the call
    got = [t.clone() for t in (st.out, st.states[0], st.state_inter, st.conv_states[0], st.conv_inter)]
    torch.cuda.synchronize()
    want = (ref.out, ref.states[0], ref.state_inter, ref.conv_states[0], ref.conv_inter)
    for a, b in zip(got, want):
        assert torch.equal(a, b)


def test_back_to_back_calls_with_kernels_between():
    """Ten windows carried in place (verify, rollback), a torch kernel producing each window's x
    just before its call, against the same windows with a synchronisation around every call."""
    d = Dims(B=3, K=8, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(4400)
    lay = make_layer(g, d, Dists())
    rnds = [make_round(g, d, Dists()) for _ in range(10)]
    ref = GdnLayerState.create(d, lay)
    for r in rnds:
        ref.load_round(r)
        torch.cuda.synchronize()
        ref.step()
        torch.cuda.synchronize()
    st = GdnLayerState.create(d, lay)
    parked = []
    for r in rnds:
        st.load_round(r)
        parked.append((st.x.clone(), st.a.clone(), st.b.clone(), st.accept_len.clone()))
    torch.cuda.synchronize()
    for x, a, b, acc in parked:
        _produce(st.x, x)
        _produce(st.a, a)
        _produce(st.b, b)
        _produce(st.accept_len, acc)
        st.step()
    torch.cuda.synchronize()
    assert torch.equal(st.state, ref.state)
    assert torch.equal(st.conv_state, ref.conv_state)
    assert torch.equal(st.out, ref.out)


def test_graph_replay_equals_eager():
    """Four windows (verify, then the rollback copy) captured in a CUDA graph, each window's
    inputs produced by kernels inside the graph: one replay gives the eager results, bit for
    bit (all three kernels are launched with programmatic dependent launch)."""
    d = Dims(B=3, K=8, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(4500)
    lay = make_layer(g, d, Dists())
    rnds = [make_round(g, d, Dists()) for _ in range(4)]
    ref = GdnLayerState.create(d, lay)
    for r in rnds:
        ref.load_round(r)
        ref.step()
    torch.cuda.synchronize()
    st = GdnLayerState.create(d, lay)
    parked = []
    for r in rnds:
        st.load_round(r)
        parked.append((st.x.clone(), st.a.clone(), st.b.clone(), st.accept_len.clone()))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        for x, a, b, acc in parked:
            _produce(st.x, x)
            _produce(st.a, a)
            _produce(st.b, b)
            _produce(st.accept_len, acc)
            st.step()
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(st.state, ref.state)
    assert torch.equal(st.conv_state, ref.conv_state)
    assert torch.equal(st.out, ref.out)
    assert torch.equal(st.state_inter, ref.state_inter)


def test_verify_right_after_prefill():
    """A prefill writes the state and conv history in place and a verify window reads them,
    launched right after it with no synchronisation (the prefill's last kernel does not signal
    its dependents early, so the verify kernel waits for its completion): the same results, bit
    for bit, as with a synchronisation in between."""
    from speculative_decode_verify_gdn_gb300.synth import make_prompts

    d = Dims(B=3, K=12, Hk=2, Hv=4, dk=128, dv=128)
    g = Gen(4700)
    lay = make_layer(g, d, Dists())
    pr = make_prompts(g, d, [200, 77, 130], Dists())
    rnd = make_round(g, d, Dists())
    pdims = gdn.make_dims(d.B, 1, d.Hk, d.Hv, d.dk, d.dv, d.W, 1.0, 1e-6, 1)
    N = int(pr.x.shape[0])
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    cu, px, pa, pb = torch.from_numpy(pr.cu).cuda(), bf(pr.x), bf(pr.a), bf(pr.b)
    pout = torch.empty((N, d.Hv, d.dv), dtype=torch.float32, device="cuda")
    pws = gdn.alloc_prefill_workspace(pdims, N)
    results = []
    for sync in (True, False):
        st = GdnLayerState.create(d, lay)
        st.load_round(rnd)
        torch.cuda.synchronize()
        gdn.gdn_prefill(pdims, cu, px, pa, pb, st.A_log, st.dt_bias, st.conv_w, st.conv_states[0], st.conv_states[0],
                        st.states[0], st.states[0], pout, pws)
        if sync:
            torch.cuda.synchronize()
        st.verify()
        torch.cuda.synchronize()
        results.append([t.clone() for t in (st.out, st.states[0], st.state_inter, st.conv_states[0], st.conv_inter)])
    for a, b in zip(*results):
        assert torch.equal(a, b)
