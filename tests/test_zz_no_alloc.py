"""The allocation-free verify entry point against the regular one.

gdn_verify_step_static_scratch serves callers that may not allocate device memory where they run
the verify step; it passes a fixed array inside the library as the workspace (the verify kernels
need none).  This file runs last
(pytest collects it after the others) so that a failure here comes after every other test has run,
and it also passes on its own in a fresh process.
"""
import pytest
import torch

from speculative_decode_verify_gdn_gb300 import gdn
from speculative_decode_verify_gdn_gb300.build import build_library
from speculative_decode_verify_gdn_gb300.runtime import GdnLayerState
from speculative_decode_verify_gdn_gb300.synth import WORKLOADS, Dims, Dists, Gen, make_layer, make_round

pytestmark = pytest.mark.gpu


def _run_pair(d, dists, seed):
    """Two windows in a row through each entry point, each side carrying its own state in place."""
    g = Gen(seed)
    lay = make_layer(g, d, dists)
    rnds = [make_round(g, d, dists) for _ in range(2)]
    ref = GdnLayerState.create(d, lay)
    nal = GdnLayerState.create(d, lay)
    for rnd in rnds:
        ref.load_round(rnd)
        ref.verify()
        nal.load_round(rnd)
        gdn.gdn_verify_step_static_scratch(nal.dims, nal.x, nal.a, nal.b, nal.A_log, nal.dt_bias, nal.conv_w,
                                           nal.conv_states[0], nal.conv_states[0], nal.conv_inter, nal.states[0],
                                           nal.states[0], nal.state_inter, nal.out)
        torch.cuda.synchronize()
        # the same kernels on the same inputs: identical results, bit for bit
        assert torch.equal(nal.out, ref.out)
        assert torch.equal(nal.state, ref.state)
        if d.K > 1:
            assert torch.equal(nal.state_inter, ref.state_inter)
        assert torch.equal(nal.conv_inter, ref.conv_inter)
        assert torch.equal(nal.conv_state, ref.conv_state)


def test_static_scratch_matches_workspace_entry_point():
    assert torch.cuda.is_available(), "GPU tests need CUDA"
    build_library()
    gdn.load_library()
    _run_pair(Dims(B=3, K=7, Hk=2, Hv=4, dk=128, dv=128), Dists(), 501)
    w = WORKLOADS["serve16"]
    _run_pair(w.dims, w.dists, 502)
    assert gdn.gdn_device_status(clear=True) == 0


def test_static_scratch_covers_every_shape():
    """The verify kernels need no scratch, so no shape is too large for the fixed array."""
    for dims in (gdn.make_dims(B=65535, K=16, Hk=64, Hv=128, dk=128, dv=128), gdn.make_dims(B=1, K=1, Hk=1, Hv=1,
                                                                                           dk=64, dv=64)):
        assert gdn.gdn_verify_workspace_size(dims) == 0
