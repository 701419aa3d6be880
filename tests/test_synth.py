"""The seeded generator: published splitmix64 values, bf16 rounding, distributions, determinism."""
import numpy as np
import torch

from speculative_decode_verify_gdn_gb300.synth import (Gen, WORKLOADS, bf16_bits_to_f32, f32_to_bf16_bits,
                                                        make_layer, make_round, splitmix64)


def test_splitmix64_published_sequence():
    # first outputs of splitmix64 seeded with 0 (the reference sequence of the generator's authors)
    assert [int(v) for v in splitmix64(0, 0, 3)] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_bf16_rounding_ties_to_even_matches_torch():
    vals = np.array([1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -2.5, 3.14159, 1e-30, 65504.0], np.float32)
    bits = f32_to_bf16_bits(vals)
    assert bits[0] == 0x3F80 and bits[1] == 0x3F80 and bits[2] == 0x3F82
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    rnd = np.random.default_rng(0).standard_normal(10000).astype(np.float32)
    ref = torch.from_numpy(rnd).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    np.testing.assert_array_equal(f32_to_bf16_bits(rnd), ref)
    np.testing.assert_array_equal(bf16_bits_to_f32(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).float().numpy())


def test_distributions_and_determinism():
    g = Gen(7)
    n = g.normal((200000,), 0.5)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 0.5) < 0.01
    u = g.uniform((200000,), -1, 1)
    assert u.min() >= -1 and u.max() < 1 and abs(u.mean()) < 0.01
    i = g.integers((100000,), 1, 16)
    assert i.min() == 1 and i.max() == 16
    a = Gen(3).normal((10,)); b = Gen(3).normal((10,))
    np.testing.assert_array_equal(a, b)


def test_workload_shapes():
    w = WORKLOADS["tiny"]
    g = Gen(w.seed)
    lay = make_layer(g, w.dims, w.dists)
    rnd = make_round(g, w.dims, w.dists)
    assert w.dims.C == 384
    assert lay.conv_w.shape == (384, 4) and lay.state.shape == (1, 2, 64, 64)
    assert rnd.x.shape == (1, 4, 384) and rnd.x.dtype == np.uint16
    assert np.all(lay.dt_bias == 0) and 0 <= rnd.accept_len.min() and rnd.accept_len.max() <= 4
    assert WORKLOADS["serve16"].dims.C == 8192
