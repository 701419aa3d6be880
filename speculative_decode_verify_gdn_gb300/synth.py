"""Seeded synthetic inputs for the GDN verify step.

This module holds no part of the method's arithmetic: it only draws random
numbers and rounds them to the storage types the step consumes (bf16 for
activations, f32 for parameters and states).  Both the CUDA path's tests and
the CPU oracle's tests take their inputs from here, so the two sides see the
same bytes.

Generator: splitmix64 (Steele, Lea & Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used counter-style, the i-th draw being the
mixing function applied to ``seed + (i + 1) * 0x9E3779B97F4A7C15``.
Uniform doubles take the top 53 bits; normals use the Box-Muller transform
(cosine branch, two uniforms per normal); bf16 values are the f32 values
rounded to nearest-even on the upper 16 bits.

The distributions of the named workloads follow the verify configurations
of the speculative-decoding pages (Luce-Org/lucebox #637, Avarok atlas #297):
activations N(0,1), conv taps N(0,0.5), A_log U(-1,1), states N(0, 0.05..0.1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def splitmix64(seed: int, start: int, n: int) -> np.ndarray:
    """Draws ``start .. start+n-1`` of the splitmix64 sequence seeded with ``seed``."""
    with np.errstate(over="ignore"):
        ctr = np.arange(start + 1, start + n + 1, dtype=np.uint64)
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + ctr * _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round f32 values to bf16 (nearest, ties to even); returns uint16 bit patterns."""
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to f32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Gen:
    """Sequential counter-based draws: each call consumes the next block of the stream."""

    def __init__(self, seed: int):
        self.seed = int(seed)
        self.ctr = 0

    def _bits(self, n: int) -> np.ndarray:
        z = splitmix64(self.seed, self.ctr, n)
        self.ctr += n
        return z

    def uniform(self, shape, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
        n = int(np.prod(shape))
        u = (self._bits(n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
        return (lo + (hi - lo) * u).reshape(shape)

    def normal(self, shape, std: float = 1.0) -> np.ndarray:
        n = int(np.prod(shape))
        z = self._bits(2 * n)
        u1 = 1.0 - (z[0::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
        u2 = (z[1::2] >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
        g = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
        return (std * g).reshape(shape)

    def integers(self, shape, lo: int, hi: int) -> np.ndarray:
        """Integers in [lo, hi] inclusive (modulo reduction; the bias is below 2^-50)."""
        n = int(np.prod(shape))
        span = np.uint64(hi - lo + 1)
        return (lo + (self._bits(n) % span).astype(np.int64)).astype(np.int32).reshape(shape)


@dataclass(frozen=True)
class Dims:
    """Shape of one GDN layer's verify step (names follow the pages' notation)."""
    B: int
    K: int
    Hk: int
    Hv: int
    dk: int
    dv: int
    W: int = 4

    @property
    def C(self) -> int:
        """Conv channels over the q|k|v slab."""
        return 2 * self.Hk * self.dk + self.Hv * self.dv


@dataclass(frozen=True)
class Dists:
    """Value distributions of one workload (standard deviations, not variances)."""
    x_std: float = 1.0
    w_std: float = 0.5
    a_std: float = 1.0
    b_std: float = 1.0
    dt_bias_std: float = 0.1          # 0 => dt_bias identically zero
    A_log_lo: float = -1.0
    A_log_hi: float = 1.0
    state_std: float = 0.05
    hist_std: float = 1.0
    accept_lo: int = 1                # accept lengths U{accept_lo .. K}


@dataclass
class Layer:
    """Per-layer parameters and carried state (host copies, storage types)."""
    conv_w: np.ndarray       # [C, W] f32
    A_log: np.ndarray        # [Hv] f32
    dt_bias: np.ndarray      # [Hv] f32
    conv_state: np.ndarray   # [B, W-1, C] f32
    state: np.ndarray        # [B, Hv, dv, dk] f32


@dataclass
class Round:
    """Per-round activations (one verify window) and the synthetic accept lengths."""
    x: np.ndarray            # [B, K, C] bf16 bits (uint16)
    a: np.ndarray            # [B, K, Hv] bf16 bits
    b: np.ndarray            # [B, K, Hv] bf16 bits
    accept_len: np.ndarray   # [B] int32


def make_layer(g: Gen, d: Dims, dist: Dists) -> Layer:
    conv_w = g.normal((d.C, d.W), dist.w_std).astype(np.float32)
    A_log = g.uniform((d.Hv,), dist.A_log_lo, dist.A_log_hi).astype(np.float32)
    if dist.dt_bias_std == 0.0:
        dt_bias = np.zeros((d.Hv,), np.float32)
    else:
        dt_bias = g.normal((d.Hv,), dist.dt_bias_std).astype(np.float32)
    conv_state = g.normal((d.B, d.W - 1, d.C), dist.hist_std).astype(np.float32)
    state = g.normal((d.B, d.Hv, d.dv, d.dk), dist.state_std).astype(np.float32)
    return Layer(conv_w, A_log, dt_bias, conv_state, state)


def make_tree(g: Gen, B: int, K: int, p_chain: float = 0.5) -> np.ndarray:
    """Random token trees in topological order: parent[b][t] in -1..t-1 (int32 [B, K]).

    With probability p_chain a node continues the previous node (a chain segment); otherwise
    its parent is drawn uniformly from -1..t-1 (a branch)."""
    parent = np.empty((B, K), np.int32)
    for bi in range(B):
        cont = g.uniform((K,)) < p_chain
        pick = g.uniform((K,))
        for t in range(K):
            parent[bi, t] = t - 1 if (t == 0 or cont[t]) else int(np.floor(pick[t] * (t + 1))) - 1
    return parent


def make_output_gate(g: Gen, d: Dims, z_std: float = 1.0, w_std: float = 0.1):
    """Inputs of the gated output norm: z [B, K, Hv, dv] as bf16 bits and the norm weight
    [dv] f32 drawn around 1."""
    z = f32_to_bf16_bits(g.normal((d.B, d.K, d.Hv, d.dv), z_std).astype(np.float32))
    w = (1.0 + g.normal((d.dv,), w_std)).astype(np.float32)
    return z, w


@dataclass
class Prompts:
    """Ragged prompts packed token-major (prompt i holds rows cu[i] .. cu[i+1]-1)."""
    cu: np.ndarray           # [B + 1] int32
    x: np.ndarray            # [N, C] bf16 bits
    a: np.ndarray            # [N, Hv] bf16 bits
    b: np.ndarray            # [N, Hv] bf16 bits


def make_prompts(g: Gen, d: Dims, lens, dist: Dists) -> Prompts:
    lens = np.asarray(lens, np.int64)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    N = int(cu[-1])
    x = f32_to_bf16_bits(g.normal((N, d.C), dist.x_std).astype(np.float32))
    a = f32_to_bf16_bits(g.normal((N, d.Hv), dist.a_std).astype(np.float32))
    b = f32_to_bf16_bits(g.normal((N, d.Hv), dist.b_std).astype(np.float32))
    return Prompts(cu, x, a, b)


def make_round(g: Gen, d: Dims, dist: Dists) -> Round:
    x = f32_to_bf16_bits(g.normal((d.B, d.K, d.C), dist.x_std).astype(np.float32))
    a = f32_to_bf16_bits(g.normal((d.B, d.K, d.Hv), dist.a_std).astype(np.float32))
    b = f32_to_bf16_bits(g.normal((d.B, d.K, d.Hv), dist.b_std).astype(np.float32))
    acc = g.integers((d.B,), dist.accept_lo, d.K)
    return Round(x, a, b, acc)


# Named workloads.  Seeds: the i-th configuration of the verify study uses seed i-1;
# the K=16, B=32 serving shape reuses the batched configuration's seed.
_DECODE_DISTS = Dists(dt_bias_std=0.1, state_std=0.05, accept_lo=1)
_TINY_DISTS = Dists(dt_bias_std=0.0, state_std=0.1, accept_lo=0)
_DFLASH_DISTS = Dists(dt_bias_std=0.0, state_std=0.1, accept_lo=1)


@dataclass(frozen=True)
class Workload:
    name: str
    dims: Dims
    dists: Dists
    seed: int
    rounds: int
    layers: int = 1
    description: str = field(default="", compare=False)


WORKLOADS = {
    "tiny": Workload("tiny", Dims(B=1, K=4, Hk=2, Hv=2, dk=64, dv=64), _TINY_DISTS, 0, 50,
                     description="tiny verify: B=1 K=4 Hk=Hv=2 dk=dv=64 C=384"),
    "decode": Workload("decode", Dims(B=1, K=1, Hk=16, Hv=32, dk=128, dv=128), _DECODE_DISTS, 1, 1000,
                       description="plain decode K=1: B=1 Hk=16 Hv=32 dk=dv=128 C=8192"),
    "dflash": Workload("dflash", Dims(B=1, K=16, Hk=16, Hv=32, dk=128, dv=128), _DFLASH_DISTS, 2, 200,
                       description="DFlash-width verify: B=1 K=16 Hk=16 Hv=32 dk=dv=128"),
    "dspark": Workload("dspark", Dims(B=32, K=8, Hk=16, Hv=32, dk=128, dv=128), _DECODE_DISTS, 3, 100,
                       description="batched verify: B=32 K=8 Hk=16 Hv=32 dk=dv=128"),
    "serve16": Workload("serve16", Dims(B=32, K=16, Hk=16, Hv=32, dk=128, dv=128), _DECODE_DISTS, 3, 100,
                        description="batched verify: B=32 K=16 Hk=16 Hv=32 dk=dv=128 W=4"),
    "stack48": Workload("stack48", Dims(B=8, K=16, Hk=16, Hv=32, dk=128, dv=128), _DECODE_DISTS, 4, 50,
                        layers=48, description="48-layer hybrid stack: B=8 K=16 Hk=16 Hv=32 dk=dv=128"),
}
