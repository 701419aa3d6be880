"""Shared pieces of the GPU parity tests: tolerances, error metrics, oracle rounds.

Tolerances (the verify step's stated bar, for bf16 activations and fp32 state):
  outputs  per (b, t, v-head) vector: max|o - o_ref| / max|o_ref| <= 2e-3 (f32 outputs);
           bf16 outputs add the bf16 rounding of the result, 2^-8.
  states   per (b, v-head) matrix:   ||S - S_ref||_F / ||S_ref||_F <= 1e-4, for the final
           state, every intermediate and every rolled-back state.
  conv history and snapshots are copies of input values: bit-exact.
"""
import numpy as np

from oracle import gdn_oracle as O
from speculative_decode_verify_gdn_gb300.synth import bf16_bits_to_f32

OUT_TOL = 2e-3
OUT_TOL_BF16 = 2e-3 + 2.0 ** -8
STATE_TOL = 1e-4


def out_rel_err(out, ref) -> float:
    out = np.asarray(out, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.max(np.abs(out - ref), axis=-1)
    den = np.max(np.abs(ref), axis=-1)
    return float(np.max(num / np.maximum(den, 1e-30)))


def state_rel_err(S, ref) -> float:
    S = np.asarray(S, np.float64)
    ref = np.asarray(ref, np.float64)
    num = np.sqrt(np.sum((S - ref) ** 2, axis=(-2, -1)))
    den = np.sqrt(np.sum(ref ** 2, axis=(-2, -1)))
    return float(np.max(num / np.maximum(den, 1e-30)))


def oracle_round(d, lay, state, conv_state, rnd, q_scale=1.0, l2_eps=1e-6):
    """One oracle verify window from the given (float64) carried state and history."""
    return O.verify_step(d, bf16_bits_to_f32(rnd.x), bf16_bits_to_f32(rnd.a), bf16_bits_to_f32(rnd.b),
                         lay.A_log, lay.dt_bias, lay.conv_w, conv_state, state, q_scale=q_scale, l2_eps=l2_eps)


def bf16_tensor_to_f32(t) -> np.ndarray:
    import torch
    return t.float().cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
