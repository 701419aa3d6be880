"""CPU oracle for the verify step of one Gated DeltaNet (GDN) layer.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import, call or
execute this module: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline / reference arm of ``bench.py`` use it.  It shares no code with the
CUDA path.

It is the plain definition of the step, computed in float64 one token at a
time, in the order the pages give it:

  a1  causal conv1d update over the q|k|v channels with its history window and
      SiLU, writing the history back and keeping one history snapshot per
      window token  (lucebox #637 "NVLink fix for PR625", commit list:
      ``ggml_ssm_conv_step`` "history window + silu(conv) + in-place history
      write-back + optional rollback window copy"; atlas #297, commit "SSM/GDN
      layer-level pieces of the K=gamma verify path":
      ``causal_conv1d_update_prefill_inter`` "writes per-token conv_state
      intermediates for partial-accept rollback")
  a2  one L2 norm over the q|k slab (lucebox #637, commit list: "single
      l2_norm over the q|k slab")
  a3  raw gates beta = sigmoid(b), g = exp(softplus(a + dt_bias) * A) with the
      softplus clipped to the identity above 20, A = -exp(A_log) (lucebox #637,
      review of ggml-cuda/gated_delta_net.cu at line 404, "raw-gate mode")
  a4  gated delta rule per v-head, q/k heads broadcast to the v heads
      (lucebox #637, commit list: "no q/k head repeat (the kernel
      broadcasts)"), keeping the state after every window token (atlas #297:
      ``gated_delta_rule_wy16.cu`` "writing final h_state and Hi_0..Hi_14
      intermediates in one pass")
  a5  rollback to the accepted length (strix-llama.cpp #14 "WIP: DSv4 +
      Qwen3.8 Flash runtime fixes", commits on recurrent snapshot planes and on
      restoring full checkpoints)

the same step over a token tree (DDTree-style window: each node continues its
parent's state and conv history; lucebox #637, ``ggml_ssm_conv_tree``), and the
prefill of whole prompts through the same recurrence (atlas #258 and #297 name the
prefill GDN paths, VARLEN-FLA / FlashInfer-GDN: ragged prompts packed token-major).

Readings taken where the pages are silent (each is also listed in the design
notes): taps are a cross-correlation with w[c, W-1] on the current token; no
conv bias; the L2 norm is x / sqrt(sum x^2 + eps); v-head h reads q/k head
h // (Hv / Hk); o_t = q_scale * S_t q_t; the state is stored [B, Hv, dv, dk]
(row = v index); conv snapshot t is the W-1 newest window rows after token t.

Every function here is pinned by ``tests/test_oracle_pins.py`` against
closed forms, invariants, special cases and brute force, not against itself.
"""
from __future__ import annotations

import numpy as np

SOFTPLUS_THRESHOLD = 20.0   # lucebox #637, review of gated_delta_net.cu:404: "(a > 20.0f) ? a : logf(1 + expf(a))"


def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z * sigmoid(z)."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def conv_step(x: np.ndarray, conv_w: np.ndarray, hist: np.ndarray):
    """a1: causal conv1d update over a window of K tokens.

    x      [B, K, C]   new inputs (values of the bf16 activations)
    conv_w [C, W]      taps; w[c, W-1] multiplies the newest row
    hist   [B, W-1, C] history, oldest row first

    Returns (y [B,K,C], conv_inter [B,K,W-1,C], hist_out [B,W-1,C]) where
    y_t[c] = SiLU(sum_j w[c,j] * win[t+j][c]) over win = [hist; x],
    conv_inter[:, t] = the W-1 newest rows of win after token t, and
    hist_out = conv_inter[:, K-1].
    """
    x = np.asarray(x, np.float64)
    w = np.asarray(conv_w, np.float64)
    hist = np.asarray(hist, np.float64)
    B, K, C = x.shape
    W = w.shape[1]
    win = np.concatenate([hist, x], axis=1)          # [B, W-1+K, C]
    y = np.empty((B, K, C))
    for t in range(K):
        acc = np.zeros((B, C))
        for j in range(W):
            acc += w[:, j] * win[:, t + j, :]
        y[:, t, :] = silu(acc)
    conv_inter = np.stack([win[:, t + 1:t + W, :] for t in range(K)], axis=1)
    hist_out = win[:, K:K + W - 1, :].copy()
    return y, conv_inter, hist_out


def split_qkv(y: np.ndarray, Hk: int, Hv: int, dk: int, dv: int):
    """Channel order of the conv slab: q | k | v, each head contiguous."""
    B, K, _ = y.shape
    q = y[..., :Hk * dk].reshape(B, K, Hk, dk)
    k = y[..., Hk * dk:2 * Hk * dk].reshape(B, K, Hk, dk)
    v = y[..., 2 * Hk * dk:2 * Hk * dk + Hv * dv].reshape(B, K, Hv, dv)
    return q, k, v


def l2_normalize(z: np.ndarray, eps: float) -> np.ndarray:
    """a2: z / sqrt(sum z^2 + eps) over the last axis."""
    return z / np.sqrt(np.sum(z * z, axis=-1, keepdims=True) + eps)


def softplus_clipped(z: np.ndarray) -> np.ndarray:
    """softplus(z) = log(1 + e^z), replaced by z itself above the threshold 20."""
    z = np.asarray(z, np.float64)
    with np.errstate(over="ignore"):
        return np.where(z > SOFTPLUS_THRESHOLD, z, np.log1p(np.exp(np.minimum(z, SOFTPLUS_THRESHOLD))))


def raw_gates(a: np.ndarray, b: np.ndarray, A_log: np.ndarray, dt_bias: np.ndarray):
    """a3: beta = sigmoid(b); g = exp(softplus(a + dt_bias) * A), A = -exp(A_log).

    a, b [B, K, Hv]; A_log, dt_bias [Hv].  Returns (beta, g), both [B, K, Hv].
    """
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    with np.errstate(over="ignore"):
        A = -np.exp(np.asarray(A_log, np.float64))
        sp = softplus_clipped(a + np.asarray(dt_bias, np.float64))
        g = np.exp(sp * A)
        beta = 1.0 / (1.0 + np.exp(-b))
    return beta, g


def delta_rule(qn, kn, v, beta, g, S0, q_scale: float = 1.0):
    """a4: the gated delta rule, one token after another.

    qn, kn [B, K, Hk, dk]  normalised queries / keys
    v      [B, K, Hv, dv]
    beta, g [B, K, Hv]
    S0     [B, Hv, dv, dk] state before the window (row = v index)

    For every v-head h (reading q/k head h // (Hv/Hk)) and token t:
        p   = S k_t
        S  <- g_t S + beta_t (v_t - g_t p) k_t^T
        o_t = q_scale * S q_t
    Returns (o [B,K,Hv,dv], states [B,K,Hv,dv,dk]) with states[:, t] the state
    after token t.
    """
    qn = np.asarray(qn, np.float64)
    kn = np.asarray(kn, np.float64)
    v = np.asarray(v, np.float64)
    B, K, Hk, dk = kn.shape
    Hv, dv = v.shape[2], v.shape[3]
    r = Hv // Hk
    kh = np.arange(Hv) // r                          # grouped broadcast of q/k heads
    S = np.array(S0, dtype=np.float64, copy=True)
    o = np.empty((B, K, Hv, dv))
    states = np.empty((B, K, Hv, dv, dk))
    for t in range(K):
        k_t = kn[:, t, kh, :]                        # [B, Hv, dk]
        q_t = qn[:, t, kh, :]
        g_t = g[:, t, :, None, None]
        b_t = beta[:, t, :, None]
        p = np.einsum("bhij,bhj->bhi", S, k_t)       # S k_t
        delta = b_t * (v[:, t] - g[:, t, :, None] * p)
        S = g_t * S + delta[..., :, None] * k_t[..., None, :]
        o[:, t] = q_scale * np.einsum("bhij,bhj->bhi", S, q_t)
        states[:, t] = S
    return o, states


def verify_step(dims, x, a, b, A_log, dt_bias, conv_w, conv_state, state,
                q_scale: float = 1.0, l2_eps: float = 1e-6):
    """a1..a4 over one window of K tokens for B sequences.

    dims: object with Hk, Hv, dk, dv.  Activations are the (bf16) values as
    floats; conv_state is [B, W-1, C]; state is [B, Hv, dv, dk].
    Returns a dict with
      out            [B, K, Hv, dv]
      states         [B, K, Hv, dv, dk]   state after each token
      state_out      [B, Hv, dv, dk]      = states[:, K-1]
      state_inter    [B, K-1, Hv, dv, dk] = states[:, :K-1]
      conv_inter     [B, K, W-1, C]
      conv_state_out [B, W-1, C]          = conv_inter[:, K-1]
      y              [B, K, C]            conv output (after SiLU)
    """
    y, conv_inter, hist_out = conv_step(x, conv_w, conv_state)
    q, k, v = split_qkv(y, dims.Hk, dims.Hv, dims.dk, dims.dv)
    qn = l2_normalize(q, l2_eps)
    kn = l2_normalize(k, l2_eps)
    beta, g = raw_gates(a, b, A_log, dt_bias)
    o, states = delta_rule(qn, kn, v, beta, g, state, q_scale)
    return {
        "out": o,
        "states": states,
        "state_out": states[:, -1],
        "state_inter": states[:, :-1],
        "conv_inter": conv_inter,
        "conv_state_out": hist_out,
        "y": y,
    }


def rollback(accept_len, state0, states, conv_state0, conv_inter):
    """a5: per sequence, keep the first L tokens of the window.

    accept_len [B] in 0..K; state0 / conv_state0 are the pre-window state and
    history; states [B,K,...] and conv_inter [B,K,W-1,C] come from verify_step.
    Returns (state, conv_state) = (S after L tokens, history after L tokens),
    which for L = 0 is the pre-window state.
    """
    accept_len = np.asarray(accept_len)
    B = accept_len.shape[0]
    K = states.shape[1]
    st = np.empty_like(np.asarray(states[:, 0], np.float64))
    cs = np.empty_like(np.asarray(conv_inter[:, 0], np.float64))
    for bi in range(B):
        L = int(accept_len[bi])
        if not 0 <= L <= K:
            raise ValueError(f"accept length {L} outside 0..{K}")
        if L == 0:
            st[bi] = state0[bi]
            cs[bi] = conv_state0[bi]
        else:
            st[bi] = states[bi, L - 1]
            cs[bi] = conv_inter[bi, L - 1]
    return st, cs


def tree_verify_step(dims, parent, x, a, b, A_log, dt_bias, conv_w, conv_state, state,
                     q_scale: float = 1.0, l2_eps: float = 1e-6):
    """Verify of a token tree (DDTree-style window; lucebox #637, review of ggml.c:
    ``ggml_ssm_conv_tree``, the tree variant of the conv step).

    parent [B, K]: parent[b][t] in -1..t-1 (-1: a child of the committed state), nodes
    in topological order.  Every node sees the sequence along its root-to-node path:
      conv window of node t = the W-1 newest rows of [history; x of the path nodes up to
      its parent], then x_t;
      state S_t = rule(S_parent) (S_{-1} = the state before the window);
      o_t = q_scale * S_t q_t.
    Returns the same dict as verify_step, with states[:, t] the state after node t,
    conv_inter[:, t] the history after node t, and the *_out entries those of node K-1.
    """
    x = np.asarray(x, np.float64)
    w = np.asarray(conv_w, np.float64)
    hist = np.asarray(conv_state, np.float64)
    parent = np.asarray(parent)
    B, K, C = x.shape
    W = w.shape[1]
    y = np.empty((B, K, C))
    conv_inter = np.empty((B, K, W - 1, C))
    for bi in range(B):
        for t in range(K):
            p = int(parent[bi, t])
            if not -1 <= p < t:
                raise ValueError(f"parent[{bi}][{t}] = {p} is not in -1..{t - 1}")
            prev = hist[bi] if p < 0 else conv_inter[bi, p]       # history after the parent
            win = np.concatenate([prev, x[bi, t:t + 1]], axis=0)  # W rows, oldest first
            y[bi, t] = silu(np.sum(w.T * win, axis=0))
            conv_inter[bi, t] = win[1:]
    q, k, v = split_qkv(y, dims.Hk, dims.Hv, dims.dk, dims.dv)
    qn = l2_normalize(q, l2_eps)
    kn = l2_normalize(k, l2_eps)
    beta, g = raw_gates(a, b, A_log, dt_bias)
    Hk, Hv = dims.Hk, dims.Hv
    kh = np.arange(Hv) // (Hv // Hk)
    S0 = np.asarray(state, np.float64)
    states = np.empty((B, K) + S0.shape[1:])
    o = np.empty((B, K, Hv, dims.dv))
    for bi in range(B):
        for t in range(K):
            p = int(parent[bi, t])
            S = S0[bi] if p < 0 else states[bi, p]
            k_t = kn[bi, t, kh]
            q_t = qn[bi, t, kh]
            g_t = g[bi, t][:, None, None]
            pk = np.einsum("hij,hj->hi", S, k_t)
            delta = beta[bi, t][:, None] * (v[bi, t] - g[bi, t][:, None] * pk)
            St = g_t * S + delta[:, :, None] * k_t[:, None, :]
            states[bi, t] = St
            o[bi, t] = q_scale * np.einsum("hij,hj->hi", St, q_t)
    return {
        "out": o,
        "states": states,
        "state_out": states[:, -1],
        "state_inter": states[:, :-1],
        "conv_inter": conv_inter,
        "conv_state_out": conv_inter[:, -1],
        "y": y,
    }


def tree_path(parent_row, t):
    """Nodes on the root-to-node path of node t, root first."""
    path = []
    n = int(t)
    while n >= 0:
        path.append(n)
        n = int(parent_row[n])
    return path[::-1]


def gated_rms_norm(o, z, weight, eps: float = 1e-6):
    """Output side of the GDN block: RMS norm of o over the v-head dim, times a learned weight
    and the SiLU of the z gate (the attn_gate half of the stacked attn_gate|attn_qkv projection,
    lucebox #637 commit list).  o, z [..., dv]; weight [dv]."""
    o = np.asarray(o, np.float64)
    z = np.asarray(z, np.float64)
    w = np.asarray(weight, np.float64)
    return o / np.sqrt(np.mean(o * o, axis=-1, keepdims=True) + eps) * w * silu(z)


def prefill(dims, cu_seqlens, x, a, b, A_log, dt_bias, conv_w, conv_state, state,
            q_scale: float = 1.0, l2_eps: float = 1e-6, block: int = 64):
    """a1..a4 over whole prompts: B prompts of ragged lengths packed token-major
    (prompt i holds rows cu_seqlens[i] .. cu_seqlens[i+1]-1 of x, a, b and out).

    x [N, C], a, b [N, Hv] (the bf16 values as floats); conv_state [B, W-1, C];
    state [B, Hv, dv, dk].  Every token takes the plain per-token update of a1..a4;
    tokens are fed in blocks of `block` only to bound the memory held, the state and
    conv history carried from one block to the next.  Only the final state and
    history of each prompt are kept.  Returns a dict with
      out            [N, Hv, dv]
      state_out      [B, Hv, dv, dk]
      conv_state_out [B, W-1, C]
    An empty prompt leaves its state and history as they were.
    """
    cu = np.asarray(cu_seqlens, np.int64)
    x = np.asarray(x, np.float64)
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    B = cu.shape[0] - 1
    N = x.shape[0]
    if cu[0] != 0 or cu[-1] != N or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must start at 0, end at N and not decrease")
    Hv, dv = dims.Hv, dims.dv
    out = np.zeros((N, Hv, dv))
    state_out = np.array(state, dtype=np.float64, copy=True)
    conv_out = np.array(conv_state, dtype=np.float64, copy=True)
    for i in range(B):
        hist = conv_out[i:i + 1]
        S = state_out[i:i + 1]
        for t0 in range(int(cu[i]), int(cu[i + 1]), block):
            t1 = min(t0 + block, int(cu[i + 1]))
            r = verify_step(dims, x[None, t0:t1], a[None, t0:t1], b[None, t0:t1], A_log, dt_bias, conv_w,
                            hist, S, q_scale=q_scale, l2_eps=l2_eps)
            out[t0:t1] = r["out"][0]
            S = r["state_out"]
            hist = r["conv_state_out"]
        state_out[i] = S[0]
        conv_out[i] = hist[0]
    return {"out": out, "state_out": state_out, "conv_state_out": conv_out}
