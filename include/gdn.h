/*
 * gdn.h - C ABI of the GB300 (sm_103a) speculative-decoding verify step of one
 * Gated DeltaNet (GDN) linear-attention layer.
 *
 * For B sequences and a window of K tokens (the seed token plus K-1 drafted
 * tokens) the step is
 *   a1  causal conv1d update over the q|k|v channels with its history window
 *       and SiLU, writing the history back and one history snapshot per token
 *       (lucebox #637 "NVLink fix for PR625", commit list: ggml_ssm_conv_step;
 *       atlas #297 "verify-step glue", commit on SSM/GDN verify kernels:
 *       causal_conv1d_update_prefill_inter),
 *   a2  one L2 norm over the q|k slab (lucebox #637, commit list),
 *   a3  raw gates beta = sigmoid(b), g = exp(softplus(a + dt_bias) * A) with
 *       A = -exp(A_log) and softplus clipped to the identity above 20
 *       (lucebox #637, review of ggml-cuda/gated_delta_net.cu line 404),
 *   a4  the gated delta rule S_t = g_t S_{t-1} + beta_t (v_t - g_t S_{t-1} k_t) k_t^T,
 *       o_t = q_scale * S_t q_t, q/k heads broadcast to the v heads
 *       (v-head h reads q/k head h / (Hv/Hk)), writing the final state and the
 *       K-1 intermediate states in one pass (atlas #297: gated_delta_rule_wy16.cu),
 *   a5  rollback of state and conv history to each sequence's accepted length
 *       (strix-llama.cpp #14 "WIP: DSv4 + Qwen3.8 Flash runtime fixes", commits
 *       on recurrent snapshot rollback and device checkpoints).
 *
 * Conventions common to every call
 *  - Layouts are row-major with the last index fastest (shapes below).
 *  - Ownership: the caller owns every buffer, scratch included.  The library
 *    allocates and frees nothing; its only state is a thread-local error
 *    message and one 32-bit device status word per GPU (see gdn_device_status).
 *  - Device reset: the library caches, per device, the device addresses of
 *    its status word and of gdn_verify_step_static_scratch's array, looked up
 *    on first use.  Do not call it across a cudaDeviceReset (or anything else
 *    that destroys and recreates the device's primary context) in one process:
 *    the cached addresses would point into the old context.
 *  - Asynchrony: calls validate on the host, enqueue kernels on `stream` and
 *    return; launch failures come back as GDN_ERR_CUDA.
 *  - Validation happens before any launch: a non-OK status means nothing was
 *    enqueued.  No call aborts the process.
 *  - Supported shapes: 1 <= K <= 16, dk and dv in {64, 128}, Hk >= 1,
 *    Hv % Hk == 0, conv width W == 4, 0 <= B <= 65535 (B == 0 is a no-op),
 *    channels C = 2*Hk*dk + Hv*dv.
 *  - Alignment: every float / bf16 buffer must be 16-byte aligned.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream handle (the same object as cudaStream_t / CUstream). NULL = legacy default stream. */
typedef struct CUstream_st* gdn_stream_t;

typedef enum {
  GDN_OK = 0,
  GDN_ERR_INVALID_ARG = 1, /* null pointer, bad size, misalignment, non-finite scalar */
  GDN_ERR_UNSUPPORTED = 2, /* shape outside the supported set above */
  GDN_ERR_ALIAS = 3,       /* buffers overlap where the call forbids it */
  GDN_ERR_NO_SNAPSHOT = 4, /* rollback asked for a snapshot that was not passed */
  GDN_ERR_CUDA = 5         /* a CUDA runtime call failed (message in gdn_last_error) */
} gdn_status;

/* Bits of the per-device status word (set by kernels, read by gdn_device_status). */
#define GDN_DEVERR_TIMEOUT 1u      /* a bounded wait in a kernel gave up; its results are invalid */
#define GDN_DEVERR_ACCEPT_RANGE 2u /* rollback saw an accept length outside 0..K; that sequence was left as is */
#define GDN_DEVERR_NO_SNAPSHOT 4u  /* rollback saw accept length 0 with no snapshot; that sequence was left as is */
#define GDN_DEVERR_TREE_PARENT 8u  /* a token tree had a parent outside -1..t-1; it was read as -1 */
#define GDN_DEVERR_SEQLENS 16u     /* gdn_prefill's cu_seqlens were not 0 = c_0 <= ... <= c_B = n_tokens; nothing was written */

typedef struct {
  int32_t B;       /* sequences */
  int32_t K;       /* window tokens: seed + drafts, 1..16 */
  int32_t Hk;      /* q/k heads */
  int32_t Hv;      /* v heads (a multiple of Hk) */
  int32_t dk;      /* q/k head dim, 64 or 128 */
  int32_t dv;      /* v head dim, 64 or 128 */
  int32_t conv_w;  /* conv taps W, must be 4 */
  float q_scale;   /* o_t = q_scale * S_t q_t (1.0 for the plain rule) */
  float l2_eps;    /* L2 norm: z / sqrt(sum z^2 + l2_eps), >= 0 */
  int32_t out_f32; /* 0: outputs in bf16, 1: outputs in f32 */
} gdn_dims;

/*
 * a1 alone: causal conv1d update with SiLU (lucebox #637 commit list,
 * ggml_ssm_conv_step: history window + silu(conv) + in-place history
 * write-back + rollback window copy).
 *   x          [B, K, C]       bf16 (uint16 bit patterns), channel fastest
 *   conv_w     [C, W]          f32; w[c][W-1] multiplies the newest row
 *   conv_state [B, W-1, C]     f32, oldest row first; read, then overwritten
 *                              in place with the history after token K-1
 *   conv_inter [B, K, W-1, C]  f32 or NULL; snapshot t = the W-1 newest
 *                              window rows after token t
 *   y          [B, K, C]       f32 if out_f32 else bf16: SiLU(conv) per token
 * No bias.  conv_inter and y must not overlap each other or the inputs.
 */
gdn_status gdn_conv_step(const gdn_dims* dims, const uint16_t* x, const float* conv_w, float* conv_state,
                         float* conv_inter, void* y, gdn_stream_t stream);

/*
 * a1..a4 fused: one verify window for B sequences.
 *   x               [B, K, C]         bf16; channel order q | k | v, each head contiguous
 *   a, b            [B, K, Hv]        bf16 raw gate inputs (alpha, beta projections)
 *   A_log, dt_bias  [Hv]              f32
 *   conv_w          [C, W]            f32
 *   conv_state_in   [B, W-1, C]       f32 history before the window
 *   conv_state_out  [B, W-1, C]       f32 history after token K-1; may equal
 *                                     conv_state_in (in place), else no overlap
 *   conv_inter      [B, K, W-1, C]    f32 or NULL: history after each token
 *   state_in        [B, Hv, dv, dk]   f32 state before the window (row = v index)
 *   state_out       [B, Hv, dv, dk]   f32 state after token K-1; may equal
 *                                     state_in (in place), else no overlap
 *   state_inter     [B, K-1, Hv, dv, dk] f32: state after tokens 0..K-2;
 *                                     NULL allowed only when K == 1
 *   out             [B, K, Hv, dv]    bf16 or f32 (out_f32): o_t = q_scale * S_t q_t
 *   workspace       unused: gdn_verify_workspace_size() reports 0 bytes and the
 *                   pointer may be NULL (the argument keeps the ABI of earlier
 *                   builds, whose kernels passed tables through it).
 * Intermediates and out must not overlap any other buffer.
 * Runs as two kernels on `stream`: a per-(sequence, v-head, 32-row tile)
 * verify kernel (conv, norms, gates and the state recurrence, which stores
 * every state straight from registers) and a per-(sequence, q/k channel
 * block) kernel that writes the q|k channels' history snapshots and new
 * history once every verify CTA has read the old ones (programmatic
 * dependent launch).  The call is complete when the second kernel is.  The
 * verify kernel is itself launched with programmatic dependent launch: it
 * reads nothing before the kernel ahead of it on the stream has completed.
 */
gdn_status gdn_verify_step(const gdn_dims* dims, const uint16_t* x, const uint16_t* a, const uint16_t* b,
                           const float* A_log, const float* dt_bias, const float* conv_w,
                           const float* conv_state_in, float* conv_state_out, float* conv_inter,
                           const float* state_in, float* state_out, float* state_inter, void* out,
                           void* workspace, uint64_t workspace_bytes, gdn_stream_t stream);

/*
 * a5 of the previous window fused into a1..a4 of the next one: rollback applied
 * on read, so the accepted state is never copied (strix-llama.cpp #14: snapshot
 * planes and rolling checkpoints; atlas #297: per-token intermediates kept for
 * partial-accept rollback).  Same result as
 *   gdn_rollback(accept_len_prev, ...) followed by gdn_verify_step(...),
 * where the previous window had the same K.  Per sequence, with
 * L = accept_len_prev[b]:
 *   L == K       S0 = state_in[b],                  history = conv_state_in[b]
 *   1 <= L < K   S0 = state_inter_prev[b][L-1],     history = conv_inter_prev[b][L-1]
 *   L == 0       S0 = state_snapshot_prev[b],       history = conv_state_snapshot_prev[b]
 * state_in / conv_state_in are the previous window's final state and history;
 * the *_prev buffers its intermediates and the pre-window snapshots (both
 * snapshots or neither; NULL makes L == 0 an error).  An out-of-range L, or
 * L == 0 without snapshots, is read as L == K and sets a device status bit.
 * In place is allowed and is the intended use: state_out may be state_in or
 * state_snapshot_prev, state_inter may be state_inter_prev, conv_state_out may
 * be conv_state_in or conv_state_snapshot_prev, conv_inter may be
 * conv_inter_prev (each state tile and v-channel history is read, then
 * rewritten, by one owner; the q|k channels' history, which every CTA of a q/k
 * head reads, is rewritten by the second kernel only after all those reads).
 * Any other overlap with an output is rejected.
 * Shapes, workspace and the remaining arguments as gdn_verify_step.
 */
gdn_status gdn_verify_resume(const gdn_dims* dims, const int32_t* accept_len_prev, const uint16_t* x,
                             const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias,
                             const float* conv_w, const float* conv_state_in, const float* conv_inter_prev,
                             const float* conv_state_snapshot_prev, float* conv_state_out, float* conv_inter,
                             const float* state_in, const float* state_inter_prev, const float* state_snapshot_prev,
                             float* state_out, float* state_inter, void* out, void* workspace,
                             uint64_t workspace_bytes, gdn_stream_t stream);

/*
 * a1..a4 over a token tree instead of a chain (DDTree-style verify; lucebox #637,
 * review of ggml.c: ggml_ssm_conv_tree, the tree variant of the conv step).
 *   parent_dev  [B, K] int32 on the device: parent[b][t] in -1..t-1 (nodes in
 *               topological order; -1 = a child of the committed state).
 * Every node sees the sequence along its root-to-node path: its conv window is
 * the W-1 newest rows of [history; x of the path nodes above it], and its state
 * is the rule applied to its parent's state (conv_state_in / state_in for -1).
 * Node t's state and history go where token t's go in gdn_verify_step
 * (state_inter[b][t] for t < K-1, state_out / conv_state_out for node K-1,
 * conv_inter[b][t]), so gdn_rollback with accept_len = n + 1 rolls a sequence
 * back to accepted node n (0 for none).  A chain (parent[t] = t-1) gives
 * gdn_verify_step's histories bit for bit and its states and outputs up to
 * f32 rounding order.  A parent outside -1..t-1 is read as -1 and sets
 * GDN_DEVERR_TREE_PARENT.  Other arguments, aliasing and workspace as
 * gdn_verify_step.
 */
gdn_status gdn_verify_tree(const gdn_dims* dims, const int32_t* parent_dev, const uint16_t* x, const uint16_t* a,
                           const uint16_t* b, const float* A_log, const float* dt_bias, const float* conv_w,
                           const float* conv_state_in, float* conv_state_out, float* conv_inter,
                           const float* state_in, float* state_out, float* state_inter, void* out,
                           void* workspace, uint64_t workspace_bytes, gdn_stream_t stream);

/*
 * gdn_verify_step with the output side of the GDN block fused into its
 * epilogue: the gated RMS norm of each token's v-head output, with the z gate
 * taken from the attn_gate half of the stacked attn_gate|attn_qkv projection
 * (lucebox #637, "NVLink fix for PR625", commit list).  Per (b, t, h):
 *   out[b,t,h,:] = o * w * SiLU(z[b,t,h,:]) / sqrt(mean_i(o_i^2) + norm_eps)
 * where o is the step's (scaled) attention output before any rounding.
 *  z        [B, K, Hv, dv] bf16, device, read only (16-byte aligned, may not
 *           overlap an output).
 *  norm_w   [dv] f32, device, read only: the norm weight, shared by all heads.
 *  norm_eps finite, >= 0.
 * Everything else (the states and histories written, aliasing, workspace,
 * errors) is as for gdn_verify_step; `out` holds the normed result only.
 * The v-head's row tiles run as one thread-block cluster, sharing the sums of
 * squares through distributed shared memory.
 */
gdn_status gdn_verify_gated(const gdn_dims* dims, const uint16_t* x, const uint16_t* a, const uint16_t* b,
                            const float* A_log, const float* dt_bias, const float* conv_w,
                            const float* conv_state_in, float* conv_state_out, float* conv_inter,
                            const float* state_in, float* state_out, float* state_inter, const uint16_t* z,
                            const float* norm_w, float norm_eps, void* out, void* workspace,
                            uint64_t workspace_bytes, gdn_stream_t stream);

/*
 * Bytes of workspace gdn_verify_step needs for `dims`: 0 (its kernels share
 * nothing through global scratch).  Validates dims like gdn_verify_step.
 */
gdn_status gdn_verify_workspace_size(const gdn_dims* dims, uint64_t* bytes);

/*
 * gdn_verify_step for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this is a convenience of this library.)
 *
 * Same arguments and results as gdn_verify_step minus the workspace.  Some
 * callers may not call cudaMalloc where they run the verify step (a runtime
 * whose memory pool forbids allocation on its hot path, a path that must not
 * synchronise the device, an embedder that only passes in tensors it owns);
 * this entry point passes a fixed array in the library's device memory as the
 * workspace instead.  The verify kernels need no scratch (see
 * gdn_verify_workspace_size), so the array is 256 bytes; dims that would need
 * more return GDN_ERR_UNSUPPORTED with a message.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current and caches it: make the
 *    first call on a device before any stream capture starts.
 *  - Nothing is allocated or freed.
 */
gdn_status gdn_verify_step_static_scratch(const gdn_dims* dims, const uint16_t* x, const uint16_t* a,
                                          const uint16_t* b, const float* A_log, const float* dt_bias,
                                          const float* conv_w, const float* conv_state_in, float* conv_state_out,
                                          float* conv_inter, const float* state_in, float* state_out,
                                          float* state_inter, void* out, gdn_stream_t stream);

/*
 * Prefill of whole prompts: a1..a4 over B prompts of any length, packed
 * token-major (the VARLEN-FLA / FlashInfer-GDN prefill paths named in atlas
 * #258 and #297; lucebox #637 speaks of long prefills through the same layer).
 * The result equals the per-token recurrence of gdn_verify_step run over each
 * prompt from its state and history; no intermediates are kept.  Prompt i holds
 * tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 of the packed tensors.
 *   dims              B = prompts (0..65535), Hk, Hv, dk, dv, conv_w, q_scale,
 *                     l2_eps, out_f32 as for gdn_verify_step; dims->K is not read
 *   n_tokens          N, 0 <= N < 2^31: the packed token count
 *   cu_seqlens_dev    [B + 1] int32 on the device, 4-byte aligned:
 *                     0 = c_0 <= c_1 <= ... <= c_B = N.  Checked on the device:
 *                     otherwise GDN_DEVERR_SEQLENS is set and nothing is written.
 *   x                 [N, C] bf16; a, b [N, Hv] bf16 (may be NULL when N == 0)
 *   A_log, dt_bias    [Hv] f32; conv_w [C, W] f32
 *   conv_state_in/out [B, W-1, C] f32: history before / after each prompt; may
 *                     be the same buffer (in place), else no overlap
 *   state_in/out      [B, Hv, dv, dk] f32: state before / after each prompt;
 *                     may be the same buffer (in place), else no overlap
 *   out               [N, Hv, dv] bf16 or f32 (may be NULL when N == 0)
 *   workspace         at least gdn_prefill_workspace_size() bytes, 16-byte
 *                     aligned, no initialisation needed, dead after the call.
 * An empty prompt passes its state and history through unchanged.
 * Runs three kernels on `stream`: a one-block check of cu_seqlens that numbers
 * the 64-token chunks; a per-(chunk, q/k head) kernel, all chunks in parallel
 * (conv, norms, gates, Gram products and the chunk's 64 x 64 triangular
 * inverse per v-head); and a per-(prompt, v-head, 64 state rows) kernel that
 * walks the prompt's chunks in order on the tensor cores (tcgen05, the state
 * in tensor memory; every product is three bf16 MMAs over hi/lo operand
 * pairs, about 2^-16 relative error per product).
 */
gdn_status gdn_prefill(const gdn_dims* dims, int64_t n_tokens, const int32_t* cu_seqlens_dev, const uint16_t* x,
                       const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias,
                       const float* conv_w, const float* conv_state_in, float* conv_state_out,
                       const float* state_in, float* state_out, void* out, void* workspace,
                       uint64_t workspace_bytes, gdn_stream_t stream);

/*
 * Bytes of workspace gdn_prefill needs for `dims` (B, Hk, Hv, dk) and N tokens:
 * with cap = ceil(N / 64) + B chunks,
 * 16 ceil((B + 5) / 4) + cap (16 + Hk * 512 * dk + Hv * 33280).
 */
gdn_status gdn_prefill_workspace_size(const gdn_dims* dims, int64_t n_tokens, uint64_t* bytes);

/*
 * a5: per sequence, keep the first L = accept_len[b] window tokens
 * (strix-llama.cpp #14: snapshot restore of the recurrent state; lucebox #637:
 * rollback window copy of the conv history).
 *   accept_len_dev          [B] int32 on the device, each in 0..K
 *   state_in_snapshot       [B, Hv, dv, dk] f32 or NULL: the state before the
 *                           window (needed only for L == 0; must not overlap state)
 *   state                   [B, Hv, dv, dk] f32, holds the state after token K-1
 *                           on entry (verify's state_out) and S_L on exit
 *   state_inter             [B, K-1, Hv, dv, dk] f32 from gdn_verify_step (NULL iff K == 1)
 *   conv_state_in_snapshot  [B, W-1, C] f32 or NULL (for L == 0; no overlap with conv_state)
 *   conv_state              [B, W-1, C] f32, history after token K-1 on entry, after L tokens on exit
 *   conv_inter              [B, K, W-1, C] f32 from gdn_verify_step (NULL iff K == 1)
 * L == K leaves a sequence untouched.  Lengths are read on the device: an
 * out-of-range length, or L == 0 with no snapshot, leaves that sequence
 * untouched and sets a bit in the device status word.
 */
gdn_status gdn_rollback(const gdn_dims* dims, const int32_t* accept_len_dev, const float* state_in_snapshot,
                        float* state, const float* state_inter, const float* conv_state_in_snapshot,
                        float* conv_state, const float* conv_inter, gdn_stream_t stream);

/*
 * Reads (and, if clear != 0, resets) the current device's status word after
 * synchronising `stream`.  *flags receives the OR of GDN_DEVERR_* bits set by
 * kernels since the last clear.
 */
gdn_status gdn_device_status(uint32_t* flags, int32_t clear, gdn_stream_t stream);

/* Message of the last non-OK status returned on this thread ("" if none). */
const char* gdn_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
