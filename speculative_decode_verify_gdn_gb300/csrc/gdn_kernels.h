// Internal launch interface between the C-ABI layer (gdn_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/gdn.h"

namespace gdn {

constexpr int kKMax = 16;  // longest verify window a launch handles
constexpr int kConvW = 4;  // conv taps
constexpr int kNCol = 2 * kKMax;  // rows of a window's q/k table: k^ in [0,16), q^ in [16,32)

struct VerifyParams {
  const uint16_t* x;
  const uint16_t* a;
  const uint16_t* b;
  const float* A_log;
  const float* dt_bias;
  const float* conv_w;
  const float* conv_state_in;
  float* conv_state_out;
  float* conv_inter;  // may be null
  const float* state_in;
  float* state_out;
  float* state_inter;  // null only when K == 1
  void* out;
  // Rollback of the previous window applied on read (all null for a plain verify step): per
  // sequence, L = accept_prev[b] selects where S0 and the conv history come from -
  // L == K: state_in / conv_state_in (the previous window's final state and history);
  // 1 <= L < K: state_inter_prev[b][L-1] / conv_inter_prev[b][L-1];
  // L == 0: state_snap_prev / conv_snap_prev (the state before the previous window).
  const int32_t* accept_prev;
  const float* state_inter_prev;
  const float* conv_inter_prev;
  const float* state_snap_prev;  // may be null (then L == 0 is an error)
  const float* conv_snap_prev;
  // Token tree (gdn_verify_tree; null for a chain window): parent[b][t] in -1..t-1.
  const int32_t* parent;
  // Gated output norm (gdn_verify_gated; z null otherwise): out = o rsqrt(mean o^2 + eps) w SiLU(z)
  const uint16_t* z;     // [B, K, Hv, dv] bf16
  const float* norm_w;   // [dv]
  float norm_eps;
  uint32_t* err;       // device status word
  int B, K, Hk, Hv, dk, dv, C;
  float q_scale, l2_eps;
  int out_f32;
};

struct ConvParams {
  const uint16_t* x;
  const float* conv_w;
  float* conv_state;
  float* conv_inter;  // may be null
  void* y;
  int B, K, C;
  int out_f32;
};

struct RollbackParams {
  const int32_t* accept_len;
  const float* state_snap;  // may be null
  float* state;
  const float* state_inter;
  const float* conv_snap;   // may be null (then state_snap is null too)
  float* conv_state;
  const float* conv_inter;
  uint32_t* err;
  int B, K;
  long long state_elems;  // per sequence: Hv*dv*dk
  long long conv_elems;   // per sequence: (W-1)*C
};

// ---- chunked prefill (gdn_prefill)
constexpr int kPrefillChunk = 64;  // tokens per chunk

// Upper bound on the chunks of B prompts holding N tokens in all.
inline long long prefill_chunk_cap(int B, long long N) { return (N + kPrefillChunk - 1) / kPrefillChunk + B; }

// Prefill workspace (operands for the tensor cores as bf16 hi/lo pairs, each block in the
// K-major core-matrix layout of 8 rows x 16 bytes):
//   meta [4 + B + 1] int32     valid flag, chunk count, -, -, first chunk of each prompt (+ total)
//   chunks [cap] int4          per chunk: prompt, first token, tokens (1..64), first token of the prompt
//   kq   [cap][Hk][4][64 x dk] k^ hi, k^ lo, q^ hi, q^ lo as [t][c] (k^ also read as [c][t])
//   wm   [cap][Hv][4][64 x 64] W hi, W lo, MQ hi, MQ lo as [t][j]
//   gd   [cap][Hv][2][64] f32  Gamma_t, then d_t = prod_{t<m<64} g_m
struct PrefillWorkspace {
  int32_t* meta;
  int4* chunks;
  uint16_t* kq;
  uint16_t* wm;
  float* gd;
  long long chunk_cap;
};

size_t prefill_workspace_bytes(int B, long long N, int Hk, int Hv, int dk);
PrefillWorkspace prefill_workspace_carve(void* base, int B, long long N, int Hk, int Hv, int dk);

struct PrefillParams {
  const int32_t* cu;  // [B + 1] token offsets of the prompts
  const uint16_t* x;  // [N, C] bf16
  const uint16_t* a;  // [N, Hv] bf16
  const uint16_t* b;
  const float* A_log;
  const float* dt_bias;
  const float* conv_w;
  const float* conv_state_in;  // [B, W-1, C]
  float* conv_state_out;
  const float* state_in;  // [B, Hv, dv, dk]
  float* state_out;
  void* out;  // [N, Hv, dv]
  PrefillWorkspace ws;
  uint32_t* err;
  int B, Hk, Hv, dk, dv, C;
  long long N;
  float q_scale, l2_eps;
  int out_f32;
};

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream);

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream);
cudaError_t launch_conv(const ConvParams& p, cudaStream_t stream);
cudaError_t launch_rollback(const RollbackParams& p, cudaStream_t stream);

// Records `msg` as this thread's gdn_last_error() text and returns `s`.
gdn_status report_error(gdn_status s, const char* msg);

}  // namespace gdn
