// Internal launch interface between the C-ABI layer (gdn_api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace gdn {

constexpr int kKMax = 16;  // longest verify window a launch handles
constexpr int kConvW = 4;  // conv taps

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

// Row tile of one v-head's state handled by one CTA of the verify kernel, for these dims.
int verify_row_tile(int dv, int r);
// Cluster size of the verify kernel (CTAs sharing one q/k head), 0 if unsupported.
int verify_cluster_size(int dv, int r);
size_t verify_smem_bytes(int dk, int dv, int r);

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream);
cudaError_t launch_conv(const ConvParams& p, cudaStream_t stream);
cudaError_t launch_rollback(const RollbackParams& p, cudaStream_t stream);

}  // namespace gdn
