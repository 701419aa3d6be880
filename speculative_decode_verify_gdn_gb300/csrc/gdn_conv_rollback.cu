// Stand-alone conv step and the rollback copy of the GDN verify library (sm_103a).
//
// Conv step: the causal conv1d update with SiLU over a window of K tokens (lucebox #637
// "NVLink fix for PR625", commit list: ggml_ssm_conv_step, "history window + silu(conv) +
// in-place history write-back + optional rollback window copy").  One thread per
// (sequence, channel) walks the window; consecutive threads take consecutive channels, so
// every load and store of a token row is coalesced.
//
// Rollback: restore each sequence's recurrent state and conv history to the point after its
// accepted prefix of L tokens (strix-llama.cpp #14 "WIP: DSv4 + Qwen3.8 Flash runtime fixes",
// commits on snapshot rollback and device-resident checkpoints; atlas #297, per-token
// conv_state intermediates for partial-accept rollback).  The source is the verify step's
// intermediate after token L-1, or the pre-window snapshot for L = 0; L = K needs no copy.
// The copy is a streaming float4 copy: each thread keeps eight 16-byte loads in flight.  It is
// launched with programmatic dependent launch, as the verify kernel is: its CTAs may be
// scheduled while the kernel ahead of it finishes, and the next verify call's while it runs.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {
namespace {

constexpr int kConvThreads = 256;
constexpr int kRbThreads = 256;
constexpr int kRbVec = 8;                                   // float4s per thread per chunk
constexpr long long kRbChunk = 4LL * kRbThreads * kRbVec;  // floats per CTA

__global__ void __launch_bounds__(kConvThreads) gdn_conv_kernel(const ConvParams p) {
  const int c = blockIdx.x * kConvThreads + threadIdx.x;
  const int b = blockIdx.y;
  if (c >= p.C) return;
  const int C = p.C;
  const int K = p.K;
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + size_t(c) * kConvW);
  float* hist = p.conv_state + size_t(b) * 3 * C + c;
  float h0 = hist[0], h1 = hist[C], h2 = hist[2 * C];
  const uint16_t* xp = p.x + size_t(b) * K * C + c;
  float* ci = p.conv_inter ? p.conv_inter + size_t(b) * K * 3 * C + c : nullptr;
  for (int t = 0; t < K; ++t) {
    const float xv = bf16_to_f32(xp[size_t(t) * C]);
    const float z = fmaf(w.w, xv, fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0)));
    const float y = silu(z);
    h0 = h1;
    h1 = h2;
    h2 = xv;
    if (ci) {
      ci[size_t(3 * t + 0) * C] = h0;
      ci[size_t(3 * t + 1) * C] = h1;
      ci[size_t(3 * t + 2) * C] = h2;
    }
    const size_t yi = (size_t(b) * K + t) * C + c;
    if (p.out_f32)
      static_cast<float*>(p.y)[yi] = y;
    else
      static_cast<uint16_t*>(p.y)[yi] = f32_to_bf16(y);
  }
  hist[0] = h0;
  hist[C] = h1;
  hist[2 * C] = h2;
}

__device__ __forceinline__ float4 ld_stream(const float4* p) {
  float4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

// grid.x: state chunks then conv chunks of one sequence; grid.y: sequence.
__global__ void __launch_bounds__(kRbThreads) gdn_rollback_kernel(const RollbackParams p, int state_chunks) {
  // the next kernel on the stream may be scheduled from here on (a verify kernel waits for this
  // grid before it reads anything); this one reads nothing before the kernel ahead of it is done
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int b = blockIdx.y;
  const int L = p.accept_len[b];
  if (L < 0 || L > p.K) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, kDevErrAcceptRange);
    return;
  }
  if (L == p.K) return;
  if (L == 0 && p.state_snap == nullptr) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(p.err, kDevErrNoSnapshot);
    return;
  }
  const bool is_state = int(blockIdx.x) < state_chunks;
  const long long n = is_state ? p.state_elems : p.conv_elems;
  const long long off = (is_state ? blockIdx.x : blockIdx.x - state_chunks) * kRbChunk;
  const float* src;
  float* dst;
  if (is_state) {
    src = (L == 0) ? p.state_snap + b * n : p.state_inter + (size_t(b) * (p.K - 1) + (L - 1)) * n;
    dst = p.state + b * n;
  } else {
    src = (L == 0) ? p.conv_snap + b * n : p.conv_inter + (size_t(b) * p.K + (L - 1)) * n;
    dst = p.conv_state + b * n;
  }
  const float4* s4 = reinterpret_cast<const float4*>(src + off);
  float4* d4 = reinterpret_cast<float4*>(dst + off);
  const long long n4 = (n - off) / 4;  // float4s left in this sequence from `off`
  float4 v[kRbVec];
#pragma unroll
  for (int k = 0; k < kRbVec; ++k) {
    const long long i = threadIdx.x + kRbThreads * k;
    if (i < n4) v[k] = ld_stream(s4 + i);
  }
#pragma unroll
  for (int k = 0; k < kRbVec; ++k) {
    const long long i = threadIdx.x + kRbThreads * k;
    if (i < n4) d4[i] = v[k];
  }
}

}  // namespace

cudaError_t launch_conv(const ConvParams& p, cudaStream_t stream) {
  dim3 grid(unsigned((p.C + kConvThreads - 1) / kConvThreads), unsigned(p.B), 1);
  gdn_conv_kernel<<<grid, kConvThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_rollback(const RollbackParams& p, cudaStream_t stream) {
  const int state_chunks = int((p.state_elems + kRbChunk - 1) / kRbChunk);
  const int conv_chunks = int((p.conv_elems + kRbChunk - 1) / kRbChunk);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(state_chunks + conv_chunks), unsigned(p.B), 1);
  cfg.blockDim = dim3(kRbThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gdn_rollback_kernel, p, state_chunks);
}

}  // namespace gdn
