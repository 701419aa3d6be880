// Verify step of one Gated DeltaNet layer on sm_103a: conv + SiLU, q|k L2 norm, raw gates and
// the chunkwise (WY) gated delta rule writing the final and every intermediate state.
//
// Method (lucebox #637 "NVLink fix for PR625", commit list: fused conv step, single l2_norm
// over q|k, raw-gate gated_delta_net with head broadcast; review of ggml-cuda/gated_delta_net.cu
// line 404 for the gate formula; atlas #297, commit on the SSM/GDN verify kernels: a K=16
// WY-chunkwise verify that writes the final state and all intermediates in one pass):
//
//   y_t   = SiLU(sum_j w[c][j] win[t+j][c])            per channel, win = [history; x]
//   q^,k^ = q / sqrt(|q|^2 + eps), k / sqrt(|k|^2 + eps)  per (token, q/k head)
//   beta  = sigmoid(b), g = exp(softplus(a + dt_bias) * -exp(A_log))
//   S_t   = g_t S_{t-1} + u_t k^_t^T,  u_t = beta_t (v_t - g_t S_{t-1} k^_t)
//   o_t   = q_scale S_t q^_t
//
// Chunk (WY) form, exact in real arithmetic: with Gamma_t = prod_{m<=t} g_m and
// D[t][j] = prod_{j<m<=t} g_m,
//   u_t = beta_t (v_t - Gamma_t S0 k^_t - sum_{j<t} D[t][j] (k^_j . k^_t) u_j)
//   o_t = q_scale Gamma_t S0 q^_t + sum_{j<=t} q_scale D[t][j] (k^_j . q^_t) u_j
// Every state row needs only its products with the window's k^ and q^ (one small product
// with S0) and a K x K forward substitution; the K states then follow as
// S_t = g_t S_{t-1} + u_t k^_t^T with no reduction between two stores.  Decay ratios are
// running products of g (all in [0, 1]), never quotients, so nothing overflows.
//
// Two kernels on the caller's stream:
//  1. qk_prologue: one CTA per (sequence, q/k head).  Conv + SiLU of the head's q|k channels
//     (each channel's history is read and rewritten by this one thread, so the in-place
//     history update is race-free), L2 norms, gates of the head's r = Hv/Hk v-heads, Gram
//     products and decay products.  Writes three small tables per head to the workspace, laid
//     out exactly as the second kernel keeps them in shared memory.
//  2. state_stream: one CTA per (sequence, v-head, 32-row tile of the state), launched with
//     programmatic dependent launch so that it starts while the prologue runs: it issues the
//     bulk async (TMA) copy of its 16 KB S0 tile and convolves its own 32 v-channels first, then
//     waits for the prologue grid and bulk-copies the tables.  From there each warp owns four
//     state rows and needs no CTA-wide barrier: products with S0, forward substitution,
//     outputs, then the K states leave straight from registers as coalesced 16-byte streaming
//     stores (512 contiguous bytes per warp instruction).
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

size_t workspace_bytes(int B, int Hk, int Hv, int dk) {
  const size_t per_head = size_t(dk) * kNCol + size_t(kKMax) * dk;
  return 4 * (size_t(B) * Hk * per_head + size_t(B) * Hv * kGateFloats);
}

Workspace workspace_carve(void* base, int B, int Hk, int Hv, int dk) {
  (void)Hv;
  Workspace w;
  w.wt = static_cast<float*>(base);
  w.kn = w.wt + size_t(B) * Hk * dk * kNCol;
  w.gate = w.kn + size_t(B) * Hk * kKMax * dk;
  return w;
}

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 32;          // state rows per CTA of the stream kernel
constexpr int kRowsPerWarp = kRows / kWarps;

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Index of q^/k^ column `col` of channel `c` in the swizzled table.
__device__ __forceinline__ int wt_idx(int c, int col) { return c * kNCol + (col ^ (c & 31)); }

// Conv + SiLU of one channel over the window; writes the channel's history snapshots and new
// history.  y[t] receives the outputs for t < K.
__device__ __forceinline__ void conv_channel(const VerifyParams& p, int b, int c, float (&y)[kKMax]) {
  const int C = p.C;
  const int K = p.K;
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + size_t(c) * kConvW);
  const float* hin = p.conv_state_in + size_t(b) * 3 * C + c;
  float h0 = hin[0], h1 = hin[C], h2 = hin[2 * C];
  const uint16_t* xp = p.x + size_t(b) * K * C + c;
  float xv[kKMax];
#pragma unroll
  for (int t = 0; t < kKMax; ++t) xv[t] = (t < K) ? bf16_to_f32(xp[size_t(t) * C]) : 0.f;
  float* ci = p.conv_inter ? p.conv_inter + size_t(b) * K * 3 * C + c : nullptr;
#pragma unroll
  for (int t = 0; t < kKMax; ++t) {
    y[t] = 0.f;
    if (t < K) {
      const float z = fmaf(w.w, xv[t], fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0)));
      y[t] = silu(z);
      h0 = h1;
      h1 = h2;
      h2 = xv[t];
      if (ci) {
        ci[size_t(3 * t + 0) * C] = h0;
        ci[size_t(3 * t + 1) * C] = h1;
        ci[size_t(3 * t + 2) * C] = h2;
      }
    }
  }
  float* hout = p.conv_state_out + size_t(b) * 3 * C + c;
  hout[0] = h0;
  hout[C] = h1;
  hout[2 * C] = h2;
}

// ------------------------------------------------------------------------------------------
// Kernel 1: per (sequence, q/k head) prologue.
template <int DK>
struct PrologueLayout {
  static constexpr int NSTRIDE = DK + 1;                    // padded rows: column reads conflict-free
  static constexpr int OFF_Y = 0;                           // raw conv outputs [32][DK] (k: 0..15, q: 16..31)
  static constexpr int OFF_N = OFF_Y + kNCol * DK;          // normalised [32][NSTRIDE]
  static constexpr int OFF_KK = OFF_N + kNCol * NSTRIDE;    // k^_t . k^_j  [16][17]
  static constexpr int OFF_KQ = OFF_KK + kKMax * kMStride;  // k^_j . q^_t  [16][17]
  static constexpr int OFF_BG = OFF_KQ + kKMax * kMStride;  // beta[16], g[16] of one v-head
  static constexpr int FLOATS = OFF_BG + 2 * kKMax;
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
};

template <int DK>
__global__ void __launch_bounds__(kThreads) gdn_qk_prologue_kernel(const VerifyParams p) {
  using L = PrologueLayout<DK>;
  extern __shared__ __align__(128) float sm[];
  float* sY = sm + L::OFF_Y;
  float* sN = sm + L::OFF_N;
  float* sKK = sm + L::OFF_KK;
  float* sKQ = sm + L::OFF_KQ;
  float* sBeta = sm + L::OFF_BG;
  float* sG = sBeta + kKMax;

  griddep_launch_dependents();  // the state kernel may start its independent work now

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kh = blockIdx.x;
  const int b = blockIdx.y;
  const int K = p.K;
  const int r = p.Hv / p.Hk;

  // a1: conv of the head's q|k channels (thread cc < 2*DK owns one channel)
  if (tid < 2 * DK) {
    const int cc = tid;
    const int c = (cc < DK) ? kh * DK + cc : p.Hk * DK + kh * DK + (cc - DK);
    float y[kKMax];
    conv_channel(p, b, c, y);
    const int n0 = (cc < DK) ? kKMax : 0;  // q rows 16..31, k rows 0..15
    const int col = cc % DK;
#pragma unroll
    for (int t = 0; t < kKMax; ++t) sY[(n0 + t) * DK + col] = y[t];
  }
  __syncthreads();

  // a2: L2 norm of each of the 2K vectors (warp per vector); rows t >= K become zero
  for (int n = warp; n < kNCol; n += kWarps) {
    const int t = n % kKMax;
    float vals[DK / 32];
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < DK / 32; ++m) {
      vals[m] = sY[n * DK + lane + 32 * m];
      ss = fmaf(vals[m], vals[m], ss);
    }
    ss = warp_sum(ss);
    const float inv = (t < K) ? 1.f / sqrtf(ss + p.l2_eps) : 0.f;
#pragma unroll
    for (int m = 0; m < DK / 32; ++m) sN[n * L::NSTRIDE + lane + 32 * m] = vals[m] * inv;
  }
  __syncthreads();

  // tables for the state kernel: swizzled [DK][32] and token-major k^ [16][DK]
  const size_t head = size_t(b) * p.Hk + kh;
  float* wt = p.ws.wt + head * DK * kNCol;
  for (int f = tid; f < DK * kNCol; f += kThreads) {
    const int c = f / kNCol;
    const int col = (f % kNCol) ^ (c & 31);
    wt[f] = sN[col * L::NSTRIDE + c];
  }
  float* kn = p.ws.kn + head * kKMax * DK;
  for (int f = tid; f < kKMax * DK; f += kThreads) kn[f] = sN[(f / DK) * L::NSTRIDE + f % DK];

  // Gram products of the window: KK[t][j] = k^_t . k^_j, KQ[t][j] = k^_j . q^_t
  {
    const int t = tid >> 4, j = tid & 15;
    const float* kt = sN + t * L::NSTRIDE;
    const float* kj = sN + j * L::NSTRIDE;
    const float* qt = sN + (kKMax + t) * L::NSTRIDE;
    float kk = 0.f, kq = 0.f;
#pragma unroll 8
    for (int c = 0; c < DK; ++c) {
      kk = fmaf(kt[c], kj[c], kk);
      kq = fmaf(qt[c], kj[c], kq);
    }
    sKK[t * kMStride + j] = kk;
    sKQ[t * kMStride + j] = kq;
  }

  // a3 and the per-v-head gate blocks
  for (int hv = 0; hv < r; ++hv) {
    const int h = kh * r + hv;
    __syncthreads();  // Gram ready (first pass); previous head's beta/g consumed
    if (tid < kKMax) {
      float beta = 0.f, g = 1.f;
      if (tid < K) {
        const float A = -expf(p.A_log[h]);
        const size_t gi = (size_t(b) * K + tid) * p.Hv + h;
        const float av = bf16_to_f32(p.a[gi]) + p.dt_bias[h];
        const float sp = (av > 20.f) ? av : log1pf(expf(av));
        g = expf(sp * A);
        beta = 1.f / (1.f + expf(-bf16_to_f32(p.b[gi])));
      }
      sBeta[tid] = beta;
      sG[tid] = g;
    }
    __syncthreads();
    float* gate = p.ws.gate + (size_t(b) * p.Hv + h) * kGateFloats;
    const int t = tid >> 4, j = tid & 15;
    float d = 1.f;
    for (int m = j + 1; m <= t; ++m) d *= sG[m];
    gate[t * kMStride + j] = (j < t) ? d * sKK[t * kMStride + j] : 0.f;
    gate[kGateOffN + t * kMStride + j] = (j <= t) ? p.q_scale * d * sKQ[t * kMStride + j] : 0.f;
    if (j == 0) gate[kGateOffGam + t] = d * sG[0];
    if (tid < kKMax) {
      gate[tid * kMStride + kKMax] = 0.f;
      gate[kGateOffN + tid * kMStride + kKMax] = 0.f;
      gate[kGateOffBeta + tid] = sBeta[tid];
      gate[kGateOffG + tid] = sG[tid];
    }
    if (tid < kGateFloats - (kGateOffGam + kKMax)) gate[kGateOffGam + kKMax + tid] = 0.f;
  }
}

// ------------------------------------------------------------------------------------------
// Kernel 2: per (sequence, v-head, 32-row tile) state stream.
template <int DK>
struct StreamLayout {
  static constexpr int PSTRIDE = kNCol + 1;
  static constexpr int OFF_S0 = 0;                               // [32][DK]      bulk copy
  static constexpr int OFF_WT = OFF_S0 + kRows * DK;             // [DK][32]      bulk copy
  static constexpr int OFF_KN = OFF_WT + DK * kNCol;             // [16][DK]      bulk copy
  static constexpr int OFF_GATE = OFF_KN + kKMax * DK;           // gate block    bulk copy
  static constexpr int OFF_V = OFF_GATE + kGateFloats;           // [warp][16][4] v conv outputs
  static constexpr int OFF_U = OFF_V + kWarps * kKMax * kRowsPerWarp;  // [warp][16][4] u
  static constexpr int OFF_P = OFF_U + kWarps * kKMax * kRowsPerWarp;  // [32][33] S0 [k^ | q^]
  static constexpr int OFF_BAR = (OFF_P + kRows * PSTRIDE + 1) & ~1;
  static constexpr int FLOATS = OFF_BAR + 2;
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
  static constexpr uint32_t S0_BYTES = kRows * DK * 4;
  static constexpr uint32_t WT_BYTES = DK * kNCol * 4;
  static constexpr uint32_t KN_BYTES = kKMax * DK * 4;
  static constexpr uint32_t GATE_BYTES = kGateFloats * 4;
  static_assert(S0_BYTES % 16 == 0 && WT_BYTES % 16 == 0 && KN_BYTES % 16 == 0 && GATE_BYTES % 16 == 0, "");
  static_assert(OFF_WT % 4 == 0 && OFF_KN % 4 == 0 && OFF_GATE % 4 == 0, "bulk destinations 16-byte aligned");
};

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 4) gdn_state_stream_kernel(const VerifyParams p) {
  using L = StreamLayout<DK>;
  extern __shared__ __align__(128) float sm[];
  float* sS0 = sm + L::OFF_S0;
  float* sWT = sm + L::OFF_WT;
  float* sKn = sm + L::OFF_KN;
  float* sGate = sm + L::OFF_GATE;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int K = p.K;
  const int b = blockIdx.y;
  constexpr int kTiles = DV / kRows;
  const int h = blockIdx.x / kTiles;
  const int r0 = (blockIdx.x % kTiles) * kRows;
  const int kh = h / (p.Hv / p.Hk);
  const size_t tile_off = ((size_t(b) * p.Hv + h) * DV + r0) * DK;
  float* sV = sm + L::OFF_V + warp * kKMax * kRowsPerWarp;
  float* sU = sm + L::OFF_U + warp * kKMax * kRowsPerWarp;

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, L::S0_BYTES + L::WT_BYTES + L::KN_BYTES + L::GATE_BYTES);
    bulk_load(sS0, p.state_in + tile_off, L::S0_BYTES, bar);
    griddep_wait();  // the prologue grid has finished and its tables are visible
    const size_t head = size_t(b) * p.Hk + kh;
    bulk_load(sWT, p.ws.wt + head * DK * kNCol, L::WT_BYTES, bar);
    bulk_load(sKn, p.ws.kn + head * kKMax * DK, L::KN_BYTES, bar);
    bulk_load(sGate, p.ws.gate + (size_t(b) * p.Hv + h) * kGateFloats, L::GATE_BYTES, bar);
  }

  // a1 for this CTA's v-channels: lanes 4..7 of warp w convolve rows 4w..4w+3
  if (lane >= 4 && lane < 4 + kRowsPerWarp) {
    const int i = warp * kRowsPerWarp + (lane - 4);
    float y[kKMax];
    conv_channel(p, b, 2 * p.Hk * DK + h * DV + r0 + i, y);
#pragma unroll
    for (int t = 0; t < kKMax; ++t) sV[t * kRowsPerWarp + (lane - 4)] = y[t];
  }
  __syncwarp();

  // S0 and the tables must have landed (bounded wait, warp-uniform outcome)
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, 0) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) {
    if (lane == 0) atomicOr(p.err, kDevErrTimeout);
    return;
  }
  (void)mbar_try_wait(bar, 0);  // every lane observes the completed phase

  const float* gM = sGate;
  const float* gN = sGate + kGateOffN;
  const float* gBeta = sGate + kGateOffBeta;
  const float* gG = sGate + kGateOffG;
  const float* gGam = sGate + kGateOffGam;
  float* sP = sm + L::OFF_P;
  const int row0 = warp * kRowsPerWarp;

  // P = S0 [k^ | q^] for this warp's rows, lane = column
  {
    float acc[kRowsPerWarp];
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) acc[m] = 0.f;
#pragma unroll 4
    for (int c = 0; c < DK; c += 4) {
      float wv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) wv[q] = sWT[wt_idx(c + q, lane)];
#pragma unroll
      for (int m = 0; m < kRowsPerWarp; ++m) {
        const float4 s = *reinterpret_cast<const float4*>(sS0 + (row0 + m) * DK + c);
        acc[m] = fmaf(s.x, wv[0], fmaf(s.y, wv[1], fmaf(s.z, wv[2], fmaf(s.w, wv[3], acc[m]))));
      }
    }
#pragma unroll
    for (int m = 0; m < kRowsPerWarp; ++m) sP[(row0 + m) * L::PSTRIDE + lane] = acc[m];
  }
  __syncwarp();

  // forward substitution for u, lanes 0..3 (one row each)
  if (lane < kRowsPerWarp) {
    const float* P = sP + (row0 + lane) * L::PSTRIDE;
    float u[kKMax];
#pragma unroll
    for (int t = 0; t < kKMax; ++t) {
      u[t] = 0.f;
      if (t < K) {
        float acc = fmaf(-gGam[t], P[t], sV[t * kRowsPerWarp + lane]);
#pragma unroll
        for (int j = 0; j < t; ++j) acc = fmaf(-gM[t * kMStride + j], u[j], acc);
        u[t] = gBeta[t] * acc;
        sU[t * kRowsPerWarp + lane] = u[t];
      }
    }
  }
  __syncwarp();

  // outputs: lane -> (row m = lane / 8, tokens t0 and t0 + 8)
  {
    const int m = lane >> 3;
    const float* P = sP + (row0 + m) * L::PSTRIDE;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int t = (lane & 7) + 8 * half;
      if (t < K) {
        float o = p.q_scale * gGam[t] * P[kKMax + t];
        for (int j = 0; j <= t; ++j) o = fmaf(gN[t * kMStride + j], sU[j * kRowsPerWarp + m], o);
        const size_t oi = (size_t(b) * K + t) * p.Hv * DV + size_t(h) * DV + r0 + row0 + m;
        if (p.out_f32)
          static_cast<float*>(p.out)[oi] = o;
        else
          static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16(o);
      }
    }
  }

  // stream the K states from registers: lane owns DK/32 float4 of the warp's 4 rows
  constexpr int F4 = DK / 32;
  constexpr int C4 = DK / 4;
  int rowq[F4];
  float4 s[F4];
  const int c4 = lane % C4;
#pragma unroll
  for (int q = 0; q < F4; ++q) {
    const int f = lane + 32 * q;
    rowq[q] = f / C4;
    s[q] = *reinterpret_cast<const float4*>(sS0 + (row0 + rowq[q]) * DK + 4 * c4);
  }
  const size_t inter_stride = size_t(p.Hv) * DV * DK;
  const size_t my_off = size_t(row0) * DK + 4 * c4;
  const size_t head_tile_off = (size_t(h) * DV + r0) * DK;  // offset of this tile inside one token's states
  float* inter = p.state_inter ? p.state_inter + size_t(b) * (K - 1) * inter_stride + head_tile_off + my_off : nullptr;
  for (int t = 0; t < K; ++t) {
    const float g = gG[t];
    const float4 kv = *reinterpret_cast<const float4*>(sKn + t * DK + 4 * c4);
    float* dst = (t == K - 1) ? p.state_out + tile_off + my_off : inter + size_t(t) * inter_stride;
#pragma unroll
    for (int q = 0; q < F4; ++q) {
      const float u = sU[t * kRowsPerWarp + rowq[q]];
      s[q].x = fmaf(u, kv.x, g * s[q].x);
      s[q].y = fmaf(u, kv.y, g * s[q].y);
      s[q].z = fmaf(u, kv.z, g * s[q].z);
      s[q].w = fmaf(u, kv.w, g * s[q].w);
      float4* d4 = reinterpret_cast<float4*>(dst + size_t(rowq[q]) * DK);
      if (t == K - 1)
        *d4 = s[q];
      else
        __stcs(d4, s[q]);
    }
  }
}

template <int DK, int DV>
cudaError_t launch_t(const VerifyParams& p, cudaStream_t stream) {
  auto k1 = gdn_qk_prologue_kernel<DK>;
  auto k2 = gdn_state_stream_kernel<DK, DV>;
  const size_t b1 = PrologueLayout<DK>::BYTES;
  const size_t b2 = StreamLayout<DK>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, int(b1));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, int(b2));
  if (e != cudaSuccess) return e;
  k1<<<dim3(unsigned(p.Hk), unsigned(p.B), 1), kThreads, b1, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.Hv * (DV / kRows)), unsigned(p.B), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = b2;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k2, p);
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream) {
  if (p.dk == 128 && p.dv == 128) return launch_t<128, 128>(p, stream);
  if (p.dk == 128 && p.dv == 64) return launch_t<128, 64>(p, stream);
  if (p.dk == 64 && p.dv == 128) return launch_t<64, 128>(p, stream);
  if (p.dk == 64 && p.dv == 64) return launch_t<64, 64>(p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace gdn
