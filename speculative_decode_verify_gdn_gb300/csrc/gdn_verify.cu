// Fused verify step of one Gated DeltaNet layer on sm_103a: conv + SiLU, q|k L2 norm,
// raw gates and the chunkwise (WY) gated delta rule writing every intermediate state.
//
// Method (lucebox #637 "NVLink fix for PR625", commit list: fused conv step, single
// l2_norm over q|k, raw-gate gated_delta_net with head broadcast; review of
// ggml-cuda/gated_delta_net.cu line 404 for the gate formula; atlas #297, commit on the
// SSM/GDN verify kernels: a K=16 WY-chunkwise verify that writes the final state and
// all intermediates in one pass):
//
//   y_t  = SiLU(sum_j w[c][j] win[t+j][c])           per channel, win = [history; x]
//   q^,k^ = q / sqrt(|q|^2 + eps), k / sqrt(|k|^2 + eps)  per (token, q/k head)
//   beta = sigmoid(b), g = exp(softplus(a + dt_bias) * -exp(A_log))
//   S_t  = g_t S_{t-1} + u_t k^_t^T,  u_t = beta_t (v_t - g_t S_{t-1} k^_t)
//   o_t  = q_scale S_t q^_t
//
// Chunk (WY) form used here, exact in real arithmetic: with Gamma_t = prod_{m<=t} g_m and
// D[t][j] = prod_{j<m<=t} g_m,
//   u_t = beta_t (v_t - Gamma_t S0 k^_t - sum_{j<t} D[t][j] (k^_j . k^_t) u_j)
//   o_t = q_scale (Gamma_t S0 q^_t + sum_{j<=t} D[t][j] (k^_j . q^_t) u_j)
// so every row of S needs only S0 k^_t and S0 q^_t (one small product with S0) and a
// K x K forward substitution; the K states then stream out as S_t = g_t S_{t-1} + u_t k^_t^T
// with no reduction on the store path.  Decay ratios are running products of g (values in
// [0, 1]), never quotients of products, so they cannot overflow or divide underflowed values.
//
// Work decomposition.  One CTA owns a tile of R rows (v indices) of one v-head's state.
// The CTAs that read the same q/k head - r = Hv/Hk v-heads x dv/R row tiles - form one
// thread-block cluster.  Each channel of the conv slab is read and written by exactly one
// thread of the whole grid: a CTA convolves its own R v-channels and a 1/G slice of its
// q/k head's channels, and pushes the q/k results to every CTA of its cluster through
// distributed shared memory.  That makes the in-place history update (conv_state_out ==
// conv_state_in) race-free and does the q/k conv once per head instead of once per CTA.
//
// Data movement.  The R x dk tile of S0 arrives by one bulk async copy (TMA, linear mode)
// on an mbarrier while the conv runs; each of the K states leaves as one 16-32 KB bulk async
// store from a ring of three shared-memory stages, so the SM keeps several stores in flight
// while it computes the next state.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kStages = 3;
constexpr int kNCol = 2 * kKMax;  // columns of the normalised q/k table: k^ in [0,16), q^ in [16,32)

template <int DK, int DV, int R>
struct Layout {
  static constexpr int TILE = R * DK;  // floats in one state tile
  static constexpr int PSTRIDE = kNCol + 1;
  static constexpr int MSTRIDE = kKMax + 1;
  // float offsets into dynamic shared memory
  static constexpr int OFF_STAGE = 0;                          // [kStages][TILE]; stage 0 receives S0
  static constexpr int OFF_QK = OFF_STAGE + 1 * TILE;          // prologue only: raw q|k conv [2][kKMax][DK]
  static constexpr int OFF_WT = OFF_STAGE + 2 * TILE;          // prologue only: q^/k^ table [DK][kNCol], swizzled
  static constexpr int OFF_KN = OFF_STAGE + kStages * TILE;    // k^ token-major [kKMax][DK]
  static constexpr int OFF_V = OFF_KN + kKMax * DK;            // v conv outputs [kKMax][R]
  static constexpr int OFF_U = OFF_V + kKMax * R;              // u [kKMax][R]
  static constexpr int OFF_P = OFF_U + kKMax * R;              // S0 k^ | S0 q^  [R][PSTRIDE]
  static constexpr int OFF_M = OFF_P + R * PSTRIDE;            // D * (k^.k^), strictly lower
  static constexpr int OFF_N = OFF_M + kKMax * MSTRIDE;        // q_scale * D * (k^.q^), lower
  static constexpr int OFF_D = OFF_N + kKMax * MSTRIDE;        // decay products D[t][j]
  static constexpr int OFF_GATE = OFF_D + kKMax * MSTRIDE;     // beta, g, Gamma (kKMax each), flag
  static constexpr int OFF_BAR = (OFF_GATE + 3 * kKMax + 4 + 1) & ~1;  // 8-byte aligned mbarrier
  static constexpr int FLOATS = OFF_BAR + 2;
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
  static_assert(2 * kKMax * DK <= TILE, "raw q|k staging must fit in one stage");
  static_assert(DK * kNCol <= TILE, "q/k table must fit in one stage");
  static_assert((TILE * 4) % 16 == 0, "bulk copies move multiples of 16 bytes");
  static_assert((TILE / 4) % kThreads == 0, "each thread owns whole float4s of the tile");
  static_assert(kThreads % (DK / 4) == 0, "a thread's float4 column is the same for every row it owns");
  static_assert(R % kWarps == 0 && R <= kThreads, "row split of the S0 products");
  static_assert(BYTES <= 227 * 1024, "shared memory per CTA");
};

// Index of q^/k^ column `col` of channel `c` in the swizzled table (conflict-free both ways).
__device__ __forceinline__ int wt_idx(int c, int col) { return c * kNCol + (col ^ (c & 31)); }

template <int DK, int DV, int R>
__global__ void __launch_bounds__(kThreads, 2) gdn_verify_kernel(const VerifyParams p) {
  using L = Layout<DK, DV, R>;
  extern __shared__ __align__(128) float sm[];
  float* stage = sm + L::OFF_STAGE;
  float* sQK = sm + L::OFF_QK;
  float* sWT = sm + L::OFF_WT;
  float* sKn = sm + L::OFF_KN;
  float* sV = sm + L::OFF_V;
  float* sU = sm + L::OFF_U;
  float* sP = sm + L::OFF_P;
  float* sM = sm + L::OFF_M;
  float* sN = sm + L::OFF_N;
  float* sD = sm + L::OFF_D;
  float* sBeta = sm + L::OFF_GATE;
  float* sG = sBeta + kKMax;
  float* sGam = sG + kKMax;
  int* sFlag = reinterpret_cast<int*>(sGam + kKMax);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int K = p.K;
  const int C = p.C;
  const int b = blockIdx.y;
  const int r = p.Hv / p.Hk;
  constexpr int kTiles = DV / R;
  const int G = r * kTiles;                 // cluster size
  const int rank = static_cast<int>(cluster_ctarank());
  const int kh = blockIdx.x / G;            // q/k head of this cluster
  const int h = kh * r + rank / kTiles;     // v head of this CTA
  const int r0 = (rank % kTiles) * R;       // first state row of this CTA
  const size_t tile_off = ((size_t(b) * p.Hv + h) * DV + r0) * DK;

  // ---- S0 tile: one bulk async copy, overlapped with the conv below
  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
    mbar_arrive_expect_tx(bar, L::TILE * 4);
    bulk_load(stage, p.state_in + tile_off, L::TILE * 4, bar);
  }
  cluster_arrive_relaxed();  // this CTA runs: peers may write its shared memory after their wait

  // ---- a1: conv over the channels this CTA owns
  const int qk_slice = (2 * DK + G - 1) / G;
  const int qk_lo = rank * qk_slice;
  const int n_qk = max(0, min(2 * DK, qk_lo + qk_slice) - qk_lo);
  const bool is_v = tid < R;
  const bool is_qk = tid >= R && tid < R + n_qk;
  float yqk[kKMax];
  if (is_v || is_qk) {
    int c;
    if (is_v) {
      c = 2 * p.Hk * DK + h * DV + r0 + tid;
    } else {
      const int cc = qk_lo + (tid - R);
      c = (cc < DK) ? kh * DK + cc : p.Hk * DK + kh * DK + (cc - DK);
    }
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
      if (t < K) {
        const float z = fmaf(w.w, xv[t], fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0)));
        const float y = silu(z);
        h0 = h1;
        h1 = h2;
        h2 = xv[t];
        if (ci) {
          ci[size_t(3 * t + 0) * C] = h0;
          ci[size_t(3 * t + 1) * C] = h1;
          ci[size_t(3 * t + 2) * C] = h2;
        }
        if (is_v) sV[t * R + tid] = y;
        yqk[t] = y;
      }
    }
    float* hout = p.conv_state_out + size_t(b) * 3 * C + c;
    hout[0] = h0;
    hout[C] = h1;
    hout[2 * C] = h2;
  }

  // ---- a3: raw gates of head h (last warp; it owns no conv channel)
  if (warp == kWarps - 1 && lane < kKMax) {
    float beta = 0.f, g = 1.f;
    if (lane < K) {
      const float A = -expf(p.A_log[h]);
      const size_t gi = (size_t(b) * K + lane) * p.Hv + h;
      const float av = bf16_to_f32(p.a[gi]) + p.dt_bias[h];
      const float sp = (av > 20.f) ? av : log1pf(expf(av));
      g = expf(sp * A);
      beta = 1.f / (1.f + expf(-bf16_to_f32(p.b[gi])));
    }
    sBeta[lane] = beta;
    sG[lane] = g;
  }

  cluster_wait_acquire();  // every CTA of the cluster has started
  if (is_qk) {
    const int cc = qk_lo + (tid - R);
    const uint32_t local = smem_addr(sQK + (cc / DK) * kKMax * DK + (cc % DK));
    for (int d = 0; d < G; ++d) {
      const uint32_t remote = map_to_rank(local, d);
#pragma unroll
      for (int t = 0; t < kKMax; ++t)
        if (t < K) st_cluster_f32(remote + t * DK * 4, yqk[t]);
    }
  }
  cluster_arrive_release();
  cluster_wait_acquire();  // all q|k conv outputs of this head are in sQK; no DSMEM access after this

  // ---- a2: L2 norm of q_t and k_t; build the swizzled table and the token-major k^
  for (int n = warp; n < kNCol; n += kWarps) {
    const int part = n / kKMax;  // 0: q, 1: k
    const int t = n % kKMax;
    const int col = part ? t : kKMax + t;
    float vals[DK / 32];
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < DK / 32; ++m) {
      vals[m] = (t < K) ? sQK[(part * kKMax + t) * DK + lane + 32 * m] : 0.f;
      ss = fmaf(vals[m], vals[m], ss);
    }
    ss = warp_sum(ss);
    const float inv = (t < K) ? 1.f / sqrtf(ss + p.l2_eps) : 0.f;
#pragma unroll
    for (int m = 0; m < DK / 32; ++m) {
      const int c = lane + 32 * m;
      const float v = vals[m] * inv;
      sWT[wt_idx(c, col)] = v;
      if (part == 1) sKn[t * DK + c] = v;
    }
  }
  // decay products D[t][j] = prod_{j<m<=t} g_m and Gamma_t = prod_{m<=t} g_m
  {
    const int t = tid >> 4, j = tid & 15;
    float d = 1.f;
    for (int m = j + 1; m <= t; ++m) d *= sG[m];
    sD[t * L::MSTRIDE + j] = (j <= t) ? d : 0.f;
    if (j == 0) sGam[t] = d * sG[0];
  }
  __syncthreads();

  // ---- Gram products of the window, scaled by the decay products
  {
    const int t = tid >> 4, j = tid & 15;
    float kk = 0.f, kq = 0.f;
#pragma unroll 8
    for (int c = 0; c < DK; ++c) {
      const float kj = sWT[wt_idx(c, j)];
      kk = fmaf(sWT[wt_idx(c, t)], kj, kk);
      kq = fmaf(sWT[wt_idx(c, kKMax + t)], kj, kq);
    }
    const float d = sD[t * L::MSTRIDE + j];
    sM[t * L::MSTRIDE + j] = (j < t) ? d * kk : 0.f;
    sN[t * L::MSTRIDE + j] = (j <= t) ? p.q_scale * d * kq : 0.f;
  }

  // ---- S0 must have landed
  if (tid == 0) {
    bool ok = mbar_wait_bounded(bar, 0);
    if (!ok) {
      atomicOr(p.err, kDevErrTimeout);
      mbar_wait_bounded(bar, 0);  // give the copy one more bounded chance to drain before exit
    }
    *sFlag = ok ? 0 : 1;
  }
  __syncthreads();
  if (*sFlag) return;  // uniform; no cluster traffic and no stores issued yet
  (void)mbar_try_wait(bar, 0);  // each thread observes the completed phase

  // ---- P = S0 [k^ | q^]: warp w owns rows w, w+8, ..., lane = column
  {
    constexpr int RPW = R / kWarps;
    float acc[RPW];
#pragma unroll
    for (int m = 0; m < RPW; ++m) acc[m] = 0.f;
#pragma unroll 2
    for (int c = 0; c < DK; c += 4) {
      float wv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) wv[q] = sWT[wt_idx(c + q, lane)];
#pragma unroll
      for (int m = 0; m < RPW; ++m) {
        const float4 s = *reinterpret_cast<const float4*>(stage + (warp + kWarps * m) * DK + c);
        acc[m] = fmaf(s.x, wv[0], fmaf(s.y, wv[1], fmaf(s.z, wv[2], fmaf(s.w, wv[3], acc[m]))));
      }
    }
#pragma unroll
    for (int m = 0; m < RPW; ++m) sP[(warp + kWarps * m) * L::PSTRIDE + lane] = acc[m];
  }
  __syncthreads();

  // ---- forward substitution for u and the outputs, one thread per row
  if (tid < R) {
    const int i = tid;
    float u[kKMax];
#pragma unroll
    for (int t = 0; t < kKMax; ++t) {
      u[t] = 0.f;
      if (t < K) {
        float acc = fmaf(-sGam[t], sP[i * L::PSTRIDE + t], sV[t * R + i]);
#pragma unroll
        for (int j = 0; j < t; ++j) acc = fmaf(-sM[t * L::MSTRIDE + j], u[j], acc);
        u[t] = sBeta[t] * acc;
        sU[t * R + i] = u[t];
      }
    }
#pragma unroll
    for (int t = 0; t < kKMax; ++t) {
      if (t < K) {
        float o = p.q_scale * sGam[t] * sP[i * L::PSTRIDE + kKMax + t];
#pragma unroll
        for (int j = 0; j <= t; ++j) o = fmaf(sN[t * L::MSTRIDE + j], u[j], o);
        const size_t oi = (size_t(b) * K + t) * p.Hv * DV + size_t(h) * DV + r0 + i;
        if (p.out_f32)
          static_cast<float*>(p.out)[oi] = o;
        else
          static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16(o);
      }
    }
  }
  __syncthreads();

  // ---- stream the K states: S_t = g_t S_{t-1} + u_t k^_t^T, one bulk store per state
  constexpr int F4 = L::TILE / 4 / kThreads;  // float4s per thread
  constexpr int C4 = DK / 4;                  // float4s per row
  float4 s[F4];
#pragma unroll
  for (int m = 0; m < F4; ++m) s[m] = reinterpret_cast<const float4*>(stage)[tid + kThreads * m];
  const int c4 = tid % C4;
  const size_t inter_stride = size_t(p.Hv) * DV * DK;  // one window token of state_inter
  float* inter_base = p.state_inter ? p.state_inter + size_t(b) * (K - 1) * inter_stride + size_t(h) * DV * DK +
                                          size_t(r0) * DK
                                    : nullptr;
  for (int t = 0; t < K; ++t) {
    float4* buf = reinterpret_cast<float4*>(stage + (t % kStages) * L::TILE);
    const float g = sG[t];
    const float4 kv = reinterpret_cast<const float4*>(sKn + t * DK)[c4];
#pragma unroll
    for (int m = 0; m < F4; ++m) {
      const float u = sU[t * R + (tid + kThreads * m) / C4];
      s[m].x = fmaf(u, kv.x, g * s[m].x);
      s[m].y = fmaf(u, kv.y, g * s[m].y);
      s[m].z = fmaf(u, kv.z, g * s[m].z);
      s[m].w = fmaf(u, kv.w, g * s[m].w);
      buf[tid + kThreads * m] = s[m];
    }
    fence_proxy_async_smem();
    // the stage written in the next iteration was last read by store t+1-kStages
    if (tid == 0) bulk_wait_read<kStages - 2>();
    __syncthreads();
    if (tid == 0) {
      float* dst = (t == K - 1) ? p.state_out + tile_off : inter_base + size_t(t) * inter_stride;
      bulk_store(dst, buf, L::TILE * 4);
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait_all<0>();
}

template <int DK, int DV, int R>
cudaError_t launch_t(const VerifyParams& p, cudaStream_t stream) {
  using L = Layout<DK, DV, R>;
  auto kern = gdn_verify_kernel<DK, DV, R>;
  const int r = p.Hv / p.Hk;
  const int G = r * (DV / R);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, int(L::BYTES));
  if (e != cudaSuccess) return e;
  if (G > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.Hk * G), unsigned(p.B), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::BYTES;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(G);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

int verify_row_tile(int dv, int r) {
  if (r * (dv / 32) <= 8) return 32;
  if (dv >= 64 && r * (dv / 64) <= 16) return 64;
  return 0;
}

int verify_cluster_size(int dv, int r) {
  const int R = verify_row_tile(dv, r);
  return R ? r * (dv / R) : 0;
}

size_t verify_smem_bytes(int dk, int dv, int r) {
  const int R = verify_row_tile(dv, r);
#define GDN_SMEM_CASE(DK_, DV_, R_) \
  if (dk == DK_ && dv == DV_ && R == R_) return Layout<DK_, DV_, R_>::BYTES;
  GDN_SMEM_CASE(64, 64, 32)
  GDN_SMEM_CASE(64, 64, 64)
  GDN_SMEM_CASE(64, 128, 32)
  GDN_SMEM_CASE(64, 128, 64)
  GDN_SMEM_CASE(128, 64, 32)
  GDN_SMEM_CASE(128, 64, 64)
  GDN_SMEM_CASE(128, 128, 32)
  GDN_SMEM_CASE(128, 128, 64)
#undef GDN_SMEM_CASE
  return 0;
}

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream) {
  const int R = verify_row_tile(p.dv, p.Hv / p.Hk);
#define GDN_LAUNCH_CASE(DK_, DV_, R_) \
  if (p.dk == DK_ && p.dv == DV_ && R == R_) return launch_t<DK_, DV_, R_>(p, stream);
  GDN_LAUNCH_CASE(64, 64, 32)
  GDN_LAUNCH_CASE(64, 64, 64)
  GDN_LAUNCH_CASE(64, 128, 32)
  GDN_LAUNCH_CASE(64, 128, 64)
  GDN_LAUNCH_CASE(128, 64, 32)
  GDN_LAUNCH_CASE(128, 64, 64)
  GDN_LAUNCH_CASE(128, 128, 32)
  GDN_LAUNCH_CASE(128, 128, 64)
#undef GDN_LAUNCH_CASE
  return cudaErrorInvalidValue;
}

}  // namespace gdn
