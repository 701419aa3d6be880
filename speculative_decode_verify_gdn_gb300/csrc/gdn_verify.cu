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
//     products and decay products.  Writes small per-head tables to the workspace, laid out as
//     the second kernel keeps them in shared memory.
//  2. state_stream: one CTA per (sequence, v-head, 32-row tile of the state), launched with
//     programmatic dependent launch so that it starts while the prologue runs: it issues the
//     bulk async (TMA) copy of its 16 KB S0 tile and convolves its own 32 v-channels first, then
//     waits for the prologue grid and bulk-copies the tables.  From there each warp owns four
//     state rows and needs no further CTA-wide barrier: products with S0, forward substitution,
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

// Columns 4j .. 4j+3 of row c of the swizzled [DK][32] q^/k^ table (element (c, col) at
// c * 32 + (col ^ (c & 31))) in plain order: one 16-byte load, whose swizzle only permutes the four
// (logical column 4j + i sits at (4j ^ (s & ~3)) + (i ^ (s & 3)) with s = c & 31).
__device__ __forceinline__ float4 unswizzled4(const float* sT, int c, int j) {
  const int x = c & 3;
  float4 v = *reinterpret_cast<const float4*>(sT + c * kNCol + ((4 * j) ^ (c & 28)));
  if (x & 1) v = make_float4(v.y, v.x, v.w, v.z);
  if (x & 2) v = make_float4(v.z, v.w, v.x, v.y);
  return v;
}

// Accepted length of the previous window for sequence b, or -1 for a plain verify step (no
// rollback applied on read).  Lengths outside 0..K, and 0 without a snapshot, read as K (the
// previous final state) after flagging the device status word.
__device__ __forceinline__ int prev_accept(const VerifyParams& p, int b, bool report) {
  if (!p.accept_prev) return -1;
  const int L = p.accept_prev[b];
  if (L < 0 || L > p.K) {
    if (report) atomicOr(p.err, kDevErrAcceptRange);
    return p.K;
  }
  if (L == 0 && !p.state_snap_prev) {
    if (report) atomicOr(p.err, kDevErrNoSnapshot);
    return p.K;
  }
  return L;
}

// Where channel c's history before this window starts, [3] rows C apart.
__device__ __forceinline__ const float* history_src(const VerifyParams& p, int b, int c, int L) {
  const int C = p.C;
  if (L < 0 || L == p.K) return p.conv_state_in + size_t(b) * 3 * C + c;
  if (L == 0) return p.conv_snap_prev + size_t(b) * 3 * C + c;
  return p.conv_inter_prev + (size_t(b) * p.K + (L - 1)) * 3 * C + c;
}

// Token-tree window (gdn_verify_tree): per node t its parent, the three window rows before x_t
// as indices into [history row 0, 1, 2, x_0 .. x_{K-1}], and the bit set of the nodes on its
// root-to-node path.  Built by one thread; a parent outside -1..t-1 reads as -1 and is flagged.
struct TreeTable {
  int parent[kKMax];
  int src[kKMax][3];
  unsigned path[kKMax];
};

__device__ __forceinline__ void build_tree(const VerifyParams& p, int b, TreeTable* tt, bool report) {
  int pr[kKMax];  // every parent index in flight at once, before the table is written
#pragma unroll
  for (int t = 0; t < kKMax; ++t) pr[t] = (t < p.K) ? p.parent[size_t(b) * p.K + t] : -1;
#pragma unroll
  for (int t = 0; t < kKMax; ++t) {
    if (t >= p.K) break;
    int par = pr[t];
    if (par < -1 || par >= t) {
      if (report) atomicOr(p.err, kDevErrTreeParent);
      par = -1;
    }
    tt->parent[t] = par;
    if (par < 0) {
      tt->src[t][0] = 0;
      tt->src[t][1] = 1;
      tt->src[t][2] = 2;
      tt->path[t] = 1u << t;
    } else {
      tt->src[t][0] = tt->src[par][1];
      tt->src[t][1] = tt->src[par][2];
      tt->src[t][2] = 3 + par;
      tt->path[t] = tt->path[par] | (1u << t);
    }
  }
}

// Conv + SiLU of one channel over the window (a chain of K tokens, or a token tree when kTree);
// writes the channel's K history snapshots and its new history (that after token / node K-1).
// y[t] receives the outputs for t < K.  A token tree reads each node's window through the
// table's indices: the three history values from registers, x_t from `scratch[t * sstride]`
// (16 floats of shared memory per thread; a register array indexed at run time would live in
// local memory).
template <bool kTree>
__device__ __forceinline__ void conv_channel(const VerifyParams& p, int b, int c, const TreeTable* tt,
                                             float (&y)[kKMax], float* scratch = nullptr, int sstride = 1) {
  if constexpr (kTree) {
    const int C = p.C;
    const int K = p.K;
    const float4 w = *reinterpret_cast<const float4*>(p.conv_w + size_t(c) * kConvW);
    const float* hin = p.conv_state_in + size_t(b) * 3 * C + c;
    const float hv0 = hin[0], hv1 = hin[C], hv2 = hin[2 * C];
    const uint16_t* xp = p.x + size_t(b) * K * C + c;
#pragma unroll
    for (int t = 0; t < kKMax; ++t) scratch[t * sstride] = (t < K) ? bf16_to_f32(xp[size_t(t) * C]) : 0.f;
    // value `idx` of [history rows 0, 1, 2, x_0 .. x_{K-1}]
    auto val = [&](int idx) { return idx < 3 ? (idx == 0 ? hv0 : (idx == 1 ? hv1 : hv2)) : scratch[(idx - 3) * sstride]; };
    float* ci = p.conv_inter ? p.conv_inter + size_t(b) * K * 3 * C + c : nullptr;
    float n0 = 0.f, n1 = 0.f, n2 = 0.f;
#pragma unroll
    for (int t = 0; t < kKMax; ++t) {
      y[t] = 0.f;
      if (t < K) {
        const float w0 = val(tt->src[t][0]), w1 = val(tt->src[t][1]), w2 = val(tt->src[t][2]);
        const float xt = scratch[t * sstride];
        y[t] = silu(fmaf(w.w, xt, fmaf(w.z, w2, fmaf(w.y, w1, w.x * w0))));
        n0 = w1;
        n1 = w2;
        n2 = xt;
        if (ci) {
          ci[size_t(3 * t + 0) * C] = n0;
          ci[size_t(3 * t + 1) * C] = n1;
          ci[size_t(3 * t + 2) * C] = n2;
        }
      }
    }
    float* hout = p.conv_state_out + size_t(b) * 3 * C + c;
    hout[0] = n0;
    hout[C] = n1;
    hout[2 * C] = n2;
    return;
  }
  (void)tt;
  (void)scratch;
  (void)sstride;
  const int C = p.C;
  const int K = p.K;
  const float4 w = *reinterpret_cast<const float4*>(p.conv_w + size_t(c) * kConvW);
  const float* hin = history_src(p, b, c, prev_accept(p, b, false));
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

// Conv + SiLU of the two adjacent channels c, c + 1 (c even) over a chain window: one 4-byte load
// per token for both x values, 8-byte history, snapshot and history stores.  The outputs go to
// dst[t * ystride], dst[t * ystride + 1] (shared memory) for t < K, zero for K <= t < 16.
__device__ __forceinline__ void conv_channel_pair(const VerifyParams& p, int b, int c, float* dst, int ystride) {
  const int C = p.C;
  const int K = p.K;
  const float4 wa = *reinterpret_cast<const float4*>(p.conv_w + size_t(c) * kConvW);
  const float4 wb = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 1) * kConvW);
  const float* hin = history_src(p, b, c, prev_accept(p, b, false));
  float2 h0 = *reinterpret_cast<const float2*>(hin);
  float2 h1 = *reinterpret_cast<const float2*>(hin + C);
  float2 h2 = *reinterpret_cast<const float2*>(hin + 2 * C);
  const uint32_t* xp = reinterpret_cast<const uint32_t*>(p.x + size_t(b) * K * C + c);
  uint32_t xv[kKMax];
#pragma unroll
  for (int t = 0; t < kKMax; ++t) xv[t] = (t < K) ? xp[size_t(t) * (C / 2)] : 0u;
  float2* ci = p.conv_inter ? reinterpret_cast<float2*>(p.conv_inter + size_t(b) * K * 3 * C + c) : nullptr;
  const size_t row2 = size_t(C) / 2;  // one history row, in float2
#pragma unroll
  for (int t = 0; t < kKMax; ++t) {
    float2 y = make_float2(0.f, 0.f);
    if (t < K) {
      const float x0 = bf16_to_f32(uint16_t(xv[t] & 0xFFFFu)), x1 = bf16_to_f32(uint16_t(xv[t] >> 16));
      y.x = silu(fmaf(wa.w, x0, fmaf(wa.z, h2.x, fmaf(wa.y, h1.x, wa.x * h0.x))));
      y.y = silu(fmaf(wb.w, x1, fmaf(wb.z, h2.y, fmaf(wb.y, h1.y, wb.x * h0.y))));
      h0 = h1;
      h1 = h2;
      h2 = make_float2(x0, x1);
      if (ci) {
        ci[(3 * t + 0) * row2] = h0;
        ci[(3 * t + 1) * row2] = h1;
        ci[(3 * t + 2) * row2] = h2;
      }
    }
    *reinterpret_cast<float2*>(dst + t * ystride) = y;
  }
  float2* hout = reinterpret_cast<float2*>(p.conv_state_out + size_t(b) * 3 * C + c);
  hout[0] = h0;
  hout[row2] = h1;
  hout[2 * row2] = h2;
}

// a3 for one (v-head, token): beta = sigmoid(b), g = exp(softplus(a + dt_bias) * -exp(A_log)) with
// the softplus clipped to the identity above 20.
__device__ __forceinline__ void raw_gate(float a, float b, float A_log, float dt_bias, float& beta, float& g) {
  const float A = -expf(A_log);
  const float av = a + dt_bias;
  const float sp = (av > 20.f) ? av : log1pf(expf(av));
  g = expf(sp * A);
  beta = 1.f / (1.f + expf(-b));
}

// a2 over the 2K q|k vectors of one q/k head, raw conv outputs in sY[32][ys] (k rows 0..15, q rows
// 16..31): warp per vector, rows t >= K become zero.  Normalised values go to the swizzled
// [DK][32] table sT and, for the k rows, token-major to kn[16][DK]; 1 / norm to sInv[32].
template <int DK>
__device__ __forceinline__ void qk_norms(const float* sY, int ys, float* sT, float* sInv, float* kn, int K,
                                         float eps, int warp, int lane) {
  for (int n = warp; n < kNCol; n += kWarps) {
    const int t = n % kKMax;
    float vals[DK / 32];
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < DK / 32; ++m) {
      vals[m] = sY[n * ys + lane + 32 * m];
      ss = fmaf(vals[m], vals[m], ss);
    }
    ss = warp_sum(ss);
    const float inv = (t < K) ? rsqrtf(ss + eps) : 0.f;
    if (lane == 0) sInv[n] = inv;
#pragma unroll
    for (int m = 0; m < DK / 32; ++m) {
      const int c = lane + 32 * m;
      sT[c * kNCol + (n ^ (c & 31))] = vals[m] * inv;
      if (n < kKMax) kn[t * DK + c] = vals[m] * inv;
    }
  }
}

// Gram products from the raw rows: thread (n, j) takes row n of [k; q] against k rows j and j + 8
// (a warp reads four n rows and sixteen k rows, all four banks apart when ys = DK + 4), paired f32
// FMAs.  qk_gram_raw returns the two unscaled sums; qk_gram_store scales them by the two inverse
// norms into KK[t][j] = k^_t . k^_j and KQ[t][j] = k^_j . q^_t.
template <int DK>
__device__ __forceinline__ float2 qk_gram_raw(const float* sY, int ys, int tid) {
  const int n = tid >> 3, j = tid & 7;
  const float* yn = sY + n * ys;
  const float* ya = sY + j * ys;
  const float* yb = sY + (j + 8) * ys;
  float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll 8
  for (int c = 0; c < DK; c += 4) {
    const float4 x = *reinterpret_cast<const float4*>(yn + c);
    const float4 u = *reinterpret_cast<const float4*>(ya + c);
    const float4 v = *reinterpret_cast<const float4*>(yb + c);
    a0 = __ffma2_rn(make_float2(x.x, x.y), make_float2(u.x, u.y), a0);
    a0 = __ffma2_rn(make_float2(x.z, x.w), make_float2(u.z, u.w), a0);
    a1 = __ffma2_rn(make_float2(x.x, x.y), make_float2(v.x, v.y), a1);
    a1 = __ffma2_rn(make_float2(x.z, x.w), make_float2(v.z, v.w), a1);
  }
  return make_float2(a0.x + a0.y, a1.x + a1.y);
}

__device__ __forceinline__ void qk_gram_store(float2 raw, const float* sInv, float* sKK, float* sKQ, int tid) {
  const int n = tid >> 3, j = tid & 7;
  const float sn = sInv[n];
  float* dst = (n < kKMax) ? sKK + n * kMStride : sKQ + (n - kKMax) * kMStride;
  dst[j] = raw.x * sn * sInv[j];
  dst[j + 8] = raw.y * sn * sInv[j + 8];
}

// One v-head's gate block, thread (t, j) = (tid / 16, tid % 16) of 256: M = D o (k^.k^) strictly
// lower, N = q_scale D o (k^.q^) lower, Gamma, beta, g, with D[t][j] = prod_{j<m<=t} g_m as a
// masked product over registers (a token tree: over the path of t below j).  bg holds beta[16]
// then g[16]; kk, kq are this thread's Gram entries.
template <bool kTree>
__device__ __forceinline__ void gate_block(const VerifyParams& p, const TreeTable* tree, const float* bg, float kk,
                                           float kq, float* gate, int tid) {
  const int t = tid >> 4, j = tid & 15;
  float g[kKMax];
#pragma unroll
  for (int m = 0; m < kKMax; m += 4) {
    const float4 v = *reinterpret_cast<const float4*>(bg + kKMax + m);
    g[m] = v.x;
    g[m + 1] = v.y;
    g[m + 2] = v.z;
    g[m + 3] = v.w;
  }
  // chain: j < t are the earlier tokens and the path below j is j+1..t; tree: j must lie on t's
  // root-to-node path, and the nodes below it are t's path minus j's (same products, same order,
  // so a chain-shaped tree gives the chain's numbers bit for bit)
  bool below = j < t, on_path = j <= t;
  unsigned down = 0;
  int root = 0;
  if constexpr (kTree) {
    const unsigned pt = tree->path[t], pj = tree->path[j];
    on_path = j <= t && ((pt >> j) & 1u);
    below = on_path && j < t;
    down = pt & ~pj;
    root = __ffs(pt) - 1;
  }
  float d = 1.f;
#pragma unroll
  for (int m = 1; m < kKMax; ++m) {
    const bool in = kTree ? ((down >> m) & 1u) : (m > j && m <= t);
    d *= in ? g[m] : 1.f;
  }
  gate[t * kMStride + j] = below ? d * kk : 0.f;
  gate[kGateOffN + t * kMStride + j] = on_path ? p.q_scale * d * kq : 0.f;
  if (j == root) gate[kGateOffGam + t] = d * g[root];
  if (tid < kKMax) {
    gate[tid * kMStride + kKMax] = 0.f;
    gate[kGateOffN + tid * kMStride + kKMax] = 0.f;
    gate[kGateOffBeta + tid] = bg[tid];
    gate[kGateOffG + tid] = bg[kKMax + tid];
  }
  if (tid < kGateFloats - (kGateOffGam + kKMax)) gate[kGateOffGam + kKMax + tid] = 0.f;
}

// ------------------------------------------------------------------------------------------
// Kernel 1: per (sequence, q/k head) prologue.
template <int DK>
struct PrologueLayout {
  static constexpr int YS = DK + 4;                         // conv row stride: rows 4 banks apart
  static constexpr int OFF_Y = 0;                           // raw conv outputs [32][YS] (k: 0..15, q: 16..31)
  static constexpr int OFF_T = OFF_Y + kNCol * YS;          // normalised table [DK][32], swizzled
  static constexpr int OFF_INV = OFF_T + DK * kNCol;        // 1 / sqrt(|y_n|^2 + eps) [32]
  static constexpr int OFF_KK = OFF_INV + kNCol;            // k^_t . k^_j  [16][17]
  static constexpr int OFF_KQ = OFF_KK + kKMax * kMStride;  // k^_j . q^_t  [16][17]
  static constexpr int OFF_BG = OFF_KQ + kKMax * kMStride;  // beta, g of up to 16 v-heads [16][2][16]
  static constexpr int OFF_TREE = OFF_BG + 16 * 2 * kKMax;  // TreeTable (token trees only)
  static constexpr int FLOATS = OFF_TREE + int(sizeof(TreeTable) / 4);
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
  static_assert(OFF_T % 4 == 0 && OFF_BG % 4 == 0 && YS % 4 == 0, "float4 access");
};

template <int DK, bool kTree>
__global__ void __launch_bounds__(kThreads, 4) gdn_qk_prologue_kernel(const VerifyParams p) {
  using L = PrologueLayout<DK>;
  extern __shared__ __align__(128) float sm[];
  float* sY = sm + L::OFF_Y;
  float* sT = sm + L::OFF_T;
  float* sInv = sm + L::OFF_INV;
  float* sKK = sm + L::OFF_KK;
  float* sKQ = sm + L::OFF_KQ;
  float* sBG = sm + L::OFF_BG;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int kh = blockIdx.x;
  const int b = blockIdx.y;
  const int K = p.K;
  const int r = p.Hv / p.Hk;
  const size_t head = size_t(b) * p.Hk + kh;
  // a small grid leaves most SMs idle: the state kernel may start on them right away (its S0
  // copies and v-channel conv then overlap this kernel; it still waits for this grid to complete
  // before it reads the tables)
  if (p.early_dependents) griddep_launch_dependents();

  // a3 inputs of up to 16 v-heads (thread = (head, token)), loaded first so that their latency
  // overlaps the conv's loads; the gates are evaluated once the conv is done
  float ga = 0.f, gb = 0.f, gA = 0.f, gdt = 0.f;
  auto gate_load = [&](int hv0) {
    const int hv = hv0 + (tid >> 4), t = tid & 15;
    if (hv < r && t < K) {
      const int h = kh * r + hv;
      const size_t gi = (size_t(b) * K + t) * p.Hv + h;
      ga = bf16_to_f32(p.a[gi]);
      gb = bf16_to_f32(p.b[gi]);
      gA = p.A_log[h];
      gdt = p.dt_bias[h];
    }
  };
  auto gate_store = [&](int hv0) {
    const int hv = hv0 + (tid >> 4), t = tid & 15;
    if (hv < r) {
      float beta = 0.f, g = 1.f;
      if (t < K) raw_gate(ga, gb, gA, gdt, beta, g);
      sBG[(hv - hv0) * 2 * kKMax + t] = beta;
      sBG[(hv - hv0) * 2 * kKMax + kKMax + t] = g;
    }
  };
  gate_load(0);
  TreeTable* tree = reinterpret_cast<TreeTable*>(sm + L::OFF_TREE);
  if constexpr (kTree) {
    if (tid == 0) build_tree(p, b, tree, kh == 0);
    __syncthreads();
  }

  // a1: conv of the head's q|k channels (each channel's history, new history and snapshots have
  // one owner thread; the snapshot stores leave from registers while the memory system is
  // otherwise idle at the start of the step).  A chain window takes two adjacent channels per
  // thread, a token tree one (its windows are gathered through the tree table)
  if constexpr (kTree) {
    if (tid < 2 * DK) {
      const int cc = tid;
      const int c = (cc < DK) ? kh * DK + cc : p.Hk * DK + kh * DK + (cc - DK);
      float y[kKMax];
      static_assert(kKMax * 2 * DK <= DK * kNCol, "16 scratch floats per conv thread fit in the table");
      conv_channel<kTree>(p, b, c, tree, y, sT + cc, 2 * DK);  // (the table is written after the conv)
      const int n0 = (cc < DK) ? kKMax : 0;  // q rows 16..31, k rows 0..15
      const int col = cc % DK;
#pragma unroll
      for (int t = 0; t < kKMax; ++t) sY[(n0 + t) * L::YS + col] = y[t];
    }
  } else {
    if (tid < DK) {
      const int cc = 2 * tid;  // q channels 0..DK-1, then k channels (pairs never straddle them)
      const int c = (cc < DK) ? kh * DK + cc : p.Hk * DK + kh * DK + (cc - DK);
      const int n0 = (cc < DK) ? kKMax : 0;  // q rows 16..31, k rows 0..15
      conv_channel_pair(p, b, c, sY + n0 * L::YS + cc % DK, L::YS);
    }
  }
  __syncthreads();

  // the Gram products of the raw rows, then a2: the L2 norm of each of the 2K vectors, straight into
  // the swizzled table (and k^ token-major to the workspace, for the state updates), and a3 for up
  // to 16 v-heads, all in one phase (the Gram sums are scaled by the inverse norms after it)
  const float2 graw = qk_gram_raw<DK>(sY, L::YS, tid);
  qk_norms<DK>(sY, L::YS, sT, sInv, p.ws.kn + head * kKMax * DK, K, p.l2_eps, warp, lane);
  gate_store(0);
  __syncthreads();

  // the [DK][32] table of k^ (columns 0..15) and q^ (16..31) for the state kernel, in plain column
  // order
  {
    float* dst = p.ws.wt + head * DK * kNCol;
    for (int f4 = tid; f4 < DK * (kNCol / 4); f4 += kThreads) {
      const int c = f4 / (kNCol / 4), j = f4 % (kNCol / 4);
      *reinterpret_cast<float4*>(dst + c * kNCol + 4 * j) = unswizzled4(sT, c, j);
    }
  }

  qk_gram_store(graw, sInv, sKK, sKQ, tid);
  __syncthreads();

  // per-v-head gate blocks
  const float kk = sKK[(tid >> 4) * kMStride + (tid & 15)];
  const float kq = sKQ[(tid >> 4) * kMStride + (tid & 15)];
  for (int hv0 = 0; hv0 < r; hv0 += 16) {
    if (hv0 > 0) {
      __syncthreads();
      gate_load(hv0);
      gate_store(hv0);
      __syncthreads();
    }
    for (int hv = hv0; hv < min(r, hv0 + 16); ++hv)
      gate_block<kTree>(p, tree, sBG + (hv - hv0) * 2 * kKMax, kk, kq,
                        p.ws.gate + (size_t(b) * p.Hv + kh * r + hv) * kGateFloats, tid);
  }
  // on a large grid the state kernel's independent work (S0 copy, v-channel conv) starts as this
  // grid finishes: earlier starts only made the two grids contend for the SMs (measured)
  if (!p.early_dependents) griddep_launch_dependents();
}

// ------------------------------------------------------------------------------------------
// Kernel 2: per (sequence, v-head, 32-row tile) state stream.
template <int DK, bool kGated = false>
struct StreamLayout {
  static constexpr int PSTRIDE = kNCol + 4;                    // 16-byte rows
  static constexpr int RSTRIDE = kKMax + 1;
  static constexpr int SSTRIDE = DK + 4;                         // S0 rows 4 banks apart
  static constexpr int OFF_S0 = 0;                               // [32][SSTRIDE] bulk copy per row
  static constexpr int OFF_WT = OFF_S0 + kRows * SSTRIDE;        // [DK][32]      bulk copy
  static constexpr int OFF_GATE = OFF_WT + DK * kNCol;           // gate block    bulk copy
  static constexpr int OFF_KN = OFF_GATE + kGateFloats;          // [16][DK] k^ token-major, bulk copy
  static constexpr int OFF_V = OFF_KN + kKMax * DK;              // [warp][16][4] v conv outputs
  static constexpr int OFF_U = OFF_V + kWarps * kKMax * kRowsPerWarp;  // [warp][16][4] u
  static constexpr int OFF_P = OFF_U + kWarps * kKMax * kRowsPerWarp;  // [32][PSTRIDE] S0 [k^ | q^]
  static constexpr int OFF_R = OFF_P + kRows * PSTRIDE;                // [32][RSTRIDE] rhs, then o (gated)
  static constexpr int OFF_X = OFF_R + kRows * RSTRIDE;                // tree table or gated-norm block
  static constexpr int OFF_TREE = OFF_X;                                 // TreeTable (token trees only)
  static constexpr int OFF_SQ = OFF_X;  // gated: sums of o^2 [tile][warp][8] float2 (tokens c, c + 8)
  static constexpr int X_FLOATS = kGated ? 4 * kWarps * kKMax : int(sizeof(TreeTable) / 4);
  static constexpr int OFF_BAR = (OFF_X + X_FLOATS + 1) & ~1;            // 8-byte aligned mbarrier(s)
  static constexpr int FLOATS = OFF_BAR + (kGated ? 4 : 2);              // gated: + the exchange mbarrier
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
  static constexpr uint32_t S0_ROW_BYTES = DK * 4;
  static constexpr uint32_t S0_BYTES = kRows * S0_ROW_BYTES;
  static constexpr uint32_t WT_BYTES = DK * kNCol * 4;
  static constexpr uint32_t GATE_BYTES = kGateFloats * 4;
  static constexpr uint32_t KN_BYTES = kKMax * DK * 4;
  static_assert(OFF_SQ % 2 == 0, "gated exchange slots 8-byte aligned");
  static_assert(S0_ROW_BYTES % 16 == 0 && (SSTRIDE * 4) % 16 == 0 && WT_BYTES % 16 == 0 && GATE_BYTES % 16 == 0 && KN_BYTES % 16 == 0, "");
  static_assert(OFF_WT % 4 == 0 && OFF_GATE % 4 == 0 && OFF_KN % 4 == 0 && OFF_P % 4 == 0,
                "bulk destinations and float4 rows 16-byte aligned");
};

template <int DK, int DV, bool kTree, bool kGated>
__global__ void __launch_bounds__(kThreads, 4) gdn_state_stream_kernel(const VerifyParams p) {
  static_assert(!(kTree && kGated), "tree and gated-norm variants are separate");
  using L = StreamLayout<DK, kGated>;
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

  TreeTable* tree = reinterpret_cast<TreeTable*>(sm + L::OFF_TREE);
  // gated: the partial sums of o^2 of all kTiles CTAs of the head land on bar_sq (8 bytes from
  // each of 8 lanes of every warp of every CTA, own included)
  uint64_t* bar_sq = bar + 1;
  constexpr uint32_t kSqBytes = uint32_t(kTiles * kWarps * 8 * 8);
  if (tid == 0) {
    mbar_init(bar, 1);
    if constexpr (kGated) {
      mbar_init(bar_sq, 1);
      mbar_arrive_expect_tx(bar_sq, kSqBytes);
    }
    fence_mbar_init();
  }
  if constexpr (kGated) cluster_arrive_relaxed();  // this CTA runs: the head's peers may write its smem later
  __syncthreads();  // the barrier is ready before any thread uses it
  if (tid == 0) {
    mbar_arrive_expect_tx(bar, L::S0_BYTES + L::WT_BYTES + L::GATE_BYTES + L::KN_BYTES);
    griddep_wait();  // the prologue grid has finished and its tables are visible
    const size_t head = size_t(b) * p.Hk + kh;
    bulk_load(sWT, p.ws.wt + head * DK * kNCol, L::WT_BYTES, bar);
    bulk_load(sGate, p.ws.gate + (size_t(b) * p.Hv + h) * kGateFloats, L::GATE_BYTES, bar);
    bulk_load(sKn, p.ws.kn + head * kKMax * DK, L::KN_BYTES, bar);
  }
  if (warp == kWarps - 1) {
    // S0: the previous final state, or (rollback applied on read) the accepted intermediate or
    // the pre-window snapshot of the previous window; one row per lane, into rows padded by four
    // banks so that the four rows a warp reads together in the products below do not conflict.
    // (A warp of its own, so that the tables' copies above do not wait behind the load of the
    // accept length; the copies' bytes may land before the expected count is set, the phase
    // completing only with thread 0's arrival.)
    const int Lp = prev_accept(p, b, blockIdx.x == 0 && lane == 0);
    const float* s0 = p.state_in + tile_off;
    if (Lp == 0)
      s0 = p.state_snap_prev + tile_off;
    else if (Lp > 0 && Lp < K)
      s0 = p.state_inter_prev + (size_t(b) * (K - 1) + (Lp - 1)) * size_t(p.Hv) * DV * DK + (size_t(h) * DV + r0) * DK;
    bulk_load(sS0 + lane * L::SSTRIDE, s0 + size_t(lane) * DK, L::S0_ROW_BYTES, bar);
  }
  // gated: the lane's two z values of the epilogue, (token cg, row m of its warp) and eight tokens
  // later, and the row's norm weight, fetched now so that they have long arrived when used (the
  // lane map (m, cg) is the one of the outputs phase below)
  uint16_t z_a = 0, z_b = 0;
  float nw = 0.f;
  if constexpr (kGated) {
    const int t0 = lane & 7, i0 = warp * kRowsPerWarp + (lane >> 3);
    const uint16_t* zp = p.z + ((size_t(b) * K + t0) * p.Hv + h) * DV + r0 + i0;
    if (t0 < K) z_a = __ldg(zp);
    if (t0 + 8 < K) z_b = __ldg(zp + size_t(8) * p.Hv * DV);
    nw = __ldg(p.norm_w + r0 + i0);
  }
  if constexpr (kTree) {  // (off thread 0, and before it waits for the prologue grid)
    if (tid == 32) build_tree(p, b, tree, false);
    __syncthreads();  // the tree table is ready before the conv reads it
  }

  // a1 for this CTA's v-channels: lanes 4..7 of warp w convolve rows 4w..4w+3
  if (lane >= 4 && lane < 4 + kRowsPerWarp) {
    const int i = warp * kRowsPerWarp + (lane - 4);
    float y[kKMax];
    // (a token tree's window values go through this row of the P table, which the warp only
    // fills after the load wait)
    conv_channel<kTree>(p, b, 2 * p.Hk * DK + h * DV + r0 + i, tree, y, sm + L::OFF_P + i * L::PSTRIDE);
#pragma unroll
    for (int t = 0; t < kKMax; ++t) sV[t * kRowsPerWarp + (lane - 4)] = y[t];
  }

  __syncwarp();

  // S0 and the tables must have landed (bounded wait, warp-uniform outcome; no CTA-wide barrier
  // follows, so each warp proceeds on its own)
  int ok = 1;
  if (lane == 0) ok = mbar_wait_bounded(bar, 0) ? 1 : 0;
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) {
    if (lane == 0) {
      atomicOr(p.err, kDevErrTimeout);
      (void)mbar_drain(bar, 0);  // the copies in flight land before this warp moves on
    }
    __syncwarp();
    if constexpr (!kGated) return;
  }
  const float* gM = sGate;
  const float* gN = sGate + kGateOffN;
  const float* gBeta = sGate + kGateOffBeta;
  const float* gG = sGate + kGateOffG;
  const float* gGam = sGate + kGateOffGam;
  float* sP = sm + L::OFF_P;
  float* sR = sm + L::OFF_R;
  const int row0 = warp * kRowsPerWarp;
  const int m = lane >> 3;   // row of this warp handled by this lane in the phases below
  const int cg = lane & 7;   // column group (P) / token (outputs)

  // (a gated CTA's warps take part in the cluster exchange below even after a timeout)
  // gated: o of (row m, tokens cg and cg + 8), scaled by w SiLU(z) once its square is taken, and
  // the squares themselves
  float o_a = 0.f, o_b = 0.f, sq_a = 0.f, sq_b = 0.f;
  // outputs o_t = q_scale Gamma_t Pq_t + sum_{j<=t} N[t][j] u_j: lane -> (row m, tokens cg, cg + 8).
  // No state depends on them, so the plain and tree variants compute them after the state
  // stream, off the path to the first store; the gated variant needs them inside the stream.
  auto outputs = [&]() {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int t = cg + 8 * half;
      if (t < K) {
        float o = p.q_scale * gGam[t] * sP[(row0 + m) * L::PSTRIDE + kKMax + t];
        for (int jj = 0; jj <= t; ++jj) o = fmaf(gN[t * kMStride + jj], sU[jj * kRowsPerWarp + m], o);
        if constexpr (kGated) {
          const float gz = nw * silu(bf16_to_f32(half ? z_b : z_a));
          if (half == 0) {
            sq_a = o * o;
            o_a = o * gz;
          } else {
            sq_b = o * o;
            o_b = o * gz;
          }
        } else {
          const size_t oi = (size_t(b) * K + t) * p.Hv * DV + size_t(h) * DV + r0 + row0 + m;
          if (p.out_f32)
            static_cast<float*>(p.out)[oi] = o;
          else
            static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16(o);
        }
      }
    }
    __syncwarp();
  };
  if (ok) {
  (void)mbar_try_wait(bar, 0);  // every lane observes the completed phase

  // P = S0 [k^ | q^]: lane (m, cg) computes columns 4cg..4cg+3 of row row0+m; for the k^
  // columns the right-hand side rhs_j = v_j - Gamma_j (S0 k^_j) right away
  {
    float2 acc01 = make_float2(0.f, 0.f), acc23 = make_float2(0.f, 0.f);
    const float* srow = sS0 + (row0 + m) * L::SSTRIDE;
    const float* wcol = sWT + 4 * cg;
#pragma unroll 4
    for (int c = 0; c < DK; c += 4) {
      const float4 sv = *reinterpret_cast<const float4*>(srow + c);
      const float sc[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 w = *reinterpret_cast<const float4*>(wcol + (c + q) * kNCol);
        const float2 ss = make_float2(sc[q], sc[q]);
        acc01 = __ffma2_rn(ss, make_float2(w.x, w.y), acc01);
        acc23 = __ffma2_rn(ss, make_float2(w.z, w.w), acc23);
      }
    }
    const float pv[4] = {acc01.x, acc01.y, acc23.x, acc23.y};
    *reinterpret_cast<float4*>(sP + (row0 + m) * L::PSTRIDE + 4 * cg) = make_float4(pv[0], pv[1], pv[2], pv[3]);
    if (cg < 4) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int jj = 4 * cg + i;
        sR[(row0 + m) * L::RSTRIDE + jj] = fmaf(-gGam[jj], pv[i], sV[jj * kRowsPerWarp + m]);
      }
    }
  }
  __syncwarp();

  // forward substitution u_t = beta_t (rhs_t - sum_{j<t} M[t][j] u_j), lanes 0..3 (one row each;
  // a version that split each step's sum over all 32 lanes with shuffles took twice as long: the
  // shuffles queue behind the shared-memory traffic of the neighbouring CTAs' state streams)
  if (lane < kRowsPerWarp) {
    const float* rh = sR + (row0 + lane) * L::RSTRIDE;
    float u[kKMax];
#pragma unroll
    for (int tt = 0; tt < kKMax; ++tt) {
      u[tt] = 0.f;
      if (tt < K) {
        float acc = rh[tt];
#pragma unroll
        for (int jj = 0; jj < tt; ++jj) acc = fmaf(-gM[tt * kMStride + jj], u[jj], acc);
        u[tt] = gBeta[tt] * acc;
        sU[tt * kRowsPerWarp + lane] = u[tt];
      }
    }
  }
  __syncwarp();

  if constexpr (kGated) outputs();
  }  // ok

  // gated: the exchange of the sums of o^2 over the warp's 4 rows (lanes m = 0..3 of one column
  // group), pushed into every CTA of the cluster as asynchronous stores that complete on the
  // receiver's bar_sq, and the output norm that waits for them; both run inside the state stream
  // (after its first and middle token) so that their latency hides behind the stores in flight
  auto gated_push = [&]() {
    sq_a += __shfl_xor_sync(0xffffffffu, sq_a, 8);
    sq_a += __shfl_xor_sync(0xffffffffu, sq_a, 16);
    sq_b += __shfl_xor_sync(0xffffffffu, sq_b, 8);
    sq_b += __shfl_xor_sync(0xffffffffu, sq_b, 16);
    cluster_wait_acquire();  // every CTA of the cluster has started and set up bar_sq
    if (lane < 8) {
      const uint32_t rank = cluster_ctarank();
      const uint32_t slot = smem_addr(sm + L::OFF_SQ + ((rank * kWarps + warp) * (kKMax / 2) + lane) * 2);
      const uint32_t sbar = smem_addr(bar_sq);
      for (int d = 0; d < kTiles; ++d) st_async_cluster_f32x2(map_to_rank(slot, d), sq_a, sq_b, map_to_rank(sbar, d));
    }
  };
  // out = o rsqrt(sum_rows o^2 / dv + eps) w SiLU(z) over the head's dv rows, which the cluster's
  // kTiles CTAs share, per warp on the o w SiLU(z) it holds.  Every CTA waits here for all pushes
  // into its shared memory, so none exits while a peer still writes to it.
  auto gated_finish = [&]() {
    const bool got = mbar_wait_bounded(bar_sq, 0);
    if (!got) {  // (the peers' pushes still land before this CTA can exit)
      if (lane == 0) atomicOr(p.err, kDevErrTimeout);
      (void)mbar_drain(bar_sq, 0);
    }
    if (ok && got) {
      // lane (m, cg) adds the partials of warps m, m + 4, ...; the xor over the m bits completes
      const float2* sSq = reinterpret_cast<const float2*>(sm + L::OFF_SQ);
      float ta = 0.f, tb = 0.f;
#pragma unroll
      for (int d = m; d < kTiles * kWarps; d += 4) {
        const float2 v = sSq[d * (kKMax / 2) + cg];
        ta += v.x;
        tb += v.y;
      }
      ta += __shfl_xor_sync(0xffffffffu, ta, 8);
      ta += __shfl_xor_sync(0xffffffffu, ta, 16);
      tb += __shfl_xor_sync(0xffffffffu, tb, 8);
      tb += __shfl_xor_sync(0xffffffffu, tb, 16);
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int t = cg + 8 * half;
        if (t < K) {
          const float inv = rsqrtf((half ? tb : ta) * (1.f / DV) + p.norm_eps);
          const float y = (half ? o_b : o_a) * inv;
          const size_t oi = (size_t(b) * K + t) * p.Hv * DV + size_t(h) * DV + r0 + row0 + m;
          if (p.out_f32)
            static_cast<float*>(p.out)[oi] = y;
          else
            static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16(y);
        }
      }
    }
  };
  (void)gated_push;
  (void)gated_finish;

  if (ok) {
  // stream the K states from registers: lane owns DK/32 float4 of the warp's 4 rows
  constexpr int F4 = DK / 32;
  constexpr int C4 = DK / 4;
  // float4 q of this lane sits in row rowq[q] of the warp's rows, column c4 (row and column are
  // compile-time constants per q when a row spans the whole warp)
  static_assert(C4 == 32 || C4 == 16, "dk = 128 or 64");
  const int row_lane = (C4 == 32) ? 0 : lane / C4;
  int rowq[F4];
  float4 s[F4];
  const int c4 = (C4 == 32) ? lane : lane % C4;
#pragma unroll
  for (int q = 0; q < F4; ++q) {
    rowq[q] = q * (32 / C4) + row_lane;
    s[q] = *reinterpret_cast<const float4*>(sS0 + (row0 + rowq[q]) * L::SSTRIDE + 4 * c4);
  }
  const size_t inter_stride = size_t(p.Hv) * DV * DK;
  const size_t my_off = size_t(row0) * DK + 4 * c4;
  const size_t head_tile_off = (size_t(h) * DV + r0) * DK;  // offset of this tile inside one token's states
  float* inter = p.state_inter ? p.state_inter + size_t(b) * (K - 1) * inter_stride + head_tile_off + my_off : nullptr;
  for (int t = 0; t < K; ++t) {
    if constexpr (kTree) {
      // a node that does not continue the previous one starts from its parent's state, rebuilt
      // from shared memory in its closed form S_par = Gamma_par S0 + sum_{j in path(par)}
      // D[par][j] u_j k^_j^T (D: the product of g over the path nodes after j), walking the path
      // upwards; no reload of the parent's intermediate from global memory
      const int par = tree->parent[t];
      if (t > 0 && par != t - 1) {
#pragma unroll
        for (int q = 0; q < F4; ++q) s[q] = make_float4(0.f, 0.f, 0.f, 0.f);
        float d = 1.f;
        for (int j = par; j >= 0; j = tree->parent[j]) {
          const float4 kj = *reinterpret_cast<const float4*>(sKn + j * DK + 4 * c4);
          float uj[F4];  // u_j of the lane's rows (one 16-byte broadcast when a row spans the warp)
          if constexpr (C4 == 32) {
            const float4 u4 = *reinterpret_cast<const float4*>(sU + j * kRowsPerWarp);
            uj[0] = u4.x;
            uj[1] = u4.y;
            uj[2] = u4.z;
            uj[3] = u4.w;
          } else {
#pragma unroll
            for (int q = 0; q < F4; ++q) uj[q] = sU[j * kRowsPerWarp + rowq[q]];
          }
#pragma unroll
          for (int q = 0; q < F4; ++q) {
            const float du = d * uj[q];
            s[q].x = fmaf(du, kj.x, s[q].x);
            s[q].y = fmaf(du, kj.y, s[q].y);
            s[q].z = fmaf(du, kj.z, s[q].z);
            s[q].w = fmaf(du, kj.w, s[q].w);
          }
          d *= gG[j];
        }
#pragma unroll
        for (int q = 0; q < F4; ++q) {
          const float4 s0v = *reinterpret_cast<const float4*>(sS0 + (row0 + rowq[q]) * L::SSTRIDE + 4 * c4);
          s[q].x = fmaf(d, s0v.x, s[q].x);
          s[q].y = fmaf(d, s0v.y, s[q].y);
          s[q].z = fmaf(d, s0v.z, s[q].z);
          s[q].w = fmaf(d, s0v.w, s[q].w);
        }
      }
    }
    const float g = gG[t];
    const float4 kv = *reinterpret_cast<const float4*>(sKn + t * DK + 4 * c4);
    float* dst = (t == K - 1) ? p.state_out + tile_off + my_off : inter + size_t(t) * inter_stride;
    float uq[F4];  // u_t of the lane's rows: one 16-byte broadcast when a row spans the warp
    if constexpr (C4 == 32) {
      static_assert(F4 == kRowsPerWarp && L::OFF_U % 4 == 0, "the warp's four u values are one float4");
      const float4 u4 = *reinterpret_cast<const float4*>(sU + t * kRowsPerWarp);
      uq[0] = u4.x;
      uq[1] = u4.y;
      uq[2] = u4.z;
      uq[3] = u4.w;
    } else {
#pragma unroll
      for (int q = 0; q < F4; ++q) uq[q] = sU[t * kRowsPerWarp + rowq[q]];
    }
#pragma unroll
    for (int q = 0; q < F4; ++q) {
      const float u = uq[q];
      {  // s = g s + u k, two lanes of f32 per instruction
        const float2 gg = make_float2(g, g), uu = make_float2(u, u);
        const float2 lo = __ffma2_rn(uu, make_float2(kv.x, kv.y), __fmul2_rn(gg, make_float2(s[q].x, s[q].y)));
        const float2 hi = __ffma2_rn(uu, make_float2(kv.z, kv.w), __fmul2_rn(gg, make_float2(s[q].z, s[q].w)));
        s[q] = make_float4(lo.x, lo.y, hi.x, hi.y);
      }
      float4* d4 = reinterpret_cast<float4*>(dst + size_t(rowq[q]) * DK);
      if (t == K - 1)
        *d4 = s[q];
      else
        __stcs(d4, s[q]);
    }
    if constexpr (kGated) {
      if (t == 0) gated_push();
      if (t == K / 2) gated_finish();
    }
  }
  if constexpr (!kGated) outputs();
  }  // ok

  if constexpr (kGated) {
    if (!ok) {  // (the exchange still runs: the peers wait for this CTA's partials)
      gated_push();
      gated_finish();
    }
  }
}

template <int DK, int DV, bool kTree, bool kGated>
cudaError_t launch_t(const VerifyParams& p, cudaStream_t stream) {
  auto k1 = gdn_qk_prologue_kernel<DK, kTree>;
  auto k2 = gdn_state_stream_kernel<DK, DV, kTree, kGated>;
  const size_t b1 = PrologueLayout<DK>::BYTES;
  const size_t b2 = StreamLayout<DK, kGated>::BYTES;
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if constexpr (kGated) {  // the row tiles of one v-head form a cluster (they share the output norm)
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = DV / kRows;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, k2, p);
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream) {
  const bool tree = p.parent != nullptr;
  const bool gated = p.z != nullptr;
#define GDN_LAUNCH(DK_, DV_)                                          \
  if (p.dk == DK_ && p.dv == DV_) {                                   \
    if (gated) return launch_t<DK_, DV_, false, true>(p, stream);     \
    if (tree) return launch_t<DK_, DV_, true, false>(p, stream);      \
    return launch_t<DK_, DV_, false, false>(p, stream);               \
  }
  GDN_LAUNCH(128, 128)
  GDN_LAUNCH(128, 64)
  GDN_LAUNCH(64, 128)
  GDN_LAUNCH(64, 64)
#undef GDN_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace gdn
