// Verify step of one Gated DeltaNet layer on sm_103a: conv + SiLU, q|k L2 norm, raw gates and
// the gated delta rule over a window of K tokens, writing the final and every intermediate state.
//
// Method (lucebox #637 "NVLink fix for PR625", commit list: fused conv step, single l2_norm
// over q|k, raw-gate gated_delta_net with head broadcast; review of ggml-cuda/gated_delta_net.cu
// line 404 for the gate formula; atlas #297, commit on the SSM/GDN verify kernels: a K=16
// verify that writes the final state and all intermediates in one pass):
//
//   y_t   = SiLU(sum_j w[c][j] win[t+j][c])            per channel, win = [history; x]
//   q^,k^ = q / sqrt(|q|^2 + eps), k / sqrt(|k|^2 + eps)  per (token, q/k head)
//   beta  = sigmoid(b), g = exp(softplus(a + dt_bias) * -exp(A_log))
//   S_t   = g_t S_{t-1} + u_t k^_t^T,  u_t = beta_t (v_t - g_t S_{t-1} k^_t)
//   o_t   = q_scale S_t q^_t
//
// Row i of S_t depends only on row i of S_{t-1}, on k^_t, q^_t, the gates and the conv output of
// v-channel i.  So each warp takes four state rows and runs the recurrence token by token from
// registers: a dot product with k^_t (over the eight lanes that hold a row), the rank-1 update,
// the store of S_t (512 contiguous bytes per warp instruction) and the dot product with q^_t for
// o_t.  Every state is produced, and stored, exactly once; nothing waits for another CTA, so the
// first states leave as soon as a CTA's own conv and norms are done.
//
// Two kernels on the caller's stream:
//  1. verify: one CTA per (sequence, v-head, 32-row tile of the state), 256 threads.  A bulk async
//     (TMA) copy of its S0 tile; conv + SiLU of the 2 dk q|k channels of its q/k head (each CTA
//     of the head computes them again: a few thousand instructions, against a table handed over
//     between CTAs whose wait would hold back every state stream) and of its own 32 v-channels;
//     the gates of its v-head; the L2 norms; then the recurrence.  Launched with programmatic
//     dependent launch (its CTAs may be scheduled while the kernel ahead of it finishes; they
//     wait for it before reading anything).
//  2. qk_history: the K history snapshots and the new history of the q|k channels, which all
//     CTAs of a q/k head read and so none of them may rewrite in place.  Launched with
//     programmatic dependent launch: it can start only once every verify CTA has passed the
//     point where it has used its q|k history (each signals right after its conv), and it
//     only reads what kernel 1 does not write.  The v-channels' snapshots and history are
//     written by kernel 1, each channel by the one thread that reads it.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRows = 32;          // state rows per CTA of the verify kernel
constexpr int kRowsPerWarp = kRows / kWarps;
constexpr int kHistThreads = 128;  // q|k channel pairs per CTA of the history kernel

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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

__device__ __forceinline__ float2 unpack_bf16x2(uint32_t v) {
  return make_float2(bf16_to_f32(uint16_t(v & 0xFFFFu)), bf16_to_f32(uint16_t(v >> 16)));
}

// Conv + SiLU of the two adjacent q|k channels c, c + 1 (c even) over the window, outputs only
// (their snapshots and new history are the history kernel's): one 4-byte load per token for both
// x values, 8-byte history loads.  The outputs go to dst[t * ystride], dst[t * ystride + 1] for
// t < K, zero for K <= t < 16.  A token tree reads each node's window through the table: the
// history from registers, the x values from `scratch[t * sstride]` (shared memory).
template <bool kTree>
__device__ __forceinline__ void qk_conv_pair(const VerifyParams& p, int b, int c, const TreeTable* tt, float* dst,
                                             int ystride, float2* scratch, int sstride) {
  const int C = p.C;
  const int K = p.K;
  const float4 wa = *reinterpret_cast<const float4*>(p.conv_w + size_t(c) * kConvW);
  const float4 wb = *reinterpret_cast<const float4*>(p.conv_w + size_t(c + 1) * kConvW);
  const float* hin = kTree ? p.conv_state_in + size_t(b) * 3 * C + c : history_src(p, b, c, prev_accept(p, b, false));
  const float2 h0 = *reinterpret_cast<const float2*>(hin);
  const float2 h1 = *reinterpret_cast<const float2*>(hin + C);
  const float2 h2 = *reinterpret_cast<const float2*>(hin + 2 * C);
  const uint32_t* xp = reinterpret_cast<const uint32_t*>(p.x + size_t(b) * K * C + c);
  uint32_t xv[kKMax];
#pragma unroll
  for (int t = 0; t < kKMax; ++t) xv[t] = (t < K) ? xp[size_t(t) * (C / 2)] : 0u;
  auto conv2 = [&](float2 w0, float2 w1, float2 w2, float2 xt) {
    return make_float2(silu(fmaf(wa.w, xt.x, fmaf(wa.z, w2.x, fmaf(wa.y, w1.x, wa.x * w0.x)))),
                       silu(fmaf(wb.w, xt.y, fmaf(wb.z, w2.y, fmaf(wb.y, w1.y, wb.x * w0.y)))));
  };
  if constexpr (kTree) {
#pragma unroll
    for (int t = 0; t < kKMax; ++t) scratch[t * sstride] = unpack_bf16x2(xv[t]);
    // value `idx` of [history rows 0, 1, 2, x_0 .. x_{K-1}]
    auto val = [&](int idx) { return idx < 3 ? (idx == 0 ? h0 : (idx == 1 ? h1 : h2)) : scratch[(idx - 3) * sstride]; };
#pragma unroll
    for (int t = 0; t < kKMax; ++t) {
      float2 y = make_float2(0.f, 0.f);
      if (t < K) y = conv2(val(tt->src[t][0]), val(tt->src[t][1]), val(tt->src[t][2]), scratch[t * sstride]);
      *reinterpret_cast<float2*>(dst + t * ystride) = y;
    }
  } else {
    (void)tt;
    (void)scratch;
    (void)sstride;
    float2 w0 = h0, w1 = h1, w2 = h2;
#pragma unroll
    for (int t = 0; t < kKMax; ++t) {
      float2 y = make_float2(0.f, 0.f);
      if (t < K) {
        const float2 xt = unpack_bf16x2(xv[t]);
        y = conv2(w0, w1, w2, xt);
        w0 = w1;
        w1 = w2;
        w2 = xt;
      }
      *reinterpret_cast<float2*>(dst + t * ystride) = y;
    }
  }
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


// The V = dk / 32 state columns a lane holds per row (a4): 16-byte pieces at dk = 128, 8-byte
// at dk = 64.
template <int V>
__device__ __forceinline__ void load_vec(const float* src, float (&v)[V]) {
  if constexpr (V == 4) {
    const float4 x = *reinterpret_cast<const float4*>(src);
    v[0] = x.x;
    v[1] = x.y;
    v[2] = x.z;
    v[3] = x.w;
  } else {
    static_assert(V == 2, "dk = 128 or 64");
    const float2 x = *reinterpret_cast<const float2*>(src);
    v[0] = x.x;
    v[1] = x.y;
  }
}

template <int V>
__device__ __forceinline__ float dot_vec(const float (&s)[V], const float (&k)[V]) {
  if constexpr (V == 4) {
    float2 acc = __fmul2_rn(make_float2(s[0], s[1]), make_float2(k[0], k[1]));
    acc = __ffma2_rn(make_float2(s[2], s[3]), make_float2(k[2], k[3]), acc);
    return acc.x + acc.y;
  } else {
    return fmaf(s[1], k[1], s[0] * k[0]);
  }
}

// s = g s + u k, two lanes of f32 per instruction
template <int V>
__device__ __forceinline__ void update_vec(float (&s)[V], float g, float u, const float (&k)[V]) {
  const float2 gg = make_float2(g, g), uu = make_float2(u, u);
#pragma unroll
  for (int e = 0; e < V; e += 2) {
    const float2 r = __ffma2_rn(uu, make_float2(k[e], k[e + 1]), __fmul2_rn(gg, make_float2(s[e], s[e + 1])));
    s[e] = r.x;
    s[e + 1] = r.y;
  }
}

// streaming (evict-first) unless `keep`
template <int V>
__device__ __forceinline__ void store_vec(float* dst, const float (&v)[V], bool keep) {
  if constexpr (V == 4) {
    const float4 x = make_float4(v[0], v[1], v[2], v[3]);
    if (keep)
      *reinterpret_cast<float4*>(dst) = x;
    else
      __stcs(reinterpret_cast<float4*>(dst), x);
  } else {
    const float2 x = make_float2(v[0], v[1]);
    if (keep)
      *reinterpret_cast<float2*>(dst) = x;
    else
      __stcs(reinterpret_cast<float2*>(dst), x);
  }
}

// For every lane l, the sum over the warp's 32 lanes of p[l / 8]: two halving rounds (partners
// 16, then 8 lanes apart, each lane keeping half of the rows it still holds and sending the other
// half) and a butterfly over the last three lane bits, 6 shuffles in all.  The eight lanes of a
// row end with the same value (each pairwise sum adds the same two numbers).
__device__ __forceinline__ float reduce4(const float (&p)[4], int lane) {
  const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
  float k0 = h16 ? p[2] : p[0];
  float k1 = h16 ? p[3] : p[1];
  const float x0 = h16 ? p[0] : p[2];
  const float x1 = h16 ? p[1] : p[3];
  k0 += __shfl_xor_sync(0xffffffffu, x0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, x1, 16);
  float k = h8 ? k1 : k0;
  const float x = h8 ? k0 : k1;
  k += __shfl_xor_sync(0xffffffffu, x, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

// Two reduce4 at once, their shuffles interleaved (the sums and their order are reduce4's).
__device__ __forceinline__ void reduce4_pair(const float (&p)[4], const float (&q)[4], int lane, float& rp,
                                             float& rq) {
  const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
  float k0 = h16 ? p[2] : p[0], k1 = h16 ? p[3] : p[1];
  float m0 = h16 ? q[2] : q[0], m1 = h16 ? q[3] : q[1];
  const float x0 = h16 ? p[0] : p[2], x1 = h16 ? p[1] : p[3];
  const float y0 = h16 ? q[0] : q[2], y1 = h16 ? q[1] : q[3];
  k0 += __shfl_xor_sync(0xffffffffu, x0, 16);
  m0 += __shfl_xor_sync(0xffffffffu, y0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, x1, 16);
  m1 += __shfl_xor_sync(0xffffffffu, y1, 16);
  float k = h8 ? k1 : k0, mm = h8 ? m1 : m0;
  const float x = h8 ? k0 : k1, y = h8 ? m0 : m1;
  k += __shfl_xor_sync(0xffffffffu, x, 8);
  mm += __shfl_xor_sync(0xffffffffu, y, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  mm += __shfl_xor_sync(0xffffffffu, mm, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  mm += __shfl_xor_sync(0xffffffffu, mm, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  mm += __shfl_xor_sync(0xffffffffu, mm, 1);
  rp = k;
  rq = mm;
}

// ------------------------------------------------------------------------------------------
// Kernel 2: the q|k channels' history snapshots and new history (thread = channel pair 2i, 2i+1
// of the 2 Hk dk q|k channels, q first).  Snapshot t of a chain window is the history after token
// t, [win[t+1], win[t+2], x_t]; of a token tree, the history after node t along its path.
template <bool kTree>
__global__ void __launch_bounds__(kHistThreads) gdn_qk_history_kernel(const VerifyParams p) {
  // the next call's verify CTAs may be scheduled from here on: each waits for this grid's
  // completion, which follows the verify grid's, before it reads anything
  griddep_launch_dependents();
  __shared__ TreeTable tree_s;
  __shared__ float2 sx[kTree ? kKMax * kHistThreads : 1];
  const int b = blockIdx.y;
  const int i = blockIdx.x * kHistThreads + threadIdx.x;
  if constexpr (kTree) {
    if (threadIdx.x == 0) build_tree(p, b, &tree_s, false);
    __syncthreads();
  }
  if (i < p.Hk * p.dk) {
    const int c = 2 * i;
    const int C = p.C;
    const int K = p.K;
    const float* hin = kTree ? p.conv_state_in + size_t(b) * 3 * C + c : history_src(p, b, c, prev_accept(p, b, false));
    float2 h0 = *reinterpret_cast<const float2*>(hin);
    float2 h1 = *reinterpret_cast<const float2*>(hin + C);
    float2 h2 = *reinterpret_cast<const float2*>(hin + 2 * C);
    const uint32_t* xp = reinterpret_cast<const uint32_t*>(p.x + size_t(b) * K * C + c);
    uint32_t xv[kKMax];
#pragma unroll
    for (int t = 0; t < kKMax; ++t) xv[t] = (t < K) ? xp[size_t(t) * (C / 2)] : 0u;
    float2* ci = p.conv_inter ? reinterpret_cast<float2*>(p.conv_inter + size_t(b) * K * 3 * C + c) : nullptr;
    const size_t row2 = size_t(C) / 2;  // one history row, in float2
    if constexpr (kTree) {
      float2* scr = sx + threadIdx.x;
#pragma unroll
      for (int t = 0; t < kKMax; ++t) scr[t * kHistThreads] = unpack_bf16x2(xv[t]);
      auto val = [&](int idx) { return idx < 3 ? (idx == 0 ? h0 : (idx == 1 ? h1 : h2)) : scr[(idx - 3) * kHistThreads]; };
      float2 n0 = h0, n1 = h1, n2 = h2;
      for (int t = 0; t < K; ++t) {
        n0 = val(tree_s.src[t][1]);
        n1 = val(tree_s.src[t][2]);
        n2 = scr[t * kHistThreads];
        if (ci) {
          ci[(3 * t + 0) * row2] = n0;
          ci[(3 * t + 1) * row2] = n1;
          ci[(3 * t + 2) * row2] = n2;
        }
      }
      h0 = n0;
      h1 = n1;
      h2 = n2;
    } else {
#pragma unroll
      for (int t = 0; t < kKMax; ++t) {
        if (t < K) {
          h0 = h1;
          h1 = h2;
          h2 = unpack_bf16x2(xv[t]);
          if (ci) {
            ci[(3 * t + 0) * row2] = h0;
            ci[(3 * t + 1) * row2] = h1;
            ci[(3 * t + 2) * row2] = h2;
          }
        }
      }
    }
    float2* hout = reinterpret_cast<float2*>(p.conv_state_out + size_t(b) * 3 * C + c);
    hout[0] = h0;
    hout[row2] = h1;
    hout[2 * row2] = h2;
  }
  // this grid ends only after the verify grid (its completion is what the next call on the
  // stream waits for)
  griddep_wait();
}

// ------------------------------------------------------------------------------------------
// Kernel 1: per (sequence, v-head, 32-row tile) verify.
template <int DK, int DV, bool kTree, bool kGated>
struct VerifyLayout {
  static constexpr int kTiles = DV / kRows;
  static constexpr int SSTRIDE = DK + 4;                  // rows 4 banks apart
  static constexpr int OFF_S0 = 0;                        // [32][SSTRIDE] S0 tile, bulk copy per row
  static constexpr int OFF_Y = OFF_S0 + kRows * SSTRIDE;  // [32][SSTRIDE] q|k conv outputs, then k^ (rows
                                                          // 0..15) and q^ (rows 16..31), zero for t >= K
  static constexpr int OFF_V = OFF_Y + kNCol * SSTRIDE;   // [16][32] v conv outputs, token-major
  static constexpr int OFF_U = OFF_V + kKMax * kRows;     // [16][32] token tree: the v conv's x values,
                                                          // then u_t (for the branch rebuilds)
  static constexpr int OFF_BG = OFF_U + kKMax * kRows;    // beta[16], g[16]
  static constexpr int OFF_X = OFF_BG + 2 * kKMax;        // token tree: q|k x values [16][dk] float2;
                                                          // gated: sums of o^2 [tile][warp][8] float2
  static constexpr int X_FLOATS = kTree ? 2 * kKMax * DK : (kGated ? 2 * kTiles * kWarps * 8 : 0);
  static constexpr int OFF_TREE = OFF_X + X_FLOATS;
  static constexpr int TREE_FLOATS = kTree ? int(sizeof(TreeTable) / 4) : 0;
  static constexpr int OFF_BAR = (OFF_TREE + TREE_FLOATS + 1) & ~1;  // 8-byte aligned mbarrier(s)
  static constexpr int FLOATS = OFF_BAR + (kGated ? 4 : 2);           // gated: + the exchange mbarrier
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
  static constexpr uint32_t S0_ROW_BYTES = DK * 4;
  static constexpr uint32_t S0_BYTES = kRows * S0_ROW_BYTES;
  static_assert((SSTRIDE * 4) % 16 == 0 && OFF_Y % 4 == 0 && S0_ROW_BYTES % 16 == 0, "16-byte rows");
  static_assert(OFF_X % 2 == 0, "float2 scratch and exchange slots 8-byte aligned");
};

// kOne: the K = 1 instantiation (plain decode), with the window length fixed at compile time; the
// token loop then has no previous output whose row sum to overlap with the next token's.
template <int DK, int DV, bool kTree, bool kGated, bool kOne>
__global__ void __launch_bounds__(kThreads, 4) gdn_verify_kernel(const VerifyParams p) {
  static_assert(!(kTree && kGated), "tree and gated-norm variants are separate");
  static_assert(!(kTree && kOne), "a one-node tree takes the tree variant");
  static_assert(DK == 64 || DK == 128, "dk = 64 or 128");
  using L = VerifyLayout<DK, DV, kTree, kGated>;
  constexpr int kTiles = L::kTiles;
  extern __shared__ __align__(128) float sm[];
  float* sS0 = sm + L::OFF_S0;
  float* sY = sm + L::OFF_Y;
  float* sV = sm + L::OFF_V;
  float* sU = sm + L::OFF_U;
  float* sBG = sm + L::OFF_BG;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);
  TreeTable* tree = reinterpret_cast<TreeTable*>(sm + L::OFF_TREE);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int K = kOne ? 1 : p.K;
  const int b = blockIdx.y;
  const int h = blockIdx.x / kTiles;
  const int r0 = (blockIdx.x % kTiles) * kRows;
  const int kh = h / (p.Hv / p.Hk);
  const size_t tile_off = ((size_t(b) * p.Hv + h) * DV + r0) * DK;
  // Launched with programmatic dependent launch, the CTA may start while the kernel before it on
  // the stream still runs: nothing is read from global memory before this wait, which returns
  // once that kernel has completed and its writes are visible.
  griddep_wait();

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
  if constexpr (kTree) {
    if (tid == 32) build_tree(p, b, tree, blockIdx.x == 0);
  }
  __syncthreads();  // the barrier (and the tree table) are ready before any thread uses them

  if (warp == kWarps - 1) {
    // S0: the previous final state, or (rollback applied on read) the accepted intermediate or
    // the pre-window snapshot of the previous window; one row per lane, into rows padded by four
    // banks
    const int Lp = prev_accept(p, b, blockIdx.x == 0 && lane == 0);
    const float* s0 = p.state_in + tile_off;
    if (Lp == 0)
      s0 = p.state_snap_prev + tile_off;
    else if (Lp > 0 && Lp < K)
      s0 = p.state_inter_prev + (size_t(b) * (K - 1) + (Lp - 1)) * size_t(p.Hv) * DV * DK + (size_t(h) * DV + r0) * DK;
    if (lane == 0) mbar_arrive_expect_tx(bar, L::S0_BYTES);
    __syncwarp();
    bulk_load(sS0 + lane * L::SSTRIDE, s0 + size_t(lane) * DK, L::S0_ROW_BYTES, bar);
  }
  // gated: the lane's two z values of the epilogue, (token cg, row m of its warp) and eight tokens
  // later, and the row's norm weight, fetched now so that they have long arrived when used (the
  // lane map (m, cg) is the one of the recurrence below)
  uint16_t z_a = 0, z_b = 0;
  float nw = 0.f;
  if constexpr (kGated) {
    const int t0 = lane & 7, i0 = warp * kRowsPerWarp + (lane >> 3);
    const uint16_t* zp = p.z + ((size_t(b) * K + t0) * p.Hv + h) * DV + r0 + i0;
    if (t0 < K) z_a = __ldg(zp);
    if (t0 + 8 < K) z_b = __ldg(zp + size_t(8) * p.Hv * DV);
    nw = __ldg(p.norm_w + r0 + i0);
  }

  // a1: threads 0 .. dk-1 convolve the q|k channel pairs of head kh (k rows 0..15 of the table,
  // q rows 16..31), warp 4 the tile's 32 v-channels (writing their snapshots and history: each
  // channel has this one owner), warp 5 evaluates the gates of v-head h (a3)
  if (tid < DK) {
    const int cc = 2 * tid;  // q channels 0..dk-1, then k channels (pairs never straddle them)
    const int c = (cc < DK) ? kh * DK + cc : p.Hk * DK + kh * DK + (cc - DK);
    const int n0 = (cc < DK) ? kKMax : 0;
    qk_conv_pair<kTree>(p, b, c, tree, sY + n0 * L::SSTRIDE + cc % DK, L::SSTRIDE,
                        reinterpret_cast<float2*>(sm + L::OFF_X) + tid, DK);
  } else if (warp == 4) {
    float y[kKMax];
    conv_channel<kTree>(p, b, 2 * p.Hk * DK + h * DV + r0 + lane, tree, y, sU + lane, kRows);
#pragma unroll
    for (int t = 0; t < kKMax; ++t) sV[t * kRows + lane] = y[t];
  } else if (warp == 5 && lane < kKMax) {
    float beta = 0.f, g = 1.f;
    if (lane < K) {
      const size_t gi = (size_t(b) * K + lane) * p.Hv + h;
      raw_gate(bf16_to_f32(p.a[gi]), bf16_to_f32(p.b[gi]), p.A_log[h], p.dt_bias[h], beta, g);
    }
    sBG[lane] = beta;
    sBG[kKMax + lane] = g;
  }
  __syncthreads();
  // every q|k history value of this CTA has been loaded and used: the history kernel may rewrite
  // them once all CTAs got here
  griddep_launch_dependents();

  // a2: L2 norm of each of the 2K vectors in place, warp per vector; rows t >= K hold the conv's
  // zeros and stay.  A chain window takes a warp's four vectors side by side, so that their
  // shuffle reductions overlap (the token-tree variant, measured slower that way, one by one).
  if constexpr (kTree) {
    for (int n = warp; n < kNCol; n += kWarps) {
      float* yr = sY + n * L::SSTRIDE;
      float vals[DK / 32];
      float ss = 0.f;
#pragma unroll
      for (int m = 0; m < DK / 32; ++m) {
        vals[m] = yr[lane + 32 * m];
        ss = fmaf(vals[m], vals[m], ss);
      }
      ss = warp_sum(ss);
      const float inv = (n % kKMax < K) ? rsqrtf(ss + p.l2_eps) : 0.f;
#pragma unroll
      for (int m = 0; m < DK / 32; ++m) yr[lane + 32 * m] = vals[m] * inv;
    }
  } else {
    constexpr int kPer = kNCol / kWarps;
    static_assert(kNCol % kWarps == 0, "whole vectors per warp");
    float vals[kPer][DK / 32], ss[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int n = warp + u * kWarps;
      ss[u] = 0.f;
#pragma unroll
      for (int m = 0; m < DK / 32; ++m) {
        vals[u][m] = (n % kKMax < K) ? sY[n * L::SSTRIDE + lane + 32 * m] : 0.f;
        ss[u] = fmaf(vals[u][m], vals[u][m], ss[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) ss[u] = warp_sum(ss[u]);
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      const int n = warp + u * kWarps;
      if (n % kKMax < K) {
        const float inv = rsqrtf(ss[u] + p.l2_eps);
#pragma unroll
        for (int m = 0; m < DK / 32; ++m) sY[n * L::SSTRIDE + lane + 32 * m] = vals[u][m] * inv;
      }
    }
  }
  __syncthreads();

  // S0 must have landed (bounded wait, warp-uniform outcome; no CTA-wide barrier follows)
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

  // a4.  Lane (m, cg) = (l / 8, l % 8) keeps o of row 4 warp + m for tokens cg and cg + 8 for the
  // epilogue.  A chain window holds row m at columns 32 f + 4 cg .. + 3 (f < dk / 32), the row's
  // dot products then needing only its eight lanes (three shuffles on the path from one token to
  // the next); a token tree holds all four rows of the warp at columns V l .. V l + V - 1 (V = dk /
  // 32), so that the k^ reads of its branch rebuilds are 32 distinct pieces instead of the same
  // 128 bytes read by four row groups, at the price of a reduction over the whole warp per dot
  // product (reduce4).  Measured at the serving shape: the tree layout took seeded 16-node trees
  // from 230.1 to 213.3 us per step, and made the chain's latency-bound shapes slower (B = 32,
  // K = 8 rounds 109.4 -> 114.7 us, the gated variant 191.8 -> 196.4 us).
  const int m = lane >> 3;
  const int cg = lane & 7;
  const int row = warp * kRowsPerWarp + m;
  float o_a = 0.f, o_b = 0.f;
  const size_t inter_stride = size_t(p.Hv) * DV * DK;
  if (ok) {
    (void)mbar_try_wait(bar, 0);  // every lane observes the completed phase
    if constexpr (kTree) {
      constexpr int V = DK / 32;
      const int row0 = warp * kRowsPerWarp;
      const int col = V * lane;
      float s[kRowsPerWarp][V];
#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) load_vec<V>(sS0 + (row0 + r) * L::SSTRIDE + col, s[r]);
      const size_t my_off = size_t(row0) * DK + col;
      float* fin = p.state_out + tile_off + my_off;
      float* inter = p.state_inter
                         ? p.state_inter + size_t(b) * (K - 1) * inter_stride + (size_t(h) * DV + r0) * DK + my_off
                         : nullptr;
      float pq[kRowsPerWarp] = {0.f, 0.f, 0.f, 0.f};
      for (int t = 0; t < K; ++t) {
        // a node that does not continue the previous one starts from its parent's state, rebuilt
        // in its closed form S_par = Gamma_par S0 + sum_{j in path(par)} D[par][j] u_j k^_j^T
        // (D: the product of g over the path nodes after j), walking the path upwards
        const int par = tree->parent[t];
        if (t > 0 && par != t - 1) {
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
            for (int e = 0; e < V; ++e) s[r][e] = 0.f;
          float d = 1.f;
          for (int j = par; j >= 0; j = tree->parent[j]) {
            const float4 uj = *reinterpret_cast<const float4*>(sU + j * kRows + row0);
            const float du[kRowsPerWarp] = {d * uj.x, d * uj.y, d * uj.z, d * uj.w};
            float kj[V];
            load_vec<V>(sY + j * L::SSTRIDE + col, kj);
#pragma unroll
            for (int r = 0; r < kRowsPerWarp; ++r)
#pragma unroll
              for (int e = 0; e < V; ++e) s[r][e] = fmaf(du[r], kj[e], s[r][e]);
            d *= sBG[kKMax + j];
          }
#pragma unroll
          for (int r = 0; r < kRowsPerWarp; ++r) {
            float sv[V];
            load_vec<V>(sS0 + (row0 + r) * L::SSTRIDE + col, sv);
#pragma unroll
            for (int e = 0; e < V; ++e) s[r][e] = fmaf(d, sv[e], s[r][e]);
          }
        }
        // S_{t-1} k^_t for the four rows (every lane ends with the same four sums), reduced
        // together with node t - 1's outputs (pq: their unreduced partials), so that the two
        // reductions' shuffles hide each other's latency (seeded 16-node trees at the serving
        // shape: 212.4 -> 203.7 us per step)
        float kv[V];
        load_vec<V>(sY + t * L::SSTRIDE + col, kv);
        float pk[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) pk[r] = dot_vec<V>(s[r], kv);
        float a_m, o_m;
        reduce4_pair(pk, pq, lane, a_m, o_m);
        if (t > 0) {
          const float o = o_m * p.q_scale;
          if (t - 1 == cg) o_a = o;
          if (t - 1 == cg + 8) o_b = o;
        }
        const float g = sBG[kKMax + t];
        const float beta = sBG[t];
        const float4 v4 = *reinterpret_cast<const float4*>(sV + t * kRows + row0);
        const float vr[kRowsPerWarp] = {v4.x, v4.y, v4.z, v4.w};
        float u[kRowsPerWarp];
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r)
          u[r] = beta * fmaf(-g, __shfl_sync(0xffffffffu, a_m, 8 * r), vr[r]);
        if (lane == 0) *reinterpret_cast<float4*>(sU + t * kRows + row0) = make_float4(u[0], u[1], u[2], u[3]);
        __syncwarp();
        // S_t = g S_{t-1} + u k^_t, stored straight from registers (the intermediates streaming,
        // evict-first; the final state with the normal policy)
        float* dst = (t == K - 1) ? fin : inter + size_t(t) * inter_stride;
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) {
          update_vec<V>(s[r], g, u[r], kv);
          store_vec<V>(dst + r * DK, s[r], t == K - 1);
        }
        // o_t = q_scale S_t q^_t: the lane's parts now, the sums with the next node's
        float qv[V];
        load_vec<V>(sY + (kKMax + t) * L::SSTRIDE + col, qv);
#pragma unroll
        for (int r = 0; r < kRowsPerWarp; ++r) pq[r] = dot_vec<V>(s[r], qv);
      }
      {
        const float o = reduce4(pq, lane) * p.q_scale;
        if (K - 1 == cg) o_a = o;
        if (K - 1 == cg + 8) o_b = o;
      }
    } else {
      constexpr int F = DK / 32;
      const int col = 4 * cg;
      const float* s0r = sS0 + row * L::SSTRIDE + col;
      float4 s[F];
#pragma unroll
      for (int f = 0; f < F; ++f) s[f] = *reinterpret_cast<const float4*>(s0r + 32 * f);
      const size_t my_off = size_t(row) * DK + col;
      float* fin = p.state_out + tile_off + my_off;
      float* inter = p.state_inter
                         ? p.state_inter + size_t(b) * (K - 1) * inter_stride + (size_t(h) * DV + r0) * DK + my_off
                         : nullptr;
      // o of token t - 1 is reduced over the row inside token t's k^ reduction (op: its unreduced
      // partial), so that the two butterflies' shuffles hide each other's latency on the path
      // from one token to the next; the sums are the same, added in the same order.  Measured
      // against reducing o in its own token: resume step 190.9 -> 189.6 us, B = 32 K = 8 rounds
      // 106.1 -> 102.0 us, 48-layer stack 2.72 -> 2.58 ms (a run-time skip of the first token's
      // zero shuffles lost on every shape; plain decode has its own K = 1 instantiation, with
      // no overlap to make)
      float op = 0.f;
      auto keep_o = [&](int tt, float ov) {
        ov *= p.q_scale;
        if (tt == cg) o_a = ov;
        if (tt == cg + 8) o_b = ov;
      };
      for (int t = 0; t < K; ++t) {
        // S_{t-1} k^_t over the row: the lane's columns, then the row's eight lanes (every lane of
        // the row ends with the same sum: the butterfly adds the same pairs in each)
        const float* kr = sY + t * L::SSTRIDE + col;
        float4 kv[F];
#pragma unroll
        for (int f = 0; f < F; ++f) kv[f] = *reinterpret_cast<const float4*>(kr + 32 * f);
        float2 a0 = make_float2(0.f, 0.f), a1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int f = 0; f < F; ++f) {
          a0 = __ffma2_rn(make_float2(s[f].x, s[f].y), make_float2(kv[f].x, kv[f].y), a0);
          a1 = __ffma2_rn(make_float2(s[f].z, s[f].w), make_float2(kv[f].z, kv[f].w), a1);
        }
        float a = (a0.x + a0.y) + (a1.x + a1.y);
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        if constexpr (!kOne) op += __shfl_xor_sync(0xffffffffu, op, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        if constexpr (!kOne) op += __shfl_xor_sync(0xffffffffu, op, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        if constexpr (!kOne) op += __shfl_xor_sync(0xffffffffu, op, 4);
        if (t > 0) keep_o(t - 1, op);
        const float g = sBG[kKMax + t];
        const float u = sBG[t] * fmaf(-g, a, sV[t * kRows + row]);
        // S_t = g S_{t-1} + u k^_t, stored straight from registers (the intermediates streaming,
        // evict-first; the final state with the normal policy)
        float* dst = (t == K - 1) ? fin : inter + size_t(t) * inter_stride;
        const float2 gg = make_float2(g, g), uu = make_float2(u, u);
#pragma unroll
        for (int f = 0; f < F; ++f) {
          const float2 lo = __ffma2_rn(uu, make_float2(kv[f].x, kv[f].y), __fmul2_rn(gg, make_float2(s[f].x, s[f].y)));
          const float2 hi = __ffma2_rn(uu, make_float2(kv[f].z, kv[f].w), __fmul2_rn(gg, make_float2(s[f].z, s[f].w)));
          s[f] = make_float4(lo.x, lo.y, hi.x, hi.y);
          float4* d4 = reinterpret_cast<float4*>(dst + 32 * f);
          if (t == K - 1)
            *d4 = s[f];
          else
            __stcs(d4, s[f]);
        }
        // o_t = q_scale S_t q^_t: the lane's part now, the row's sum in the next token
        const float* qr = sY + (kKMax + t) * L::SSTRIDE + col;
        float2 b0 = make_float2(0.f, 0.f), b1 = make_float2(0.f, 0.f);
#pragma unroll
        for (int f = 0; f < F; ++f) {
          const float4 qv = *reinterpret_cast<const float4*>(qr + 32 * f);
          b0 = __ffma2_rn(make_float2(s[f].x, s[f].y), make_float2(qv.x, qv.y), b0);
          b1 = __ffma2_rn(make_float2(s[f].z, s[f].w), make_float2(qv.z, qv.w), b1);
        }
        op = (b0.x + b0.y) + (b1.x + b1.y);
      }
      op += __shfl_xor_sync(0xffffffffu, op, 1);
      op += __shfl_xor_sync(0xffffffffu, op, 2);
      op += __shfl_xor_sync(0xffffffffu, op, 4);
      keep_o(K - 1, op);
    }
    if constexpr (!kGated) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int t = cg + 8 * half;
        if (t < K) {
          const float o = half ? o_b : o_a;
          const size_t oi = (size_t(b) * K + t) * p.Hv * DV + size_t(h) * DV + r0 + row;
          if (p.out_f32)
            static_cast<float*>(p.out)[oi] = o;
          else
            static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16(o);
        }
      }
    }
  }  // ok

  if constexpr (kGated) {
    // out = o rsqrt(sum_rows o^2 / dv + eps) w SiLU(z) over the head's dv rows, which the cluster's
    // kTiles CTAs share: the sums of o^2 over each warp's 4 rows (lanes m = 0..3 of one column
    // group) go into every CTA of the cluster as asynchronous stores that complete on the
    // receiver's bar_sq.  A warp that timed out above still takes part with zeros: the peers
    // wait for its partials.
    float sq_a = o_a * o_a, sq_b = o_b * o_b;
    o_a *= nw * silu(bf16_to_f32(z_a));
    o_b *= nw * silu(bf16_to_f32(z_b));
    sq_a += __shfl_xor_sync(0xffffffffu, sq_a, 8);
    sq_a += __shfl_xor_sync(0xffffffffu, sq_a, 16);
    sq_b += __shfl_xor_sync(0xffffffffu, sq_b, 8);
    sq_b += __shfl_xor_sync(0xffffffffu, sq_b, 16);
    cluster_wait_acquire();  // every CTA of the cluster has started and set up bar_sq
    if (lane < 8) {
      const uint32_t rank = cluster_ctarank();
      const uint32_t slot = smem_addr(sm + L::OFF_X + ((rank * kWarps + warp) * (kKMax / 2) + lane) * 2);
      const uint32_t sbar = smem_addr(bar_sq);
      for (int d = 0; d < kTiles; ++d) st_async_cluster_f32x2(map_to_rank(slot, d), sq_a, sq_b, map_to_rank(sbar, d));
    }
    // every CTA waits here for all pushes into its shared memory, so none exits while a peer
    // still writes to it
    const bool got = mbar_wait_bounded(bar_sq, 0);
    if (!got) {  // (the peers' pushes still land before this CTA can exit)
      if (lane == 0) atomicOr(p.err, kDevErrTimeout);
      (void)mbar_drain(bar_sq, 0);
    }
    if (ok && got) {
      // lane (m, cg) adds the partials of warps m, m + 4, ...; the xor over the m bits completes
      const float2* sSq = reinterpret_cast<const float2*>(sm + L::OFF_X);
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
          const size_t oi = (size_t(b) * K + t) * p.Hv * DV + size_t(h) * DV + r0 + row;
          if (p.out_f32)
            static_cast<float*>(p.out)[oi] = y;
          else
            static_cast<uint16_t*>(p.out)[oi] = f32_to_bf16(y);
        }
      }
    }
  }
}

template <int DK, int DV, bool kTree, bool kGated, bool kOne>
cudaError_t launch_t(const VerifyParams& p, cudaStream_t stream) {
  auto k1 = gdn_verify_kernel<DK, DV, kTree, kGated, kOne>;
  const size_t b1 = VerifyLayout<DK, DV, kTree, kGated>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, int(b1));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(p.Hv * (DV / kRows)), unsigned(p.B), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = b1;
  cfg.stream = stream;
  // programmatic dependent launch: the CTAs may be scheduled while the previous kernel on the
  // stream finishes (they wait for it before any global read)
  cudaLaunchAttribute attr[2];
  cfg.attrs = attr;
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if constexpr (kGated) {  // the row tiles of one v-head form a cluster (they share the output norm)
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = DV / kRows;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  e = cudaLaunchKernelEx(&cfg, k1, p);
  if (e != cudaSuccess) return e;
  // the q|k histories, rewritten once every verify CTA has read them
  cudaLaunchConfig_t c2 = {};
  c2.gridDim = dim3(unsigned((p.Hk * DK + kHistThreads - 1) / kHistThreads), unsigned(p.B), 1);
  c2.blockDim = dim3(kHistThreads, 1, 1);
  c2.dynamicSmemBytes = 0;
  c2.stream = stream;
  cudaLaunchAttribute a2[1];
  a2[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a2[0].val.programmaticStreamSerializationAllowed = 1;
  c2.attrs = a2;
  c2.numAttrs = 1;
  return cudaLaunchKernelEx(&c2, gdn_qk_history_kernel<kTree>, p);
}

}  // namespace

cudaError_t launch_verify(const VerifyParams& p, cudaStream_t stream) {
  const bool tree = p.parent != nullptr;
  const bool gated = p.z != nullptr;
#define GDN_LAUNCH(DK_, DV_)                                          \
  if (p.dk == DK_ && p.dv == DV_) {                                   \
    if (tree) return launch_t<DK_, DV_, true, false, false>(p, stream); \
    if (p.K == 1)                                                       \
      return gated ? launch_t<DK_, DV_, false, true, true>(p, stream)   \
                   : launch_t<DK_, DV_, false, false, true>(p, stream); \
    return gated ? launch_t<DK_, DV_, false, true, false>(p, stream)    \
                 : launch_t<DK_, DV_, false, false, false>(p, stream);  \
  }
  GDN_LAUNCH(128, 128)
  GDN_LAUNCH(128, 64)
  GDN_LAUNCH(64, 128)
  GDN_LAUNCH(64, 64)
#undef GDN_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace gdn
