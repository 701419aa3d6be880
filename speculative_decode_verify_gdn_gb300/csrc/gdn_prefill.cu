// Chunked prefill of whole prompts through the GDN layer (sm_103a).
//
// The same recurrence as the verify step - causal conv1d + SiLU, L2 norm of q and k, raw
// gates, gated delta rule - over prompts of any length, packed token-major with cu_seqlens
// offsets (the packed layout of the VARLEN-FLA / FlashInfer-GDN prefill paths named in atlas
// #258 and #297).  Tokens are taken in chunks of 64 with the chunkwise (WY) form of the rule:
// per chunk, with Gamma_t = prod_{m<=t} g_m and D[t][j] = prod_{j<m<=t} g_m,
//   U   = W (V - diag(Gamma) K S^T)         W  = (I + diag(beta) (D o K K^T)_strict)^-1 diag(beta)
//   O   = q_scale (diag(Gamma) Q S^T + MQ U)  MQ = (D o Q K^T)_lower incl. diagonal
//   S' = Gamma_63 S + (diag(d) U)^T K         d_t = D[63][t]
// (rows of U, O are tokens; S is [dv x dk] with row = v index).
//
// Three kernels:
//   gdn_prefill_index_kernel   one CTA: checks cu_seqlens, numbers the chunks of all prompts;
//   gdn_prefill_chunk_kernel   one CTA per (chunk, q/k head), all chunks in parallel: conv of the
//                              q|k channels, L2 norms, Gram products, gates, decay products and
//                              the 64 x 64 triangular inverse of every v-head of the group;
//   gdn_prefill_state_kernel   one CTA per (prompt, v-head, 32 state rows): walks the prompt's
//                              chunks in order with the state tile in shared memory, the next
//                              chunk's tables arriving by bulk copy (double-buffered) while
//                              the current one is computed; convolves its own v channels.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kCh = kPrefillChunk;   // 64 tokens per chunk
constexpr int kAS = kCh + 1;         // row stride of the packed W | MQ block
constexpr int kTileRows = 32;        // state rows per state-kernel CTA

__device__ __forceinline__ long long min_ll(long long a, long long b) { return a < b ? a : b; }

__device__ __forceinline__ float gate_g(float a, float A_log, float dt_bias) {
  const float A = -expf(A_log);
  const float av = a + dt_bias;
  const float sp = (av > 20.f) ? av : log1pf(expf(av));
  return expf(sp * A);
}

__device__ __forceinline__ float gate_beta(float b) { return 1.f / (1.f + expf(-b)); }

// Position (in floats) of element (t, c) of a 64 x DK token-major table: float4 groups are
// XOR-swizzled with t & 7 so that eight rows read at the same column hit different banks.
template <int DK>
__device__ __forceinline__ int swz(int t, int c4) {
  return t * DK + ((c4 ^ (t & 7)) << 2);
}

// ------------------------------------------------------------------------------------------
// Kernel 0: cu_seqlens check and chunk numbering (one CTA of 1024 threads).
__global__ void __launch_bounds__(1024) gdn_prefill_index_kernel(const PrefillParams p) {
  __shared__ long long part[1024];
  __shared__ int bad;
  const int tid = threadIdx.x;
  if (tid == 0) bad = 0;
  __syncthreads();
  const int B = p.B;
  const int per = (B + 1023) / 1024;
  const int i0 = min(B, tid * per), i1 = min(B, i0 + per);
  long long sum = 0;
  int my_bad = 0;
  for (int i = i0; i < i1; ++i) {
    const long long s = p.cu[i], e = p.cu[i + 1];
    if (e < s)
      my_bad = 1;
    else
      sum += (e - s + kCh - 1) / kCh;
  }
  if (tid == 0 && (p.cu[0] != 0 || p.cu[B] != p.N)) my_bad = 1;
  if (my_bad) atomicOr(&bad, 1);
  part[tid] = sum;
  __syncthreads();
  for (int off = 1; off < 1024; off <<= 1) {  // inclusive scan of the per-thread chunk counts
    const long long v = tid >= off ? part[tid - off] : 0;
    __syncthreads();
    part[tid] += v;
    __syncthreads();
  }
  int32_t* base = p.ws.meta + 4;
  long long run = tid ? part[tid - 1] : 0;
  for (int i = i0; i < i1; ++i) {
    base[i] = int32_t(run);
    const long long s = p.cu[i], e = p.cu[i + 1];
    if (e >= s) run += (e - s + kCh - 1) / kCh;
  }
  if (tid == 1023) {
    const bool ok = !bad && part[1023] <= p.ws.chunk_cap;
    base[B] = int32_t(part[1023]);
    p.ws.meta[1] = ok ? int32_t(part[1023]) : 0;
    p.ws.meta[0] = ok ? 1 : 0;
    if (!ok) atomicOr(p.err, kDevErrSeqlens);
  }
}

// Prompt i holding global chunk c: the largest i with base[i] <= c (empty prompts share their
// successor's base, so the largest one is the prompt that owns the chunk).
__device__ __forceinline__ int prompt_of_chunk(const int32_t* base, int B, int c) {
  int lo = 0, hi = B - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= c)
      lo = mid;
    else
      hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------------------------------------
// Kernel 1: per (chunk, q/k head).
template <int DK>
struct ChunkLayout {
  static constexpr int YS = 2 * DK + 4;                       // row stride of the q|k conv table
  static constexpr int Y_FLOATS = kCh * YS;
  static constexpr int MAT = kCh * kAS;                       // one 64 x 65 matrix
  static constexpr int OFF_Y = 0;                             // [64][YS]: q (0..DK-1) | k (DK..2DK-1)
  static constexpr int OFF_D = 0;                             // after the Gram products: D, then X
  static constexpr int OFF_L = MAT;                           //   beta D (k.k), strictly lower
  static constexpr int R_FLOATS = (Y_FLOATS > 2 * MAT) ? Y_FLOATS : 2 * MAT;
  static constexpr int OFF_KK = R_FLOATS;                     // [64][65] k^_t . k^_j
  static constexpr int OFF_QK = OFF_KK + MAT;                 // [64][65] q^_t . k^_j
  static constexpr int OFF_BG = OFF_QK + MAT;                 // beta[64], g[64], Gamma[64]
  static constexpr int FLOATS = OFF_BG + 3 * kCh;
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
};

template <int DK>
__global__ void __launch_bounds__(kThreads, 2) gdn_prefill_chunk_kernel(const PrefillParams p) {
  using L = ChunkLayout<DK>;
  extern __shared__ __align__(128) float sm[];
  const int tid = threadIdx.x;
  const int c = blockIdx.x;
  const int kh = blockIdx.y;
  const int32_t* meta = p.ws.meta;
  if (meta[0] == 0 || c >= meta[1]) return;
  const int32_t* base = meta + 4;
  const int i = prompt_of_chunk(base, p.B, c);
  const long long s0 = p.cu[i], s1 = p.cu[i + 1];
  const long long tok0 = s0 + (long long)(c - base[i]) * kCh;
  const int len = int(min_ll(kCh, s1 - tok0));
  const size_t C = size_t(p.C);
  const int r = p.Hv / p.Hk;

  // a1 for the head's 2 DK q|k channels, one thread per channel walking the chunk; the three
  // rows before the chunk come from the prompt itself or, at its start, from the history
  float* sY = sm + L::OFF_Y;
  for (int ch = tid; ch < 2 * DK; ch += kThreads) {
    const size_t gch = (ch < DK) ? size_t(kh) * DK + ch : size_t(p.Hk) * DK + size_t(kh) * DK + (ch - DK);
    const float4 w = *reinterpret_cast<const float4*>(p.conv_w + gch * kConvW);
    float h[3];
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const long long pos = tok0 - 3 + m;
      h[m] = (pos >= s0) ? bf16_to_f32(p.x[size_t(pos) * C + gch])
                         : p.conv_state_in[(size_t(i) * 3 + size_t(pos - s0 + 3)) * C + gch];
    }
    float h0 = h[0], h1 = h[1], h2 = h[2];
#pragma unroll 8
    for (int t = 0; t < kCh; ++t) {
      const float xv = (t < len) ? bf16_to_f32(p.x[size_t(tok0 + t) * C + gch]) : 0.f;
      const float z = fmaf(w.w, xv, fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0)));
      sY[t * L::YS + ch] = (t < len) ? silu(z) : 0.f;
      h0 = h1;
      h1 = h2;
      h2 = xv;
    }
  }
  __syncthreads();

  // a2: one warp per (token, q|k) vector
  {
    const int warp = tid >> 5, lane = tid & 31;
    for (int v = warp; v < 2 * kCh; v += kThreads / 32) {
      const int t = v >> 1, off = (v & 1) * DK;
      float* row = sY + t * L::YS + off;
      float ss = 0.f;
#pragma unroll
      for (int e = lane; e < DK; e += 32) ss = fmaf(row[e], row[e], ss);
      ss = warp_sum(ss);
      const float inv = (t < len) ? rsqrtf(ss + p.l2_eps) : 0.f;
#pragma unroll
      for (int e = lane; e < DK; e += 32) row[e] *= inv;
    }
  }
  __syncthreads();

  // normalised k^ and q^ to the workspace, token-major and swizzled: [2][64][DK]
  {
    float* dst = p.ws.kq + (size_t(c) * p.Hk + kh) * 2 * kCh * DK;
    constexpr int C4 = DK / 4;
    for (int idx = tid; idx < 2 * kCh * C4; idx += kThreads) {
      const int part = idx / (kCh * C4);           // 0: k^, 1: q^
      const int t = (idx / C4) % kCh, c4 = idx % C4;
      const float4 v = *reinterpret_cast<const float4*>(sY + t * L::YS + (part ? 0 : DK) + 4 * c4);
      *reinterpret_cast<float4*>(dst + size_t(part) * kCh * DK + swz<DK>(t, c4)) = v;
    }
  }

  // Gram products k^_t . k^_j and q^_t . k^_j: thread (tb, jb) takes t = tb + 16a, j = jb + 16b
  {
    const int tb = tid >> 4, jb = tid & 15;
    float kk[4][4], qk[4][4];
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) kk[a][bb] = qk[a][bb] = 0.f;
#pragma unroll 2
    for (int c4 = 0; c4 < DK / 4; ++c4) {
      float4 kt[4], qt[4], kj[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) {
        kt[a] = *reinterpret_cast<const float4*>(sY + (tb + 16 * a) * L::YS + DK + 4 * c4);
        qt[a] = *reinterpret_cast<const float4*>(sY + (tb + 16 * a) * L::YS + 4 * c4);
        kj[a] = *reinterpret_cast<const float4*>(sY + (jb + 16 * a) * L::YS + DK + 4 * c4);
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          kk[a][bb] = fmaf(kt[a].x, kj[bb].x, fmaf(kt[a].y, kj[bb].y, fmaf(kt[a].z, kj[bb].z, fmaf(kt[a].w, kj[bb].w, kk[a][bb]))));
          qk[a][bb] = fmaf(qt[a].x, kj[bb].x, fmaf(qt[a].y, kj[bb].y, fmaf(qt[a].z, kj[bb].z, fmaf(qt[a].w, kj[bb].w, qk[a][bb]))));
        }
    }
#pragma unroll
    for (int a = 0; a < 4; ++a)
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {
        sm[L::OFF_KK + (tb + 16 * a) * kAS + jb + 16 * bb] = kk[a][bb];
        sm[L::OFF_QK + (tb + 16 * a) * kAS + jb + 16 * bb] = qk[a][bb];
      }
  }
  __syncthreads();  // the q|k table is dead from here: its space holds D, X and beta D (k.k)

  float* sD = sm + L::OFF_D;  // D[t][j] (j <= t), later X = (I + beta D o KK)^-1
  float* sL = sm + L::OFF_L;
  float* sBeta = sm + L::OFF_BG;
  float* sG = sBeta + kCh;
  float* sGam = sG + kCh;
  for (int e = 0; e < r; ++e) {
    const int h = kh * r + e;
    // a3 for this v-head (padding tokens: beta = 0, g = 1, so they change nothing)
    if (tid < kCh) {
      float beta = 0.f, g = 1.f;
      if (tid < len) {
        const size_t gi = size_t(tok0 + tid) * p.Hv + h;
        g = gate_g(bf16_to_f32(p.a[gi]), p.A_log[h], p.dt_bias[h]);
        beta = gate_beta(bf16_to_f32(p.b[gi]));
      }
      sBeta[tid] = beta;
      sG[tid] = g;
    }
    __syncthreads();
    // decay products: column j runs down the rows; thread 64 forms Gamma
    if (tid < kCh) {
      const int j = tid;
      float dcur = 1.f;
      sD[j * kAS + j] = 1.f;
      for (int t = j + 1; t < kCh; ++t) {
        dcur *= sG[t];
        sD[t * kAS + j] = dcur;
      }
    } else if (tid == kCh) {
      float gam = 1.f;
      for (int t = 0; t < kCh; ++t) {
        gam *= sG[t];
        sGam[t] = gam;
      }
    }
    __syncthreads();
    float* A = p.ws.wm + (size_t(c) * p.Hv + h) * (kCh * kAS);
    float* gd = p.ws.gd + (size_t(c) * p.Hv + h) * (2 * kCh);
    // beta_t D (k.k) strictly below the diagonal; MQ[t][j] = D (q.k) to A[j][t + 1]; Gamma, d
    for (int idx = tid; idx < kCh * kCh; idx += kThreads) {
      const int j = idx / kCh, t = idx % kCh;
      if (j < t) sL[t * kAS + j] = sBeta[t] * sD[t * kAS + j] * sm[L::OFF_KK + t * kAS + j];
      if (j <= t) A[j * kAS + t + 1] = sD[t * kAS + j] * sm[L::OFF_QK + t * kAS + j];
    }
    if (tid < kCh) {
      gd[tid] = sGam[tid];
      gd[kCh + tid] = sD[(kCh - 1) * kAS + tid];
    }
    __syncthreads();
    // X = (I + L)^-1 by forward substitution, column j by four lanes (m split mod 4); X
    // overwrites D (each lane reads back only the X entries it wrote itself)
    {
      const int j = tid >> 2, part = tid & 3;
      const unsigned mask = 0xFu << (threadIdx.x & 28);
      if (part == 0) sD[j * kAS + j] = 1.f;
      for (int t = j + 1; t < kCh; ++t) {
        float s = 0.f;
        for (int m = j + part; m < t; m += 4) s = fmaf(sL[t * kAS + m], sD[m * kAS + j], s);
        s += __shfl_xor_sync(mask, s, 1);
        s += __shfl_xor_sync(mask, s, 2);
        if (part == ((t - j) & 3)) sD[t * kAS + j] = -s;
      }
    }
    __syncthreads();
    // W = X diag(beta) on and below the diagonal
    for (int idx = tid; idx < kCh * kCh; idx += kThreads) {
      const int t = idx / kCh, j = idx % kCh;
      if (j <= t) A[t * kAS + j] = sD[t * kAS + j] * sBeta[j];
    }
    __syncthreads();
  }
}

// ------------------------------------------------------------------------------------------
// Kernel 2: per (prompt, v-head, 32 state rows), sequential over the prompt's chunks.
template <int DK>
struct StateLayout {
  static constexpr int KQ = 2 * kCh * DK;                     // k^ then q^, swizzled
  static constexpr int STAGE = KQ + kCh * kAS + 2 * kCh;      // + W|MQ + Gamma, d
  static constexpr int SS = DK + 4;                           // state tile row stride
  static constexpr int XS = 36;                               // raw x row stride
  static constexpr int OFF_ST = 0;                            // two stages
  static constexpr int OFF_S = 2 * STAGE;                     // [32][SS]
  static constexpr int OFF_X = OFF_S + kTileRows * SS;        // [67][XS]: 3 history rows, 64 tokens
  static constexpr int OFF_VRU = OFF_X + ((67 * XS + 3) & ~3);  // [32][65]: v, then r, then u
  static constexpr int OFF_PQO = OFF_VRU + ((kTileRows * kAS + 3) & ~3);  // [32][65]: S q^, then o
  static constexpr int OFF_TAP = OFF_PQO + ((kTileRows * kAS + 3) & ~3);  // [32][4] conv taps
  static constexpr int OFF_BAR = OFF_TAP + kTileRows * 4;     // two mbarriers
  static constexpr int FLOATS = OFF_BAR + 4;
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
  static constexpr uint32_t KQ_BYTES = KQ * 4;
  static constexpr uint32_t A_BYTES = kCh * kAS * 4;
  static constexpr uint32_t GD_BYTES = 2 * kCh * 4;
  static_assert(STAGE % 4 == 0 && (KQ + kCh * kAS) % 4 == 0 && OFF_S % 4 == 0 && OFF_X % 4 == 0, "16-byte alignment");
  static_assert(A_BYTES % 16 == 0, "bulk copy size");
};

template <int DK>
__device__ __forceinline__ void issue_chunk(const PrefillParams& p, float* stage, uint64_t* bar, int c, int kh, int h) {
  using L = StateLayout<DK>;
  mbar_arrive_expect_tx(bar, L::KQ_BYTES + L::A_BYTES + L::GD_BYTES);
  bulk_load(stage, p.ws.kq + (size_t(c) * p.Hk + kh) * L::KQ, L::KQ_BYTES, bar);
  bulk_load(stage + L::KQ, p.ws.wm + (size_t(c) * p.Hv + h) * (kCh * kAS), L::A_BYTES, bar);
  bulk_load(stage + L::KQ + kCh * kAS, p.ws.gd + (size_t(c) * p.Hv + h) * (2 * kCh), L::GD_BYTES, bar);
}

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads, 1) gdn_prefill_state_kernel(const PrefillParams p) {
  using L = StateLayout<DK>;
  extern __shared__ __align__(128) float sm[];
  constexpr int kTiles = DV / kTileRows;
  const int tid = threadIdx.x;
  const int i = blockIdx.y;
  const int h = blockIdx.x / kTiles;
  const int tile = blockIdx.x % kTiles;
  const int r0 = tile * kTileRows;
  const int kh = h / (p.Hv / p.Hk);
  if (p.ws.meta[0] == 0) return;
  const int32_t* base = p.ws.meta + 4;
  const int c_first = base[i], n_chunks = base[i + 1] - base[i];
  const long long s0 = p.cu[i], s1 = p.cu[i + 1];
  const size_t C = size_t(p.C);
  const size_t vch0 = size_t(2) * p.Hk * DK + size_t(h) * DV + r0;  // first conv channel of the tile
  float* sS = sm + L::OFF_S;
  float* sX = sm + L::OFF_X;
  float* sVRU = sm + L::OFF_VRU;
  float* sPQO = sm + L::OFF_PQO;
  float* sTap = sm + L::OFF_TAP;
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);

  if (tid == 0) {
    mbar_init(bar, 1);
    mbar_init(bar + 1, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    for (int q = 0; q < 2 && q < n_chunks; ++q) issue_chunk<DK>(p, sm + q * L::STAGE, bar + q, c_first + q, kh, h);
  }
  // state tile, conv taps and the three history rows of the tile's v channels
  {
    const float* src = p.state_in + ((size_t(i) * p.Hv + h) * DV + r0) * DK;
    for (int idx = tid; idx < kTileRows * DK / 4; idx += kThreads) {
      const int row = idx / (DK / 4), c4 = idx % (DK / 4);
      *reinterpret_cast<float4*>(sS + row * L::SS + 4 * c4) = *reinterpret_cast<const float4*>(src + size_t(row) * DK + 4 * c4);
    }
    if (tid < kTileRows) *reinterpret_cast<float4*>(sTap + 4 * tid) = *reinterpret_cast<const float4*>(p.conv_w + (vch0 + tid) * kConvW);
    if (tid < 3 * kTileRows) {
      const int m = tid / kTileRows, ch = tid % kTileRows;
      sX[m * L::XS + ch] = p.conv_state_in[(size_t(i) * 3 + m) * C + vch0 + ch];
    }
  }
  // raw x of the tile's 32 channels for one chunk: thread = (token tid / 4, 8 channels)
  const int xt = tid >> 2, xg = tid & 3;
  uint4 xr = make_uint4(0, 0, 0, 0);
  if (n_chunks > 0 && xt < min_ll(kCh, s1 - s0))
    xr = *reinterpret_cast<const uint4*>(p.x + size_t(s0 + xt) * C + vch0 + 8 * xg);
  __syncthreads();

  int len = 0;
  for (int lc = 0; lc < n_chunks; ++lc) {
    const int st = lc & 1;
    float* stage = sm + st * L::STAGE;
    const float* sK = stage;
    const float* sQ = stage + kCh * DK;
    const float* sA = stage + L::KQ;
    const float* sGam = sA + kCh * kAS;
    const float* sd = sGam + kCh;
    const long long tok0 = s0 + (long long)lc * kCh;
    len = int(min_ll(kCh, s1 - tok0));

    // raw x of this chunk to rows 3..66; the next chunk's x is fetched meanwhile
    {
      const uint32_t wv[4] = {xr.x, xr.y, xr.z, xr.w};
      float* row = sX + (xt + 3) * L::XS + 8 * xg;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        row[2 * q] = (xt < len) ? bf16_to_f32(uint16_t(wv[q] & 0xFFFFu)) : 0.f;
        row[2 * q + 1] = (xt < len) ? bf16_to_f32(uint16_t(wv[q] >> 16)) : 0.f;
      }
      const long long nt = tok0 + kCh + xt;
      if (lc + 1 < n_chunks && nt < s1) xr = *reinterpret_cast<const uint4*>(p.x + size_t(nt) * C + vch0 + 8 * xg);
    }
    // the chunk's tables (bounded wait; the outcome is made uniform over the CTA)
    const bool ok = mbar_wait_bounded(bar + st, (lc >> 1) & 1);
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        atomicOr(p.err, kDevErrTimeout);
        (void)mbar_wait_bounded(bar + (st ^ 1), ((lc + 1) >> 1) & 1);  // copies still in flight
      }
      return;
    }

    // a1 for the v channels: v[ch][t] = SiLU(taps . rows t..t+3)
    {
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int ch = 8 * xg + q;
        const float4 w = *reinterpret_cast<const float4*>(sTap + 4 * ch);
        const float z = fmaf(w.w, sX[(xt + 3) * L::XS + ch],
                             fmaf(w.z, sX[(xt + 2) * L::XS + ch], fmaf(w.y, sX[(xt + 1) * L::XS + ch], w.x * sX[xt * L::XS + ch])));
        sVRU[ch * kAS + xt] = silu(z);
      }
    }
    __syncthreads();

    // S [k^ | q^]: thread (part, rb, tb) takes rows rb + 8a, tokens tb + 16b; for k^ the
    // epilogue forms r = v - Gamma (S k^) in place of v, for q^ it keeps S q^
    {
      const int part = tid >> 7, rb = (tid >> 4) & 7, tb = tid & 15;
      const float* tab = part ? sQ : sK;
      float acc[4][4];
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) acc[a][bb] = 0.f;
#pragma unroll 2
      for (int c4 = 0; c4 < DK / 4; ++c4) {
        float4 sv[4], kv[4];
#pragma unroll
        for (int a = 0; a < 4; ++a) sv[a] = *reinterpret_cast<const float4*>(sS + (rb + 8 * a) * L::SS + 4 * c4);
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) kv[bb] = *reinterpret_cast<const float4*>(tab + swz<DK>(tb + 16 * bb, c4));
#pragma unroll
        for (int a = 0; a < 4; ++a)
#pragma unroll
          for (int bb = 0; bb < 4; ++bb)
            acc[a][bb] = fmaf(sv[a].x, kv[bb].x, fmaf(sv[a].y, kv[bb].y, fmaf(sv[a].z, kv[bb].z, fmaf(sv[a].w, kv[bb].w, acc[a][bb]))));
      }
#pragma unroll
      for (int a = 0; a < 4; ++a)
#pragma unroll
        for (int bb = 0; bb < 4; ++bb) {
          const int row = rb + 8 * a, t = tb + 16 * bb;
          if (part == 0)
            sVRU[row * kAS + t] = fmaf(-sGam[t], acc[a][bb], sVRU[row * kAS + t]);
          else
            sPQO[row * kAS + t] = acc[a][bb];
        }
      // the last three rows become the next chunk's history (the conv above is done with them)
      if (tid < 3 * kTileRows && len == kCh) {
        const int m = tid / kTileRows, ch = tid % kTileRows;
        sX[m * L::XS + ch] = sX[(kCh + m) * L::XS + ch];
      }
    }
    __syncthreads();

    // u = W r: thread (row, tg) takes tokens tg + 8k
    const int urow = tid >> 3, tg = tid & 7;
    {
      float u[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) u[k] = 0.f;
      for (int j = 0; j < kCh; ++j) {
        const float rj = sVRU[urow * kAS + j];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int t = tg + 8 * k;
          u[k] = fmaf((j <= t) ? sA[t * kAS + j] : 0.f, rj, u[k]);
        }
      }
      __syncthreads();  // every r is read
#pragma unroll
      for (int k = 0; k < 8; ++k) sVRU[urow * kAS + tg + 8 * k] = u[k];
    }
    __syncthreads();

    // o = q_scale (Gamma S q^ + MQ u), in place of S q^
    {
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const int t = tg + 8 * k;
        o[k] = sGam[t] * sPQO[urow * kAS + t];
      }
      for (int j = 0; j < kCh; ++j) {
        const float uj = sVRU[urow * kAS + j];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int t = tg + 8 * k;
          o[k] = fmaf((j <= t) ? sA[j * kAS + t + 1] : 0.f, uj, o[k]);
        }
      }
#pragma unroll
      for (int k = 0; k < 8; ++k) sPQO[urow * kAS + tg + 8 * k] = p.q_scale * o[k];
    }
    // S <- Gamma_63 S + sum_t d_t u_t k^_t^T: thread (row, q8) owns float4 columns q8 + 8m
    {
      constexpr int NF = DK / 32;
      float4 s[NF];
      const float gl = sGam[kCh - 1];
#pragma unroll
      for (int m = 0; m < NF; ++m) {
        const float4 v = *reinterpret_cast<const float4*>(sS + urow * L::SS + 4 * (tg + 8 * m));
        s[m] = make_float4(gl * v.x, gl * v.y, gl * v.z, gl * v.w);
      }
      for (int t = 0; t < kCh; ++t) {
        const float cu = sd[t] * sVRU[urow * kAS + t];
#pragma unroll
        for (int m = 0; m < NF; ++m) {
          const float4 kv = *reinterpret_cast<const float4*>(sK + swz<DK>(t, tg + 8 * m));
          s[m].x = fmaf(cu, kv.x, s[m].x);
          s[m].y = fmaf(cu, kv.y, s[m].y);
          s[m].z = fmaf(cu, kv.z, s[m].z);
          s[m].w = fmaf(cu, kv.w, s[m].w);
        }
      }
#pragma unroll
      for (int m = 0; m < NF; ++m) *reinterpret_cast<float4*>(sS + urow * L::SS + 4 * (tg + 8 * m)) = s[m];
    }
    __syncthreads();  // stage st is free; o is complete

    if (tid == 0 && lc + 2 < n_chunks) issue_chunk<DK>(p, stage, bar + st, c_first + lc + 2, kh, h);
    // outputs: thread = (token xt, rows 8 xg .. 8 xg + 7)
    if (xt < len) {
      float ov[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) ov[q] = sPQO[(8 * xg + q) * kAS + xt];
      const size_t oi = size_t(tok0 + xt) * p.Hv * DV + size_t(h) * DV + r0 + 8 * xg;
      if (p.out_f32) {
        float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi);
        o4[0] = make_float4(ov[0], ov[1], ov[2], ov[3]);
        o4[1] = make_float4(ov[4], ov[5], ov[6], ov[7]);
      } else {
        uint4 pk;
        pk.x = uint32_t(f32_to_bf16(ov[0])) | (uint32_t(f32_to_bf16(ov[1])) << 16);
        pk.y = uint32_t(f32_to_bf16(ov[2])) | (uint32_t(f32_to_bf16(ov[3])) << 16);
        pk.z = uint32_t(f32_to_bf16(ov[4])) | (uint32_t(f32_to_bf16(ov[5])) << 16);
        pk.w = uint32_t(f32_to_bf16(ov[6])) | (uint32_t(f32_to_bf16(ov[7])) << 16);
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + oi) = pk;
      }
    }
  }

  // final state tile
  {
    float* dst = p.state_out + ((size_t(i) * p.Hv + h) * DV + r0) * DK;
    for (int idx = tid; idx < kTileRows * DK / 4; idx += kThreads) {
      const int row = idx / (DK / 4), c4 = idx % (DK / 4);
      *reinterpret_cast<float4*>(dst + size_t(row) * DK + 4 * c4) = *reinterpret_cast<const float4*>(sS + row * L::SS + 4 * c4);
    }
  }
  // conv history: the v channels from the last three rows held in shared memory (rows len ..
  // len + 2 of the last chunk, or the untouched history of an empty prompt)
  if (tid < 3 * kTileRows) {
    const int m = tid / kTileRows, ch = tid % kTileRows;
    p.conv_state_out[(size_t(i) * 3 + m) * C + vch0 + ch] = sX[(len + m) * L::XS + ch];
  }
  // the q|k channels of the head group, split over the first v-head's row tiles; every value
  // is read before this thread writes, and no other thread of this grid reads them
  if (h % (p.Hv / p.Hk) == 0) {
    constexpr int kPer = 2 * DK / kTiles;
    for (int q = tid; q < kPer; q += kThreads) {
      const int ch = tile * kPer + q;
      const size_t gch = (ch < DK) ? size_t(kh) * DK + ch : size_t(p.Hk) * DK + size_t(kh) * DK + (ch - DK);
      float hv[3];
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        const long long pos = s1 - 3 + m;
        hv[m] = (pos >= s0) ? bf16_to_f32(p.x[size_t(pos) * C + gch])
                            : p.conv_state_in[(size_t(i) * 3 + size_t(pos - s0 + 3)) * C + gch];
      }
#pragma unroll
      for (int m = 0; m < 3; ++m) p.conv_state_out[(size_t(i) * 3 + m) * C + gch] = hv[m];
    }
  }
}

template <int DK, int DV>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t stream) {
  auto k1 = gdn_prefill_chunk_kernel<DK>;
  auto k2 = gdn_prefill_state_kernel<DK, DV>;
  const size_t b1 = ChunkLayout<DK>::BYTES, b2 = StateLayout<DK>::BYTES;
  cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, int(b1));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, int(b2));
  if (e != cudaSuccess) return e;
  gdn_prefill_index_kernel<<<1, 1024, 0, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k1<<<dim3(unsigned(p.ws.chunk_cap), unsigned(p.Hk), 1), kThreads, b1, stream>>>(p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k2<<<dim3(unsigned(p.Hv * (DV / kTileRows)), unsigned(p.B), 1), kThreads, b2, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_workspace_bytes(int B, long long N, int Hk, int Hv, int dk) {
  const long long cap = prefill_chunk_cap(B, N);
  const size_t meta = ((size_t(B) + 5 + 3) & ~size_t(3)) * 4;
  return meta + size_t(cap) * 4 * (size_t(Hk) * 2 * kCh * dk + size_t(Hv) * (kCh * kAS + 2 * kCh));
}

PrefillWorkspace prefill_workspace_carve(void* base, int B, long long N, int Hk, int Hv, int dk) {
  PrefillWorkspace w;
  w.chunk_cap = prefill_chunk_cap(B, N);
  char* p = static_cast<char*>(base);
  w.meta = reinterpret_cast<int32_t*>(p);
  p += ((size_t(B) + 5 + 3) & ~size_t(3)) * 4;
  w.kq = reinterpret_cast<float*>(p);
  p += size_t(w.chunk_cap) * Hk * 2 * kCh * dk * 4;
  w.wm = reinterpret_cast<float*>(p);
  p += size_t(w.chunk_cap) * Hv * kCh * kAS * 4;
  w.gd = reinterpret_cast<float*>(p);
  return w;
}

cudaError_t launch_prefill(const PrefillParams& p, cudaStream_t stream) {
#define GDN_PF_LAUNCH(DK_, DV_) \
  if (p.dk == DK_ && p.dv == DV_) return launch_prefill_t<DK_, DV_>(p, stream);
  GDN_PF_LAUNCH(128, 128)
  GDN_PF_LAUNCH(128, 64)
  GDN_PF_LAUNCH(64, 128)
  GDN_PF_LAUNCH(64, 64)
#undef GDN_PF_LAUNCH
  return cudaErrorInvalidValue;
}

}  // namespace gdn
