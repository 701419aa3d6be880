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
//   gdn_prefill_state128_kernel (dv = 128) one CTA per (prompt, v-head), the whole state as one
//                              M = 128 tile; gdn_prefill_state_kernel (dv = 64) one CTA per
//                              (prompt, v-head, 64 state rows), M = 64: both walk the prompt's
//                              chunks in order on the tensor cores with the state in tensor
//                              memory, the next chunk's operands arriving by bulk copy while the
//                              current one is computed, and convolve their own v channels.
#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace gdn {
namespace {

__device__ __forceinline__ long long min_ll(long long a, long long b) { return a < b ? a : b; }

constexpr int kThreads = 256;
constexpr int kCh = kPrefillChunk;   // 64 tokens per chunk
constexpr int kAS = kCh + 4;         // row stride of the chunk kernel's 64 x 64 D, L and X tables: 16-byte
                                     // rows four banks apart, so a quarter-warp's 16-byte accesses to eight
                                     // consecutive rows (or to one row) meet no bank twice
constexpr int kY2S = 36;             // row stride of the inverse's 32 x 32 product temp (same reason)
constexpr int kTileRows = 64;        // state rows per state-kernel CTA (the MMA M)
constexpr int kKqBlocks = 4;         // k^ hi, lo, q^ hi, lo per (chunk, q/k head)
constexpr int kAbHeads = 2;          // v-heads per q/k head whose gate inputs the chunk kernel prefetches

__device__ __forceinline__ float gate_beta(float b) { return 1.f / (1.f + expf(-b)); }

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
  const bool valid = !bad && part[1023] <= p.ws.chunk_cap;
  for (int i = i0; i < i1; ++i) {
    base[i] = int32_t(run);
    const long long s = p.cu[i], e = p.cu[i + 1];
    if (e >= s) {
      const int n = int((e - s + kCh - 1) / kCh);
      if (valid)  // one record per chunk: prompt, first token, tokens, first token of the prompt
        for (int lc = 0; lc < n; ++lc)
          p.ws.chunks[run + lc] = make_int4(i, int(s) + lc * kCh, int(min_ll(kCh, e - s - lc * kCh)), int(s));
      run += n;
    }
  }
  if (tid == 1023) {
    base[B] = int32_t(part[1023]);
    p.ws.meta[1] = valid ? int32_t(part[1023]) : 0;
    p.ws.meta[0] = valid ? 1 : 0;
    if (!valid) atomicOr(p.err, kDevErrSeqlens);
  }
}

// One product of the chunk form as three bf16 MMA chains over hi/lo operand pairs (hi.hi, hi.lo,
// lo.hi) of KSTEPS steps of K = 16 each.  Descriptors are formed once; a K step moves the start
// address field by 256 bytes (two core matrices).
template <int KSTEPS>
__device__ __forceinline__ void umma_split3(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                            uint32_t sbo, uint32_t idesc, bool accumulate) {
  const uint64_t dah = umma_smem_desc(a_hi, 128, sbo), dal = umma_smem_desc(a_lo, 128, sbo);
  const uint64_t dbh = umma_smem_desc(b_hi, 128, sbo), dbl = umma_smem_desc(b_lo, 128, sbo);
#pragma unroll
  for (int sp = 0; sp < 3; ++sp) {
    const uint64_t da = (sp == 2) ? dal : dah;
    const uint64_t db = (sp == 1) ? dbl : dbh;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk)
      umma_bf16(d, da + uint64_t(16 * kk), db + uint64_t(16 * kk), idesc, (accumulate || sp > 0 || kk > 0) ? 1u : 0u);
  }
}

// ------------------------------------------------------------------------------------------
// Kernel 1: per (chunk, q/k head).
template <int DK>
struct ChunkLayout {
  static constexpr int YS = 2 * DK + 4;                       // row stride of the q|k conv table
  static_assert(YS % 4 == 0, "16-byte rows");
  static constexpr int Y_FLOATS = kCh * YS;
  static constexpr int MAT = kCh * kAS;                       // one 64 x 68 matrix
  static constexpr int OFF_Y = 0;                             // [64][YS]: q (0..DK-1) | k (DK..2DK-1)
  // after the Gram products, per v-head group g (two v-heads at a time): D, then X, at
  // OFF_D + 2 g MAT, and beta D (k.k) strictly lower just after it
  static constexpr int OFF_D = 0;
  static constexpr int R_FLOATS = (Y_FLOATS > 4 * MAT) ? Y_FLOATS : 4 * MAT;
  static constexpr int OFF_KK = R_FLOATS;                     // [64][64] k^_t . k^_j, swizzled (gram_off)
  static constexpr int OFF_QK = OFF_KK + kCh * kCh;           // [64][64] q^_t . k^_j, swizzled
  static constexpr int OFF_BG = OFF_QK + kCh * kCh;           // per group: beta[64], g[64], Gamma[64]
  static constexpr int OFF_Y2 = OFF_BG + 2 * 3 * kCh;         // per group: [32][kY2S] product temp of the inverse
  static constexpr int OFF_AB = OFF_Y2 + 2 * 32 * kY2S;       // a, b of the first kAbHeads v-heads [e][2][64]
  static constexpr int OFF_QKD = OFF_AB + kAbHeads * 2 * kCh; // q^_t . k^_t in f32 [64]
  static constexpr int OFF_BAR = (OFF_QKD + kCh + 1) & ~1;    // 2 mbarriers, the TMEM slot
  static constexpr int FLOATS = OFF_BAR + 6;
  static_assert(4 * kCh * DK * 2 <= R_FLOATS * 4, "the split q|k operands fit in the conv table's space");
  static_assert(MAT % 4 == 0 && OFF_KK % 4 == 0 && OFF_BG % 4 == 0 && OFF_Y2 % 4 == 0 && (32 * kY2S) % 4 == 0,
                "16-byte aligned tables");
  static constexpr size_t BYTES = size_t(FLOATS) * 4;
  // two CTAs per SM: each takes its bytes plus 1 KB reserved, in 128-byte units, of the SM's 228 KB
  static_assert(2 * ((BYTES + 1024 + 127) / 128 * 128) <= 228 * 1024, "two chunk-kernel CTAs per SM");
};

// Offset of element (t, j) in the k^.k^ and q^.k^ tables: rows of 64 floats whose 16-byte groups
// are XOR-swizzled by t mod 8, so that the row-per-thread writes from tensor memory and the
// eight-row reads of the operand loop both spread a quarter-warp over all 32 banks.
__device__ __forceinline__ int gram_off(int t, int j) { return t * kCh + 4 * ((j >> 2) ^ (t & 7)) + (j & 3); }

// four / eight consecutive floats of shared memory at a 16-byte aligned address
__device__ __forceinline__ void ld4(const float* src, float* v) {
  const float4 a = *reinterpret_cast<const float4*>(src);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
}
__device__ __forceinline__ void ld8(const float* src, float* v) {
  ld4(src, v);
  ld4(src + 4, v + 4);
}
__device__ __forceinline__ void st8(float* dst, const float* v) {
  *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

template <int DK>
__global__ void __launch_bounds__(kThreads, 2) gdn_prefill_chunk_kernel(const PrefillParams p) {
  using L = ChunkLayout<DK>;
  extern __shared__ __align__(128) float sm[];
  const int tid = threadIdx.x;
  const int c = blockIdx.x;
  const int kh = blockIdx.y;
  if (c >= p.ws.meta[1]) return;  // (0 when cu_seqlens were rejected)
  uint64_t* sbar = reinterpret_cast<uint64_t*>(sm + L::OFF_BAR);  // [0] operand copies, [1] Gram MMAs
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sbar + 2);
  if (tid == 0) {
    mbar_init(sbar, 1);
    mbar_init(sbar + 1, 1);
    fence_mbar_init();
  }
  if ((tid >> 5) == 0) tmem_alloc(tslot, kCh);  // the Gram accumulators: 128 lanes x 64 columns
  const int4 rec = p.ws.chunks[c];
  const int i = rec.x, len = rec.z;
  const long long tok0 = rec.y, s0 = rec.w;
  const size_t C = size_t(p.C);
  const int r = p.Hv / p.Hk;

  // the gate inputs of the group's first v-heads, fetched now so that they arrive during the conv
  float* sAB = sm + L::OFF_AB;
  for (int idx = tid; idx < min(r, kAbHeads) * kCh; idx += kThreads) {
    const int e = idx / kCh, t = idx % kCh;
    const size_t gi = size_t(tok0 + t) * p.Hv + size_t(kh) * r + e;
    sAB[(2 * e) * kCh + t] = (t < len) ? bf16_to_f32(p.a[gi]) : 0.f;
    sAB[(2 * e + 1) * kCh + t] = (t < len) ? bf16_to_f32(p.b[gi]) : 0.f;
  }

  // a1 for the head's 2 DK q|k channels.  The raw x tile [64 tokens][2 DK] (q channels, then k)
  // comes in with 16-byte loads, staged in the space of the conv table; then one thread per
  // channel reads its column into registers and walks the chunk.  The three rows before the
  // chunk come from the prompt itself or, at its start, from the history.
  float* sY = sm + L::OFF_Y;
  static_assert(2 * DK <= kThreads, "one thread per q|k channel");
  const int ch = tid;  // (threads beyond the 2 DK channels only join the barriers)
  const bool own = ch < 2 * DK;
  const size_t gch = (ch < DK) ? size_t(kh) * DK + ch : size_t(p.Hk) * DK + size_t(kh) * DK + (ch - DK);
  float4 w = make_float4(0.f, 0.f, 0.f, 0.f);
  float h[3] = {0.f, 0.f, 0.f};
  {
    // every load of the tile, and the channel's taps and history, in flight at once
    uint16_t* sXr = reinterpret_cast<uint16_t*>(sY);
    constexpr int V8 = 2 * DK / 8;  // 16-byte groups per token row
    constexpr int kPer = kCh * V8 / kThreads;
    static_assert(kCh * V8 % kThreads == 0, "whole 16-byte groups per thread");
    uint4 v[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int idx = tid + q * kThreads;
      const int t = idx / V8, ch0 = 8 * (idx % V8);
      const size_t gch0 = (ch0 < DK) ? size_t(kh) * DK + ch0 : size_t(p.Hk) * DK + size_t(kh) * DK + (ch0 - DK);
      v[q] = make_uint4(0, 0, 0, 0);
      if (t < len) v[q] = *reinterpret_cast<const uint4*>(p.x + size_t(tok0 + t) * C + gch0);
    }
    if (own) {
      w = *reinterpret_cast<const float4*>(p.conv_w + gch * kConvW);
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        const long long pos = tok0 - 3 + m;
        h[m] = (pos >= s0) ? bf16_to_f32(p.x[size_t(pos) * C + gch])
                           : p.conv_state_in[(size_t(i) * 3 + size_t(pos - s0 + 3)) * C + gch];
      }
    }
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
      const int idx = tid + q * kThreads;
      const int t = idx / V8, ch0 = 8 * (idx % V8);
      *reinterpret_cast<uint4*>(sXr + t * 2 * DK + ch0) = v[q];
    }
  }
  __syncthreads();
  {
    float h0 = h[0], h1 = h[1], h2 = h[2];
    uint16_t xs[kCh];
    if (own) {
      const uint16_t* sXr = reinterpret_cast<const uint16_t*>(sY);
#pragma unroll
      for (int t = 0; t < kCh; ++t) xs[t] = sXr[t * 2 * DK + ch];
    }
    __syncthreads();  // every column is read before the conv outputs overwrite the staging
    if (own) {
#pragma unroll
      for (int t = 0; t < kCh; ++t) {
        const float xv = bf16_to_f32(xs[t]);
        const float z = fmaf(w.w, xv, fmaf(w.z, h2, fmaf(w.y, h1, w.x * h0)));
        sY[t * L::YS + ch] = (t < len) ? silu(z) : 0.f;
        h0 = h1;
        h1 = h2;
        h2 = xv;
      }
    }
  }
  __syncthreads();

  // a2: one warp per (token, q|k) vector, four vectors of a warp in flight together so that
  // their shuffle reductions overlap
  {
    const int warp = tid >> 5, lane = tid & 31;
    constexpr int kWarpsC = kThreads / 32;
    constexpr int kPerWarp = 2 * kCh / kWarpsC;
    static_assert(kPerWarp % 4 == 0, "four vectors at a time");
    for (int k0 = 0; k0 < kPerWarp; k0 += 4) {
      float x[4][DK / 32], ss[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = warp + (k0 + u) * kWarpsC;
        const float* row = sY + (v >> 1) * L::YS + (v & 1) * DK;
        ss[u] = 0.f;
#pragma unroll
        for (int e = 0; e < DK / 32; ++e) {
          x[u][e] = row[lane + 32 * e];
          ss[u] = fmaf(x[u][e], x[u][e], ss[u]);
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) ss[u] = warp_sum(ss[u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int v = warp + (k0 + u) * kWarpsC, t = v >> 1;
        float* row = sY + t * L::YS + (v & 1) * DK;
        const float inv = (t < len) ? rsqrtf(ss[u] + p.l2_eps) : 0.f;
#pragma unroll
        for (int e = 0; e < DK / 32; ++e) row[lane + 32 * e] = x[u][e] * inv;
      }
    }
  }
  __syncthreads();

  // q^_t . k^_t in f32 from the normalised table: the diagonal of MQ.  Where a token's decay is 0
  // its output is this one product times beta v, and a three-pass bf16 product's absolute error
  // (about 2^-21 here) would be a large part of it when q^ and k^ are nearly orthogonal.
  float* sQKd = sm + L::OFF_QKD;
  {
    const int warp = tid >> 5, lane = tid & 31;
    for (int t = warp; t < kCh; t += kThreads / 32) {
      const float* row = sY + t * L::YS;
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < DK / 32; ++e) acc = fmaf(row[lane + 32 * e], row[DK + lane + 32 * e], acc);
      acc = warp_sum(acc);
      if (lane == 0) sQKd[t] = acc;
    }
  }

  // normalised k^ and q^ to the workspace as bf16 hi/lo MMA operands (K-major core-matrix
  // layout, [t][c] with K = DK): k^ hi, k^ lo, q^ hi, q^ lo.  The state kernel also reads the k^
  // blocks as the MN-major operand [c][t] of its state update.  Eight consecutive threads fill
  // one 128-byte core matrix.
  {
    uint8_t* dst = reinterpret_cast<uint8_t*>(p.ws.kq) + (size_t(c) * p.Hk + kh) * kKqBlocks * (kCh * DK * 2);
    constexpr int BLK = kCh * DK * 2;
    for (int idx = tid; idx < 2 * kCh * (DK / 8); idx += kThreads) {
      const int part = idx / (kCh * (DK / 8));  // 0: k^, 1: q^
      const int cm = (idx >> 3) % (kCh * DK / 64), r8 = idx & 7;
      const int t = (cm / (DK / 8)) * 8 + r8, cb = cm % (DK / 8);
      float v[8];
      {  // (16-byte aligned: YS and DK are multiples of 4)
        const float4* src = reinterpret_cast<const float4*>(sY + t * L::YS + (part ? 0 : DK) + 8 * cb);
        const float4 a0 = src[0], a1 = src[1];
        v[0] = a0.x; v[1] = a0.y; v[2] = a0.z; v[3] = a0.w;
        v[4] = a1.x; v[5] = a1.y; v[6] = a1.z; v[7] = a1.w;
      }
      uint4 hi, lo;
      split8(v, hi, lo);
      const uint32_t off = kmajor_off(t, 8 * cb, DK);
      *reinterpret_cast<uint4*>(dst + (2 * part) * BLK + off) = hi;
      *reinterpret_cast<uint4*>(dst + (2 * part + 1) * BLK + off) = lo;
    }
  }

  // Gram products k^_t . k^_j and q^_t . k^_j on the tensor cores, from the split operands just
  // written (three bf16 MMAs over the hi/lo pairs, as in the state kernel).  They come back from
  // L2 into the conv table's space, dead once split, as [k^ hi | q^ hi | k^ lo | q^ lo]: k^ and
  // q^ then read as one M = 128 operand and k^ alone as the N = 64 one.  TMEM lane r holds row r
  // of [k^ k^T ; q^ k^T].
  {
    constexpr uint32_t BLK = kCh * DK * 2;
    uint8_t* sOp = reinterpret_cast<uint8_t*>(sY);
    const uint8_t* src = reinterpret_cast<const uint8_t*>(p.ws.kq) + (size_t(c) * p.Hk + kh) * kKqBlocks * BLK;
    asm volatile("fence.proxy.async.global;" ::: "memory");  // this thread's operand stores, before the copies
    tc_fence_before();
    __syncthreads();  // every operand store fenced, every read of the conv table done
    tc_fence_after();
    const uint32_t tmem = *tslot;
    bool issued = false;  // (thread 0: the Gram MMAs were issued)
    if (tid == 0) {
      mbar_arrive_expect_tx(sbar, 4 * BLK);
      bulk_load(sOp, src, BLK, sbar);                     // k^ hi
      bulk_load(sOp + BLK, src + 2 * BLK, BLK, sbar);     // q^ hi
      bulk_load(sOp + 2 * BLK, src + BLK, BLK, sbar);     // k^ lo
      bulk_load(sOp + 3 * BLK, src + 3 * BLK, BLK, sbar); // q^ lo
      if (mbar_wait_bounded(sbar, 0)) {
        tc_fence_after();
        const uint32_t a0 = smem_addr(sOp);
        umma_split3<DK / 16>(tmem, a0, a0 + 2 * BLK, a0, a0 + 2 * BLK, (DK / 8) * 128, umma_idesc_bf16(2 * kCh, kCh),
                             false);
        umma_commit(sbar + 1);
        issued = true;
      }
    }
    const bool ok = !__syncthreads_or(!mbar_wait_bounded(sbar + 1, 0));
    tc_fence_after();
    if (!ok) {
      if (tid == 0) {  // the copies and MMAs in flight finish before the TMEM is freed and the CTA exits
        atomicOr(p.err, kDevErrTimeout);
        (void)mbar_drain(sbar, 0);
        if (issued) (void)mbar_drain(sbar + 1, 0);
      }
    } else if (tid < 2 * kCh) {  // warps 0..3: thread = TMEM lane = row
      const int row = tid & (kCh - 1);
      float* dst = sm + ((tid < kCh) ? L::OFF_KK : L::OFF_QK);
      const uint32_t lane_sel = uint32_t(32 * (tid >> 5)) << 16;
#pragma unroll
      for (int c0 = 0; c0 < kCh; c0 += 32) {
        float v[32];
        tmem_ld32(tmem + lane_sel + c0, v);
#pragma unroll
        for (int q = 0; q < 32; q += 4)
          *reinterpret_cast<float4*>(dst + gram_off(row, c0 + q)) = make_float4(v[q], v[q + 1], v[q + 2], v[q + 3]);
      }
    }
    tc_fence_before();
  }
  __syncthreads();  // the q|k table is dead from here: its space holds D, X and beta D (k.k)

  // Per v-head work, two v-heads at a time: threads 0..127 take the even one, 128..255 the odd one,
  // each half synchronising on a named barrier of its own (the phases below are chains of short
  // steps, so two of them side by side fill the SM better than one after the other)
  const int grp = tid >> 7, gt = tid & 127;
  auto gsync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(1 + grp) : "memory"); };
  float* sD = sm + L::OFF_D + grp * 2 * L::MAT;  // D[t][j] (j <= t), later X = (I + beta D o KK)^-1
  float* sL = sD + L::MAT;
  float* sBeta = sm + L::OFF_BG + grp * 3 * kCh;
  float* sG = sBeta + kCh;  // g
  float* sGam = sG + kCh;
  float* sY2 = sm + L::OFF_Y2 + grp * 32 * kY2S;
  for (int e0 = 0; e0 < r; e0 += 2) {
    const int e = e0 + grp;
    if (e >= r) break;  // (an odd r leaves the second half idle on the last pair)
    const int h = kh * r + e;
    // a3 for this v-head (padding tokens: beta = 0, g = 1, so they change nothing)
    if (gt < kCh) {
      float beta = 0.f, g = 1.f;
      if (gt < len) {
        float av, bv;
        if (e < kAbHeads) {
          av = sAB[(2 * e) * kCh + gt];
          bv = sAB[(2 * e + 1) * kCh + gt];
        } else {
          const size_t gi = size_t(tok0 + gt) * p.Hv + h;
          av = bf16_to_f32(p.a[gi]);
          bv = bf16_to_f32(p.b[gi]);
        }
        const float A = -expf(p.A_log[h]);
        const float z = av + p.dt_bias[h];
        g = expf(((z > 20.f) ? z : log1pf(expf(z))) * A);
        beta = gate_beta(bv);
      }
      sBeta[gt] = beta;
      sG[gt] = g;
    }
    gsync();
    // decay products D[t][j] = prod_{j<m<=t} g_m, a running product down each column (thread j),
    // zeros above the diagonal (the blocked inverse relies on them); Gamma_t = prod_{m<=t} g_m
    // (thread 64).  Every factor is in [0, 1]: nothing overflows, nothing cancels (a difference
    // of running sums of log g would lose digits once those sums are large, and gives NaN after
    // a token with g = 0), and a product that underflows is below anything it is added to.
    // (the g values come in as sixteen 16-byte broadcasts before the products, so that the chain
    // of 64 multiplies does not wait on a shared-memory load at every step)
    if (gt <= kCh) {
      float gv[kCh];
#pragma unroll
      for (int t = 0; t < kCh; t += 4) {
        const float4 q4 = *reinterpret_cast<const float4*>(sG + t);
        gv[t] = q4.x;
        gv[t + 1] = q4.y;
        gv[t + 2] = q4.z;
        gv[t + 3] = q4.w;
      }
      if (gt < kCh) {
        const int j = gt;
        float d = 1.f;
#pragma unroll
        for (int t = 0; t < kCh; ++t) {
          if (t > j) d *= gv[t];
          sD[t * kAS + j] = (t < j) ? 0.f : d;
        }
      } else {
        float gam = 1.f;
#pragma unroll
        for (int t = 0; t < kCh; ++t) {
          gam *= gv[t];
          sGam[t] = gam;
        }
      }
    }
    gsync();
    // per v-head operands: W hi, W lo, MQ hi, MQ lo, each [t][j] (K = 64), zero above the diagonal
    uint8_t* wq = reinterpret_cast<uint8_t*>(p.ws.wm) + (size_t(c) * p.Hv + h) * (4 * kCh * kCh * 2);
    float* gd = p.ws.gd + (size_t(c) * p.Hv + h) * (2 * kCh);
    // beta_t D (k.k) strictly below the diagonal; MQ = D (q.k) on and below it (D = 1 on the
    // diagonal, where q.k is the f32 product); Gamma, d
    // (thread = row t, eight columns 8 jb.. 8 jb + 7: 16-byte reads and writes)
    for (int idx = gt; idx < kCh * (kCh / 8); idx += 128) {
      const int cm = idx >> 3, r8 = idx & 7;
      const int t = (cm >> 3) * 8 + r8, jb = cm & 7;
      float d[8], kk[8], qk[8], l[8], v[8];
      ld8(sD + t * kAS + 8 * jb, d);
      ld4(sm + L::OFF_KK + gram_off(t, 8 * jb), kk);
      ld4(sm + L::OFF_KK + gram_off(t, 8 * jb + 4), kk + 4);
      ld4(sm + L::OFF_QK + gram_off(t, 8 * jb), qk);
      ld4(sm + L::OFF_QK + gram_off(t, 8 * jb + 4), qk + 4);
      const float bt = sBeta[t];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = 8 * jb + q;
        l[q] = (j < t) ? bt * d[q] * kk[q] : 0.f;
        v[q] = (j < t) ? d[q] * qk[q] : ((j == t) ? sQKd[t] : 0.f);
      }
      st8(sL + t * kAS + 8 * jb, l);
      uint4 hi, lo;
      split8(v, hi, lo);
      const uint32_t off = kmajor_off(t, 8 * jb, kCh);
      *reinterpret_cast<uint4*>(wq + 2 * (kCh * kCh * 2) + off) = hi;
      *reinterpret_cast<uint4*>(wq + 3 * (kCh * kCh * 2) + off) = lo;
    }
    if (gt < kCh) {
      gd[gt] = sGam[gt];
      gd[kCh + gt] = sD[(kCh - 1) * kAS + gt];
    }
    gsync();
    // X = (I + L)^-1, blocked.  The four 16 x 16 diagonal blocks: one thread per column, forward
    // substitution unrolled in registers (x_t = 0 above the diagonal, 1 on it).  Then
    // X21 = -X22 (L21 X11) for the 16 x 16 and the 32 x 32 off-diagonal blocks, whose upper
    // triangles are zero.  X overwrites D.
    if (gt < kCh) {
      const int jb = gt & ~15, jj = gt & 15;
      float x[16];
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        float acc = 0.f;
#pragma unroll
        for (int m = 0; m < t; ++m) acc = fmaf(sL[(jb + t) * kAS + jb + m], x[m], acc);
        x[t] = (t < jj) ? 0.f : ((t == jj) ? 1.f : -acc);
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) sD[(jb + t) * kAS + gt] = x[t];
    }
    gsync();
    {  // 16 x 16 off-diagonal blocks of the two 32 x 32 blocks: thread = (row, 2 columns), both blocks
      const int ii = gt >> 3, jj = 2 * (gt & 7);
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int o = 32 * blk;
        float y0 = 0.f, y1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float l = sL[(o + 16 + ii) * kAS + o + k];
          y0 = fmaf(l, sD[(o + k) * kAS + o + jj], y0);
          y1 = fmaf(l, sD[(o + k) * kAS + o + jj + 1], y1);
        }
        sY2[(16 * blk + ii) * kY2S + jj] = y0;
        sY2[(16 * blk + ii) * kY2S + jj + 1] = y1;
      }
      gsync();
#pragma unroll
      for (int blk = 0; blk < 2; ++blk) {
        const int o = 32 * blk;
        float x0 = 0.f, x1 = 0.f;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          const float xv = sD[(o + 16 + ii) * kAS + o + 16 + k];
          x0 = fmaf(xv, sY2[(16 * blk + k) * kY2S + jj], x0);
          x1 = fmaf(xv, sY2[(16 * blk + k) * kY2S + jj + 1], x1);
        }
        sD[(o + 16 + ii) * kAS + o + jj] = -x0;
        sD[(o + 16 + ii) * kAS + o + jj + 1] = -x1;
      }
    }
    gsync();
    {  // the 32 x 32 off-diagonal block: thread = (row, 8 columns), the columns read 16 bytes at a time
      const int ii = gt >> 2, jj = 8 * (gt & 3);
      float y[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float l = sL[(32 + ii) * kAS + k];
        float xr[8];
        ld8(sD + k * kAS + jj, xr);
#pragma unroll
        for (int q = 0; q < 8; ++q) y[q] = fmaf(l, xr[q], y[q]);
      }
      st8(sY2 + ii * kY2S + jj, y);
      gsync();
      float x[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float xv = sD[(32 + ii) * kAS + 32 + k];
        float yr[8];
        ld8(sY2 + k * kY2S + jj, yr);
#pragma unroll
        for (int q = 0; q < 8; ++q) x[q] = fmaf(xv, yr[q], x[q]);
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) x[q] = -x[q];
      st8(sD + (32 + ii) * kAS + jj, x);
    }
    gsync();
    for (int idx = gt; idx < kCh * (kCh / 8); idx += 128) {
      const int cm = idx >> 3, r8 = idx & 7;
      const int t = (cm >> 3) * 8 + r8, jb = cm & 7;
      float x[8], bj[8], v[8];
      ld8(sD + t * kAS + 8 * jb, x);
      ld8(sBeta + 8 * jb, bj);
#pragma unroll
      for (int q = 0; q < 8; ++q) v[q] = (8 * jb + q <= t) ? x[q] * bj[q] : 0.f;
      uint4 hi, lo;
      split8(v, hi, lo);
      const uint32_t off = kmajor_off(t, 8 * jb, kCh);
      *reinterpret_cast<uint4*>(wq + off) = hi;
      *reinterpret_cast<uint4*>(wq + (kCh * kCh * 2) + off) = lo;
    }
    gsync();
  }
  tc_fence_after();
  if ((tid >> 5) == 0) tmem_dealloc(*tslot, kCh);
}

// ------------------------------------------------------------------------------------------
// Kernel 2: per (prompt, v-head, 64 state rows), sequential over the prompt's chunks, on the
// tensor cores.  The f32 state lives in TMEM (64 lanes x DK columns, the M = 64 accumulator
// layout: row m in lane 32 (m / 16) + m % 16).  Each product of the chunk form is three bf16
// MMAs over hi/lo operand pairs (hi.hi + hi.lo + lo.hi), about 2^-16 relative per product:
//   P  = S [k^ | q^]^T   (A = S hi/lo in shared memory, B = k^ / q^ hi/lo from kernel 1)
//   u  = r W^T           (r = v - Gamma o P_k, written by the threads)
//   S  = Gamma_63 S + (d o u) k^   (accumulated into the TMEM state, B = the k^ blocks read
//                                   MN-major)
//   o' = u MQ^T          (out = q_scale (Gamma o P_q + o'))
// Thread roles: warps 0..7 run the epilogues (warp w reaches TMEM lanes 32 (w % 4) ..; warps w
// and w + 4 split the columns); a ninth warp's first thread issues the bulk copies and the
// MMAs in a loop of its own, so that its stalls on the MMA queue delay no epilogue.
template <int DK>
struct TcLayout {
  static constexpr int BLK_KQ = kCh * DK * 2;            // one 64 x DK bf16 operand
  static constexpr int BLK = kCh * kCh * 2;              // one 64 x 64 bf16 operand
  // k^ of two chunks (buffers 0 and 1) around q^ of one: hi parts [k^0 | q^ | k^1], then the lo
  // parts in the same order, so that k^ of either buffer and q^ are adjacent (one N = 128 operand)
  static constexpr int OFF_KH = 0;
  static constexpr int OFF_KL = OFF_KH + 3 * BLK_KQ;
  static constexpr int OFF_W = OFF_KL + 3 * BLK_KQ;      // W hi, lo
  static constexpr int OFF_MQ = OFF_W + 2 * BLK;         // MQ hi, lo
  static constexpr int OFF_GD = OFF_MQ + 2 * BLK;        // two buffers of Gamma[64], d[64]
  static constexpr int OFF_S = OFF_GD + 2 * 2 * kCh * 4; // S hi, lo (64 x DK)
  static constexpr int OFF_RD = OFF_S + 2 * BLK_KQ;      // r hi, lo; later (d o u) hi, lo
  static constexpr int OFF_U = OFF_RD + 2 * BLK;         // u hi, lo
  static constexpr int OFF_X = OFF_U + 2 * BLK;          // raw x [67][64] f32 (3 history rows)
  static constexpr int OFF_TAP = OFF_X + 67 * kTileRows * 4;  // conv taps [64][4]
  static constexpr int OFF_BAR = OFF_TAP + kTileRows * 16;    // mbarriers
  static constexpr int NBAR = 14;
  static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_TSLOT + 16;
  static_assert(OFF_TAP % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
};

// TMEM columns: the state, two buffers of P = [P_k | P_q] (chunk parity), u, o'
constexpr uint32_t kColS = 0, kColP0 = 128, kColU = 384, kColO = 448, kTmemCols = 512;
// mbarriers
enum { kBarK0 = 0, kBarK1, kBarQ, kBarW, kBarMQ, kBarGD0, kBarGD1, kBarPk, kBarU, kBarO, kBarS, kRdyR, kRdyU, kRdyS,
       kNumBars };
constexpr uint32_t kEpiThreads = kThreads;  // arrivals on the kRdy* (operand written) barriers

// every thread waits (bounded); true when any thread of the CTA gave up
__device__ __forceinline__ bool wait_failed(uint64_t* bar, uint32_t parity) {
  const bool ok = mbar_wait_bounded(bar, parity);
  return __syncthreads_or(!ok) != 0;
}

// Named barrier 1 over the state kernel's 256 epilogue threads (warps 0..7), plain and with an
// or-reduction of a predicate.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool epi_any(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.or.pred q, 1, 256, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(v))
      : "memory");
  return r != 0;
}

// The same with an MN-major B operand (the k^ blocks read as [c][t]): LBO is the byte step between
// core matrices along K (eight tokens), SBO along N (eight channels), and a K step moves the B
// start address by two core-matrix rows along K.
template <int KSTEPS>
__device__ __forceinline__ void umma_split3_bmn(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t a_sbo, uint32_t b_hi,
                                                uint32_t b_lo, uint32_t b_lbo, uint32_t b_sbo, uint32_t idesc,
                                                bool accumulate) {
  const uint64_t dah = umma_smem_desc(a_hi, 128, a_sbo), dal = umma_smem_desc(a_lo, 128, a_sbo);
  const uint64_t dbh = umma_smem_desc(b_hi, b_lbo, b_sbo), dbl = umma_smem_desc(b_lo, b_lbo, b_sbo);
  const uint64_t bstep = uint64_t((2 * b_lbo) >> 4);
#pragma unroll
  for (int sp = 0; sp < 3; ++sp) {
    const uint64_t da = (sp == 2) ? dal : dah;
    const uint64_t db = (sp == 1) ? dbl : dbh;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk)
      umma_bf16(d, da + uint64_t(16 * kk), db + bstep * kk, idesc, (accumulate || sp > 0 || kk > 0) ? 1u : 0u);
  }
}

// Row-swizzled [rows][64] f32 tables (raw x, staged outputs): element (t, c) at t * 64 +
// (c ^ swz(t)); the swizzle spreads the 16x256b thread layout's four token columns over all
// banks and keeps groups of four consecutive c together.
__device__ __forceinline__ int swz(int t) { return ((t >> 1) & 3) << 3; }

constexpr int kIssuer = kThreads;  // the state kernel's copy / MMA issuing thread (first of warp 8)

template <int DK, int DV>
__global__ void __launch_bounds__(kThreads + 32, 1) gdn_prefill_state_kernel(const PrefillParams p) {
  using L = TcLayout<DK>;
  extern __shared__ __align__(128) uint8_t smb[];
  constexpr int kHalves = DV / kTileRows;
  constexpr int SC = DK / 2;      // state columns per epilogue thread (two warps per row quarter)
  constexpr int SREP = SC / 32;   // 16x256b x4 accesses per state half
  static_assert(SREP == 1 || SREP == 2, "dk = 64 or 128");
  static_assert(L::NBAR >= kNumBars, "mbarrier slots");
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.y;
  const int h = blockIdx.x / kHalves;
  const int r0 = (blockIdx.x % kHalves) * kTileRows;
  const int kh = h / (p.Hv / p.Hk);
  if (p.ws.meta[0] == 0) return;
  const int32_t* base = p.ws.meta + 4;
  const int c_first = base[i], n_chunks = base[i + 1] - base[i];
  const long long s0 = p.cu[i], s1 = p.cu[i + 1];
  const size_t C = size_t(p.C);
  const size_t vch0 = size_t(2) * p.Hk * DK + size_t(h) * DV + r0;  // first conv channel of the tile
  float* sX = reinterpret_cast<float*>(smb + L::OFF_X);
  float* sTap = reinterpret_cast<float*>(smb + L::OFF_TAP);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smb + L::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smb + L::OFF_TSLOT);
  const uint32_t sbase = smem_addr(smb);

  // epilogue coordinates.  32x32b accesses (state in and out): row m (lanes 0..15), column half
  // hh.  16x256b accesses (the chunk loop): rows ra, rb = ra + 8, columns 2 c4 + e of each
  // 8-column block of the half.
  const int quad = warp & 3, hh = warp >> 2;
  const int m = 16 * quad + (lane & 15);
  const bool epi = warp < kThreads / 32;  // an epilogue warp (not the issuing warp)
  const bool act = epi && lane < 16;
  const uint32_t lane_sel = uint32_t(32 * quad) << 16;
  const int ra = 16 * quad + (lane >> 2), rb = ra + 8, c4 = lane & 3;

  if (tid == 0) {
    for (int q = 0; q < kNumBars; ++q) mbar_init(bar + q, q >= kRdyR ? kEpiThreads : 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  // phases armed per barrier (thread kIssuer only), so that a failed CTA can wait for what it started
  int armed[kNumBars] = {};
  auto kq_src = [&](int c) {
    return reinterpret_cast<const uint8_t*>(p.ws.kq) + (size_t(c) * p.Hk + kh) * kKqBlocks * L::BLK_KQ;
  };
  auto issue_k = [&](int c, int b) {  // k^ hi, lo of chunk c into buffer b
    ++armed[kBarK0 + b];
    mbar_arrive_expect_tx(bar + kBarK0 + b, 2 * L::BLK_KQ);
    bulk_load(smb + L::OFF_KH + 2 * b * L::BLK_KQ, kq_src(c), L::BLK_KQ, bar + kBarK0 + b);
    bulk_load(smb + L::OFF_KL + 2 * b * L::BLK_KQ, kq_src(c) + L::BLK_KQ, L::BLK_KQ, bar + kBarK0 + b);
  };
  auto issue_q = [&](int c) {
    ++armed[kBarQ];
    mbar_arrive_expect_tx(bar + kBarQ, 2 * L::BLK_KQ);
    bulk_load(smb + L::OFF_KH + L::BLK_KQ, kq_src(c) + 2 * L::BLK_KQ, L::BLK_KQ, bar + kBarQ);
    bulk_load(smb + L::OFF_KL + L::BLK_KQ, kq_src(c) + 3 * L::BLK_KQ, L::BLK_KQ, bar + kBarQ);
  };
  auto wq_src = [&](int c) {
    return reinterpret_cast<const uint8_t*>(p.ws.wm) + (size_t(c) * p.Hv + h) * (4 * L::BLK);
  };
  auto issue_w = [&](int c) {
    ++armed[kBarW];
    mbar_arrive_expect_tx(bar + kBarW, 2 * L::BLK);
    bulk_load(smb + L::OFF_W, wq_src(c), 2 * L::BLK, bar + kBarW);
  };
  auto issue_mq = [&](int c) {
    ++armed[kBarMQ];
    mbar_arrive_expect_tx(bar + kBarMQ, 2 * L::BLK);
    bulk_load(smb + L::OFF_MQ, wq_src(c) + 2 * L::BLK, 2 * L::BLK, bar + kBarMQ);
  };
  auto issue_gd = [&](int lc) {  // buffer lc & 1 holds local chunk lc
    const int b = lc & 1, c = c_first + lc;
    ++armed[kBarGD0 + b];
    mbar_arrive_expect_tx(bar + kBarGD0 + b, 2 * kCh * 4);
    bulk_load(smb + L::OFF_GD + b * 2 * kCh * 4, p.ws.gd + (size_t(c) * p.Hv + h) * (2 * kCh), 2 * kCh * 4,
              bar + kBarGD0 + b);
  };
  if (tid == kIssuer && n_chunks > 0) {
    issue_k(c_first, 0);
    issue_q(c_first);
    issue_w(c_first);
    issue_mq(c_first);
    issue_gd(0);
    if (n_chunks > 1) {
      issue_gd(1);
      issue_k(c_first + 1, 1);
    }
  }

  // S hi/lo operand stores of this thread's columns [c0, c0 + n) of row m (32x32b layout)
  auto store_pair = [&](int off, int row, int k0, int kdim, const float* v, int n) {
    for (int q = 0; q < n; q += 8) {
      uint4 hi, lo;
      split8(v + q, hi, lo);
      const uint32_t o = kmajor_off(row, k0 + q, kdim);
      *reinterpret_cast<uint4*>(smb + off + o) = hi;
      *reinterpret_cast<uint4*>(smb + off + (kdim == DK ? L::BLK_KQ : L::BLK) + o) = lo;
    }
  };
  // hi/lo operand stores of a 16x256b register block: 4 reps x (rows ra, rb) x 2 columns from
  // column k0 of a K-major operand with kdim columns (lo block `lo_off` bytes after hi)
  auto store_block = [&](int off, uint32_t lo_off, int k0, int kdim, const float (&v)[16]) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int k = k0 + 8 * j + 2 * c4;
      uint32_t hi, lo;
      split2(v[4 * j], v[4 * j + 1], hi, lo);
      uint32_t o = kmajor_off(ra, k, kdim);
      *reinterpret_cast<uint32_t*>(smb + off + o) = hi;
      *reinterpret_cast<uint32_t*>(smb + off + lo_off + o) = lo;
      split2(v[4 * j + 2], v[4 * j + 3], hi, lo);
      o = kmajor_off(rb, k, kdim);
      *reinterpret_cast<uint32_t*>(smb + off + o) = hi;
      *reinterpret_cast<uint32_t*>(smb + off + lo_off + o) = lo;
    }
  };

  // the state tile into TMEM and, split, into the S operand; taps; the v channels' history
  {
    const float* src = p.state_in + ((size_t(i) * p.Hv + h) * DV + r0 + m) * DK + hh * SC;
#pragma unroll
    for (int c0 = 0; c0 < SC && epi; c0 += 16) {
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; q += 4) {
        float4 f = act ? *reinterpret_cast<const float4*>(src + c0 + q) : make_float4(0.f, 0.f, 0.f, 0.f);
        v[q] = f.x; v[q + 1] = f.y; v[q + 2] = f.z; v[q + 3] = f.w;
      }
      tmem_st16(tmem + lane_sel + kColS + hh * SC + c0, v);
      if (act) store_pair(L::OFF_S, m, hh * SC + c0, DK, v, 16);
    }
    if (tid < kTileRows) *reinterpret_cast<float4*>(sTap + 4 * tid) = *reinterpret_cast<const float4*>(p.conv_w + (vch0 + tid) * kConvW);
    for (int idx = tid; idx < 3 * kTileRows; idx += kThreads) {
      const int mm = idx / kTileRows, ch = idx % kTileRows;
      sX[mm * kTileRows + (ch ^ swz(mm))] = p.conv_state_in[(size_t(i) * 3 + mm) * C + vch0 + ch];
    }
  }
  // raw x of the tile's 64 channels for one chunk: thread = (token tid / 4, 16 channels)
  const int xt = tid >> 2, xg = tid & 3;
  uint4 xr0 = make_uint4(0, 0, 0, 0), xr1 = xr0;
  if (n_chunks > 0 && xt < min_ll(kCh, s1 - s0)) {
    const uint4* src = reinterpret_cast<const uint4*>(p.x + size_t(s0 + xt) * C + vch0 + 16 * xg);
    xr0 = src[0];
    xr1 = src[1];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t id_n64 = umma_idesc_bf16(kTileRows, kCh), id_ndk = umma_idesc_bf16(kTileRows, DK);
  const uint32_t id_n128 = umma_idesc_bf16(kTileRows, 2 * kCh);
  const uint32_t id_ndk_bmn = id_ndk | (1u << 16);  // B MN-major
  bool failed = false;
  if (n_chunks > 0) {
    // the state in TMEM is kept pre-scaled by the current chunk's Gamma_63, so that the update
    // MMA can accumulate onto it
    if (wait_failed(bar + kBarGD0, 0)) {
      failed = true;
    } else {
      tc_fence_after();
      if (epi) {
        const float gl = reinterpret_cast<const float*>(smb + L::OFF_GD)[kCh - 1];
#pragma unroll
        for (int c0 = 0; c0 < SC; c0 += 32) {
          float sv[32];
          tmem_ld32(tmem + lane_sel + kColS + hh * SC + c0, sv);
#pragma unroll
          for (int q = 0; q < 32; ++q) sv[q] *= gl;
          tmem_st32(tmem + lane_sel + kColS + hh * SC + c0, sv);
        }
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  }

  // From here the issuing thread and the epilogue warps run separate loops: the epilogue warps
  // synchronise among themselves on named barrier 1 and hand each finished operand to the issuer
  // through an mbarrier (256 arrivals), so that an issuer blocked on a full MMA queue never holds
  // up an epilogue.
  int len = 0;
  if (tid == kIssuer) {
    for (int lc = 0; lc < n_chunks && !failed; ++lc) {
      const uint32_t par = lc & 1;
      const uint32_t colP = kColP0 + 128 * par;
      const bool more = lc + 1 < n_chunks;
      // P = S [k^ | q^]^T into this chunk's P buffer, once the S operand is written: k^ (buffer
      // lc & 1) and q^ are adjacent, so they read as one N = 128 operand ([k^0 | q^] for even
      // chunks, P_k in the first 64 columns; [q^ | k^1] for odd ones, P_k in the second 64).  One
      // N = 128 MMA reads the A tile once for both halves: the M = 64 MMAs here are bound by
      // shared-memory reads, not by the tensor core.
      if ((lc > 0 && !mbar_wait_bounded(bar + kRdyS, (lc - 1) & 1)) ||
          !mbar_wait_bounded(bar + kBarK0 + par, (lc >> 1) & 1) || !mbar_wait_bounded(bar + kBarQ, par)) {
        failed = true;
        break;
      }
      tc_fence_after();
      {
        const uint32_t sS = sbase + L::OFF_S, bo = (par ? 1 : 0) * L::BLK_KQ;
        umma_split3<DK / 16>(tmem + colP, sS, sS + L::BLK_KQ, sbase + L::OFF_KH + bo, sbase + L::OFF_KL + bo,
                             (DK / 8) * 128, id_n128, false);
        umma_commit(bar + kBarPk);
        ++armed[kBarPk];
      }
      // Bulk copies are issued only right after an MMA group, while it runs: issuing one can hold
      // this thread for hundreds of cycles, which must not delay the next MMA group.  The
      // previous chunk's o' and update MMAs are done by now: this chunk's MQ, and the next
      // chunk's k^ into the buffer the previous chunk used.
      if (lc > 0) {
        if (!mbar_wait_bounded(bar + kBarO, (lc - 1) & 1)) {
          failed = true;
          break;
        }
        issue_mq(c_first + lc);
        if (more) {
          if (!mbar_wait_bounded(bar + kBarS, (lc - 1) & 1)) {
            failed = true;
            break;
          }
          issue_k(c_first + lc + 1, (lc + 1) & 1);
        }
      }
      // u = r W^T; then the next chunk's q^ (the P MMAs are done with it: the epilogue waited)
      if (!mbar_wait_bounded(bar + kRdyR, par) || !mbar_wait_bounded(bar + kBarW, par)) {
        failed = true;
        break;
      }
      tc_fence_after();
      umma_split3<kCh / 16>(tmem + kColU, sbase + L::OFF_RD, sbase + L::OFF_RD + L::BLK, sbase + L::OFF_W,
                            sbase + L::OFF_W + L::BLK, 1024, id_n64, false);
      umma_commit(bar + kBarU);
      ++armed[kBarU];
      if (more) issue_q(c_first + lc + 1);
      // S += (d o u) k^ (k^ of this chunk's buffer, read MN-major), then o' = u MQ^T; then the
      // next chunk's W (the epilogue waited for the u MMAs) and Gamma, d of chunk lc + 2
      // (chunk lc's are read)
      if (!mbar_wait_bounded(bar + kRdyU, par)) {
        failed = true;
        break;
      }
      tc_fence_after();
      umma_split3_bmn<kCh / 16>(tmem + kColS, sbase + L::OFF_RD, sbase + L::OFF_RD + L::BLK, 1024,
                                sbase + L::OFF_KH + 2 * par * L::BLK_KQ, sbase + L::OFF_KL + 2 * par * L::BLK_KQ,
                                (DK / 8) * 128, 128, id_ndk_bmn, true);
      umma_commit(bar + kBarS);
      ++armed[kBarS];
      if (!mbar_wait_bounded(bar + kBarMQ, par)) {
        failed = true;
        break;
      }
      umma_split3<kCh / 16>(tmem + kColO, sbase + L::OFF_U, sbase + L::OFF_U + L::BLK, sbase + L::OFF_MQ,
                            sbase + L::OFF_MQ + L::BLK, 1024, id_n64, false);
      umma_commit(bar + kBarO);
      ++armed[kBarO];
      if (more) issue_w(c_first + lc + 1);
      if (lc + 2 < n_chunks) issue_gd(lc + 2);
    }
  } else if (epi && !failed && n_chunks > 0) {
    // raw x of a chunk into rows 3..66 (zero past the prompt's end), then the next chunk's x is
    // fetched: thread = (token xt, 16 channels)
    auto stage_x = [&](long long tok0, int n) {
      const uint32_t wv[8] = {xr0.x, xr0.y, xr0.z, xr0.w, xr1.x, xr1.y, xr1.z, xr1.w};
      const int t = xt + 3, sw = swz(t);
      float* row = sX + t * kTileRows;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float4 f;
        f.x = (xt < n) ? bf16_to_f32(uint16_t(wv[2 * q] & 0xFFFFu)) : 0.f;
        f.y = (xt < n) ? bf16_to_f32(uint16_t(wv[2 * q] >> 16)) : 0.f;
        f.z = (xt < n) ? bf16_to_f32(uint16_t(wv[2 * q + 1] & 0xFFFFu)) : 0.f;
        f.w = (xt < n) ? bf16_to_f32(uint16_t(wv[2 * q + 1] >> 16)) : 0.f;
        *reinterpret_cast<float4*>(row + ((16 * xg + 4 * q) ^ sw)) = f;
      }
      const long long nt = tok0 + kCh + xt;
      if (nt < s1) {
        const uint4* src = reinterpret_cast<const uint4*>(p.x + size_t(nt) * C + vch0 + 16 * xg);
        xr0 = src[0];
        xr1 = src[1];
      }
    };
    // conv + SiLU of the v channels at this thread's (row, token) cells
    float v[16];
    auto conv = [&]() {
      const float4 wa = *reinterpret_cast<const float4*>(sTap + 4 * ra);
      const float4 wb = *reinterpret_cast<const float4*>(sTap + 4 * rb);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 32 * hh + 8 * j + 2 * c4 + (e & 1);
          const int row = (e < 2) ? ra : rb;
          const float4 w = (e < 2) ? wa : wb;
          const float z = fmaf(w.w, sX[(t + 3) * kTileRows + (row ^ swz(t + 3))],
                               fmaf(w.z, sX[(t + 2) * kTileRows + (row ^ swz(t + 2))],
                                    fmaf(w.y, sX[(t + 1) * kTileRows + (row ^ swz(t + 1))],
                                         w.x * sX[t * kTileRows + (row ^ swz(t))])));
          v[4 * j + e] = silu(z);
        }
    };
    // outputs o = q_scale (Gamma o P_q + o'), staged token-major in the u operand buffer (the o'
    // MMAs are done with it), then written out as 16-byte stores
    float* sOut = reinterpret_cast<float*>(smb + L::OFF_U);  // [64 tokens][64 rows], row-swizzled
    auto out_chunk = [&](int lc, long long tok0, const float (&gam)[8]) {
      float o[16], pq[16];
      tmem_ld16x256_2x4(tmem + lane_sel + kColO + 32 * hh,
                        tmem + lane_sel + kColP0 + 128 * (lc & 1) + ((lc & 1) ? 0 : kCh) + 32 * hh, o, pq);
#pragma unroll
      for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int t = 32 * hh + 8 * j + 2 * c4 + (e & 1);
          const int row = (e < 2) ? ra : rb;
          sOut[t * kTileRows + (row ^ swz(t))] = p.q_scale * fmaf(gam[2 * j + (e & 1)], pq[4 * j + e], o[4 * j + e]);
        }
      epi_sync();
      if (xt < len) {  // thread = (token xt, rows 16 xg .. 16 xg + 15)
        const float* src = sOut + xt * kTileRows;
        const int sw = swz(xt);
        const size_t oi = size_t(tok0 + xt) * p.Hv * DV + size_t(h) * DV + r0 + 16 * xg;
        float4 f[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) f[q] = *reinterpret_cast<const float4*>(src + ((16 * xg + 4 * q) ^ sw));
        if (p.out_f32) {
          float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi);
#pragma unroll
          for (int q = 0; q < 4; ++q) o4[q] = f[q];
        } else {
          uint32_t w[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const __nv_bfloat162 b0 = __floats2bfloat162_rn(f[q].x, f[q].y);
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(f[q].z, f[q].w);
            w[2 * q] = *reinterpret_cast<const uint32_t*>(&b0);
            w[2 * q + 1] = *reinterpret_cast<const uint32_t*>(&b1);
          }
          uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + oi);
          o4[0] = make_uint4(w[0], w[1], w[2], w[3]);
          o4[1] = make_uint4(w[4], w[5], w[6], w[7]);
        }
      }
    };
    // every epilogue thread hands its operand writes to the tensor core and arrives
    auto hand_over = [&](uint64_t* rdy) {
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(rdy);
    };

    stage_x(s0, int(min_ll(kCh, s1 - s0)));
    epi_sync();
    conv();
    for (int lc = 0; lc < n_chunks; ++lc) {
      const uint32_t par = lc & 1;
      const uint32_t colP = kColP0 + 128 * par;
      const float* sGam = reinterpret_cast<const float*>(smb + L::OFF_GD + (lc & 1) * 2 * kCh * 4);
      const float* sd = sGam + kCh;
      const long long tok0 = s0 + (long long)lc * kCh;
      len = int(min_ll(kCh, s1 - tok0));
      const bool more = lc + 1 < n_chunks;

      // (a) r = v - Gamma o P_k -> operand; the last three raw rows become the next chunk's
      // history (every conv read of this chunk is done: the barrier of the wait)
      if (epi_any(!mbar_wait_bounded(bar + kBarPk, par))) {
        failed = true;
        break;
      }
      tc_fence_after();
      float gam[8];
      {
        float pk[16];
        tmem_ld16x256_x4(tmem + lane_sel + colP + (par ? kCh : 0) + 32 * hh, pk);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          gam[2 * j] = sGam[32 * hh + 8 * j + 2 * c4];
          gam[2 * j + 1] = sGam[32 * hh + 8 * j + 2 * c4 + 1];
#pragma unroll
          for (int e = 0; e < 4; ++e) pk[4 * j + e] = fmaf(-gam[2 * j + (e & 1)], pk[4 * j + e], v[4 * j + e]);
        }
        store_block(L::OFF_RD, L::BLK, 32 * hh, kCh, pk);
      }
      if (len == kCh && tid < 3 * kTileRows) {
        const int mm = tid / kTileRows, ch = tid % kTileRows;
        sX[mm * kTileRows + (ch ^ swz(mm))] = sX[(kCh + mm) * kTileRows + (ch ^ swz(kCh + mm))];
      }
      hand_over(bar + kRdyR);
      // (b) u and d o u -> operands
      if (epi_any(!mbar_wait_bounded(bar + kBarU, par))) {
        failed = true;
        break;
      }
      tc_fence_after();
      {
        float u[16];
        tmem_ld16x256_x4(tmem + lane_sel + kColU + 32 * hh, u);
        store_block(L::OFF_U, L::BLK, 32 * hh, kCh, u);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float d0 = sd[32 * hh + 8 * j + 2 * c4], d1 = sd[32 * hh + 8 * j + 2 * c4 + 1];
          u[4 * j] *= d0;
          u[4 * j + 1] *= d1;
          u[4 * j + 2] *= d0;
          u[4 * j + 3] *= d1;
        }
        store_block(L::OFF_RD, L::BLK, 32 * hh, kCh, u);  // r is dead: the u MMAs are done
      }
      hand_over(bar + kRdyU);
      // (c) while the state update runs: the next chunk's raw x and conv
      if (more) {
        stage_x(tok0 + kCh, int(min_ll(kCh, s1 - tok0 - kCh)));
        epi_sync();
        conv();
      }
      // (d) the new state: split into the S operand of the next chunk, and pre-scaled in TMEM by
      // the next chunk's Gamma_63
      {
        bool ok = mbar_wait_bounded(bar + kBarS, par);
        if (more) ok = ok && mbar_wait_bounded(bar + kBarGD0 + ((lc + 1) & 1), ((lc + 1) >> 1) & 1);
        if (epi_any(!ok)) {
          failed = true;
          break;
        }
      }
      tc_fence_after();
      {
        const float gl = more ? reinterpret_cast<const float*>(smb + L::OFF_GD + ((lc + 1) & 1) * 2 * kCh * 4)[kCh - 1] : 1.f;
        const uint32_t cs = tmem + lane_sel + kColS + hh * SC;
        float sv[SREP][16];
        if constexpr (SREP == 2)
          tmem_ld16x256_2x4(cs, cs + 32, sv[0], sv[1]);
        else
          tmem_ld16x256_x4(cs, sv[0]);
#pragma unroll
        for (int q = 0; q < SREP; ++q) store_block(L::OFF_S, L::BLK_KQ, hh * SC + 32 * q, DK, sv[q]);
        if (more) {
          uint32_t w[SREP][16];
#pragma unroll
          for (int q = 0; q < SREP; ++q)
#pragma unroll
            for (int e = 0; e < 16; ++e) w[q][e] = __float_as_uint(sv[q][e] * gl);
          if constexpr (SREP == 2)
            tmem_st16x256_2x4(cs, cs + 32, w[0], w[1]);
          else
            tmem_st16x256_x4(cs, w[0]);
        }
      }
      hand_over(bar + kRdyS);
      // (e) this chunk's outputs, while the next chunk's P runs
      if (epi_any(!mbar_wait_bounded(bar + kBarO, par))) {
        failed = true;
        break;
      }
      tc_fence_after();
      out_chunk(lc, tok0, gam);
    }
  }
  // (the issuer's and the epilogue's failure flags meet here; warp 8's other lanes idled)
  __syncwarp();
  failed = __syncthreads_or(failed) != 0;

  if (failed) {
    if (tid == kIssuer) {  // every copy and MMA group still in flight lands before TMEM is freed
      atomicOr(p.err, kDevErrTimeout);
      for (int q = 0; q < kNumBars; ++q)
        if (armed[q] > 0) (void)mbar_drain(bar + q, uint32_t(armed[q] - 1) & 1u);
    }
  } else {
    // final state from TMEM
    float* dst = p.state_out + ((size_t(i) * p.Hv + h) * DV + r0 + m) * DK + hh * SC;
#pragma unroll
    for (int c0 = 0; c0 < SC && epi; c0 += 32) {
      float sv[32];
      tmem_ld32(tmem + lane_sel + kColS + hh * SC + c0, sv);
      if (act)
#pragma unroll
        for (int q = 0; q < 32; q += 4) *reinterpret_cast<float4*>(dst + c0 + q) = make_float4(sv[q], sv[q + 1], sv[q + 2], sv[q + 3]);
    }
    // conv history: the v channels from the last three raw rows (rows len .. len + 2 of the
    // last chunk, or the untouched history of an empty prompt); epilogue threads only, which
    // know len
    for (int idx = tid; idx < 3 * kTileRows; idx += kThreads) {
      const int mm = idx / kTileRows, ch = idx % kTileRows;
      p.conv_state_out[(size_t(i) * 3 + mm) * C + vch0 + ch] = sX[(len + mm) * kTileRows + (ch ^ swz(len + mm))];
    }
    // the q|k channels of the head group, split over the first v-head's row tiles; every value
    // is read before this thread writes, and no other thread of this grid reads them
    if (h % (p.Hv / p.Hk) == 0) {
      constexpr int kPer = 2 * DK / kHalves;
      for (int q = tid; q < kPer; q += kThreads) {
        const int ch = (r0 / kTileRows) * kPer + q;
        const size_t gch = (ch < DK) ? size_t(kh) * DK + ch : size_t(p.Hk) * DK + size_t(kh) * DK + (ch - DK);
        float hv[3];
#pragma unroll
        for (int mm = 0; mm < 3; ++mm) {
          const long long pos = s1 - 3 + mm;
          hv[mm] = (pos >= s0) ? bf16_to_f32(p.x[size_t(pos) * C + gch])
                               : p.conv_state_in[(size_t(i) * 3 + size_t(pos - s0 + 3)) * C + gch];
        }
#pragma unroll
        for (int mm = 0; mm < 3; ++mm) p.conv_state_out[(size_t(i) * 3 + mm) * C + gch] = hv[mm];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------------
// Kernel 2 at dv = 128: one CTA per (prompt, v-head), the whole 128-row state as one M = 128
// accumulator (row m in TMEM lane m), so that every MMA does twice the work of an M = 64 one in
// the same time and 256 CTAs make 2 waves where 512 made 4.  The operand space this needs is
// found in tensor memory: the S operand's hi and lo halves live there as the A operand of the P
// product (row m in lane m, two bf16 per 32-bit column), and P needs one buffer because the
// epilogue turns its q^ half into the initial value Gamma o P_q of the o accumulator, onto which
// the o' MMA then adds.  TMEM: the state (dk columns), P (128), u (64), o (64), S hi and lo
// (dk / 2 each) - all 512 columns at dk = 128.  Epilogue warp w reaches lanes 32 (w % 4) ..
// + 31 (rows) with the 32x32b shape; warps w and w + 4 split the columns.  Raw x is staged as
// bf16 (it is bf16), the three history rows as f32.
template <int DK>
struct Tc128Layout {
  static constexpr int ROWS = 128;
  static constexpr int BLK_KQ = kCh * DK * 2;               // one 64 x DK bf16 operand
  static constexpr int BLK_R = ROWS * kCh * 2;              // one 128 x 64 bf16 operand (r, d o u, u)
  static constexpr int BLK = kCh * kCh * 2;                 // one 64 x 64 bf16 operand (W, MQ)
  static constexpr int OFF_KH = 0;                          // [k^0 | q^ | k^1] hi
  static constexpr int OFF_KL = OFF_KH + 3 * BLK_KQ;        // the same, lo
  static constexpr int OFF_W = OFF_KL + 3 * BLK_KQ;         // W hi, lo
  static constexpr int OFF_MQ = OFF_W + 2 * BLK;            // MQ hi, lo
  static constexpr int OFF_GD = OFF_MQ + 2 * BLK;           // two buffers of Gamma[64], d[64]
  static constexpr int OFF_RD = OFF_GD + 2 * 2 * kCh * 4;   // r hi, lo; later (d o u) hi, lo
  static constexpr int OFF_U = OFF_RD + 2 * BLK_R;          // u hi, lo; later the staged outputs
  static constexpr int OFF_H = OFF_U + 2 * BLK_R;           // three history rows [3][128] f32
  static constexpr int OFF_X = OFF_H + 3 * ROWS * 4;        // raw x of a chunk [64][128] bf16
  static constexpr int OFF_TAP = OFF_X + kCh * ROWS * 2;    // conv taps [128][4]
  static constexpr int OFF_BAR = OFF_TAP + ROWS * 16;       // mbarriers
  static constexpr int NBAR = 16;
  static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_TSLOT + 16;
  static_assert(2 * BLK_R >= kCh * ROWS * 4, "the staged outputs fit in the u operand's space");
  static_assert(OFF_X % 16 == 0 && OFF_TAP % 16 == 0 && OFF_BAR % 8 == 0, "alignment");
  static_assert(BYTES <= 227 * 1024, "one CTA per SM");
};

// TMEM columns of the M = 128 kernel
constexpr uint32_t kC8S = 0, kC8P = 128, kC8U = 256, kC8O = 320, kC8SH = 384, kC8SL = 448;
// its extra mbarrier: the u operand written (the o' MMA waits for it; the update MMA, on the
// chain, waits only for d o u)
constexpr int kRdyUo = kNumBars;

// Three-pass split product with the A operand in TMEM (hi and lo halves at a_hi, a_lo; a K step
// of 16 is 8 columns) and the B operand K-major in shared memory.
template <int KSTEPS>
__device__ __forceinline__ void umma_split3_at(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hi, uint32_t b_lo,
                                               uint32_t b_sbo, uint32_t idesc) {
  const uint64_t dbh = umma_smem_desc(b_hi, 128, b_sbo), dbl = umma_smem_desc(b_lo, 128, b_sbo);
#pragma unroll
  for (int sp = 0; sp < 3; ++sp) {
    const uint32_t a = (sp == 2) ? a_lo : a_hi;
    const uint64_t db = (sp == 1) ? dbl : dbh;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const uint32_t acc = (sp > 0 || kk > 0) ? 1u : 0u;
      asm volatile(
          "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
          "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
          "r"(a + 8 * kk), "l"(db + uint64_t(16 * kk)), "r"(idesc), "r"(acc)
          : "memory");
    }
  }
}

// The staged output table [64 tokens][128 rows] f32: row (token) t, column c at t * 128 +
// (c ^ sw) with the column bits 5-6 and the token's low bit folded into bits 2-4, so that both
// the row-per-lane writes and the 16-byte reads of 32 columns per lane are free of conflicts.
__device__ __forceinline__ int out_col(int t, int c) { return c ^ ((((c >> 5) & 3) | ((t & 1) << 2)) << 2); }

template <int DK>
__global__ void __launch_bounds__(kThreads + 32, 1) gdn_prefill_state128_kernel(const PrefillParams p) {
  using L = Tc128Layout<DK>;
  constexpr int ROWS = L::ROWS;
  constexpr int SC = DK / 2;   // state columns per epilogue thread (two warps per lane quarter)
  constexpr int SP = DK / 4;   // packed bf16 pairs of them
  static_assert(SC == 32 || SC == 64, "dk = 64 or 128");
  extern __shared__ __align__(128) uint8_t smb[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int i = blockIdx.y;
  const int h = blockIdx.x;
  const int kh = h / (p.Hv / p.Hk);
  if (p.ws.meta[0] == 0) return;
  const int32_t* base = p.ws.meta + 4;
  const int c_first = base[i], n_chunks = base[i + 1] - base[i];
  const long long s0 = p.cu[i], s1 = p.cu[i + 1];
  const size_t C = size_t(p.C);
  const size_t vch0 = size_t(2) * p.Hk * DK + size_t(h) * ROWS;  // first conv channel of the head
  float* sH = reinterpret_cast<float*>(smb + L::OFF_H);
  uint16_t* sX = reinterpret_cast<uint16_t*>(smb + L::OFF_X);
  float* sTap = reinterpret_cast<float*>(smb + L::OFF_TAP);
  uint64_t* bar = reinterpret_cast<uint64_t*>(smb + L::OFF_BAR);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smb + L::OFF_TSLOT);
  const uint32_t sbase = smem_addr(smb);

  // epilogue coordinates: row m = lane 32 quad + lane, column half hh (tokens 32 hh .. + 31 of a
  // chunk, state columns hh SC .. + SC - 1)
  const int quad = warp & 3, hh = warp >> 2;
  const int m = 32 * quad + lane;
  const bool epi = warp < kThreads / 32;
  const uint32_t lane_sel = uint32_t(32 * quad) << 16;

  static_assert(L::NBAR > kRdyUo, "mbarrier slots");
  if (tid == 0) {
    for (int q = 0; q <= kRdyUo; ++q) mbar_init(bar + q, q >= kRdyR ? kEpiThreads : 1);
    fence_mbar_init();
  }
  if (warp == 0) tmem_alloc(tslot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  int armed[kNumBars] = {};
  auto kq_src = [&](int c) {
    return reinterpret_cast<const uint8_t*>(p.ws.kq) + (size_t(c) * p.Hk + kh) * kKqBlocks * L::BLK_KQ;
  };
  auto issue_k = [&](int c, int b) {
    ++armed[kBarK0 + b];
    mbar_arrive_expect_tx(bar + kBarK0 + b, 2 * L::BLK_KQ);
    bulk_load(smb + L::OFF_KH + 2 * b * L::BLK_KQ, kq_src(c), L::BLK_KQ, bar + kBarK0 + b);
    bulk_load(smb + L::OFF_KL + 2 * b * L::BLK_KQ, kq_src(c) + L::BLK_KQ, L::BLK_KQ, bar + kBarK0 + b);
  };
  auto issue_q = [&](int c) {
    ++armed[kBarQ];
    mbar_arrive_expect_tx(bar + kBarQ, 2 * L::BLK_KQ);
    bulk_load(smb + L::OFF_KH + L::BLK_KQ, kq_src(c) + 2 * L::BLK_KQ, L::BLK_KQ, bar + kBarQ);
    bulk_load(smb + L::OFF_KL + L::BLK_KQ, kq_src(c) + 3 * L::BLK_KQ, L::BLK_KQ, bar + kBarQ);
  };
  auto wq_src = [&](int c) {
    return reinterpret_cast<const uint8_t*>(p.ws.wm) + (size_t(c) * p.Hv + h) * (4 * L::BLK);
  };
  auto issue_w = [&](int c) {
    ++armed[kBarW];
    mbar_arrive_expect_tx(bar + kBarW, 2 * L::BLK);
    bulk_load(smb + L::OFF_W, wq_src(c), 2 * L::BLK, bar + kBarW);
  };
  auto issue_mq = [&](int c) {
    ++armed[kBarMQ];
    mbar_arrive_expect_tx(bar + kBarMQ, 2 * L::BLK);
    bulk_load(smb + L::OFF_MQ, wq_src(c) + 2 * L::BLK, 2 * L::BLK, bar + kBarMQ);
  };
  auto issue_gd = [&](int lc) {  // buffer lc & 1 holds local chunk lc
    const int b = lc & 1, c = c_first + lc;
    ++armed[kBarGD0 + b];
    mbar_arrive_expect_tx(bar + kBarGD0 + b, 2 * kCh * 4);
    bulk_load(smb + L::OFF_GD + b * 2 * kCh * 4, p.ws.gd + (size_t(c) * p.Hv + h) * (2 * kCh), 2 * kCh * 4,
              bar + kBarGD0 + b);
  };
  if (tid == kIssuer && n_chunks > 0) {
    issue_k(c_first, 0);
    issue_q(c_first);
    issue_w(c_first);
    issue_mq(c_first);
    issue_gd(0);
    if (n_chunks > 1) {
      issue_gd(1);
      issue_k(c_first + 1, 1);
    }
  }

  // hi/lo operand stores of 32 consecutive K values (this thread's tokens) of row m of a K-major
  // [128][64] operand (lo block BLK_R bytes after hi)
  auto store_row32 = [&](int off, const float* v) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      uint4 hi, lo;
      split8(v + 8 * g, hi, lo);
      const uint32_t o = kmajor_off(m, 32 * hh + 8 * g, kCh);
      *reinterpret_cast<uint4*>(smb + off + o) = hi;
      *reinterpret_cast<uint4*>(smb + off + L::BLK_R + o) = lo;
    }
  };
  // state columns hh SC + 32 q .. + 31 of this thread's row: loaded, stored, and split into the S
  // operand (packed two per TMEM column), one 32-column slice at a time
  auto ld_state = [&](int q, float (&sv)[32]) { tmem_ld32(tmem + lane_sel + kC8S + hh * SC + 32 * q, sv); };
  auto st_state = [&](int q, const float (&sv)[32]) { tmem_st32(tmem + lane_sel + kC8S + hh * SC + 32 * q, sv); };
  auto store_s_operand = [&](int q, const float (&sv)[32]) {
    float ph[16], pl[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      uint32_t hi, lo;
      split2(sv[2 * e], sv[2 * e + 1], hi, lo);
      ph[e] = __uint_as_float(hi);
      pl[e] = __uint_as_float(lo);
    }
    tmem_st16(tmem + lane_sel + kC8SH + hh * SP + 16 * q, ph);
    tmem_st16(tmem + lane_sel + kC8SL + hh * SP + 16 * q, pl);
  };

  // the state into TMEM and, split, into the S operand; taps; the v channels' history
  if (epi) {
    const float* src = p.state_in + ((size_t(i) * p.Hv + h) * ROWS + m) * DK + hh * SC;
#pragma unroll
    for (int q = 0; q < SC / 32; ++q) {
      float sv[32];
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const float4 f = *reinterpret_cast<const float4*>(src + 32 * q + e);
        sv[e] = f.x;
        sv[e + 1] = f.y;
        sv[e + 2] = f.z;
        sv[e + 3] = f.w;
      }
      st_state(q, sv);
      store_s_operand(q, sv);
    }
  }
  if (tid < ROWS) *reinterpret_cast<float4*>(sTap + 4 * tid) = *reinterpret_cast<const float4*>(p.conv_w + (vch0 + tid) * kConvW);
  for (int idx = tid; idx < 3 * ROWS; idx += kThreads + 32) {
    const int mm = idx / ROWS, ch = idx % ROWS;
    sH[idx] = p.conv_state_in[(size_t(i) * 3 + mm) * C + vch0 + ch];
  }
  // raw x of the head's 128 channels for one chunk: thread = (channels 8 xc .. + 7, tokens
  // xr0 + 16 q), so that each quarter-warp's 16-byte stores fill 128 contiguous bytes of a row
  const int xc = tid & 15, xr0 = (tid >> 4) & 15;
  uint4 xr[4] = {};
  if (epi && n_chunks > 0) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (xr0 + 16 * q < min_ll(kCh, s1 - s0))
        xr[q] = *reinterpret_cast<const uint4*>(p.x + size_t(s0 + xr0 + 16 * q) * C + vch0 + 8 * xc);
  }
  // the output write-out: thread = (token xt, rows 32 xg .. + 31)
  const int xt = tid >> 2, xg = tid & 3;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  const uint32_t id_n64 = umma_idesc_bf16(ROWS, kCh);
  const uint32_t id_n128 = umma_idesc_bf16(ROWS, 2 * kCh);
  const uint32_t id_ndk_bmn = umma_idesc_bf16(ROWS, DK) | (1u << 16);  // B MN-major
  bool failed = false;
  if (n_chunks > 0) {
    // the state in TMEM is kept pre-scaled by the current chunk's Gamma_63, so that the update
    // MMA can accumulate onto it (the S operand holds it unscaled)
    if (wait_failed(bar + kBarGD0, 0)) {
      failed = true;
    } else {
      tc_fence_after();
      if (epi) {
        const float gl = reinterpret_cast<const float*>(smb + L::OFF_GD)[kCh - 1];
#pragma unroll
        for (int q = 0; q < SC / 32; ++q) {
          float sv[32];
          ld_state(q, sv);
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[e] *= gl;
          st_state(q, sv);
        }
      }
      tc_fence_before();
      __syncthreads();
      tc_fence_after();
    }
  }

  int len = 0;
  if (tid == kIssuer) {
    for (int lc = 0; lc < n_chunks && !failed; ++lc) {
      const uint32_t par = lc & 1;
      const bool more = lc + 1 < n_chunks;
      // P = S [k^ | q^]^T with S from TMEM, once the S operand is written (and the previous
      // chunk's P has been read: the same hand-over); [k^0 | q^] for even chunks, P_k in the
      // first 64 columns, [q^ | k^1] for odd ones, P_k in the second 64
      if ((lc > 0 && !mbar_wait_bounded(bar + kRdyS, (lc - 1) & 1)) ||
          !mbar_wait_bounded(bar + kBarK0 + par, (lc >> 1) & 1) || !mbar_wait_bounded(bar + kBarQ, par)) {
        failed = true;
        break;
      }
      tc_fence_after();
      {
        const uint32_t bo = (par ? 1 : 0) * L::BLK_KQ;
        umma_split3_at<DK / 16>(tmem + kC8P, tmem + kC8SH, tmem + kC8SL, sbase + L::OFF_KH + bo,
                                sbase + L::OFF_KL + bo, (DK / 8) * 128, id_n128);
        umma_commit(bar + kBarPk);
        ++armed[kBarPk];
      }
      // copies only right after an MMA group: this chunk's MQ, the next chunk's k^
      if (lc > 0) {
        if (!mbar_wait_bounded(bar + kBarO, (lc - 1) & 1)) {
          failed = true;
          break;
        }
        issue_mq(c_first + lc);
        if (more) {
          if (!mbar_wait_bounded(bar + kBarS, (lc - 1) & 1)) {
            failed = true;
            break;
          }
          issue_k(c_first + lc + 1, (lc + 1) & 1);
        }
      }
      // u = r W^T; then the next chunk's q^
      if (!mbar_wait_bounded(bar + kRdyR, par) || !mbar_wait_bounded(bar + kBarW, par)) {
        failed = true;
        break;
      }
      tc_fence_after();
      umma_split3<kCh / 16>(tmem + kC8U, sbase + L::OFF_RD, sbase + L::OFF_RD + L::BLK_R, sbase + L::OFF_W,
                            sbase + L::OFF_W + L::BLK, 1024, id_n64, false);
      umma_commit(bar + kBarU);
      ++armed[kBarU];
      if (more) issue_q(c_first + lc + 1);
      // S += (d o u) k^, then o += u MQ^T (onto Gamma o P_q); then the next W and Gamma, d
      if (!mbar_wait_bounded(bar + kRdyU, par)) {
        failed = true;
        break;
      }
      tc_fence_after();
      umma_split3_bmn<kCh / 16>(tmem + kC8S, sbase + L::OFF_RD, sbase + L::OFF_RD + L::BLK_R, 1024,
                                sbase + L::OFF_KH + 2 * par * L::BLK_KQ, sbase + L::OFF_KL + 2 * par * L::BLK_KQ,
                                (DK / 8) * 128, 128, id_ndk_bmn, true);
      umma_commit(bar + kBarS);
      ++armed[kBarS];
      if (!mbar_wait_bounded(bar + kBarMQ, par) || !mbar_wait_bounded(bar + kRdyUo, par)) {
        failed = true;
        break;
      }
      tc_fence_after();
      umma_split3<kCh / 16>(tmem + kC8O, sbase + L::OFF_U, sbase + L::OFF_U + L::BLK_R, sbase + L::OFF_MQ,
                            sbase + L::OFF_MQ + L::BLK, 1024, id_n64, true);
      umma_commit(bar + kBarO);
      ++armed[kBarO];
      if (more) issue_w(c_first + lc + 1);
      if (lc + 2 < n_chunks) issue_gd(lc + 2);
    }
  } else if (epi && !failed && n_chunks > 0) {
    // raw x of a chunk into the staging table (zero past the prompt's end), then the next
    // chunk's x is fetched
    auto stage_x = [&](long long tok0, int n) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int t = xr0 + 16 * q;
        *reinterpret_cast<uint4*>(sX + t * ROWS + 8 * xc) = (t < n) ? xr[q] : make_uint4(0, 0, 0, 0);
        const long long nt = tok0 + kCh + t;
        if (nt < s1) xr[q] = *reinterpret_cast<const uint4*>(p.x + size_t(nt) * C + vch0 + 8 * xc);
      }
    };
    // value idx of the chunk's window [history rows 0..2, x_0 .. x_63] for channel m
    auto win = [&](int idx) { return idx < 3 ? sH[idx * ROWS + m] : bf16_to_f32(sX[(idx - 3) * ROWS + m]); };
    // conv + SiLU of channel m at this thread's 32 tokens
    float v[32];
    auto conv = [&]() {
      const float4 w = *reinterpret_cast<const float4*>(sTap + 4 * m);
      float a0 = win(32 * hh), a1 = win(32 * hh + 1), a2 = win(32 * hh + 2);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float a3 = win(32 * hh + j + 3);
        v[j] = silu(fmaf(w.w, a3, fmaf(w.z, a2, fmaf(w.y, a1, w.x * a0))));
        a0 = a1;
        a1 = a2;
        a2 = a3;
      }
    };
    float* sOut = reinterpret_cast<float*>(smb + L::OFF_U);  // [64 tokens][128 rows], out_col order
    auto hand_over = [&](uint64_t* rdy) {
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(rdy);
    };

    stage_x(s0, int(min_ll(kCh, s1 - s0)));
    epi_sync();
    conv();
    for (int lc = 0; lc < n_chunks; ++lc) {
      const uint32_t par = lc & 1;
      const float* sGam = reinterpret_cast<const float*>(smb + L::OFF_GD + (lc & 1) * 2 * kCh * 4);
      const float* sd = sGam + kCh;
      const long long tok0 = s0 + (long long)lc * kCh;
      len = int(min_ll(kCh, s1 - tok0));
      const bool more = lc + 1 < n_chunks;

      // (a) r = v - Gamma o P_k -> operand (on the chain); then o = Gamma o P_q into the o
      // accumulator (the o' MMA adds onto it) and the last three raw rows become the next
      // chunk's history
      if (epi_any(!mbar_wait_bounded(bar + kBarPk, par))) {
        failed = true;
        break;
      }
      tc_fence_after();
      {
        float pk[32];
        tmem_ld32(tmem + lane_sel + kC8P + (par ? kCh : 0) + 32 * hh, pk);
#pragma unroll
        for (int j = 0; j < 32; ++j) pk[j] = fmaf(-sGam[32 * hh + j], pk[j], v[j]);
        store_row32(L::OFF_RD, pk);
      }
      hand_over(bar + kRdyR);
      {
        float pq[32];
        tmem_ld32(tmem + lane_sel + kC8P + (par ? 0 : kCh) + 32 * hh, pq);
#pragma unroll
        for (int j = 0; j < 32; ++j) pq[j] *= sGam[32 * hh + j];
        tmem_st32(tmem + lane_sel + kC8O + 32 * hh, pq);
      }
      if (len == kCh) {
        for (int idx = tid; idx < 3 * ROWS; idx += kThreads) sH[idx] = bf16_to_f32(sX[(kCh - 3) * ROWS + idx]);
      }
      // (b) d o u -> the update's operand (on the chain), then u -> the o' MMA's
      if (epi_any(!mbar_wait_bounded(bar + kBarU, par))) {
        failed = true;
        break;
      }
      tc_fence_after();
      {
        float u[32], du[32];
        tmem_ld32(tmem + lane_sel + kC8U + 32 * hh, u);
#pragma unroll
        for (int j = 0; j < 32; ++j) du[j] = u[j] * sd[32 * hh + j];
        store_row32(L::OFF_RD, du);  // r is dead: the u MMAs are done
        hand_over(bar + kRdyU);
        store_row32(L::OFF_U, u);
      }
      hand_over(bar + kRdyUo);
      // (c) while the state update runs: the next chunk's raw x and conv
      if (more) {
        stage_x(tok0 + kCh, int(min_ll(kCh, s1 - tok0 - kCh)));
        epi_sync();
        conv();
      }
      // (d) the new state: split into the S operand of the next chunk (unscaled), and pre-scaled
      // in TMEM by the next chunk's Gamma_63
      {
        bool ok = mbar_wait_bounded(bar + kBarS, par);
        if (more) ok = ok && mbar_wait_bounded(bar + kBarGD0 + ((lc + 1) & 1), ((lc + 1) >> 1) & 1);
        if (epi_any(!ok)) {
          failed = true;
          break;
        }
      }
      tc_fence_after();
      // (the S operand first: the next P waits for it; the update that adds onto the re-scaled
      // state is issued only after this chunk's hand-overs)
      if (more) {
#pragma unroll
        for (int q = 0; q < SC / 32; ++q) {
          float sv[32];
          ld_state(q, sv);
          store_s_operand(q, sv);
        }
      }
      hand_over(bar + kRdyS);
      if (more) {
        const float gl = reinterpret_cast<const float*>(smb + L::OFF_GD + ((lc + 1) & 1) * 2 * kCh * 4)[kCh - 1];
#pragma unroll
        for (int q = 0; q < SC / 32; ++q) {
          float sv[32];
          ld_state(q, sv);
#pragma unroll
          for (int e = 0; e < 32; ++e) sv[e] *= gl;
          st_state(q, sv);
        }
      }
      // (e) this chunk's outputs, while the next chunk's P runs: o = q_scale (Gamma o P_q + o'),
      // staged token-major in the u operand's space (the o' MMAs are done with it), then
      // written out as 16-byte stores, thread = (token xt, 32 rows)
      if (epi_any(!mbar_wait_bounded(bar + kBarO, par))) {
        failed = true;
        break;
      }
      tc_fence_after();
      {
        float o[32];
        tmem_ld32(tmem + lane_sel + kC8O + 32 * hh, o);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int t = 32 * hh + j;
          sOut[t * ROWS + out_col(t, m)] = p.q_scale * o[j];
        }
      }
      epi_sync();
      if (xt < len) {
        const float* src = sOut + xt * ROWS;
        const size_t oi = size_t(tok0 + xt) * p.Hv * ROWS + size_t(h) * ROWS + 32 * xg;
        float4 f[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) f[q] = *reinterpret_cast<const float4*>(src + out_col(xt, 32 * xg + 4 * q));
        if (p.out_f32) {
          float4* o4 = reinterpret_cast<float4*>(static_cast<float*>(p.out) + oi);
#pragma unroll
          for (int q = 0; q < 8; ++q) o4[q] = f[q];
        } else {
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const __nv_bfloat162 b0 = __floats2bfloat162_rn(f[q].x, f[q].y);
            const __nv_bfloat162 b1 = __floats2bfloat162_rn(f[q].z, f[q].w);
            w[2 * q] = *reinterpret_cast<const uint32_t*>(&b0);
            w[2 * q + 1] = *reinterpret_cast<const uint32_t*>(&b1);
          }
          uint4* o4 = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) + oi);
#pragma unroll
          for (int q = 0; q < 4; ++q) o4[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
        }
      }
      // (the staging space is next written as the u operand in (b), behind the barrier of (a))
    }
  }
  __syncwarp();
  failed = __syncthreads_or(failed) != 0;

  if (failed) {
    if (tid == kIssuer) {  // every copy and MMA group still in flight lands before TMEM is freed
      atomicOr(p.err, kDevErrTimeout);
      for (int q = 0; q < kNumBars; ++q)
        if (armed[q] > 0) (void)mbar_drain(bar + q, uint32_t(armed[q] - 1) & 1u);
    }
  } else {
    // final state from TMEM (the last update left it unscaled)
    if (epi) {
      float* dst = p.state_out + ((size_t(i) * p.Hv + h) * ROWS + m) * DK + hh * SC;
#pragma unroll
      for (int q = 0; q < SC / 32; ++q) {
        float sv[32];
        ld_state(q, sv);
#pragma unroll
        for (int e = 0; e < 32; e += 4)
          *reinterpret_cast<float4*>(dst + 32 * q + e) = make_float4(sv[e], sv[e + 1], sv[e + 2], sv[e + 3]);
      }
    }
    // conv history: the v channels from window rows len .. len + 2 of the last chunk (the
    // untouched history of an empty prompt)
    for (int idx = tid; epi && idx < 3 * ROWS; idx += kThreads) {  // (epilogue threads know len)
      const int mm = idx / ROWS, ch = idx % ROWS, row = len + mm;
      p.conv_state_out[(size_t(i) * 3 + mm) * C + vch0 + ch] =
          row < 3 ? sH[row * ROWS + ch] : bf16_to_f32(sX[(row - 3) * ROWS + ch]);
    }
    // the q|k channels of the head group, by the group's first v-head; every value is read
    // before this thread writes, and no other thread of this grid reads them
    if (h % (p.Hv / p.Hk) == 0) {
      for (int q = tid; q < 2 * DK; q += kThreads + 32) {
        const size_t gch = (q < DK) ? size_t(kh) * DK + q : size_t(p.Hk) * DK + size_t(kh) * DK + (q - DK);
        float hv[3];
#pragma unroll
        for (int mm = 0; mm < 3; ++mm) {
          const long long pos = s1 - 3 + mm;
          hv[mm] = (pos >= s0) ? bf16_to_f32(p.x[size_t(pos) * C + gch])
                               : p.conv_state_in[(size_t(i) * 3 + size_t(pos - s0 + 3)) * C + gch];
        }
#pragma unroll
        for (int mm = 0; mm < 3; ++mm) p.conv_state_out[(size_t(i) * 3 + mm) * C + gch] = hv[mm];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int DK, int DV>
cudaError_t launch_prefill_t(const PrefillParams& p, cudaStream_t stream) {
  auto k1 = gdn_prefill_chunk_kernel<DK>;
  // dv = 128: the whole v-head per CTA (M = 128); dv = 64: the M = 64 kernel, also one CTA per head
  constexpr bool kM128 = DV == 128;
  auto k2 = kM128 ? gdn_prefill_state128_kernel<DK> : gdn_prefill_state_kernel<DK, DV>;
  const size_t b1 = ChunkLayout<DK>::BYTES, b2 = kM128 ? size_t(Tc128Layout<DK>::BYTES) : size_t(TcLayout<DK>::BYTES);
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
  k2<<<dim3(unsigned(p.Hv * (kM128 ? 1 : DV / kTileRows)), unsigned(p.B), 1), kThreads + 32, b2, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_workspace_bytes(int B, long long N, int Hk, int Hv, int dk) {
  const long long cap = prefill_chunk_cap(B, N);
  const size_t meta = ((size_t(B) + 5 + 3) & ~size_t(3)) * 4;
  return meta + size_t(cap) * (16 + size_t(Hk) * kKqBlocks * kCh * dk * 2 + size_t(Hv) * (4 * kCh * kCh * 2 + 2 * kCh * 4));
}

PrefillWorkspace prefill_workspace_carve(void* base, int B, long long N, int Hk, int Hv, int dk) {
  PrefillWorkspace w;
  w.chunk_cap = prefill_chunk_cap(B, N);
  char* p = static_cast<char*>(base);
  w.meta = reinterpret_cast<int32_t*>(p);
  p += ((size_t(B) + 5 + 3) & ~size_t(3)) * 4;
  w.chunks = reinterpret_cast<int4*>(p);
  p += size_t(w.chunk_cap) * 16;
  w.kq = reinterpret_cast<uint16_t*>(p);
  p += size_t(w.chunk_cap) * Hk * kKqBlocks * kCh * dk * 2;
  w.wm = reinterpret_cast<uint16_t*>(p);
  p += size_t(w.chunk_cap) * Hv * 4 * kCh * kCh * 2;
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
