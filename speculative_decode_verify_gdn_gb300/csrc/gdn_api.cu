// C ABI of the GDN verify library: host-side validation, launches, error reporting.
//
// Every entry point checks its arguments completely before it enqueues anything, so a
// non-OK status always means that nothing ran.  Checks: shapes inside the supported set,
// 16-byte alignment of every buffer (bulk async copies and float4 accesses need it), the
// aliasing rules of each call, finite scalars.  See include/gdn.h for the contract.
#include <climits>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "gdn_common.cuh"
#include "gdn_kernels.h"

namespace {

thread_local std::string g_last_error;

// Per-device status word; kernels OR error bits into it.
__device__ uint32_t g_device_status;

gdn_status fail(gdn_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

gdn_status ok() {
  g_last_error.clear();
  return GDN_OK;
}

// Device address of g_device_status on the current device (looked up once per device).
gdn_status status_word(uint32_t** out) {
  constexpr int kMaxDevices = 64;
  static uint32_t* cache[kMaxDevices] = {};
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(GDN_ERR_UNSUPPORTED, "device ordinal %d", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_device_status);
    if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "cudaGetSymbolAddress: %s", cudaGetErrorString(e));
    cache[dev] = static_cast<uint32_t*>(ptr);
  }
  *out = cache[dev];
  return GDN_OK;
}

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
  bool valid() const { return lo != 0 && hi > lo; }
};

Range range_of(const void* p, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return Range{a, p ? a + bytes : 0};
}

bool overlap(Range a, Range b) { return a.valid() && b.valid() && a.lo < b.hi && b.lo < a.hi; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_dims(const gdn_dims* d, bool need_gates, bool check_K = true) {
  if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 0 || d->B > 65535) return fail(GDN_ERR_INVALID_ARG, "B=%d outside 0..65535", d->B);
  if (check_K && (d->K < 1 || d->K > gdn::kKMax))
    return fail(GDN_ERR_UNSUPPORTED, "K=%d outside 1..%d", d->K, gdn::kKMax);
  if (d->conv_w != gdn::kConvW) return fail(GDN_ERR_UNSUPPORTED, "conv width %d (only 4)", d->conv_w);
  if (d->Hk < 1 || d->Hv < 1) return fail(GDN_ERR_INVALID_ARG, "Hk=%d Hv=%d must be >= 1", d->Hk, d->Hv);
  if (d->Hv % d->Hk != 0) return fail(GDN_ERR_UNSUPPORTED, "Hv=%d not a multiple of Hk=%d", d->Hv, d->Hk);
  if (d->dk != 64 && d->dk != 128) return fail(GDN_ERR_UNSUPPORTED, "dk=%d (64 or 128)", d->dk);
  if (d->dv != 64 && d->dv != 128) return fail(GDN_ERR_UNSUPPORTED, "dv=%d (64 or 128)", d->dv);
  if (d->out_f32 != 0 && d->out_f32 != 1) return fail(GDN_ERR_INVALID_ARG, "out_f32=%d (0 or 1)", d->out_f32);
  const long long C = 2LL * d->Hk * d->dk + 1LL * d->Hv * d->dv;
  if (C > (1LL << 24)) return fail(GDN_ERR_UNSUPPORTED, "C=%lld channels too many", C);
  if (need_gates) {
    if (!std::isfinite(d->q_scale)) return fail(GDN_ERR_INVALID_ARG, "q_scale not finite");
    if (!std::isfinite(d->l2_eps) || d->l2_eps < 0.f) return fail(GDN_ERR_INVALID_ARG, "l2_eps must be finite, >= 0");
  }
  return GDN_OK;
}

#define GDN_CHECK_PTR(p, name)                                                                     \
  do {                                                                                             \
    if (!(p)) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", name);                                \
    if (!aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name);        \
  } while (0)

#define GDN_CHECK_OPT_PTR(p, name)                                                                 \
  do {                                                                                             \
    if ((p) && !aligned16(p)) return fail(GDN_ERR_INVALID_ARG, "%s is not 16-byte aligned", name); \
  } while (0)

// Arguments of the verify step; the *_prev and snapshot fields are used by gdn_verify_resume only.
struct VerifyArgs {
  bool resume;
  const int32_t* accept_prev;
  const int32_t* parent;  // token tree (gdn_verify_tree) or null
  const uint16_t* z;      // gated output norm (gdn_verify_gated) or null
  const float* norm_w;
  float norm_eps;
  const uint16_t *x, *a, *b;
  const float *A_log, *dt_bias, *conv_w;
  const float* conv_state_in;
  const float* conv_inter_prev;
  const float* conv_snap_prev;
  float* conv_state_out;
  float* conv_inter;
  const float* state_in;
  const float* state_inter_prev;
  const float* state_snap_prev;
  float* state_out;
  float* state_inter;
  void* out;
};

struct Buf {
  const char* name;
  Range r;
  bool output;
};

gdn_status verify_impl(const gdn_dims* dims, const VerifyArgs& v, gdn_stream_t stream) {
  gdn_status s = check_dims(dims, true);
  if (s != GDN_OK) return s;
  const gdn_dims& d = *dims;
  if (d.B == 0) return ok();
  GDN_CHECK_PTR(v.x, "x");
  GDN_CHECK_PTR(v.a, "a");
  GDN_CHECK_PTR(v.b, "b");
  GDN_CHECK_PTR(v.A_log, "A_log");
  GDN_CHECK_PTR(v.dt_bias, "dt_bias");
  GDN_CHECK_PTR(v.conv_w, "conv_w");
  GDN_CHECK_PTR(v.conv_state_in, "conv_state_in");
  GDN_CHECK_PTR(v.conv_state_out, "conv_state_out");
  GDN_CHECK_OPT_PTR(v.conv_inter, "conv_inter");
  GDN_CHECK_PTR(v.state_in, "state_in");
  GDN_CHECK_PTR(v.state_out, "state_out");
  GDN_CHECK_OPT_PTR(v.state_inter, "state_inter");
  GDN_CHECK_PTR(v.out, "out");
  if (d.K > 1 && !v.state_inter) return fail(GDN_ERR_INVALID_ARG, "state_inter is NULL with K=%d > 1", d.K);
  if (v.resume) {
    if (!v.accept_prev) return fail(GDN_ERR_INVALID_ARG, "accept_len_prev is NULL");
    if (reinterpret_cast<uintptr_t>(v.accept_prev) & 3u) return fail(GDN_ERR_INVALID_ARG, "accept_len_prev misaligned");
    GDN_CHECK_OPT_PTR(v.state_inter_prev, "state_inter_prev");
    GDN_CHECK_OPT_PTR(v.conv_inter_prev, "conv_inter_prev");
    GDN_CHECK_OPT_PTR(v.state_snap_prev, "state_snapshot_prev");
    GDN_CHECK_OPT_PTR(v.conv_snap_prev, "conv_state_snapshot_prev");
    if (d.K > 1 && (!v.state_inter_prev || !v.conv_inter_prev))
      return fail(GDN_ERR_INVALID_ARG, "state_inter_prev and conv_inter_prev are required when K=%d > 1", d.K);
    if ((v.state_snap_prev == nullptr) != (v.conv_snap_prev == nullptr))
      return fail(GDN_ERR_NO_SNAPSHOT, "pass both snapshots or neither");
  }
  if (v.parent && (reinterpret_cast<uintptr_t>(v.parent) & 3u))
    return fail(GDN_ERR_INVALID_ARG, "parent misaligned");
  if (v.z) {
    GDN_CHECK_PTR(v.norm_w, "norm_w");
    if (!std::isfinite(v.norm_eps) || v.norm_eps < 0.f)
      return fail(GDN_ERR_INVALID_ARG, "norm_eps must be finite, >= 0");
  }

  const size_t C = 2ull * d.Hk * d.dk + size_t(d.Hv) * d.dv;
  const size_t B = size_t(d.B), K = size_t(d.K);
  const size_t S = size_t(d.Hv) * d.dv * d.dk;  // state floats per sequence
  const bool k1 = d.K == 1;
  const Buf bufs[] = {
      {"x", range_of(v.x, B * K * C * 2), false},
      {"a", range_of(v.a, B * K * d.Hv * 2), false},
      {"b", range_of(v.b, B * K * d.Hv * 2), false},
      {"A_log", range_of(v.A_log, size_t(d.Hv) * 4), false},
      {"dt_bias", range_of(v.dt_bias, size_t(d.Hv) * 4), false},
      {"conv_w", range_of(v.conv_w, C * 4 * 4), false},
      {"conv_state_in", range_of(v.conv_state_in, B * 3 * C * 4), false},
      {"conv_inter_prev", range_of(k1 ? nullptr : v.conv_inter_prev, B * K * 3 * C * 4), false},
      {"conv_state_snapshot_prev", range_of(v.conv_snap_prev, B * 3 * C * 4), false},
      {"state_in", range_of(v.state_in, B * S * 4), false},
      {"state_inter_prev", range_of(k1 ? nullptr : v.state_inter_prev, B * (K - 1) * S * 4), false},
      {"state_snapshot_prev", range_of(v.state_snap_prev, B * S * 4), false},
      {"accept_len_prev", range_of(v.accept_prev, B * 4), false},
      {"parent", range_of(v.parent, B * K * 4), false},
      {"z", range_of(v.z, B * K * d.Hv * d.dv * 2), false},
      {"norm_w", range_of(v.z ? v.norm_w : nullptr, size_t(d.dv) * 4), false},
      {"conv_state_out", range_of(v.conv_state_out, B * 3 * C * 4), true},
      {"conv_inter", range_of(v.conv_inter, B * K * 3 * C * 4), true},
      {"state_out", range_of(v.state_out, B * S * 4), true},
      {"state_inter", range_of(k1 ? nullptr : v.state_inter, B * (K - 1) * S * 4), true},
      {"out", range_of(v.out, B * K * d.Hv * d.dv * (d.out_f32 ? 4 : 2)), true},
  };
  // (output, input) pairs that may be the very same buffer: every state tile and every history
  // channel is read, then rewritten, by one owner, so working in place is race-free
  const char* in_place[][2] = {{"conv_state_out", "conv_state_in"},       {"state_out", "state_in"},
                               {"conv_inter", "conv_inter_prev"},         {"state_inter", "state_inter_prev"},
                               {"conv_state_out", "conv_state_snapshot_prev"}, {"state_out", "state_snapshot_prev"}};
  const int n = int(sizeof(bufs) / sizeof(bufs[0]));
  for (int i = 0; i < n; ++i) {
    if (!bufs[i].output) continue;
    for (int j = 0; j < n; ++j) {
      if (i == j || (bufs[j].output && j < i) || !overlap(bufs[i].r, bufs[j].r)) continue;
      bool allowed = false;
      if (!bufs[j].output && bufs[i].r.lo == bufs[j].r.lo && bufs[i].r.hi == bufs[j].r.hi)
        for (const auto& pr : in_place)
          if (!strcmp(pr[0], bufs[i].name) && !strcmp(pr[1], bufs[j].name)) allowed = true;
      if (!allowed) return fail(GDN_ERR_ALIAS, "%s overlaps %s", bufs[i].name, bufs[j].name);
    }
  }

  uint32_t* err = nullptr;
  s = status_word(&err);
  if (s != GDN_OK) return s;
  gdn::VerifyParams p{};
  p.x = v.x;
  p.a = v.a;
  p.b = v.b;
  p.A_log = v.A_log;
  p.dt_bias = v.dt_bias;
  p.conv_w = v.conv_w;
  p.conv_state_in = v.conv_state_in;
  p.conv_state_out = v.conv_state_out;
  p.conv_inter = v.conv_inter;
  p.state_in = v.state_in;
  p.state_out = v.state_out;
  p.state_inter = k1 ? nullptr : v.state_inter;
  p.out = v.out;
  p.parent = v.parent;
  p.z = v.z;
  p.norm_w = v.z ? v.norm_w : nullptr;
  p.norm_eps = v.norm_eps;
  if (v.resume) {
    p.accept_prev = v.accept_prev;
    p.state_inter_prev = k1 ? nullptr : v.state_inter_prev;
    p.conv_inter_prev = k1 ? nullptr : v.conv_inter_prev;
    p.state_snap_prev = v.state_snap_prev;
    p.conv_snap_prev = v.conv_snap_prev;
  }
  p.err = err;
  p.B = d.B;
  p.K = d.K;
  p.Hk = d.Hk;
  p.Hv = d.Hv;
  p.dk = d.dk;
  p.dv = d.dv;
  p.C = int(C);
  p.q_scale = d.q_scale;
  p.l2_eps = d.l2_eps;
  p.out_f32 = d.out_f32;
  cudaError_t e = gdn::launch_verify(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "verify launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // namespace

namespace gdn {
gdn_status report_error(gdn_status s, const char* msg) { return fail(s, "%s", msg); }
}  // namespace gdn

extern "C" {

const char* gdn_last_error(void) { return g_last_error.c_str(); }

gdn_status gdn_device_status(uint32_t* flags, int32_t clear, gdn_stream_t stream) {
  if (!flags) return fail(GDN_ERR_INVALID_ARG, "flags is NULL");
  uint32_t* word = nullptr;
  gdn_status s = status_word(&word);
  if (s != GDN_OK) return s;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = cudaMemcpyAsync(flags, word, sizeof(uint32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess && clear) e = cudaMemsetAsync(word, 0, sizeof(uint32_t), st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "device status: %s", cudaGetErrorString(e));
  return ok();
}

gdn_status gdn_conv_step(const gdn_dims* dims, const uint16_t* x, const float* conv_w, float* conv_state,
                         float* conv_inter, void* y, gdn_stream_t stream) {
  gdn_status s = check_dims(dims, false);
  if (s != GDN_OK) return s;
  const gdn_dims& d = *dims;
  if (d.B == 0) return ok();
  GDN_CHECK_PTR(x, "x");
  GDN_CHECK_PTR(conv_w, "conv_w");
  GDN_CHECK_PTR(conv_state, "conv_state");
  GDN_CHECK_OPT_PTR(conv_inter, "conv_inter");
  GDN_CHECK_PTR(y, "y");
  const size_t C = 2ull * d.Hk * d.dk + size_t(d.Hv) * d.dv;
  const size_t BKC = size_t(d.B) * d.K * C;
  const Range rx = range_of(x, BKC * 2), rw = range_of(conv_w, C * 4 * 4),
              rh = range_of(conv_state, size_t(d.B) * 3 * C * 4),
              ri = range_of(conv_inter, BKC * 3 * 4), ry = range_of(y, BKC * (d.out_f32 ? 4 : 2));
  const Range outs[3] = {rh, ri, ry};
  const Range ins[2] = {rx, rw};
  for (int i = 0; i < 3; ++i) {
    for (int j = 0; j < 2; ++j)
      if (overlap(outs[i], ins[j])) return fail(GDN_ERR_ALIAS, "conv_step: an output overlaps an input");
    for (int j = i + 1; j < 3; ++j)
      if (overlap(outs[i], outs[j])) return fail(GDN_ERR_ALIAS, "conv_step: outputs overlap");
  }
  gdn::ConvParams p{x, conv_w, conv_state, conv_inter, y, d.B, d.K, int(C), d.out_f32};
  cudaError_t e = gdn::launch_conv(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "conv_step launch: %s", cudaGetErrorString(e));
  return ok();
}

gdn_status gdn_verify_workspace_size(const gdn_dims* dims, uint64_t* bytes) {
  gdn_status s = check_dims(dims, true);
  if (s != GDN_OK) return s;
  if (!bytes) return fail(GDN_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = 0;  // the verify kernels keep everything they share in shared memory
  return ok();
}

gdn_status gdn_verify_step(const gdn_dims* dims, const uint16_t* x, const uint16_t* a, const uint16_t* b,
                           const float* A_log, const float* dt_bias, const float* conv_w,
                           const float* conv_state_in, float* conv_state_out, float* conv_inter,
                           const float* state_in, float* state_out, float* state_inter, void* out,
                           void* workspace, uint64_t workspace_bytes, gdn_stream_t stream) {
  VerifyArgs v{};
  v.x = x;
  v.a = a;
  v.b = b;
  v.A_log = A_log;
  v.dt_bias = dt_bias;
  v.conv_w = conv_w;
  v.conv_state_in = conv_state_in;
  v.conv_state_out = conv_state_out;
  v.conv_inter = conv_inter;
  v.state_in = state_in;
  v.state_out = state_out;
  v.state_inter = state_inter;
  v.out = out;
  (void)workspace;  // (needs 0 bytes: see gdn_verify_workspace_size)
  (void)workspace_bytes;
  return verify_impl(dims, v, stream);
}

gdn_status gdn_verify_tree(const gdn_dims* dims, const int32_t* parent_dev, const uint16_t* x, const uint16_t* a,
                           const uint16_t* b, const float* A_log, const float* dt_bias, const float* conv_w,
                           const float* conv_state_in, float* conv_state_out, float* conv_inter,
                           const float* state_in, float* state_out, float* state_inter, void* out,
                           void* workspace, uint64_t workspace_bytes, gdn_stream_t stream) {
  if (dims && dims->B > 0 && !parent_dev) return fail(GDN_ERR_INVALID_ARG, "parent is NULL");
  VerifyArgs v{};
  v.parent = parent_dev;
  v.x = x;
  v.a = a;
  v.b = b;
  v.A_log = A_log;
  v.dt_bias = dt_bias;
  v.conv_w = conv_w;
  v.conv_state_in = conv_state_in;
  v.conv_state_out = conv_state_out;
  v.conv_inter = conv_inter;
  v.state_in = state_in;
  v.state_out = state_out;
  v.state_inter = state_inter;
  v.out = out;
  (void)workspace;  // (needs 0 bytes: see gdn_verify_workspace_size)
  (void)workspace_bytes;
  return verify_impl(dims, v, stream);
}

gdn_status gdn_verify_gated(const gdn_dims* dims, const uint16_t* x, const uint16_t* a, const uint16_t* b,
                            const float* A_log, const float* dt_bias, const float* conv_w,
                            const float* conv_state_in, float* conv_state_out, float* conv_inter,
                            const float* state_in, float* state_out, float* state_inter, const uint16_t* z,
                            const float* norm_w, float norm_eps, void* out, void* workspace,
                            uint64_t workspace_bytes, gdn_stream_t stream) {
  if (dims && dims->B > 0) GDN_CHECK_PTR(z, "z");
  VerifyArgs v{};
  v.z = z;
  v.norm_w = norm_w;
  v.norm_eps = norm_eps;
  v.x = x;
  v.a = a;
  v.b = b;
  v.A_log = A_log;
  v.dt_bias = dt_bias;
  v.conv_w = conv_w;
  v.conv_state_in = conv_state_in;
  v.conv_state_out = conv_state_out;
  v.conv_inter = conv_inter;
  v.state_in = state_in;
  v.state_out = state_out;
  v.state_inter = state_inter;
  v.out = out;
  (void)workspace;  // (needs 0 bytes: see gdn_verify_workspace_size)
  (void)workspace_bytes;
  return verify_impl(dims, v, stream);
}

gdn_status gdn_verify_resume(const gdn_dims* dims, const int32_t* accept_len_prev, const uint16_t* x,
                             const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias,
                             const float* conv_w, const float* conv_state_in, const float* conv_inter_prev,
                             const float* conv_state_snapshot_prev, float* conv_state_out, float* conv_inter,
                             const float* state_in, const float* state_inter_prev, const float* state_snapshot_prev,
                             float* state_out, float* state_inter, void* out, void* workspace,
                             uint64_t workspace_bytes, gdn_stream_t stream) {
  VerifyArgs v{};
  v.resume = true;
  v.accept_prev = accept_len_prev;
  v.x = x;
  v.a = a;
  v.b = b;
  v.A_log = A_log;
  v.dt_bias = dt_bias;
  v.conv_w = conv_w;
  v.conv_state_in = conv_state_in;
  v.conv_inter_prev = conv_inter_prev;
  v.conv_snap_prev = conv_state_snapshot_prev;
  v.conv_state_out = conv_state_out;
  v.conv_inter = conv_inter;
  v.state_in = state_in;
  v.state_inter_prev = state_inter_prev;
  v.state_snap_prev = state_snapshot_prev;
  v.state_out = state_out;
  v.state_inter = state_inter;
  v.out = out;
  (void)workspace;  // (needs 0 bytes: see gdn_verify_workspace_size)
  (void)workspace_bytes;
  return verify_impl(dims, v, stream);
}

gdn_status gdn_prefill_workspace_size(const gdn_dims* dims, int64_t n_tokens, uint64_t* bytes) {
  gdn_status s = check_dims(dims, true, false);
  if (s != GDN_OK) return s;
  if (n_tokens < 0 || n_tokens > INT32_MAX) return fail(GDN_ERR_INVALID_ARG, "n_tokens=%lld outside 0..2^31-1", (long long)n_tokens);
  if (!bytes) return fail(GDN_ERR_INVALID_ARG, "bytes is NULL");
  *bytes = gdn::prefill_workspace_bytes(dims->B, n_tokens, dims->Hk, dims->Hv, dims->dk);
  return ok();
}

gdn_status gdn_prefill(const gdn_dims* dims, int64_t n_tokens, const int32_t* cu_seqlens_dev, const uint16_t* x,
                       const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias,
                       const float* conv_w, const float* conv_state_in, float* conv_state_out,
                       const float* state_in, float* state_out, void* out, void* workspace,
                       uint64_t workspace_bytes, gdn_stream_t stream) {
  gdn_status s = check_dims(dims, true, false);
  if (s != GDN_OK) return s;
  const gdn_dims& d = *dims;
  if (n_tokens < 0 || n_tokens > INT32_MAX) return fail(GDN_ERR_INVALID_ARG, "n_tokens=%lld outside 0..2^31-1", (long long)n_tokens);
  if (d.B == 0) {
    if (n_tokens != 0) return fail(GDN_ERR_INVALID_ARG, "n_tokens=%lld with no prompts", (long long)n_tokens);
    return ok();
  }
  if (!cu_seqlens_dev) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens is NULL");
  if (reinterpret_cast<uintptr_t>(cu_seqlens_dev) & 3u) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens misaligned");
  if (n_tokens > 0) {
    GDN_CHECK_PTR(x, "x");
    GDN_CHECK_PTR(a, "a");
    GDN_CHECK_PTR(b, "b");
    GDN_CHECK_PTR(out, "out");
  } else {
    GDN_CHECK_OPT_PTR(x, "x");
    GDN_CHECK_OPT_PTR(a, "a");
    GDN_CHECK_OPT_PTR(b, "b");
    GDN_CHECK_OPT_PTR(out, "out");
  }
  GDN_CHECK_PTR(A_log, "A_log");
  GDN_CHECK_PTR(dt_bias, "dt_bias");
  GDN_CHECK_PTR(conv_w, "conv_w");
  GDN_CHECK_PTR(conv_state_in, "conv_state_in");
  GDN_CHECK_PTR(conv_state_out, "conv_state_out");
  GDN_CHECK_PTR(state_in, "state_in");
  GDN_CHECK_PTR(state_out, "state_out");
  GDN_CHECK_PTR(workspace, "workspace");
  const size_t ws_need = gdn::prefill_workspace_bytes(d.B, n_tokens, d.Hk, d.Hv, d.dk);
  if (workspace_bytes < ws_need)
    return fail(GDN_ERR_INVALID_ARG, "workspace has %llu bytes, needs %zu", (unsigned long long)workspace_bytes, ws_need);

  const size_t C = 2ull * d.Hk * d.dk + size_t(d.Hv) * d.dv;
  const size_t B = size_t(d.B), N = size_t(n_tokens);
  const size_t S = size_t(d.Hv) * d.dv * d.dk;
  const Buf bufs[] = {
      {"cu_seqlens", range_of(cu_seqlens_dev, (B + 1) * 4), false},
      {"x", range_of(x, N * C * 2), false},
      {"a", range_of(a, N * d.Hv * 2), false},
      {"b", range_of(b, N * d.Hv * 2), false},
      {"A_log", range_of(A_log, size_t(d.Hv) * 4), false},
      {"dt_bias", range_of(dt_bias, size_t(d.Hv) * 4), false},
      {"conv_w", range_of(conv_w, C * 4 * 4), false},
      {"conv_state_in", range_of(conv_state_in, B * 3 * C * 4), false},
      {"state_in", range_of(state_in, B * S * 4), false},
      {"conv_state_out", range_of(conv_state_out, B * 3 * C * 4), true},
      {"state_out", range_of(state_out, B * S * 4), true},
      {"out", range_of(out, N * d.Hv * d.dv * (d.out_f32 ? 4 : 2)), true},
      {"workspace", range_of(workspace, ws_need), true},
  };
  const char* in_place[][2] = {{"conv_state_out", "conv_state_in"}, {"state_out", "state_in"}};
  const int n = int(sizeof(bufs) / sizeof(bufs[0]));
  for (int i = 0; i < n; ++i) {
    if (!bufs[i].output) continue;
    for (int j = 0; j < n; ++j) {
      if (i == j || (bufs[j].output && j < i) || !overlap(bufs[i].r, bufs[j].r)) continue;
      bool allowed = false;
      if (!bufs[j].output && bufs[i].r.lo == bufs[j].r.lo && bufs[i].r.hi == bufs[j].r.hi)
        for (const auto& pr : in_place)
          if (!strcmp(pr[0], bufs[i].name) && !strcmp(pr[1], bufs[j].name)) allowed = true;
      if (!allowed) return fail(GDN_ERR_ALIAS, "%s overlaps %s", bufs[i].name, bufs[j].name);
    }
  }

  uint32_t* err = nullptr;
  s = status_word(&err);
  if (s != GDN_OK) return s;
  gdn::PrefillParams p{};
  p.cu = cu_seqlens_dev;
  p.x = x;
  p.a = a;
  p.b = b;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.conv_w = conv_w;
  p.conv_state_in = conv_state_in;
  p.conv_state_out = conv_state_out;
  p.state_in = state_in;
  p.state_out = state_out;
  p.out = out;
  p.ws = gdn::prefill_workspace_carve(workspace, d.B, n_tokens, d.Hk, d.Hv, d.dk);
  p.err = err;
  p.B = d.B;
  p.Hk = d.Hk;
  p.Hv = d.Hv;
  p.dk = d.dk;
  p.dv = d.dv;
  p.C = int(C);
  p.N = n_tokens;
  p.q_scale = d.q_scale;
  p.l2_eps = d.l2_eps;
  p.out_f32 = d.out_f32;
  cudaError_t e = gdn::launch_prefill(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "prefill launch: %s", cudaGetErrorString(e));
  return ok();
}

gdn_status gdn_rollback(const gdn_dims* dims, const int32_t* accept_len_dev, const float* state_in_snapshot,
                        float* state, const float* state_inter, const float* conv_state_in_snapshot,
                        float* conv_state, const float* conv_inter, gdn_stream_t stream) {
  gdn_status s = check_dims(dims, false);
  if (s != GDN_OK) return s;
  const gdn_dims& d = *dims;
  if (d.B == 0) return ok();
  if (!accept_len_dev) return fail(GDN_ERR_INVALID_ARG, "accept_len is NULL");
  if (reinterpret_cast<uintptr_t>(accept_len_dev) & 3u) return fail(GDN_ERR_INVALID_ARG, "accept_len misaligned");
  GDN_CHECK_OPT_PTR(state_in_snapshot, "state_in_snapshot");
  GDN_CHECK_PTR(state, "state");
  GDN_CHECK_OPT_PTR(state_inter, "state_inter");
  GDN_CHECK_OPT_PTR(conv_state_in_snapshot, "conv_state_in_snapshot");
  GDN_CHECK_PTR(conv_state, "conv_state");
  GDN_CHECK_OPT_PTR(conv_inter, "conv_inter");
  if (d.K > 1 && (!state_inter || !conv_inter))
    return fail(GDN_ERR_INVALID_ARG, "state_inter and conv_inter are required when K=%d > 1", d.K);
  if ((state_in_snapshot == nullptr) != (conv_state_in_snapshot == nullptr))
    return fail(GDN_ERR_NO_SNAPSHOT, "pass both snapshots or neither");

  const size_t C = 2ull * d.Hk * d.dk + size_t(d.Hv) * d.dv;
  const size_t B = size_t(d.B), K = size_t(d.K);
  const size_t S = size_t(d.Hv) * d.dv * d.dk;
  const Range r_len = range_of(accept_len_dev, B * 4), r_snap = range_of(state_in_snapshot, B * S * 4),
              r_st = range_of(state, B * S * 4), r_sx = range_of(d.K > 1 ? state_inter : nullptr, B * (K - 1) * S * 4),
              r_csnap = range_of(conv_state_in_snapshot, B * 3 * C * 4), r_cs = range_of(conv_state, B * 3 * C * 4),
              r_ci = range_of(d.K > 1 ? conv_inter : nullptr, B * K * 3 * C * 4);
  const Range srcs[5] = {r_len, r_snap, r_sx, r_csnap, r_ci};
  for (int j = 0; j < 5; ++j) {
    if (overlap(r_st, srcs[j])) return fail(GDN_ERR_ALIAS, "state overlaps a rollback source");
    if (overlap(r_cs, srcs[j])) return fail(GDN_ERR_ALIAS, "conv_state overlaps a rollback source");
  }
  if (overlap(r_st, r_cs)) return fail(GDN_ERR_ALIAS, "state overlaps conv_state");

  uint32_t* err = nullptr;
  s = status_word(&err);
  if (s != GDN_OK) return s;
  gdn::RollbackParams p{};
  p.accept_len = accept_len_dev;
  p.state_snap = state_in_snapshot;
  p.state = state;
  p.state_inter = state_inter;
  p.conv_snap = conv_state_in_snapshot;
  p.conv_state = conv_state;
  p.conv_inter = conv_inter;
  p.err = err;
  p.B = d.B;
  p.K = d.K;
  p.state_elems = (long long)S;
  p.conv_elems = 3LL * (long long)C;
  cudaError_t e = gdn::launch_rollback(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "rollback launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"
