// C ABI of the GDN verify library: host-side validation, launches, error reporting.
//
// Every entry point checks its arguments completely before it enqueues anything, so a
// non-OK status always means that nothing ran.  Checks: shapes inside the supported set,
// 16-byte alignment of every buffer (bulk async copies and float4 accesses need it), the
// aliasing rules of each call, finite scalars.  See include/gdn.h for the contract.
#include <cmath>
#include <cstdarg>
#include <cstdio>
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

gdn_status check_dims(const gdn_dims* d, bool need_gates) {
  if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
  if (d->B < 0 || d->B > 65535) return fail(GDN_ERR_INVALID_ARG, "B=%d outside 0..65535", d->B);
  if (d->K < 1 || d->K > gdn::kKMax) return fail(GDN_ERR_UNSUPPORTED, "K=%d outside 1..%d", d->K, gdn::kKMax);
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
  *bytes = gdn::workspace_bytes(dims->B, dims->Hk, dims->Hv, dims->dk);
  return ok();
}

gdn_status gdn_verify_step(const gdn_dims* dims, const uint16_t* x, const uint16_t* a, const uint16_t* b,
                           const float* A_log, const float* dt_bias, const float* conv_w,
                           const float* conv_state_in, float* conv_state_out, float* conv_inter,
                           const float* state_in, float* state_out, float* state_inter, void* out,
                           void* workspace, uint64_t workspace_bytes, gdn_stream_t stream) {
  gdn_status s = check_dims(dims, true);
  if (s != GDN_OK) return s;
  const gdn_dims& d = *dims;
  if (d.B == 0) return ok();
  GDN_CHECK_PTR(x, "x");
  GDN_CHECK_PTR(a, "a");
  GDN_CHECK_PTR(b, "b");
  GDN_CHECK_PTR(A_log, "A_log");
  GDN_CHECK_PTR(dt_bias, "dt_bias");
  GDN_CHECK_PTR(conv_w, "conv_w");
  GDN_CHECK_PTR(conv_state_in, "conv_state_in");
  GDN_CHECK_PTR(conv_state_out, "conv_state_out");
  GDN_CHECK_OPT_PTR(conv_inter, "conv_inter");
  GDN_CHECK_PTR(state_in, "state_in");
  GDN_CHECK_PTR(state_out, "state_out");
  GDN_CHECK_OPT_PTR(state_inter, "state_inter");
  GDN_CHECK_PTR(out, "out");
  GDN_CHECK_PTR(workspace, "workspace");
  if (d.K > 1 && !state_inter) return fail(GDN_ERR_INVALID_ARG, "state_inter is NULL with K=%d > 1", d.K);
  const size_t ws_need = gdn::workspace_bytes(d.B, d.Hk, d.Hv, d.dk);
  if (workspace_bytes < ws_need)
    return fail(GDN_ERR_INVALID_ARG, "workspace has %llu bytes, needs %zu", (unsigned long long)workspace_bytes, ws_need);

  const size_t C = 2ull * d.Hk * d.dk + size_t(d.Hv) * d.dv;
  const size_t B = size_t(d.B), K = size_t(d.K);
  const size_t S = size_t(d.Hv) * d.dv * d.dk;  // state floats per sequence
  const Range r_x = range_of(x, B * K * C * 2), r_a = range_of(a, B * K * d.Hv * 2),
              r_b = range_of(b, B * K * d.Hv * 2), r_alog = range_of(A_log, size_t(d.Hv) * 4),
              r_dt = range_of(dt_bias, size_t(d.Hv) * 4), r_w = range_of(conv_w, C * 4 * 4),
              r_csi = range_of(conv_state_in, B * 3 * C * 4), r_cso = range_of(conv_state_out, B * 3 * C * 4),
              r_ci = range_of(conv_inter, B * K * 3 * C * 4), r_si = range_of(state_in, B * S * 4),
              r_so = range_of(state_out, B * S * 4),
              r_sx = range_of(d.K > 1 ? state_inter : nullptr, B * (K - 1) * S * 4),
              r_o = range_of(out, B * K * d.Hv * d.dv * (d.out_f32 ? 4 : 2)), r_ws = range_of(workspace, ws_need);
  // in-place pairs: identical start or disjoint
  if (conv_state_out != conv_state_in && overlap(r_cso, r_csi))
    return fail(GDN_ERR_ALIAS, "conv_state_out partially overlaps conv_state_in");
  if (state_out != state_in && overlap(r_so, r_si))
    return fail(GDN_ERR_ALIAS, "state_out partially overlaps state_in");
  const Range ins[7] = {r_x, r_a, r_b, r_alog, r_dt, r_w, r_csi};
  const Range writes[6] = {r_cso, r_ci, r_so, r_sx, r_o, r_ws};
  const char* wname[6] = {"conv_state_out", "conv_inter", "state_out", "state_inter", "out", "workspace"};
  for (int i = 0; i < 6; ++i) {
    for (int j = 0; j < 7; ++j) {
      if (i == 0 && j == 6) continue;  // conv_state_out vs conv_state_in handled above
      if (overlap(writes[i], ins[j])) return fail(GDN_ERR_ALIAS, "%s overlaps an input", wname[i]);
    }
    if (i != 2 && overlap(writes[i], r_si)) return fail(GDN_ERR_ALIAS, "%s overlaps state_in", wname[i]);
    for (int j = i + 1; j < 6; ++j)
      if (overlap(writes[i], writes[j])) return fail(GDN_ERR_ALIAS, "%s overlaps %s", wname[i], wname[j]);
  }

  uint32_t* err = nullptr;
  s = status_word(&err);
  if (s != GDN_OK) return s;
  gdn::VerifyParams p{};
  p.x = x;
  p.a = a;
  p.b = b;
  p.A_log = A_log;
  p.dt_bias = dt_bias;
  p.conv_w = conv_w;
  p.conv_state_in = conv_state_in;
  p.conv_state_out = conv_state_out;
  p.conv_inter = conv_inter;
  p.state_in = state_in;
  p.state_out = state_out;
  p.state_inter = d.K > 1 ? state_inter : nullptr;
  p.out = out;
  p.ws = gdn::workspace_carve(workspace, d.B, d.Hk, d.Hv, d.dk);
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
  if (e != cudaSuccess) return fail(GDN_ERR_CUDA, "verify_step launch: %s", cudaGetErrorString(e));
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
