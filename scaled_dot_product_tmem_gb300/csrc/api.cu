// api.cu -- the C ABI declared in include/sdpa_tmem.h: argument validation,
// TMA tensor-map creation, workspace carving and kernel dispatch.  No compute.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "../../include/sdpa_tmem.h"
#include "attn_kernels.h"
#include "tmap.h"

namespace {

// Text of the last failure seen by this thread (which call, and CUDA's message).
thread_local char g_last_error[256] = "";

void set_error(const char* what, cudaError_t e) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what, cudaGetErrorString(e), (int)e);
}
void set_error(const char* what) { snprintf(g_last_error, sizeof(g_last_error), "%s", what); }

__device__ int g_device_error;  // one word per GPU: 0 or kErrTimeoutBase + site

constexpr int kMaxDevices = 64;

int* device_error_ptr() {
  static int* ptrs[kMaxDevices] = {nullptr};
  static std::mutex mu;  // first calls on one device from several threads fill its entry once
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    set_error("cudaGetDevice", e);
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("device index out of the library's range (64 devices)");
    return nullptr;
  }
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) {
      set_error("cudaGetSymbolAddress(device error word)", e);
      return nullptr;
    }
    ptrs[dev] = static_cast<int*>(p);
  }
  return ptrs[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct WsLayout {
  size_t nlse2, dsum, dq_acc, dk_part, dv_part, counter, total;
  int ns;  // query-head splits of the kv kernel
};

WsLayout ws_layout(int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, bool need_dq_acc) {
  const size_t s_pad = (static_cast<size_t>(S_q) + 127) / 128 * 128;
  const size_t rows = static_cast<size_t>(B) * H_q * s_pad;
  WsLayout w;
  w.nlse2 = 0;
  w.dsum = round256(rows * sizeof(float));
  w.dq_acc = w.dsum + round256(rows * sizeof(float));
  w.dk_part = w.dq_acc + (need_dq_acc ? round256(static_cast<size_t>(B) * S_q * H_q * d_qk * sizeof(float)) : 0);
  w.ns = S_q > 0 && S_kv > 0 ? sdpa::bwd_kv_head_splits(B, S_kv, H_kv, H_q / H_kv) : 1;
  const size_t kv_rows = static_cast<size_t>(w.ns > 1 ? w.ns : 0) * B * S_kv * H_kv;
  w.dv_part = w.dk_part + round256(kv_rows * d_qk * sizeof(float));
  // tile counters of the persistent kv and dQ kernels
  w.counter = w.dv_part + round256(kv_rows * d_v * sizeof(float));
  w.total = w.counter + 256;
  return w;
}

bool use_fused_dq(int d_qk, int d_v, int deterministic) {
  return !deterministic && sdpa::bwd_kv_supports_fused_dq(d_qk, d_v);
}

// ---------------------------------------------------------------------------
// Optional timing of every kernel launch (CUDA events on the launch stream).
// Events come from a pool that attn_timing_read refills, so after the first
// timed steps a launch costs two event records and no event creation.
// ---------------------------------------------------------------------------
struct TimingRec {
  cudaEvent_t a, b;
  int kind, launches;
};
std::mutex g_timing_mu;
bool g_timing_on = false;
std::vector<TimingRec> g_timing;
std::vector<cudaEvent_t> g_event_pool;

// An event from the pool, or a new one (null if CUDA cannot make one).  Caller holds g_timing_mu.
cudaEvent_t pooled_event() {
  if (!g_event_pool.empty()) {
    cudaEvent_t e = g_event_pool.back();
    g_event_pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  return cudaEventCreate(&e) == cudaSuccess ? e : nullptr;
}

// Runs `launch` (which enqueues `nlaunch` kernels of class `kind` on stream s);
// brackets it with events when timing is on.
template <class F>
int timed(int kind, int nlaunch, cudaStream_t s, F&& launch) {
  cudaEvent_t a = nullptr, b = nullptr;
  {
    std::lock_guard<std::mutex> g(g_timing_mu);
    if (!g_timing_on) return launch();
    a = pooled_event();
    b = pooled_event();
    if (!a || !b) {
      if (a) g_event_pool.push_back(a);
      if (b) g_event_pool.push_back(b);
      return -1;
    }
  }
  cudaEventRecord(a, s);
  const int rc = launch();
  cudaEventRecord(b, s);
  std::lock_guard<std::mutex> g(g_timing_mu);
  g_timing.push_back({a, b, kind, nlaunch});
  return rc;
}

}  // namespace

namespace sdpa {
// The device error word of the current device, for the other host files of the library.
int* device_error_word() { return device_error_ptr(); }

bool dims_supported(int d_qk, int d_v) {
  return (d_qk == 64 || d_qk == 128 || d_qk == 192) && (d_v == 64 || d_v == 128);
}

// Shared validation of sizes and flags.  Returns ATTN_OK or an error status.
int check_common(int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, int causal, int window,
                 int softmax_type, const float* softmax_offset) {
  if (B < 0 || S_q < 0 || S_kv < 0 || H_q <= 0 || H_kv <= 0) return ATTN_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (softmax_type < ATTN_SOFTMAX_VANILLA || softmax_type > ATTN_SOFTMAX_LEARNABLE) return ATTN_ERR_INVALID_ARG;
  if (softmax_type == ATTN_SOFTMAX_LEARNABLE && softmax_offset == nullptr) return ATTN_ERR_INVALID_ARG;
  if (!dims_supported(d_qk, d_v)) return ATTN_ERR_UNSUPPORTED;
  if (window >= 0 && !causal) return ATTN_ERR_UNSUPPORTED;
  if (B > 65535 || H_q > 65535) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

float resolve_scale(float scale, int d_qk) {
  if (!(scale > 0.f) || std::isinf(scale)) return 1.0f / std::sqrt(static_cast<float>(d_qk));
  return scale;
}
}  // namespace sdpa

using sdpa::check_common;
using sdpa::resolve_scale;

// The drop threshold t of dropout probability p: 16-bit uniforms below t are dropped,
// so p is realised as t / 65536 with t = floor(p * 65536 + 1/2).  -1 when p is not in
// [0, 1) or rounds to 1.
static int drop_threshold(float p) {
  if (!(p >= 0.f) || !(p < 1.f)) return -1;
  const double t = std::floor(static_cast<double>(p) * 65536.0 + 0.5);
  return t > 65535.0 ? -1 : static_cast<int>(t);
}

// Dropout arguments into the kernel parameters: ATTN_OK, or an error status.
template <class P>
static int set_dropout(P& prm, float dropout_p, const unsigned long long* rng_state) {
  const int t = drop_threshold(dropout_p);
  if (t < 0) return ATTN_ERR_INVALID_ARG;
  prm.drop_t = static_cast<unsigned>(t);
  prm.drop_scale = t > 0 ? static_cast<float>(65536.0 / (65536.0 - t)) : 1.f;
  prm.rng = t > 0 ? rng_state : nullptr;
  if (t > 0 && !rng_state) return ATTN_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(rng_state) & 7u) return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

extern "C" {

const char* attn_last_error_message(void) { return g_last_error; }

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer (16-byte alignment required)";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_DEVICE_TIMEOUT: return "device pipeline wait timed out";
    case ATTN_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
    default: return "unknown status";
  }
}

int attn_last_device_error(void* stream, int* site) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_CUDA;
  int* p = device_error_ptr();
  if (!p) return ATTN_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (site) *site = v;
  if (v == 0) return ATTN_OK;
  const int zero = 0;
  if (cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return ATTN_ERR_CUDA;
  return ATTN_ERR_DEVICE_TIMEOUT;
}

// Checks of an additive bias [bias_B, bias_H, S_q, S_kv] (bf16, 16-byte aligned) and
// its element strides (0 along a broadcast dim).
static int check_bias(const void* bias, int bias_B, int bias_H, int B, int H_q, int d_qk, int d_v, long long* sb,
                      long long* sh, int S_q, int S_kv) {
  if (!bias || (bias_B != 1 && bias_B != B) || (bias_H != 1 && bias_H != H_q)) return ATTN_ERR_INVALID_ARG;
  if (!((d_qk == d_v && (d_qk == 64 || d_qk == 128)) || (d_qk == 192 && d_v == 128))) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(bias)) return ATTN_ERR_MISALIGNED;
  *sh = bias_H == 1 ? 0 : (long long)S_q * S_kv;
  *sb = bias_B == 1 ? 0 : (long long)bias_H * S_q * S_kv;
  return ATTN_OK;
}

static int fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q, int S_kv,
                    int H_q, int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                    const float* softmax_offset, const int* seq_lens_q, const int* seq_lens_kv, const void* bias,
                    int bias_B, int bias_H, void* stream, float dropout_p = 0.f,
                    const unsigned long long* rng_state = nullptr) {
  int st = check_common(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, causal, window, softmax_type, softmax_offset);
  if (st != ATTN_OK) return st;
  sdpa::FwdParams p;
  st = set_dropout(p, dropout_p, rng_state);
  if (st != ATTN_OK) return st;
  long long bsb = 0, bsh = 0;
  if (bias) {
    st = check_bias(bias, bias_B, bias_H, B, H_q, d_qk, d_v, &bsb, &bsh, S_q, S_kv);
    if (st != ATTN_OK) return st;
  }
  if (B == 0 || S_q == 0) return ATTN_OK;
  if (!q || !o || !lse || (S_kv > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(k) || !aligned16(v) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens_q) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens_kv) & 3u))
    return ATTN_ERR_MISALIGNED;
  int* err = device_error_ptr();
  if (!err) return ATTN_ERR_CUDA;
  // TMA maps need a non-empty tensor; with S_kv == 0 no kv tile is ever loaded.
  const int skv_map = S_kv > 0 ? S_kv : 1;
  const void* kk = S_kv > 0 ? k : q;
  const void* vv = S_kv > 0 ? v : q;
  CUtensorMap tq, tk, tv;
  if (!sdpa::make_bshd_map(&tq, q, B, S_q, H_q, d_qk, 128) ||
      !sdpa::make_bshd_map(&tk, kk, B, skv_map, S_kv > 0 ? H_kv : H_q, d_qk, 128) ||
      !sdpa::make_bshd_map(&tv, vv, B, skv_map, S_kv > 0 ? H_kv : H_q, S_kv > 0 ? d_v : d_qk, 128)) {
    set_error("cuTensorMapEncodeTiled (forward operands)");
    return ATTN_ERR_CUDA;
  }
  p.B = B; p.S_q = S_q; p.S_kv = S_kv; p.H_q = H_q; p.H_kv = H_kv; p.G = H_q / H_kv;
  p.scale_log2 = resolve_scale(scale, d_qk) * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.window = window < 0 ? -1 : window;
  p.softmax_type = softmax_type;
  p.offset = softmax_offset;
  p.seq_q = seq_lens_q;
  p.seq_kv = seq_lens_kv;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.bias_sb = bsb;
  p.bias_sh = bsh;
  // head dims up to 128 stage the bias tiles by TMA when the rows are whole 16-byte units
  CUtensorMap tb;
  p.bias_tma = bias && d_qk <= 128 && S_kv > 0 && S_kv % 8 == 0 ? 1 : 0;
  if (p.bias_tma && !sdpa::make_bias_map_sw128(&tb, bias, bias_B, bias_H, S_q, S_kv)) {
    set_error("cuTensorMapEncodeTiled (bias)");
    return ATTN_ERR_CUDA;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int rc = timed(ATTN_KERNEL_FWD, 1, s, [&] {
    return p.drop_t ? sdpa::launch_attn_fwd_dropout(d_qk, d_v, tq, tk, tv, p, s)
                    : sdpa::launch_attn_fwd(d_qk, d_v, tq, tk, tv, p, s, p.bias_tma ? &tb : nullptr);
  });
  if (rc == -2) return ATTN_ERR_UNSUPPORTED;
  if (rc != 0) {
    set_error("forward kernel launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q, int S_kv,
                    int H_q, int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                    const float* softmax_offset, const int* seq_lens_q, const int* seq_lens_kv, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal, window, softmax_type,
                  softmax_offset, seq_lens_q, seq_lens_kv, nullptr, 1, 1, stream);
}

int attn_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse, const void* bias, int bias_B,
                  int bias_H, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, float scale, int causal,
                  int window, int softmax_type, const float* softmax_offset, void* stream) {
  if (!bias) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal, window, softmax_type,
                  softmax_offset, nullptr, nullptr, bias, bias_B, bias_H, stream);
}

int attn_fwd_varlen_bias(const void* q, const void* k, const void* v, void* o, float* lse, const void* bias,
                         int bias_B, int bias_H, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v,
                         float scale, int causal, int window, int softmax_type, const float* softmax_offset,
                         const int* seq_lens_q, const int* seq_lens_kv, void* stream) {
  if (!bias) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal, window, softmax_type,
                  softmax_offset, seq_lens_q, seq_lens_kv, bias, bias_B, bias_H, stream);
}

int attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q, int S_kv,
                     int H_q, int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                     const float* softmax_offset, float dropout_p, const unsigned long long* rng_state, void* stream) {
  return fwd_impl(q, k, v, o, lse, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal, window, softmax_type,
                  softmax_offset, nullptr, nullptr, nullptr, 1, 1, stream, dropout_p, rng_state);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q, int S_kv, int H_q,
             int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
             const float* softmax_offset, void* stream) {
  return attn_fwd_varlen(q, k, v, o, lse, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal, window, softmax_type,
                         softmax_offset, nullptr, nullptr, stream);
}

size_t attn_bwd_workspace_size(int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, int deterministic) {
  if (check_common(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, 1, -1, 0, nullptr) != ATTN_OK) return 0;
  return ws_layout(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, use_fused_dq(d_qk, d_v, deterministic)).total;
}

static int bwd_impl(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                    void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv,
                    int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                    const float* softmax_offset, const int* seq_lens_q, const int* seq_lens_kv, const void* bias,
                    int bias_B, int bias_H, float* dbias, int deterministic, void* workspace, size_t workspace_bytes,
                    void* stream, float dropout_p = 0.f, const unsigned long long* rng_state = nullptr) {
  if ((reinterpret_cast<uintptr_t>(seq_lens_q) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens_kv) & 3u) ||
      (reinterpret_cast<uintptr_t>(dbias) & 3u))
    return ATTN_ERR_MISALIGNED;
  int st = check_common(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, causal, window, softmax_type, softmax_offset);
  if (st != ATTN_OK) return st;
  sdpa::BwdParams p;
  st = set_dropout(p, dropout_p, rng_state);
  if (st != ATTN_OK) return st;
  long long bsb = 0, bsh = 0;
  if (bias) {
    st = check_bias(bias, bias_B, bias_H, B, H_q, d_qk, d_v, &bsb, &bsh, S_q, S_kv);
    if (st != ATTN_OK) return st;
    // a broadcast dbias sums several (b, h) with fp32 atomics: not bitwise reproducible
    if (deterministic && dbias && ((bias_B == 1 && B > 1) || (bias_H == 1 && H_q > 1))) return ATTN_ERR_UNSUPPORTED;
  }
  const size_t dbias_bytes = bias && dbias ? sizeof(float) * (size_t)bias_B * bias_H * S_q * S_kv : 0;
  if (softmax_type == ATTN_SOFTMAX_LEARNABLE && !d_offset) return ATTN_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B == 0 || (S_q == 0 && S_kv == 0)) {
    if (d_offset && cudaMemsetAsync(d_offset, 0, sizeof(float) * H_q, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  // dbias accumulates with atomics from zero (no visible pair: it stays zero)
  if (dbias_bytes && cudaMemsetAsync(dbias, 0, dbias_bytes, s) != cudaSuccess) return ATTN_ERR_CUDA;
  if ((S_q > 0 && (!q || !o || !dout || !lse || !dq)) || (S_kv > 0 && (!k || !v || !dk || !dv)))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(d_offset) & 3u))
    return ATTN_ERR_MISALIGNED;
  const bool fused = use_fused_dq(d_qk, d_v, deterministic);
  const WsLayout w = ws_layout(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, fused);
  if (!workspace || workspace_bytes < w.total || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;
  int* err = device_error_ptr();
  if (!err) return ATTN_ERR_CUDA;

  // No query rows: dK = dV = 0 (no key is seen); no key: dQ = 0.
  if (S_q == 0) {
    if (cudaMemsetAsync(dk, 0, (size_t)B * S_kv * H_kv * d_qk * 2, s) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, (size_t)B * S_kv * H_kv * d_v * 2, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (d_offset && cudaMemsetAsync(d_offset, 0, sizeof(float) * H_q, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.B = B; p.S_q = S_q; p.S_kv = S_kv; p.H_q = H_q; p.H_kv = H_kv; p.G = H_q / H_kv;
  p.scale = resolve_scale(scale, d_qk);
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.window = window < 0 ? -1 : window;
  p.softmax_type = softmax_type;
  p.S_pad = (S_q + 127) / 128 * 128;
  p.offset = softmax_offset;
  p.seq_q = seq_lens_q;
  p.seq_kv = seq_lens_kv;
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.nlse2 = reinterpret_cast<float*>(ws + w.nlse2);
  p.Dsum = reinterpret_cast<float*>(ws + w.dsum);
  p.d_offset = d_offset;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dq_acc = fused ? reinterpret_cast<float*>(ws + w.dq_acc) : nullptr;
  p.tile_counter = reinterpret_cast<int*>(ws + w.counter);
  p.tile_counter_q = reinterpret_cast<int*>(ws + w.counter) + 1;
  p.bias = static_cast<const __nv_bfloat16*>(bias);
  p.bias_sb = bsb;
  p.bias_sh = bsh;
  p.dbias = bias ? dbias : nullptr;
  p.ns = w.ns;
  p.dk_part = w.ns > 1 ? reinterpret_cast<float*>(ws + w.dk_part) : nullptr;
  p.dv_part = w.ns > 1 ? reinterpret_cast<float*>(ws + w.dv_part) : nullptr;
  p.err = err;

  const int n_pre = 1 + (softmax_type == ATTN_SOFTMAX_LEARNABLE ? 1 : 0);
  if (timed(ATTN_KERNEL_BWD_PREPROCESS, n_pre, s, [&] { return sdpa::launch_bwd_preprocess(d_v, p, s); }) != 0) {
    set_error("backward preprocess launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  if (fused && cudaMemsetAsync(p.dq_acc, 0, sizeof(float) * (size_t)B * S_q * H_q * d_qk, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (S_kv == 0) {
    // Every row is empty: O = 0 so D = 0, dQ = 0, d_offset = 0 (written by preprocess).
    if (cudaMemsetAsync(dq, 0, (size_t)B * S_q * H_q * d_qk * 2, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  CUtensorMap tq, tk, tv, tdo;
  const int bq_rows = 64;  // query-tile rows of the kv-stationary kernel
  if (!sdpa::make_bshd_map(&tq, q, B, S_q, H_q, d_qk, bq_rows) ||
      !sdpa::make_bshd_map(&tdo, dout, B, S_q, H_q, d_v, bq_rows) ||
      !sdpa::make_bshd_map(&tk, k, B, S_kv, H_kv, d_qk, 128) ||
      !sdpa::make_bshd_map(&tv, v, B, S_kv, H_kv, d_v, 128)) {
    set_error("cuTensorMapEncodeTiled (backward operands)");
    return ATTN_ERR_CUDA;
  }
  CUtensorMap tdq = tq;
  if (fused && !sdpa::make_f32_bshd_map(&tdq, p.dq_acc, B, S_q, H_q, d_qk, bq_rows)) {
    set_error("cuTensorMapEncodeTiled (dQ accumulator)");
    return ATTN_ERR_CUDA;
  }
  // the kv kernel stages its bias tiles (64 query rows x 128 keys) by TMA when the rows
  // are a multiple of 16 bytes long; otherwise each thread loads its key's column itself
  CUtensorMap tb = tq;
  p.bias_tma = bias && S_kv % 8 == 0 ? 1 : 0;
  if (p.bias_tma && !sdpa::make_bias_map(&tb, bias, bias_B, bias_H, S_q, S_kv, bq_rows, 128)) {
    set_error("cuTensorMapEncodeTiled (bias)");
    return ATTN_ERR_CUDA;
  }
  // the query-stationary dQ kernel's maps (128-row boxes); the deterministic path's kv
  // kernel uses them too where its 128-row-step form applies
  CUtensorMap tq128 = tq, tdo128 = tdo;
  if (!fused && (!sdpa::make_bshd_map(&tq128, q, B, S_q, H_q, d_qk, 128) ||
                 !sdpa::make_bshd_map(&tdo128, dout, B, S_q, H_q, d_v, 128))) {
    set_error("cuTensorMapEncodeTiled (backward operands, 128 rows)");
    return ATTN_ERR_CUDA;
  }
  const bool wide = !fused && !bias && !p.drop_t && sdpa::bwd_kv_wide_supported(d_qk, d_v);
  int rc = timed(ATTN_KERNEL_BWD_KV, 1, s, [&] {
    if (wide) return sdpa::launch_bwd_kv_wide(d_qk, d_v, tq128, tk, tv, tdo128, p, s);
    return p.drop_t ? sdpa::launch_bwd_kv_dropout(d_qk, d_v, tq, tk, tv, tdo, tdq, tb, p, fused, s)
                    : sdpa::launch_bwd_kv(d_qk, d_v, tq, tk, tv, tdo, tdq, tb, p, fused, s);
  });
  if (rc == -2) return ATTN_ERR_UNSUPPORTED;
  if (rc != 0) {
    set_error("backward kv kernel launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  if (p.ns > 1 &&
      timed(ATTN_KERNEL_BWD_DQ_CONVERT, 1, s, [&] { return sdpa::launch_bwd_kv_combine(d_qk, d_v, p, s); }) != 0) {
    set_error("dK/dV split combine launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  if (fused) {
    if (timed(ATTN_KERNEL_BWD_DQ_CONVERT, 1, s, [&] { return sdpa::launch_bwd_dq_convert(d_qk, p, s); }) != 0) {
      set_error("dQ convert launch", cudaGetLastError());
      return ATTN_ERR_CUDA;
    }
  } else {
    rc = timed(ATTN_KERNEL_BWD_Q, 1, s, [&] {
      return p.drop_t ? sdpa::launch_bwd_q_dropout(d_qk, d_v, tq128, tk, tv, tdo128, p, s)
                      : sdpa::launch_bwd_q(d_qk, d_v, tq128, tk, tv, tdo128, p, s);
    });
    if (rc == -2) return ATTN_ERR_UNSUPPORTED;
    if (rc != 0) {
      set_error("backward dQ kernel launch", cudaGetLastError());
      return ATTN_ERR_CUDA;
    }
  }
  return ATTN_OK;
}

int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                    void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv,
                    int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                    const float* softmax_offset, const int* seq_lens_q, const int* seq_lens_kv, int deterministic,
                    void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, d_offset, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal,
                  window, softmax_type, softmax_offset, seq_lens_q, seq_lens_kv, nullptr, 1, 1, nullptr,
                  deterministic, workspace, workspace_bytes, stream);
}

int attn_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, float* d_offset, const void* bias, int bias_B, int bias_H,
                  float* dbias, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, float scale,
                  int causal, int window, int softmax_type, const float* softmax_offset, int deterministic,
                  void* workspace, size_t workspace_bytes, void* stream) {
  if (!bias) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, d_offset, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal,
                  window, softmax_type, softmax_offset, nullptr, nullptr, bias, bias_B, bias_H, dbias,
                  deterministic, workspace, workspace_bytes, stream);
}

int attn_bwd_varlen_bias(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, float* d_offset, const void* bias, int bias_B,
                         int bias_H, float* dbias, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v,
                         float scale, int causal, int window, int softmax_type, const float* softmax_offset,
                         const int* seq_lens_q, const int* seq_lens_kv, int deterministic, void* workspace,
                         size_t workspace_bytes, void* stream) {
  if (!bias) return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, d_offset, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal,
                  window, softmax_type, softmax_offset, seq_lens_q, seq_lens_kv, bias, bias_B, bias_H, dbias,
                  deterministic, workspace, workspace_bytes, stream);
}

int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv,
                     int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                     const float* softmax_offset, float dropout_p, const unsigned long long* rng_state,
                     int deterministic, void* workspace, size_t workspace_bytes, void* stream) {
  return bwd_impl(q, k, v, o, dout, lse, dq, dk, dv, d_offset, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale, causal,
                  window, softmax_type, softmax_offset, nullptr, nullptr, nullptr, 1, 1, nullptr, deterministic,
                  workspace, workspace_bytes, stream, dropout_p, rng_state);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk,
             int d_v, float scale, int causal, int window, int softmax_type, const float* softmax_offset,
             int deterministic, void* workspace, size_t workspace_bytes, void* stream) {
  return attn_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, d_offset, B, S_q, S_kv, H_q, H_kv, d_qk, d_v, scale,
                         causal, window, softmax_type, softmax_offset, nullptr, nullptr, deterministic, workspace,
                         workspace_bytes, stream);
}

int attn_fp8_vt_row_bytes(int S) { return S <= 0 ? 0 : (S + 15) / 16 * 16; }

int attn_fp8_amax(const void* x, size_t n, float* amax, void* stream) {
  if (!amax || (n > 0 && !x)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || (reinterpret_cast<uintptr_t>(amax) & 3u)) return ATTN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (timed(ATTN_KERNEL_FP8_QUANT, n > 0 ? 1 : 0, s, [&] {
        return sdpa::launch_fp8_amax(static_cast<const __nv_bfloat16*>(x), n, amax, s);
      }) != 0) {
    set_error("fp8 amax launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

static int fp8_quantize_impl(const void* x, void* x8, int B, int S, int H, int d, int transpose, const float* amax,
                             float* descale, float* amax_out, void* stream, bool e5m2, void* x8_nat = nullptr) {
  if (B < 0 || S < 0 || H <= 0 || d <= 0 || d % 8 != 0 || !amax || !descale) return ATTN_ERR_INVALID_ARG;
  if (transpose && d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if ((size_t)B * S * H * d > 0 && (!x || !x8)) return ATTN_ERR_INVALID_ARG;
  if (x8_nat && (x8_nat == x8 || !transpose)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(x8) || !aligned16(x8_nat) || (reinterpret_cast<uintptr_t>(amax) & 3u) ||
      (reinterpret_cast<uintptr_t>(descale) & 3u) || (reinterpret_cast<uintptr_t>(amax_out) & 3u))
    return ATTN_ERR_MISALIGNED;
  if (amax_out && (amax_out == amax || amax_out == descale)) return ATTN_ERR_INVALID_ARG;
  if ((size_t)B * S * H * d == 0) return ATTN_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rc = timed(ATTN_KERNEL_FP8_QUANT, 1, s, [&] {
    return sdpa::launch_fp8_quantize(static_cast<const __nv_bfloat16*>(x), static_cast<uint8_t*>(x8), B, S, H, d,
                                     transpose != 0, attn_fp8_vt_row_bytes(S), amax, descale, amax_out, s, e5m2,
                                     static_cast<uint8_t*>(x8_nat));
  });
  if (rc == -2) return ATTN_ERR_UNSUPPORTED;
  if (rc != 0) {
    set_error("fp8 quantize launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

int attn_fp8_quantize(const void* x, void* x8, int B, int S, int H, int d, int transpose, const float* amax,
                      float* descale, float* amax_out, void* stream) {
  return fp8_quantize_impl(x, x8, B, S, H, d, transpose, amax, descale, amax_out, stream, false);
}

int attn_fp8_quantize_e5m2(const void* x, void* x8, int B, int S, int H, int d, int transpose, const float* amax,
                           float* descale, float* amax_out, void* stream) {
  return fp8_quantize_impl(x, x8, B, S, H, d, transpose, amax, descale, amax_out, stream, true);
}

int attn_fp8_quantize_both(const void* x, void* x8, void* x8t, int B, int S, int H, int d, int e5m2,
                           const float* amax, float* descale, float* amax_out, void* stream) {
  if ((size_t)B * S * H * d > 0 && !x8) return ATTN_ERR_INVALID_ARG;
  return fp8_quantize_impl(x, x8t, B, S, H, d, 1, amax, descale, amax_out, stream, e5m2 != 0, x8);
}

int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* descale_q, const float* descale_k,
                 const float* descale_v, void* o, float* lse, int B, int S_q, int S_kv, int H_q, int H_kv, int d,
                 float scale, int causal, int window, int softmax_type, const float* softmax_offset, void* stream) {
  int st = check_common(B, S_q, S_kv, H_q, H_kv, d, d, causal, window, softmax_type, softmax_offset);
  if (st != ATTN_OK) return st;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || S_q == 0) return ATTN_OK;
  if (!q8 || !o || !lse || !descale_q || !descale_k || !descale_v || (S_kv > 0 && (!k8 || !vt8)))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(vt8) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u) || (reinterpret_cast<uintptr_t>(descale_q) & 3u) ||
      (reinterpret_cast<uintptr_t>(descale_k) & 3u) || (reinterpret_cast<uintptr_t>(descale_v) & 3u))
    return ATTN_ERR_MISALIGNED;
  int* err = device_error_ptr();
  if (!err) return ATTN_ERR_CUDA;
  // TMA maps need a non-empty tensor; with S_kv == 0 no kv tile is ever loaded.
  const int skv_map = S_kv > 0 ? S_kv : 1;
  const void* kk = S_kv > 0 ? k8 : q8;
  CUtensorMap tq, tk, tv;
  bool ok = sdpa::make_bshd_map_e4m3(&tq, q8, B, S_q, H_q, d, 128) &&
            sdpa::make_bshd_map_e4m3(&tk, kk, B, skv_map, S_kv > 0 ? H_kv : H_q, d, 128);
  if (S_kv > 0)
    ok = ok && sdpa::make_vt_map_e4m3(&tv, vt8, B, S_kv, attn_fp8_vt_row_bytes(S_kv), H_kv, d);
  else
    tv = tk;
  if (!ok) {
    set_error("cuTensorMapEncodeTiled (fp8 forward operands)");
    return ATTN_ERR_CUDA;
  }
  sdpa::FwdParams p;
  p.B = B; p.S_q = S_q; p.S_kv = S_kv; p.H_q = H_q; p.H_kv = H_kv; p.G = H_q / H_kv;
  p.scale_log2 = resolve_scale(scale, d) * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.window = window < 0 ? -1 : window;
  p.softmax_type = softmax_type;
  p.offset = softmax_offset;
  p.seq_q = nullptr;
  p.seq_kv = nullptr;
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.err = err;
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int rc = timed(ATTN_KERNEL_FWD, 1, s, [&] { return sdpa::launch_attn_fwd_fp8(d, tq, tk, tv, p, s); });
  if (rc == -2) return ATTN_ERR_UNSUPPORTED;
  if (rc != 0) {
    set_error("fp8 forward kernel launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

size_t attn_bwd_fp8_workspace_size(int B, int S_q, int H_q) {
  if (B < 0 || S_q < 0 || H_q <= 0) return 0;
  const size_t rows = static_cast<size_t>(B) * H_q * ((static_cast<size_t>(S_q) + 127) / 128 * 128);
  return 2 * round256(rows * sizeof(float));
}

int attn_bwd_fp8(const void* q8, const void* k8, const void* v8, const void* do8, const void* qt8, const void* kt8,
                 const void* dot8, const float* descale_q, const float* descale_k, const float* descale_v,
                 const float* descale_do, const void* o, const float* lse, const float* ds_amax, float* ds_amax_out,
                 void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv, int d,
                 float scale, int causal, int window, int softmax_type, const float* softmax_offset, void* workspace,
                 size_t workspace_bytes, void* stream) {
  int st = check_common(B, S_q, S_kv, H_q, H_kv, d, d, causal, window, softmax_type, softmax_offset);
  if (st != ATTN_OK) return st;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (softmax_type == ATTN_SOFTMAX_LEARNABLE && !d_offset) return ATTN_ERR_INVALID_ARG;
  if (!descale_q || !descale_k || !descale_v || !descale_do || !ds_amax) return ATTN_ERR_INVALID_ARG;
  if (ds_amax_out && ds_amax_out == ds_amax) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(descale_q) & 3u) || (reinterpret_cast<uintptr_t>(descale_k) & 3u) ||
      (reinterpret_cast<uintptr_t>(descale_v) & 3u) || (reinterpret_cast<uintptr_t>(descale_do) & 3u) ||
      (reinterpret_cast<uintptr_t>(ds_amax) & 3u) || (reinterpret_cast<uintptr_t>(ds_amax_out) & 3u) ||
      (reinterpret_cast<uintptr_t>(d_offset) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_MISALIGNED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B == 0 || (S_q == 0 && S_kv == 0)) {
    if (d_offset && cudaMemsetAsync(d_offset, 0, sizeof(float) * H_q, s) != cudaSuccess) return ATTN_ERR_CUDA;
    if (ds_amax_out && cudaMemsetAsync(ds_amax_out, 0, sizeof(float), s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  if ((S_q > 0 && (!q8 || !qt8 || !do8 || !dot8 || !o || !lse || !dq)) ||
      (S_kv > 0 && (!k8 || !kt8 || !v8 || !dk || !dv)))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q8) || !aligned16(k8) || !aligned16(v8) || !aligned16(do8) || !aligned16(qt8) ||
      !aligned16(kt8) || !aligned16(dot8) || !aligned16(o) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_MISALIGNED;
  const size_t need = attn_bwd_fp8_workspace_size(B, S_q, H_q);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return ATTN_ERR_WORKSPACE;
  int* err = device_error_ptr();
  if (!err) return ATTN_ERR_CUDA;
  // this call's max |dS| is taken with atomic maxima from zero (0 when nothing is visible)
  if (ds_amax_out && cudaMemsetAsync(ds_amax_out, 0, sizeof(float), s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (S_q == 0) {  // no query row sees a key: dK = dV = 0
    if (cudaMemsetAsync(dk, 0, (size_t)B * S_kv * H_kv * d * 2, s) != cudaSuccess ||
        cudaMemsetAsync(dv, 0, (size_t)B * S_kv * H_kv * d * 2, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    if (d_offset && cudaMemsetAsync(d_offset, 0, sizeof(float) * H_q, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  sdpa::BwdParams p;
  p.B = B; p.S_q = S_q; p.S_kv = S_kv; p.H_q = H_q; p.H_kv = H_kv; p.G = H_q / H_kv;
  p.scale = resolve_scale(scale, d);
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.window = window < 0 ? -1 : window;
  p.softmax_type = softmax_type;
  p.S_pad = (S_q + 127) / 128 * 128;
  p.offset = softmax_offset;
  p.seq_q = nullptr;
  p.seq_kv = nullptr;
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dout = nullptr;
  p.lse = lse;
  p.nlse2 = reinterpret_cast<float*>(ws);
  p.Dsum = reinterpret_cast<float*>(ws + need / 2);
  p.d_offset = d_offset;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.ns = 1;
  p.dk_part = nullptr;
  p.dv_part = nullptr;
  p.dq_acc = nullptr;
  p.err = err;
  p.do8 = static_cast<const uint8_t*>(do8);
  p.descale_q = descale_q;
  p.descale_k = descale_k;
  p.descale_v = descale_v;
  p.descale_do = descale_do;
  p.ds_amax = ds_amax;
  p.ds_amax_out = ds_amax_out;
  const int n_pre = 1 + (softmax_type == ATTN_SOFTMAX_LEARNABLE ? 1 : 0);
  if (timed(ATTN_KERNEL_BWD_PREPROCESS, n_pre, s, [&] { return sdpa::launch_bwd_preprocess_fp8(d, p, s); }) != 0) {
    set_error("fp8 backward preprocess launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  if (S_kv == 0) {  // every row is empty: O = 0 so D = 0 and dQ = 0
    if (cudaMemsetAsync(dq, 0, (size_t)B * S_q * H_q * d * 2, s) != cudaSuccess) return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  const int tq_row = attn_fp8_vt_row_bytes(S_q), tk_row = attn_fp8_vt_row_bytes(S_kv);
  // kv kernel: 64-query Q / dO tiles, 128-key K / V tiles; dQ kernel: 128-row Q / dO tiles,
  // 64-key K / V / K^T tiles
  CUtensorMap tq64, tdo64, tq128, tdo128, tk, tv, tk64, tv64, tqt, tdot, tkt;
  if (!sdpa::make_bshd_map_e4m3(&tq64, q8, B, S_q, H_q, d, 64) ||
      !sdpa::make_bshd_map_e4m3(&tdo64, do8, B, S_q, H_q, d, 64) ||
      !sdpa::make_bshd_map_e4m3(&tq128, q8, B, S_q, H_q, d, 128) ||
      !sdpa::make_bshd_map_e4m3(&tdo128, do8, B, S_q, H_q, d, 128) ||
      !sdpa::make_bshd_map_e4m3(&tk, k8, B, S_kv, H_kv, d, 128) ||
      !sdpa::make_bshd_map_e4m3(&tv, v8, B, S_kv, H_kv, d, 128) ||
      !sdpa::make_bshd_map_e4m3(&tk64, k8, B, S_kv, H_kv, d, 64) ||
      !sdpa::make_bshd_map_e4m3(&tv64, v8, B, S_kv, H_kv, d, 64) ||
      !sdpa::make_t_map_fp8(&tqt, qt8, B, S_q, tq_row, H_q, d, 64) ||
      !sdpa::make_t_map_fp8(&tdot, dot8, B, S_q, tq_row, H_q, d, 64) ||
      !sdpa::make_t_map_fp8(&tkt, kt8, B, S_kv, tk_row, H_kv, d, 64)) {
    set_error("cuTensorMapEncodeTiled (fp8 backward operands)");
    return ATTN_ERR_CUDA;
  }
  int rc = timed(ATTN_KERNEL_BWD_KV, 1, s,
                 [&] { return sdpa::launch_bwd_kv_fp8(d, tq64, tk, tv, tdo64, tqt, tdot, p, s); });
  if (rc == 0)
    rc = timed(ATTN_KERNEL_BWD_Q, 1, s, [&] { return sdpa::launch_bwd_q_fp8(d, tq128, tk64, tv64, tdo128, tkt, p, s); });
  if (rc == -2) return ATTN_ERR_UNSUPPORTED;
  if (rc != 0) {
    set_error("fp8 backward kernel launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

int attn_selftest_wait_timeout(int site, void* stream) {
  if (site < 0 || site > 0xFF) return ATTN_ERR_INVALID_ARG;
  int* err = device_error_ptr();
  if (!err) return ATTN_ERR_CUDA;
  if (sdpa::launch_selftest_wait(err, site, static_cast<cudaStream_t>(stream)) != 0) {
    set_error("self-test launch", cudaGetLastError());
    return ATTN_ERR_CUDA;
  }
  return ATTN_OK;
}

int attn_timing_enable(int on) {
  std::lock_guard<std::mutex> g(g_timing_mu);
  g_timing_on = on != 0;
  return ATTN_OK;
}

int attn_timing_read(double* ms, int* launches, int n) {
  std::vector<TimingRec> recs;
  {
    std::lock_guard<std::mutex> g(g_timing_mu);
    recs.swap(g_timing);
  }
  for (int k = 0; k < n; ++k) {
    if (ms) ms[k] = 0.0;
    if (launches) launches[k] = 0;
  }
  int status = ATTN_OK;
  for (const TimingRec& r : recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
      status = ATTN_ERR_CUDA;
    if (r.kind >= 0 && r.kind < n) {
      if (ms) ms[r.kind] += t;
      if (launches) launches[r.kind] += r.launches;
    }
  }
  std::lock_guard<std::mutex> g(g_timing_mu);
  for (const TimingRec& r : recs) {  // back to the pool for the next timed launches
    g_event_pool.push_back(r.a);
    g_event_pool.push_back(r.b);
  }
  return status;
}

}  // extern "C"
