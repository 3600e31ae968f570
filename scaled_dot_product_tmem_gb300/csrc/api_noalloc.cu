// api_noalloc.cu -- attn_bwd_noalloc: the attention backward for callers that
// cannot allocate device memory.
//
// attn_bwd needs a caller-provided workspace for two fp32 rows per query row
// (LSE * log2 e and D = rowsum(dO * O)).  Some callers have no way to provide one:
// runtimes that fix their device-memory footprint when they start and forbid
// allocation on the launch path (inference-engine plugins, for example), and
// plain C callers with no device allocator of their own.  This entry point keeps
// that scratch in one fixed array inside the library instead, so it allocates
// nothing at all.  It always takes the deterministic backward (query-stationary
// dQ), whose scratch is small; the fp32 dQ accumulator of the atomic path would
// not fit a fixed array.
//
// The array is kScratchBytes (8 MiB) per GPU, reserved on every GPU that loads
// the library until the process exits.  Problems needing more are rejected.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/sdpa_tmem.h"
#include "attn_kernels.h"
#include "tmap.h"

namespace {

constexpr size_t kScratchBytes = size_t(8) << 20;

// The shared scratch.  In host code this name is only a host-side stand-in for
// the device array, never a device address: host code must use the pointer
// cudaGetSymbolAddress returns for the current device (scratch_ptr below).
static __device__ __align__(256) unsigned char g_bwd_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned char* g_scratch_ptr[kMaxDevices] = {nullptr};

thread_local char g_msg[256] = "";

// Set-up, once per device, with that device current: look up the device address
// of g_bwd_scratch.  Runs on the first call made on each device.
unsigned char* scratch_ptr(int* status) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) {
    snprintf(g_msg, sizeof(g_msg), "attn_bwd_noalloc: cudaGetDevice failed: %s", cudaGetErrorString(e));
    *status = ATTN_ERR_CUDA;
    return nullptr;
  }
  if (dev < 0 || dev >= kMaxDevices) {
    snprintf(g_msg, sizeof(g_msg), "attn_bwd_noalloc: device %d is past the %d devices the library tracks", dev,
             kMaxDevices);
    *status = ATTN_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess || p == nullptr) {
      snprintf(g_msg, sizeof(g_msg), "attn_bwd_noalloc: cudaGetSymbolAddress(scratch) failed on device %d: %s",
               dev, cudaGetErrorString(e));
      *status = ATTN_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
  }
  return g_scratch_ptr[dev];
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Records which CUDA call failed and why; returns ATTN_ERR_CUDA.
int cuda_failed(const char* what, cudaError_t e) {
  snprintf(g_msg, sizeof(g_msg), "attn_bwd_noalloc: %s failed: %s (%d)", what, cudaGetErrorString(e), (int)e);
  return ATTN_ERR_CUDA;
}
// The same for a kernel launch (the reason is CUDA's last error).
int launch_failed(const char* what) { return cuda_failed(what, cudaGetLastError()); }

// cudaMemsetAsync(dst, 0, bytes) on s; ATTN_OK or ATTN_ERR_CUDA with the message set.
int zero_async(void* dst, size_t bytes, cudaStream_t s) {
  const cudaError_t e = cudaMemsetAsync(dst, 0, bytes, s);
  return e == cudaSuccess ? ATTN_OK : cuda_failed("cudaMemsetAsync", e);
}

}  // namespace

extern "C" {

size_t attn_bwd_noalloc_max_scratch_bytes(void) { return kScratchBytes; }

const char* attn_bwd_noalloc_message(void) { return g_msg; }

int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv,
                     int H_q, int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                     const float* softmax_offset, void* stream) {
  g_msg[0] = '\0';
  // The argument rules of attn_bwd (the same checks, shared with the other entry points).
  const int st = sdpa::check_common(B, S_q, S_kv, H_q, H_kv, d_qk, d_v, causal, window, softmax_type,
                                    softmax_offset);
  if (st != ATTN_OK) return st;
  if (softmax_type == ATTN_SOFTMAX_LEARNABLE && !d_offset) return ATTN_ERR_INVALID_ARG;
  const size_t s_pad = (static_cast<size_t>(S_q) + 127) / 128 * 128;
  const size_t rows = static_cast<size_t>(B) * H_q * s_pad;
  const size_t need = 2 * round256(rows * sizeof(float));
  if (need > kScratchBytes) {
    snprintf(g_msg, sizeof(g_msg),
             "attn_bwd_noalloc: this problem needs %zu bytes of scratch (8 bytes per (batch, head, query row "
             "padded to 128)); the built-in array holds %zu bytes; use attn_bwd with a workspace",
             need, kScratchBytes);
    return ATTN_ERR_WORKSPACE;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (B == 0 || (S_q == 0 && S_kv == 0)) return d_offset ? zero_async(d_offset, sizeof(float) * H_q, s) : ATTN_OK;
  if ((S_q > 0 && (!q || !o || !dout || !lse || !dq)) || (S_kv > 0 && (!k || !v || !dk || !dv)))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3u) ||
      (reinterpret_cast<uintptr_t>(d_offset) & 3u))
    return ATTN_ERR_MISALIGNED;
  if (S_q == 0) {
    int rc = zero_async(dk, (size_t)B * S_kv * H_kv * d_qk * 2, s);
    if (rc == ATTN_OK) rc = zero_async(dv, (size_t)B * S_kv * H_kv * d_v * 2, s);
    if (rc == ATTN_OK && d_offset) rc = zero_async(d_offset, sizeof(float) * H_q, s);
    return rc;
  }
  int status = ATTN_OK;
  unsigned char* scratch = scratch_ptr(&status);
  if (!scratch) return status;
  int* err = sdpa::device_error_word();
  if (!err) {
    snprintf(g_msg, sizeof(g_msg), "attn_bwd_noalloc: the device error word is unavailable (%s)",
             attn_last_error_message());
    return ATTN_ERR_CUDA;
  }

  // Every word of the scratch that the kernels read is written earlier in the
  // same call: the preprocess kernel writes both arrays for every real row and
  // every padding row (D = 0, LSE * log2 e = -inf past S_q), so nothing left by a
  // previous call is ever read and nothing needs clearing.  Calls that overlap on
  // the GPU (other streams, other threads) share the array and race.
  sdpa::BwdParams p;
  p.B = B; p.S_q = S_q; p.S_kv = S_kv; p.H_q = H_q; p.H_kv = H_kv; p.G = H_q / H_kv;
  p.scale = sdpa::resolve_scale(scale, d_qk);
  p.scale_log2 = p.scale * 1.4426950408889634f;
  p.causal = causal ? 1 : 0;
  p.window = window < 0 ? -1 : window;
  p.softmax_type = softmax_type;
  p.S_pad = static_cast<int>(s_pad);
  p.offset = softmax_offset;
  p.o = static_cast<const __nv_bfloat16*>(o);
  p.dout = static_cast<const __nv_bfloat16*>(dout);
  p.lse = lse;
  p.nlse2 = reinterpret_cast<float*>(scratch);
  p.Dsum = reinterpret_cast<float*>(scratch + round256(rows * sizeof(float)));
  p.d_offset = d_offset;
  p.dq = static_cast<__nv_bfloat16*>(dq);
  p.dk = static_cast<__nv_bfloat16*>(dk);
  p.dv = static_cast<__nv_bfloat16*>(dv);
  p.dq_acc = nullptr;
  p.ns = 1;  // no scratch for split partials: one CTA per (kv tile, kv head)
  p.dk_part = p.dv_part = nullptr;
  p.seq_q = nullptr;
  p.seq_kv = nullptr;
  p.err = err;

  if (sdpa::launch_bwd_preprocess(d_v, p, s) != 0) return launch_failed("backward preprocess launch");
  if (S_kv == 0) return zero_async(dq, (size_t)B * S_q * H_q * d_qk * 2, s);
  CUtensorMap tq64, tdo64, tq128, tdo128, tk, tv;
  if (!sdpa::make_bshd_map(&tq64, q, B, S_q, H_q, d_qk, 64) || !sdpa::make_bshd_map(&tdo64, dout, B, S_q, H_q, d_v, 64) ||
      !sdpa::make_bshd_map(&tq128, q, B, S_q, H_q, d_qk, 128) ||
      !sdpa::make_bshd_map(&tdo128, dout, B, S_q, H_q, d_v, 128) ||
      !sdpa::make_bshd_map(&tk, k, B, S_kv, H_kv, d_qk, 128) || !sdpa::make_bshd_map(&tv, v, B, S_kv, H_kv, d_v, 128)) {
    snprintf(g_msg, sizeof(g_msg), "attn_bwd_noalloc: cuTensorMapEncodeTiled failed");
    return ATTN_ERR_CUDA;
  }
  // the same kv kernel as attn_bwd's deterministic path
  int rc = sdpa::bwd_kv_wide_supported(d_qk, d_v)
               ? sdpa::launch_bwd_kv_wide(d_qk, d_v, tq128, tk, tv, tdo128, p, s)
               : sdpa::launch_bwd_kv(d_qk, d_v, tq64, tk, tv, tdo64, tq64, tq64, p, false, s);
  if (rc == -2) return ATTN_ERR_UNSUPPORTED;
  if (rc != 0) return launch_failed("backward kv kernel launch");
  rc = sdpa::launch_bwd_q(d_qk, d_v, tq128, tk, tv, tdo128, p, s);
  if (rc == -2) return ATTN_ERR_UNSUPPORTED;
  if (rc != 0) return launch_failed("backward dQ kernel launch");
  return ATTN_OK;
}

}  // extern "C"
