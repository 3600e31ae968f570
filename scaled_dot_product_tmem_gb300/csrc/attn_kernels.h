// attn_kernels.h -- internal launch interface between the C-ABI layer (api.cu)
// and the kernel translation units.  Not part of the public header.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace sdpa {

struct FwdParams {
  int B, S_q, S_kv, H_q, H_kv, G;
  float scale_log2;  // scale * log2(e)
  int causal, window, softmax_type;
  const float* offset;  // [H_q], learnable only
  const int* seq_q;     // [B] query lengths of a padded batch, or null (all S_q)
  const int* seq_kv;    // [B] key lengths of a padded batch, or null (all S_kv)
  __nv_bfloat16* o;     // [B, S_q, H_q, d_v]
  float* lse;           // [B, H_q, S_q]
  int* err;             // device error word
  // E4M3 forward only: device scalars that undo the per-tensor scaling of Q, K, V
  const float* descale_q = nullptr;
  const float* descale_k = nullptr;
  const float* descale_v = nullptr;
  // additive bias [Bb, Hb, S_q, S_kv] (bf16) or null; element strides of batch and head
  // (0 along a broadcast dim)
  const __nv_bfloat16* bias = nullptr;
  long long bias_sb = 0, bias_sh = 0;
  int bias_tma = 0;  // head dims <= 128: the bias tiles are staged by TMA (S_kv % 8 == 0)
  // attention dropout (drop_t > 0): rng = device [seed, offset] (the Philox key and counter), drop
  // threshold t (16-bit uniforms below it are dropped), kept values scaled by drop_scale
  const unsigned long long* rng = nullptr;
  unsigned drop_t = 0;
  float drop_scale = 1.f;
};

// Returns 0 on a successful launch, -2 for an unsupported (d_qk, d_v), -1 on a
// CUDA launch error.
// tb: the bias map (boxes of 64 keys x 128 rows, 128-byte swizzle) when p.bias_tma, else null.
int launch_attn_fwd(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                    const FwdParams& p, cudaStream_t stream, const CUtensorMap* tb = nullptr);
// E4M3 forward, d_qk = d_v = d in {64, 128}; tvt maps V^T [B, H_kv, d, S_kv_pad].
int launch_attn_fwd_fp8(int d, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tvt,
                        const FwdParams& p, cudaStream_t stream);
// amax[0] = max |x| over n bf16 values (amax must be zeroed first).
int launch_fp8_amax(const __nv_bfloat16* x, size_t n, float* amax, cudaStream_t stream);
// x8 = E4M3(x * scale), scale = 448 / amax[0] (1 if amax is 0 or not finite),
// descale[0] = 1 / scale.  transpose: x [B, S, H, d] -> x8 [B, H, d, S_pad].
// amax_out (may be null): receives max |x| of this tensor, recorded during the cast.
// e5m2: E5M2 codes with scale = 57344 / amax instead.  x8_nat (transpose only, may be
// null): the same codes in x's BSHD layout as well, from the same read of x.
int launch_fp8_quantize(const __nv_bfloat16* x, uint8_t* x8, int B, int S, int H, int d, bool transpose, int S_pad,
                        const float* amax, float* descale, float* amax_out, cudaStream_t stream, bool e5m2 = false,
                        uint8_t* x8_nat = nullptr);

struct BwdParams {
  int B, S_q, S_kv, H_q, H_kv, G;
  float scale;       // softmax scale
  float scale_log2;  // scale * log2(e)
  int causal, window, softmax_type;
  int S_pad;                  // S_q rounded up to 128: row length of nlse2 / Dsum
  const float* offset;        // [H_q]
  const int* seq_q;           // [B] query lengths of a padded batch, or null (all S_q)
  const int* seq_kv;          // [B] key lengths of a padded batch, or null (all S_kv)
  const __nv_bfloat16* o;     // [B, S_q, H_q, d_v]
  const __nv_bfloat16* dout;  // [B, S_q, H_q, d_v]
  const float* lse;           // [B, H_q, S_q] (natural log)
  float* nlse2;               // [B, H_q, S_pad] workspace: -LSE * log2(e), -inf padding
  float* Dsum;                // [B, H_q, S_pad] workspace: rowsum(dO * O), 0 padding
  float* d_offset;            // [H_q] (learnable) or null
  __nv_bfloat16* dq;          // [B, S_q, H_q, d_qk]
  __nv_bfloat16* dk;          // [B, S_kv, H_kv, d_qk]
  __nv_bfloat16* dv;          // [B, S_kv, H_kv, d_v]
  int ns;                     // query-head splits of the kv kernel (1: a CTA walks every head of its group)
  float* dk_part;             // ns > 1: [ns, B, S_kv, H_kv, d_qk] fp32 partial dK (scaled), one slice per split
  float* dv_part;             // ns > 1: [ns, B, S_kv, H_kv, d_v] fp32 partial dV
  float* dq_acc;              // [B, S_q, H_q, d_qk] fp32 workspace (atomic dQ path) or null
  // next tile of the persistent kv kernel and of the persistent dQ kernel (workspace ints
  // the preprocess zeroes; null: those kernels run one CTA per tile)
  int* tile_counter = nullptr;
  int* tile_counter_q = nullptr;
  int* err;
  // additive bias [Bb, Hb, S_q, S_kv] (bf16) or null, with the element strides of batch
  // and head (0 along a broadcast dim); dbias: fp32, same shape and strides, zeroed by
  // the caller, accumulated with fp32 atomics (null: not wanted)
  const __nv_bfloat16* bias = nullptr;
  long long bias_sb = 0, bias_sh = 0;
  float* dbias = nullptr;
  int bias_tma = 0;  // the kv kernel stages its bias tiles by TMA (S_kv % 8 == 0), else loads them itself
  // attention dropout, as in FwdParams (the same rng state regenerates the forward's decisions)
  const unsigned long long* rng = nullptr;
  unsigned drop_t = 0;
  float drop_scale = 1.f;
  // FP8 backward: the E5M2 dO codes (for D), the per-tensor descales (device scalars), the
  // dS scaling statistic (device scalar: scale = 57344 / *ds_amax) and where this step's
  // max |dS| is recorded (may be null)
  const uint8_t* do8 = nullptr;
  const float* descale_q = nullptr;
  const float* descale_k = nullptr;
  const float* descale_v = nullptr;
  const float* descale_do = nullptr;
  const float* ds_amax = nullptr;
  float* ds_amax_out = nullptr;
};

int launch_bwd_preprocess(int d_v, const BwdParams& p, cudaStream_t stream);
// tdq: fp32 map of dq_acc (box d_qk x 64 rows) when fuse_dq, else any valid map (unused).
// tb: the bias map (box 128 keys x 64 rows) when p.bias_tma, else any valid map (unused).
int launch_bwd_kv(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                  const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tb, const BwdParams& p,
                  bool fuse_dq, cudaStream_t stream);
// Query-head splits of the kv kernel for these sizes: a grid of fewer than 3 CTAs
// per SM (few kv heads, as with MQA) is bound by its longest CTA, so each CTA's
// head loop is halved until the grid has 6 CTAs per SM; 1 = no split.
int bwd_kv_head_splits(int B, int S_kv, int H_kv, int G);
// ns > 1: dK, dV (bf16) = the sum of the ns fp32 partial slices, in slice order.
int launch_bwd_kv_combine(int d_qk, int d_v, const BwdParams& p, cudaStream_t stream);
// dK/dV only, with 128-row query steps (the deterministic path's kv kernel where it
// applies): d_qk = d_v in {64, 128}, no bias, no dropout; tq128/tdo128 have boxes of 64
// columns x 128 rows.  -2 when not applicable (the 64-row kernel is used then).
bool bwd_kv_wide_supported(int d_qk, int d_v);
int launch_bwd_kv_wide(int d_qk, int d_v, const CUtensorMap& tq128, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo128, const BwdParams& p, cudaStream_t stream);
int launch_bwd_q(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream);
int launch_bwd_dq_convert(int d_qk, const BwdParams& p, cudaStream_t stream);
bool bwd_kv_supports_fused_dq(int d_qk, int d_v);

// Bias instantiations (full-length or padded batches, bf16; (d_qk, d_v) in {(64, 64),
// (128, 128), (192, 128)}; the fused dQ for 64 and 128): the same contracts as above.
int launch_attn_fwd_bias(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t stream, const CUtensorMap* tb);
int launch_bwd_kv_bias(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tb, const BwdParams& p,
                       bool fuse_dq, cudaStream_t stream);
int launch_bwd_q_bias(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                      const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream);

// Dropout instantiations (full-length batches, bf16, no bias; (d_qk, d_v) in
// {(64, 64), (128, 128), (192, 128)}): the same contracts as the launchers above.
int launch_attn_fwd_dropout(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, cudaStream_t stream);
int launch_bwd_kv_dropout(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tb, const BwdParams& p,
                          bool fuse_dq, cudaStream_t stream);
int launch_bwd_q_dropout(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream);

// FP8 backward (E4M3 Q, K, V; E5M2 dO), d_qk = d_v = d in {64, 128}, full-length batches:
// the preprocess (D from the dequantised dO8 and the bf16 O), the kv-stationary kernel (dK,
// dV) and the query-stationary kernel (dQ).  Maps: tq8/tk8/tv8/tdo8 natural BSHD codes
// (boxes of the whole head dim x 64 rows for Q/dO, x 128 rows for K/V in the kv kernel, x 64
// rows for K/V in the dQ kernel); tqt8/tdot8 the transposed Q / dO codes [B, H_q, d, S_pad]
// (boxes of 64 queries x d); tkt8 the transposed K codes [B, H_kv, d, S_pad] (boxes of 64
// keys x d); tq8_128/tdo8_128 the natural Q/dO with 128-row boxes for the dQ kernel.
int launch_bwd_preprocess_fp8(int d, const BwdParams& p, cudaStream_t stream);
int launch_bwd_kv_fp8(int d, const CUtensorMap& tq8, const CUtensorMap& tk8, const CUtensorMap& tv8,
                      const CUtensorMap& tdo8, const CUtensorMap& tqt8, const CUtensorMap& tdot8, const BwdParams& p,
                      cudaStream_t stream);
int launch_bwd_q_fp8(int d, const CUtensorMap& tq8_128, const CUtensorMap& tk8, const CUtensorMap& tv8,
                     const CUtensorMap& tdo8_128, const CUtensorMap& tkt8, const BwdParams& p, cudaStream_t stream);

// One warp waits on an mbarrier nobody arrives at: after the wait limit it records
// kErrTimeoutBase + site in *err and returns (the failure path, without a fault).
int launch_selftest_wait(int* err, int site, cudaStream_t stream);

// Device error word of the current device (null if CUDA cannot report it).
int* device_error_word();

// Argument rules shared by every entry point (sizes, flags, head dims): ATTN_OK or an
// error status of the public header.
int check_common(int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, int causal, int window,
                 int softmax_type, const float* softmax_offset);
// The softmax scale to use: `scale` when finite and positive, else 1 / sqrt(d_qk).
float resolve_scale(float scale, int d_qk);

}  // namespace sdpa
