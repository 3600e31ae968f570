/*
 * sdpa_tmem.h -- C ABI of the GB300 (sm_103a) fused scaled-dot-product attention
 * library libsdpa_tmem.so: forward and backward of
 *
 *     O = softmax(scale * Q K^T + mask) V      on BSHD tensors,
 *
 * with grouped-query heads, a causal mask with an optional left sliding window,
 * distinct Q/K and V head dims, and three sink softmax types; plus padded batches
 * with per-entry lengths (attn_fwd_varlen / attn_bwd_varlen), an additive bias with
 * its gradient (attn_fwd_bias / attn_bwd_bias), attention dropout (attn_fwd_dropout /
 * attn_bwd_dropout), an E4M3 forward with per-tensor scaling (attn_fp8_amax,
 * attn_fp8_quantize, attn_fwd_fp8) and its FP8 backward (attn_fp8_quantize_e5m2,
 * attn_bwd_fp8).
 *
 * Where each operation is defined:
 *   - the attention itself: "Speed up attention on GPU with cuDNN and
 *     TransformerEngine", section "How attention works" (score, scale + softmax,
 *     attend, output of Q's shape), step 7 (causal: query i sees keys j <= i);
 *   - BSHD layout, GQA (num_gqa_groups: each K/V head serves H_q/H_kv query
 *     heads), causal sliding window, MLA head dims (Q/K dim != V dim, layout
 *     bshd_bshd_bshd), scale_factor defaulting to 1/sqrt(head_dim), sink softmax
 *     types and deterministic backward: "JAX: Single-GPU Attention with
 *     TransformerEngine", sections 1, 2, 4 and "Other attention knobs";
 *   - the sink softmax denominators and the learnable offset's gradient:
 *     "[JAX] Add support for sink attention in JAX #2225", Greptile summaries
 *     (vanilla exp(S_i)/sum exp(S); off-by-one exp(S_i)/(1 + sum exp(S));
 *     learnable exp(S_ji)/(exp(alpha_j) + sum_i exp(S_ji)), the backward
 *     returning grad_softmax_offset).
 *
 * Conventions shared by every call:
 *   - All pointers are DEVICE pointers owned by the caller; the library allocates
 *     no device memory.  Its only state is one device error word per GPU.
 *   - Big tensors are contiguous BSHD bf16: Q [B,S_q,H_q,d_qk], K [B,S_kv,H_kv,d_qk],
 *     V [B,S_kv,H_kv,d_v], O and dO [B,S_q,H_q,d_v]; their base addresses must be
 *     16-byte aligned.  LSE is fp32 [B,H_q,S_q] (natural log, scaled-logit units,
 *     the sink included); softmax_offset and d_offset are fp32 [H_q].
 *   - Query head h uses K/V head h / (H_q / H_kv).
 *   - Masking: key j is visible to query i iff j < S_kv, and (causal == 0 or
 *     j <= i), and (window < 0 or j >= i - window).  A window needs causal != 0.
 *     A row that sees no key gets O = 0 and LSE = sink logit (-inf for vanilla).
 *   - scale <= 0 (or NaN) selects 1/sqrt(d_qk).
 *   - softmax_type: ATTN_SOFTMAX_VANILLA (no sink), ATTN_SOFTMAX_OFF_BY_ONE (a sink
 *     logit 0, i.e. +1 in the denominator), ATTN_SOFTMAX_LEARNABLE (sink logit
 *     softmax_offset[h], not multiplied by scale; softmax_offset required).
 *   - Supported head dims: d_qk in {64, 128, 192}, d_v in {64, 128}; H_q % H_kv == 0;
 *     B, H_q <= 65535.  Anything else returns ATTN_ERR_UNSUPPORTED (no fallback).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  Outputs are overwritten, never accumulated.  A status other than
 *     ATTN_OK means nothing was launched, except ATTN_ERR_CUDA, which reports the
 *     CUDA error of a launch.
 *   - Kernels never trap.  A pipeline wait that does not complete within about a
 *     second sets the device error word and the kernel exits; read it with
 *     attn_last_device_error().
 */
#ifndef SDPA_TMEM_H
#define SDPA_TMEM_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ATTN_SOFTMAX_VANILLA = 0, ATTN_SOFTMAX_OFF_BY_ONE = 1, ATTN_SOFTMAX_LEARNABLE = 2 };

enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,   /* null pointer, negative size, bad enum, H_q % H_kv != 0 */
  ATTN_ERR_UNSUPPORTED = 2,   /* head dims, window without causal, grid limits */
  ATTN_ERR_MISALIGNED = 3,    /* a BSHD base address not 16-byte aligned */
  ATTN_ERR_CUDA = 4,          /* a CUDA runtime / driver call failed */
  ATTN_ERR_DEVICE_TIMEOUT = 5, /* reported by attn_last_device_error() */
  ATTN_ERR_WORKSPACE = 6      /* workspace missing, too small or misaligned */
};

/*
 * Forward.  Writes o [B,S_q,H_q,d_v] (bf16) and lse [B,H_q,S_q] (fp32).
 * q, k, v: bf16 BSHD inputs.  softmax_offset: fp32 [H_q] for LEARNABLE, else
 * ignored (may be NULL).  Empty problems (B == 0 or S_q == 0) return ATTN_OK
 * without launching.
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q, int S_kv, int H_q,
             int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
             const float* softmax_offset, void* stream);

/*
 * Bytes of device workspace attn_bwd needs for these sizes (256-byte aligned
 * pointer required).  deterministic != 0 selects the recompute path for dQ, which
 * needs no fp32 dQ accumulator.  When the kv-stationary grid would be small (few
 * kv heads, as with MQA) the query heads of a group are split across several CTAs
 * and the workspace also holds their fp32 partial dK/dV; the combine that sums
 * them is fixed-order, so results stay reproducible.  Returns 0 for sizes that
 * attn_bwd rejects.
 */
size_t attn_bwd_workspace_size(int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, int deterministic);

/*
 * Backward of attn_fwd for the same arguments.  Inputs: q, k, v, o (the forward
 * output), dout = dL/dO (bf16 BSHD) and lse (the forward's fp32 LSE).  Outputs:
 * dq [B,S_q,H_q,d_qk], dk [B,S_kv,H_kv,d_qk], dv [B,S_kv,H_kv,d_v] (bf16, dK/dV
 * summed over the query heads of each group) and, for LEARNABLE, d_offset [H_q]
 * (fp32, summed over batch and rows; NULL is allowed for the other types and is
 * then not written; for them a non-NULL d_offset receives zeros).
 * deterministic != 0: bitwise-reproducible results (dQ by a query-stationary
 * recompute pass); 0: dQ accumulated with fp32 reductions for (d_qk, d_v) = (64, 64)
 * and (128, 128); the other head dims take the deterministic path either way.
 * workspace: device scratch of at least attn_bwd_workspace_size() bytes.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
             void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk,
             int d_v, float scale, int causal, int window, int softmax_type, const float* softmax_offset,
             int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Padded batches ("JAX: Single-GPU Attention with TransformerEngine", section 1:
 * the sequence descriptor gives each sequence's length and its padding).  Same as
 * attn_fwd / attn_bwd, plus seq_lens_q and seq_lens_kv: device int32 arrays [B]
 * (4-byte aligned, read by the kernels, owned by the caller) holding how many of
 * entry b's S_q query rows and S_kv key rows are real; they sit at the front of the
 * entry's rows and the rest is padding.  Values are clamped to [0, S_q] and
 * [0, S_kv].  NULL means every entry is full length (then these calls are exactly
 * attn_fwd / attn_bwd).  Entry b computes as if its tensors held only its real
 * rows; a padded query row sees no key, so o = 0 and lse = the sink logit (-inf
 * for VANILLA, 0 for OFF_BY_ONE, offset[h] for LEARNABLE) there; padded rows and
 * padded keys get zero dq / dk / dv and add nothing to d_offset.  Work outside
 * each entry's lengths is skipped.  Same workspace as attn_bwd.
 */
int attn_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q, int S_kv,
                    int H_q, int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                    const float* softmax_offset, const int* seq_lens_q, const int* seq_lens_kv, void* stream);
int attn_bwd_varlen(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                    void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv,
                    int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                    const float* softmax_offset, const int* seq_lens_q, const int* seq_lens_kv, int deterministic,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Human-readable name of a status code (static storage). */
const char* attn_status_string(int status);

/* Description of the last failure this thread saw inside the library (which call
   failed and CUDA's message), or "" (thread-local storage, valid until the next call). */
const char* attn_last_error_message(void);

/*
 * Synchronises `stream`, then returns and clears the current device's error word:
 * 0 when no kernel reported a failure, ATTN_ERR_DEVICE_TIMEOUT when a pipeline
 * wait timed out (the site is written to *site if site != NULL), ATTN_ERR_CUDA if
 * the synchronisation itself failed.
 */
int attn_last_device_error(void* stream, int* site);

/*
 * attn_bwd_noalloc -- the backward of attn_fwd for callers that cannot allocate
 * device memory.  (The pages have no counterpart: this is a packaging variant of
 * attn_bwd, not part of the method.)
 *
 * attn_bwd needs a caller-provided workspace.  Some callers cannot provide one:
 * runtimes that fix their device-memory footprint at start-up and forbid any
 * allocation on the launch path (inference-engine plugins, for example), and plain
 * C callers that have no device allocator of their own.  This entry point takes the
 * same arguments as attn_bwd minus `deterministic` and the workspace, allocates
 * nothing (no cudaMalloc, no cudaFree, no allocating library call), and keeps its
 * scratch in one fixed array inside the library: attn_bwd_noalloc_max_scratch_bytes()
 * bytes (8 MiB) per GPU, held by every GPU that loads the library until the process
 * exits.  It always runs the deterministic backward (query-stationary dQ), and it
 * is itself bitwise reproducible.  Its results match attn_bwd with deterministic != 0
 * within the gradient tolerance.  They are bitwise equal to it whenever attn_bwd walks
 * every query head of a kv group in one CTA.  attn_bwd instead splits the group's heads
 * across CTAs when its kv grid has fewer than 456 CTAs (3 per SM) and the group has
 * more than one query head.  The split sums partial dK/dV slices in another fp32
 * order; this entry point has no scratch for those slices and never splits.
 *
 * Limits and rules:
 *   - the scratch holds 8 bytes per (batch, query head, query row padded up to a
 *     multiple of 128): B * H_q * ceil(S_q/128)*128 <= 1,048,576 rows (for example
 *     B=4, H_q=32, S_q=8192).  Larger problems return ATTN_ERR_WORKSPACE without
 *     launching; attn_bwd_noalloc_message() then says how much was needed.
 *   - the first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current; make that first call before
 *     any stream capture.
 *   - every call on a device shares the one array.  Each call writes every word it
 *     later reads, so a previous call's contents never leak into a result, but
 *     calls whose kernels overlap on the GPU (different streams or threads) race on
 *     the array: order them on one stream.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                     const float* lse, void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv,
                     int H_q, int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                     const float* softmax_offset, void* stream);
/* Size in bytes of attn_bwd_noalloc's built-in scratch array. */
size_t attn_bwd_noalloc_max_scratch_bytes(void);
/* Why the last attn_bwd_noalloc call on this thread failed, or "" (thread-local). */
const char* attn_bwd_noalloc_message(void);

/*
 * Attention dropout.  Source: "JAX: Single-GPU Attention with TransformerEngine",
 * section "Other attention knobs" (`attention_dropout`); the sequence diagrams of
 * "[JAX] Add support for sink attention in JAX #2225" (the fused forward returns an
 * rng_state that the fused backward takes).
 *
 * Each probability P_ij after the softmax (sink included in the normaliser) is
 * dropped or kept; a kept one is scaled by 1/(1 - p):
 *   O_i = sum_j P_ij M_ij v_j,   M_ij = keep_ij * 65536 / (65536 - t),
 * while LSE (and p_sink) are those of the undropped softmax.  The backward uses
 *   dS_ij = P_ij (M_ij dO_i . v_j - D_i),   D_i = dO_i . O_i,   dV_j = sum_i P_ij M_ij dO_i.
 * The decisions come from a counter-based generator, so the backward regenerates
 * them: Philox4x32-10 (Salmon et al., SC'11).  With rng_state = (seed, offset), the key
 * is the seed (low 32 bits, high 32 bits); pair (b, h, i, j) uses the counter
 * (j / 2, i / 4, 65536 b + h, offset mod 2^32), output word i % 4, 16-bit field j % 2
 * as a uniform u in [0, 65536), and is kept iff u >= t.
 *
 * dropout_p: drop probability in [0, 1), realised as t / 65536 with
 *   t = floor(dropout_p * 65536 + 1/2) (from the float value); t = 0 runs the plain
 *   kernels; a value outside [0, 1), or one that rounds to t = 65536, returns
 *   ATTN_ERR_INVALID_ARG.
 * rng_state: DEVICE pointer to two uint64 values, seed then offset, 8-byte aligned,
 *   read by the kernels when they run (so a caller can advance the offset in place
 *   between steps).  Only the offset's low 32 bits are used: offsets that differ by a
 *   multiple of 2^32 give the same decisions.  Pass the same state to the forward and
 *   the backward of a step.
 * Otherwise as attn_fwd / attn_bwd (same workspace as attn_bwd).  Supported: full-length
 * batches, no bias, (d_qk, d_v) in {(64, 64), (128, 128), (192, 128)}; other head dims
 * return ATTN_ERR_UNSUPPORTED.
 */
int attn_fwd_dropout(const void* q, const void* k, const void* v, void* o, float* lse, int B, int S_q, int S_kv,
                     int H_q, int H_kv, int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                     const float* softmax_offset, float dropout_p, const unsigned long long* rng_state, void* stream);
int attn_bwd_dropout(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                     void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv,
                     int d_qk, int d_v, float scale, int causal, int window, int softmax_type,
                     const float* softmax_offset, float dropout_p, const unsigned long long* rng_state,
                     int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/*
 * Additive attention bias.  Source: "JAX: Single-GPU Attention with
 * TransformerEngine", section "Other attention knobs" (pass `bias` with an
 * `attn_bias_type`), and the sequence diagrams of "[JAX] Add support for sink
 * attention in JAX #2225" (the fused forward takes the bias, the fused backward
 * returns grad_bias next to dq, dk, dv).
 *
 * bias: bf16 [bias_B, bias_H, S_q, S_kv], contiguous, 16-byte aligned, with
 *   bias_B in {1, B} and bias_H in {1, H_q} (1 = broadcast over that dim).  It is
 *   added to the scaled scores before the masks and the softmax (post-scale):
 *   s_ij = scale * q_i . k_j + bias[b][h][i][j]; a -inf entry removes that key.
 * attn_fwd_bias: otherwise as attn_fwd.  attn_bwd_bias: as attn_bwd, plus
 *   dbias: fp32, the bias's shape (NULL: not computed) = dL/ds summed over the
 *   (b, h) that share each entry; the call zeroes it and accumulates it with fp32
 *   atomics, so with a broadcast bias (bias_B = 1 < B or bias_H = 1 < H_q) dbias is
 *   not bitwise reproducible and deterministic != 0 is rejected
 *   (ATTN_ERR_UNSUPPORTED).  Same workspace as attn_bwd.
 * attn_fwd_varlen_bias / attn_bwd_varlen_bias: the same on a padded batch (per-entry
 *   lengths as for attn_fwd_varlen).  The bias keeps the padded shape [bias_B, bias_H,
 *   S_q, S_kv]; entry b uses the top-left [Lq[b], Lkv[b]] corner of its planes, and dbias
 *   is zero outside those corners.
 * Supported head dims: (d_qk, d_v) in {(64, 64), (128, 128), (192, 128)}; others return
 * ATTN_ERR_UNSUPPORTED.
 */
int attn_fwd_bias(const void* q, const void* k, const void* v, void* o, float* lse, const void* bias, int bias_B,
                  int bias_H, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, float scale, int causal,
                  int window, int softmax_type, const float* softmax_offset, void* stream);
int attn_bwd_bias(const void* q, const void* k, const void* v, const void* o, const void* dout, const float* lse,
                  void* dq, void* dk, void* dv, float* d_offset, const void* bias, int bias_B, int bias_H,
                  float* dbias, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v, float scale,
                  int causal, int window, int softmax_type, const float* softmax_offset, int deterministic,
                  void* workspace, size_t workspace_bytes, void* stream);
int attn_fwd_varlen_bias(const void* q, const void* k, const void* v, void* o, float* lse, const void* bias,
                         int bias_B, int bias_H, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v,
                         float scale, int causal, int window, int softmax_type, const float* softmax_offset,
                         const int* seq_lens_q, const int* seq_lens_kv, void* stream);
int attn_bwd_varlen_bias(const void* q, const void* k, const void* v, const void* o, const void* dout,
                         const float* lse, void* dq, void* dk, void* dv, float* d_offset, const void* bias, int bias_B,
                         int bias_H, float* dbias, int B, int S_q, int S_kv, int H_q, int H_kv, int d_qk, int d_v,
                         float scale, int causal, int window, int softmax_type, const float* softmax_offset,
                         const int* seq_lens_q, const int* seq_lens_kv, int deterministic, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * FP8 (E4M3) forward.  Source: "Speed up attention on GPU with cuDNN and
 * TransformerEngine", step 10 ("Benchmark NVIDIA TransformerEngine and FP8"),
 * section "Inspect the FP8 path": the forward runs on E4M3 tensors (4 exponent,
 * 3 mantissa bits) with per-tensor scaling factors from the absolute maximum
 * (DelayedScaling, margin 0); the output stays bf16.
 *
 * E4M3 here is the OCP 8-bit float: bias 7, no infinities, largest finite 448;
 * conversions round to nearest even and saturate to +-448.  All scalars below
 * (amax, descale) are single fp32 values in DEVICE memory, so a step needs no
 * host synchronisation.
 *
 * attn_fp8_amax: amax[0] = max |x| over n bf16 values at x (16-byte aligned).
 *   A caller with an amax history writes the history's max into amax instead.
 * attn_fp8_quantize: scale = 448 / amax[0] (1 when amax is 0 or not finite);
 *   x8 = E4M3(fp32(x) * scale) and descale[0] = 1 / scale (fp32, correctly
 *   rounded).  amax_out, when not NULL, receives max |x| of this tensor, taken
 *   during the same pass (delayed scaling: amax holds the history's max from
 *   earlier steps, amax_out records this step's; it must not alias amax or
 *   descale).  x is bf16 BSHD [B, S, H, d].  transpose = 0: x8 has the same
 *   layout; transpose = 1 (d = 64 or 128): x8 is [B, H, d, S_pad], keys
 *   innermost, S_pad = attn_fp8_vt_row_bytes(S), zeros past S — the layout
 *   attn_fwd_fp8 takes V in.  x and x8 16-byte aligned.
 * attn_fwd_fp8: O (bf16 BSHD [B, S_q, H_q, d]) and LSE (fp32 [B, H_q, S_q]) of
 *   softmax(scale * Q K^T) V over the dequantised tensors Q = q8 * descale_q,
 *   K = k8 * descale_k, V = vt8 * descale_v, with the same masks, grouped heads
 *   and sink types as attn_fwd.  q8 [B, S_q, H_q, d], k8 [B, S_kv, H_kv, d]
 *   E4M3 BSHD; vt8 [B, H_kv, d, S_pad] from attn_fp8_quantize(transpose = 1).
 *   d = d_qk = d_v in {64, 128}.  The kernel rounds the softmax numerators to
 *   E4M3 for the P.V product while the normaliser and the LSE use their fp32
 *   values; the departure from the exact O this causes is bounded per row by
 *   2^-4 * sum_j P_j |v_j| + sum_j min(2^-10 * e^(M - LSE), P_j) |v_j|
 *   (P_j the probabilities, M the row's largest logit or sink).
 * Errors as attn_fwd; d outside {64, 128} is ATTN_ERR_UNSUPPORTED.
 */
int attn_fp8_amax(const void* x, size_t n, float* amax, void* stream);
int attn_fp8_quantize(const void* x, void* x8, int B, int S, int H, int d, int transpose, const float* amax,
                      float* descale, float* amax_out, void* stream);
/* Row length in bytes of the transposed E4M3 V: S rounded up to a multiple of 16. */
int attn_fp8_vt_row_bytes(int S);
int attn_fwd_fp8(const void* q8, const void* k8, const void* vt8, const float* descale_q, const float* descale_k,
                 const float* descale_v, void* o, float* lse, int B, int S_q, int S_kv, int H_q, int H_kv, int d,
                 float scale, int causal, int window, int softmax_type, const float* softmax_offset, void* stream);

/*
 * FP8 backward (E4M3 Q, K, V; E5M2 dO).  Source: "Speed up attention on GPU with
 * cuDNN and TransformerEngine", step 10, section "Inspect the FP8 path": the hybrid
 * recipe keeps the forward's tensors in E4M3 and takes gradients in E5M2 (5 exponent,
 * 2 mantissa bits, the wider range), each with a per-tensor scale from its absolute
 * maximum (DelayedScaling, margin 0).
 *
 * E5M2 here is the OCP 8-bit float: bias 15, largest finite 57344; conversions round
 * to nearest even and saturate to +-57344.
 *
 * attn_fp8_quantize_e5m2: attn_fp8_quantize with E5M2 codes and scale = 57344 /
 *   amax[0] (1 when amax is 0 or not finite); the same layouts, alignment and errors.
 * attn_bwd_fp8_workspace_size: bytes of device workspace attn_bwd_fp8 needs (256-byte
 *   aligned; two fp32 rows per (b, h) of S_q rounded up to 128).
 * attn_bwd_fp8: dQ, dK, dV (bf16 BSHD, as attn_bwd) and d_offset of the attention
 *   whose forward attn_fwd_fp8 computed (o, lse its outputs), over the dequantised
 *   Q = q8 descale_q, K = k8 descale_k, V = v8 descale_v and dO = do8 descale_do.
 *   Per (b, h) with P = exp(scale Q K^T - LSE) masked as in the forward:
 *     D = rowsum(dO * O); dP = dO V^T; dS = P (dP - D) (fp32);
 *     P~ = E4M3(2^8 P) / 2^8 and dS~ = E5M2(s dS) / s with s = 57344 / ds_amax[0]
 *       (1 when ds_amax[0] is 0 or not finite: delayed scaling from earlier steps);
 *     dV = P~^T dO, dK = scale dS~^T Q, dQ = scale dS~ K (fp32 accumulation), summed
 *       over the query heads of a group for dK, dV; d_offset as attn_bwd.
 *   Operands: q8 [B, S_q, H_q, d], k8, v8 [B, S_kv, H_kv, d] E4M3 BSHD; do8 [B, S_q,
 *   H_q, d] E5M2 BSHD; qt8, dot8 [B, H_q, d, attn_fp8_vt_row_bytes(S_q)] and kt8 [B,
 *   H_kv, d, attn_fp8_vt_row_bytes(S_kv)], the same codes transposed (quantize calls
 *   with transpose = 1 and the same amax); o bf16 BSHD; lse fp32 [B, H_q, S_q].  All
 *   scalars are fp32 in device memory.  ds_amax_out, when not NULL, receives max |dS|
 *   (before rounding) over the whole call, for the next step's ds_amax; it must not
 *   alias ds_amax.  d = d_qk = d_v in {64, 128}; full-length batches, no bias or
 *   dropout.  The results are deterministic (no atomics in dQ, dK, dV).
 *   Errors as attn_bwd; d outside {64, 128} is ATTN_ERR_UNSUPPORTED.
 */
int attn_fp8_quantize_e5m2(const void* x, void* x8, int B, int S, int H, int d, int transpose, const float* amax,
                           float* descale, float* amax_out, void* stream);
/*
 * attn_fp8_quantize_both: both layouts of one cast from a single read of x: x8 [B, S, H, d]
 * (BSHD) and x8t [B, H, d, attn_fp8_vt_row_bytes(S)] (transposed), E4M3 (e5m2 = 0) or E5M2
 * (e5m2 != 0), with the same codes, scale, descale and amax_out as the two separate calls
 * of attn_fp8_quantize / attn_fp8_quantize_e5m2.  d = 64 or 128; x8 and x8t distinct and
 * 16-byte aligned.  Errors as attn_fp8_quantize.
 */
int attn_fp8_quantize_both(const void* x, void* x8, void* x8t, int B, int S, int H, int d, int e5m2,
                           const float* amax, float* descale, float* amax_out, void* stream);
size_t attn_bwd_fp8_workspace_size(int B, int S_q, int H_q);
int attn_bwd_fp8(const void* q8, const void* k8, const void* v8, const void* do8, const void* qt8, const void* kt8,
                 const void* dot8, const float* descale_q, const float* descale_k, const float* descale_v,
                 const float* descale_do, const void* o, const float* lse, const float* ds_amax, float* ds_amax_out,
                 void* dq, void* dk, void* dv, float* d_offset, int B, int S_q, int S_kv, int H_q, int H_kv, int d,
                 float scale, int causal, int window, int softmax_type, const float* softmax_offset, void* workspace,
                 size_t workspace_bytes, void* stream);

/*
 * Failure-path self-test.  Every pipeline wait in the kernels is bounded (about one
 * second); on expiry the kernel stores 0x100 + a site code in a per-GPU device error
 * word, every other wait gives up at once, in-flight copies and MMAs are drained with
 * bounded waits, TMEM is freed and the kernel returns, so the CUDA context stays
 * usable and attn_last_device_error() reports ATTN_ERR_DEVICE_TIMEOUT with the site.
 * attn_selftest_wait_timeout enqueues one warp that waits on a barrier nobody
 * arrives at, through that same bounded wait, so the path can be checked without a
 * fault: after it, attn_last_device_error() returns ATTN_ERR_DEVICE_TIMEOUT with
 * site 0x100 + `site` (0..255) and clears the word.
 */
int attn_selftest_wait_timeout(int site, void* stream);

/*
 * Measurement aid (off by default).  While enabled, the attn_fwd*, attn_bwd* and
 * attn_fp8_* calls record
 * a pair of CUDA events on their launch stream around each class of kernel they
 * enqueue.  attn_timing_read() waits for those events, writes per class the
 * summed milliseconds (ms[k]) and the number of kernels launched (launches[k])
 * for k < n, discards the records and returns ATTN_OK (or ATTN_ERR_CUDA).
 * Classes: the ATTN_KERNEL_* values below.  Either output pointer may be NULL.
 */
enum {
  ATTN_KERNEL_FWD = 0,             /* forward kernel */
  ATTN_KERNEL_BWD_PREPROCESS = 1,  /* D = rowsum(dO*O), LSE rescale, d_offset */
  ATTN_KERNEL_BWD_KV = 2,          /* kv-stationary dK/dV (+ atomic dQ) kernel */
  ATTN_KERNEL_BWD_Q = 3,           /* query-stationary deterministic dQ kernel */
  ATTN_KERNEL_BWD_DQ_CONVERT = 4,  /* fp32 dQ accumulator -> bf16; split dK/dV combine */
  ATTN_KERNEL_FP8_QUANT = 5,       /* E4M3 amax and quantisation */
  ATTN_KERNEL_CLASSES = 6
};
int attn_timing_enable(int on);
int attn_timing_read(double* ms, int* launches, int n);

#ifdef __cplusplus
}
#endif

#endif /* SDPA_TMEM_H */
