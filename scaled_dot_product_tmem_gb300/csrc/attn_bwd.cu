// attn_bwd.cu -- fused BSHD attention backward for sm_103a.
//
// With P_ij = exp(scale * q_i.k_j - LSE_i) (the forward's probabilities, sink
// included in LSE), dP_ij = dO_i.v_j, D_i = dO_i.O_i and dS_ij = P_ij (dP_ij - D_i):
//   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_{h in group} sum_i dS_ij q_i,
//   dV_j = sum_{h in group} sum_i P_ij dO_i,
//   d offset_h = -sum_{b,i} exp(offset_h - LSE_i) D_i        (learnable sink).
// The pages name these outputs ("[JAX] Add support for sink attention in JAX
// #2225", Greptile sequence diagrams: the backward returns grad_q, grad_k,
// grad_v, grad_bias, grad_softmax_offset); the formulas follow from the forward
// definition ("Speed up attention on GPU with cuDNN and TransformerEngine",
// section "How attention works").  The sink has no value vector, so D_i = dO_i.O_i
// and the dS formula are unchanged by it.
//
// Kernels:
//   bwd_preprocess   D and LSE*log2(e) into padded [B, H_q, S_pad] rows.
//   bwd_doffset      deterministic per-head reduction for d offset.
//   bwd_kv           kv-stationary: one CTA per (b, kv head, 128 keys) walks the
//                    query heads of the group x 64-row query tiles that see those
//                    keys; dK/dV accumulate in TMEM (the GQA head sum is free).
//                    Optionally also dQ^T = K^T dS^T per step, added into an fp32
//                    accumulator by TMA bulk reductions (non-deterministic path).
//   bwd_q            query-stationary deterministic dQ: recomputes S, P, dP, dS
//                    for one 128-row query tile over its kv tiles.
//   bwd_dq_convert   dQ = bf16(scale * fp32 accumulator).
#include <cuda_runtime.h>

#include "attn_bwd_kernels.cuh"

namespace sdpa {

// =============================================================================
// Preprocess: D = rowsum(dO * O) (fp32) and nlse2 = -LSE * log2(e), one block per
// (64 query rows, head, batch) so the per-row values are read and written as
// contiguous runs.  Rows are padded to S_pad: D = 0 and nlse2 = -inf there, so
// padded query rows get P = exp2(s + nlse2) = 0 in the main kernels.  In a padded
// batch, an entry's rows past its own query length are padding in the same way.
// =============================================================================
template <int D_V>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  constexpr int TPR = D_V / 8;     // threads per row, 8 bf16 (16 bytes) each
  constexpr int RPP = 256 / TPR;   // rows per pass of the block
  constexpr int TILE = 64;
  __shared__ float dsum[TILE];
  const int i0 = blockIdx.x * TILE, h = blockIdx.y, b = blockIdx.z;
  // the kv and dQ kernels that follow on this stream take their tiles from these counters
  if (blockIdx.x == 0 && h == 0 && b == 0 && threadIdx.x == 0) {
    if (p.tile_counter) *p.tile_counter = 0;
    if (p.tile_counter_q) *p.tile_counter_q = 0;
  }
  const int Lq = entry_len(p.seq_q, b, p.S_q);  // rows past it are padding, like rows past S_q
  const int sub = threadIdx.x % TPR;
  constexpr int NR = TILE / RPP;  // rows per thread
  uint4 a[NR], g[NR];
#pragma unroll
  for (int k = 0; k < NR; ++k) {  // every load of this thread first, then the math
    const int i = i0 + threadIdx.x / TPR + k * RPP;
    a[k] = g[k] = make_uint4(0u, 0u, 0u, 0u);
    if (i < Lq) {
      const size_t off = (((size_t)b * p.S_q + i) * p.H_q + h) * D_V + sub * 8;
      a[k] = __ldcs(reinterpret_cast<const uint4*>(p.o + off));
      g[k] = __ldcs(reinterpret_cast<const uint4*>(p.dout + off));
    }
  }
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    const int r = threadIdx.x / TPR + k * RPP;
    float acc = 0.f;
    {
      const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
      const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g[k]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 fa = __bfloat1622float2(a2[e]);
        const float2 fg = __bfloat1622float2(g2[e]);
        acc = fmaf(fa.x, fg.x, acc);
        acc = fmaf(fa.y, fg.y, acc);
      }
    }
    // the TPR lanes of a row are consecutive lanes of one warp
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0) dsum[r] = acc;
  }
  __syncthreads();
  if (threadIdx.x < TILE) {
    const int i = i0 + threadIdx.x;
    const size_t bh = (size_t)b * p.H_q + h;
    const bool real = i < Lq;
    p.Dsum[bh * p.S_pad + i] = real ? dsum[threadIdx.x] : 0.f;
    // a row with no probability mass (LSE = -inf: no visible key, or a bias of -inf on
    // every key) gets -inf too, so every P of it is exp2(-inf) = 0 without a NaN
    const float l = real ? p.lse[bh * p.S_q + i] : -INFINITY;
    p.nlse2[bh * p.S_pad + i] = l == -INFINITY ? -INFINITY : -l * kLog2e;
  }
}

// d offset_h = -sum_{b,i} exp(offset_h - LSE_{b,h,i}) D_{b,h,i}.  One block per
// head; fixed assignment of terms to threads and a fixed reduction tree, so the
// result is bitwise reproducible.
__global__ void __launch_bounds__(256) bwd_doffset_kernel(const BwdParams p) {
  const int h = blockIdx.x;
  const float c2 = p.offset[h] * kLog2e;
  float acc = 0.f;
  for (int b = 0; b < p.B; ++b) {
    const float* nl2 = p.nlse2 + ((size_t)b * p.H_q + h) * p.S_pad;
    const float* dd = p.Dsum + ((size_t)b * p.H_q + h) * p.S_pad;
    for (int i = threadIdx.x; i < p.S_q; i += blockDim.x) acc = fmaf(ex2(c2 + nl2[i]), dd[i], acc);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  __shared__ float part[8];
  if ((threadIdx.x & 31) == 0) part[threadIdx.x / 32] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += part[w];
    p.d_offset[h] = -s;
  }
}

int launch_bwd_preprocess(int d_v, const BwdParams& p, cudaStream_t stream) {
  if ((long long)p.B * p.S_q * p.H_q > 0) {
    const dim3 grid(p.S_pad / 64, p.H_q, p.B);
    if (d_v == 64)
      bwd_preprocess_kernel<64><<<grid, 256, 0, stream>>>(p);
    else if (d_v == 128)
      bwd_preprocess_kernel<128><<<grid, 256, 0, stream>>>(p);
    else
      return -2;
  }
  if (p.softmax_type == 2)
    bwd_doffset_kernel<<<p.H_q, 256, 0, stream>>>(p);
  else if (p.d_offset)
    cudaMemsetAsync(p.d_offset, 0, sizeof(float) * p.H_q, stream);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

bool bwd_kv_supports_fused_dq(int d_qk, int d_v) { return (d_qk == 128 || d_qk == 64) && (d_v == 128 || d_v == 64); }

int launch_bwd_kv(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                  const CUtensorMap& tdo, const CUtensorMap& tdq, const CUtensorMap& tb, const BwdParams& p,
                  bool fuse_dq, cudaStream_t stream) {
  if (p.bias) return launch_bwd_kv_bias(d_qk, d_v, tq, tk, tv, tdo, tdq, tb, p, fuse_dq, stream);
  if (fuse_dq) {
    if (d_qk == 128 && d_v == 128) return launch_kv_t<128, 128, true>(tq, tk, tv, tdo, tdq, tb, p, stream);
    if (d_qk == 128 && d_v == 64) return launch_kv_t<128, 64, true>(tq, tk, tv, tdo, tdq, tb, p, stream);
    if (d_qk == 64 && d_v == 64) return launch_kv_t<64, 64, true>(tq, tk, tv, tdo, tdq, tb, p, stream);
    if (d_qk == 64 && d_v == 128) return launch_kv_t<64, 128, true>(tq, tk, tv, tdo, tdq, tb, p, stream);
    return -2;
  }
  if (d_qk == 128 && d_v == 128) return launch_kv_t<128, 128, false>(tq, tk, tv, tdo, tdq, tb, p, stream);
  if (d_qk == 64 && d_v == 64) return launch_kv_t<64, 64, false>(tq, tk, tv, tdo, tdq, tb, p, stream);
  if (d_qk == 192 && d_v == 128) return launch_kv_t<192, 128, false>(tq, tk, tv, tdo, tdq, tb, p, stream);
  if (d_qk == 128 && d_v == 64) return launch_kv_t<128, 64, false>(tq, tk, tv, tdo, tdq, tb, p, stream);
  if (d_qk == 64 && d_v == 128) return launch_kv_t<64, 128, false>(tq, tk, tv, tdo, tdq, tb, p, stream);
  if (d_qk == 192 && d_v == 64) return launch_kv_t<192, 64, false>(tq, tk, tv, tdo, tdq, tb, p, stream);
  return -2;
}

int launch_bwd_q(int d_qk, int d_v, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                 const CUtensorMap& tdo, const BwdParams& p, cudaStream_t stream) {
  if (p.bias) return launch_bwd_q_bias(d_qk, d_v, tq, tk, tv, tdo, p, stream);
  if (d_qk == 128 && d_v == 128) return launch_q_t<128, 128>(tq, tk, tv, tdo, p, stream);
  if (d_qk == 64 && d_v == 64) return launch_q_t<64, 64>(tq, tk, tv, tdo, p, stream);
  if (d_qk == 192 && d_v == 128) return launch_q_t<192, 128>(tq, tk, tv, tdo, p, stream);
  if (d_qk == 128 && d_v == 64) return launch_q_t<128, 64>(tq, tk, tv, tdo, p, stream);
  if (d_qk == 64 && d_v == 128) return launch_q_t<64, 128>(tq, tk, tv, tdo, p, stream);
  if (d_qk == 192 && d_v == 64) return launch_q_t<192, 64>(tq, tk, tv, tdo, p, stream);
  return -2;
}

int bwd_kv_head_splits(int B, int S_kv, int H_kv, int G) {
  constexpr long long kSms = 152;  // GB300
  const long long ctas = (long long)((S_kv + 127) / 128) * H_kv * B;
  int ns = 1;
  if (ctas >= 3 * kSms) return ns;  // enough CTAs: the split's fp32 partials cost more than they balance
  while (2 * ns <= G && G % (2 * ns) == 0 && ctas * ns < 6 * kSms) ns *= 2;
  return ns;
}

// dK, dV = bf16(sum over the head splits of the fp32 partial slices), slice 0 first.
__global__ void __launch_bounds__(256) bwd_kv_combine_kernel(const float4* __restrict__ part,
                                                             uint2* __restrict__ out, size_t n4, int ns) {
  for (size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x; t < n4; t += (size_t)gridDim.x * blockDim.x) {
    float4 a = part[t];
    for (int s = 1; s < ns; ++s) {
      const float4 b = part[(size_t)s * n4 + t];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    out[t] = make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
  }
}

int launch_bwd_kv_combine(int d_qk, int d_v, const BwdParams& p, cudaStream_t stream) {
  const size_t rows = (size_t)p.B * p.S_kv * p.H_kv;
  for (int w = 0; w < 2; ++w) {
    const size_t n4 = rows * (w == 0 ? d_qk : d_v) / 4;
    if (n4 == 0) continue;
    const unsigned blocks = (unsigned)((n4 + 255) / 256 < 152 * 16 ? (n4 + 255) / 256 : 152 * 16);
    bwd_kv_combine_kernel<<<blocks, 256, 0, stream>>>(
        reinterpret_cast<const float4*>(w == 0 ? p.dk_part : p.dv_part),
        reinterpret_cast<uint2*>(w == 0 ? p.dk : p.dv), n4, p.ns);
  }
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

// =============================================================================
// dQ = bf16(scale * accumulator)
// =============================================================================
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(const float4* __restrict__ acc,
                                                             uint4* __restrict__ dq, size_t n8, float scale) {
  // one thread: 8 consecutive floats -> one 16-byte store
  const size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (t < n8) {
    const float4 a0 = __ldcs(acc + 2 * t), a1 = __ldcs(acc + 2 * t + 1);
    dq[t] = make_uint4(pack_bf16x2(a0.x * scale, a0.y * scale), pack_bf16x2(a0.z * scale, a0.w * scale),
                       pack_bf16x2(a1.x * scale, a1.y * scale), pack_bf16x2(a1.z * scale, a1.w * scale));
  }
}

int launch_bwd_dq_convert(int d_qk, const BwdParams& p, cudaStream_t stream) {
  const size_t n8 = (size_t)p.B * p.S_q * p.H_q * d_qk / 8;  // d_qk is a multiple of 64
  if (n8 == 0) return 0;
  bwd_dq_convert_kernel<<<(unsigned)((n8 + 255) / 256), 256, 0, stream>>>(reinterpret_cast<const float4*>(p.dq_acc),
                                                                          reinterpret_cast<uint4*>(p.dq), n8, p.scale);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sdpa
