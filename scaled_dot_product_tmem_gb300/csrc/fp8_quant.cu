// fp8_quant.cu -- per-tensor FP8 quantisation: E4M3 for the FP8 forward's inputs and
// the backward's Q, K, V; E5M2 for the backward's dO (the hybrid recipe: gradients in
// E5M2, with max finite 57344 in place of 448 below).
//
// Source: "Speed up attention on GPU with cuDNN and TransformerEngine", step 10,
// section "Inspect the FP8 path": the forward takes E4M3 tensors whose per-tensor
// scaling factors come from the absolute maximum (DelayedScaling, margin 0).
//   amax   = max |x|                       (fp8_amax_kernel)
//   scale  = 448 / amax  (1 if amax is 0 or not finite), descale = 1 / scale
//   x8     = E4M3(x * scale), round to nearest even, saturating to +-448
// With delayed scaling the scale comes from earlier steps' amax and the cast also
// records this tensor's amax (amax_out), so a step reads each tensor once.
// Both kernels are HBM-bound streams of 16-byte loads and stores.  The transposing form writes V as [B, H, d, S_pad] (keys
// innermost, rows padded to 16 bytes with zeros), the layout in which the forward's
// P.V product reads V as a K-major operand.
#include <cuda_runtime.h>

#include "attn_kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr unsigned kGridCap = 152 * 8;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Block-wide max of `m` into *out (skipped when out is null); every thread calls it.
__device__ __forceinline__ void block_amax(unsigned m, unsigned* out) {
  if (!out) return;
  m = __reduce_max_sync(0xffffffffu, m);
  __shared__ unsigned wm[32];
  if ((threadIdx.x & 31) == 0) wm[threadIdx.x / 32] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int w = 1; w < (int)(blockDim.x / 32); ++w) m = max(m, wm[w]);
    atomicMax(out, m);
  }
}

__device__ __forceinline__ unsigned abs_bits(float v) { return __float_as_uint(fabsf(v)); }

// |x| of non-negative floats orders like their bit patterns, so an unsigned max
// over the bits is a float max (a NaN input ends up above every finite value).
__global__ void __launch_bounds__(256) fp8_amax_kernel(const uint4* __restrict__ x8, const __nv_bfloat16* __restrict__ x,
                                                       size_t n, unsigned* __restrict__ amax_bits) {
  unsigned m = 0;
  const size_t n8 = n / 8;
  for (size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += (size_t)gridDim.x * blockDim.x) {
    const uint4 w = __ldcs(x8 + t);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) m = max(m, max(abs_bits(bf16_lo(ws[q])), abs_bits(bf16_hi(ws[q]))));
  }
  if (blockIdx.x == 0)
    for (size_t t = n8 * 8 + threadIdx.x; t < n; t += blockDim.x) m = max(m, abs_bits(__bfloat162float(x[t])));
  block_amax(m, amax_bits);
}

// E5: the E5M2 format (else E4M3).
template <bool E5>
__device__ __forceinline__ float scale_of(const float* amax) {
  const float a = *amax;
  return (a > 0.f && a <= 3.402823466e38f) ? __fdiv_rn(E5 ? 57344.f : 448.f, a) : 1.f;
}

template <bool E5>
__device__ __forceinline__ uint32_t pack4(float a, float b, float c, float d) {
  return E5 ? pack_e5m2x4(a, b, c, d) : pack_e4m3x4(a, b, c, d);
}

template <bool E5>
__global__ void __launch_bounds__(256) fp8_quant_kernel(const uint4* __restrict__ x8, const __nv_bfloat16* __restrict__ x,
                                                        uint2* __restrict__ out8, uint8_t* __restrict__ out, size_t n,
                                                        const float* __restrict__ amax, float* __restrict__ descale,
                                                        unsigned* __restrict__ amax_out) {
  const float sc = scale_of<E5>(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *descale = __fdiv_rn(1.f, sc);
  const size_t n8 = n / 8;
  unsigned m = 0;
  for (size_t t = (size_t)blockIdx.x * blockDim.x + threadIdx.x; t < n8; t += (size_t)gridDim.x * blockDim.x) {
    const uint4 w = __ldcs(x8 + t);
    if (amax_out) {
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) m = max(m, max(abs_bits(bf16_lo(ws[q])), abs_bits(bf16_hi(ws[q]))));
    }
    const uint32_t lo = pack4<E5>(__fmul_rn(bf16_lo(w.x), sc), __fmul_rn(bf16_hi(w.x), sc),
                                  __fmul_rn(bf16_lo(w.y), sc), __fmul_rn(bf16_hi(w.y), sc));
    const uint32_t hi = pack4<E5>(__fmul_rn(bf16_lo(w.z), sc), __fmul_rn(bf16_hi(w.z), sc),
                                  __fmul_rn(bf16_lo(w.w), sc), __fmul_rn(bf16_hi(w.w), sc));
    out8[t] = make_uint2(lo, hi);
  }
  if (blockIdx.x == 0)
    for (size_t t = n8 * 8 + threadIdx.x; t < n; t += blockDim.x) {
      const float xv = __bfloat162float(x[t]);
      m = max(m, abs_bits(xv));
      out[t] = (uint8_t)(pack4<E5>(__fmul_rn(xv, sc), 0.f, 0.f, 0.f) & 0xFFu);
    }
  block_amax(m, amax_out);
}

// One block per (b, h, 128-key tile).  Phase 1 reads the tile's 128 x d bf16 values
// as 16-byte chunks (coalesced along d), converts them and stores the codes row by
// row (key-major) in shared memory.  Phase 2 gives each thread 4 head dims x 16 keys:
// sixteen 4-byte reads, 4 x 4 byte transposes with byte permutes, and one 16-byte
// store per head dim into V^T (keys past S are zeros; keys past S_pad are not written).
// out_nat (may be null): the same codes in the input's own BSHD layout, written in phase 1,
// so one read of x gives both layouts.
template <int D, bool E5>
__global__ void __launch_bounds__(256) fp8_quant_t_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ out,
                                                          int S, int H, int S_pad, const float* __restrict__ amax,
                                                          float* __restrict__ descale, unsigned* __restrict__ amax_out,
                                                          uint8_t* __restrict__ out_nat) {
  constexpr int KT = 128;          // keys per tile
  constexpr int ROW = D + 4;       // bytes per key row in shared memory (4-byte aligned, skews the banks)
  __shared__ __align__(16) uint8_t tile[KT * ROW];
  const float sc = scale_of<E5>(amax);
  if (blockIdx.x == 0 && threadIdx.x == 0) *descale = __fdiv_rn(1.f, sc);
  const int n_tiles = (S_pad + KT - 1) / KT;
  const int kt = blockIdx.x % n_tiles, bh = blockIdx.x / n_tiles;
  const int h = bh % H, b = bh / H;
  const int k0 = kt * KT;
  constexpr int CPR = D / 8;  // 16-byte chunks per key row
  unsigned m = 0;
  for (int c = threadIdx.x; c < KT * CPR; c += blockDim.x) {
    const int kk = c / CPR, d0 = (c % CPR) * 8;
    const int key = k0 + kk;
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (key < S) w = __ldcs(reinterpret_cast<const uint4*>(x + (((size_t)b * S + key) * H + h) * D + d0));
    m = max(m, max(max(abs_bits(bf16_lo(w.x)), abs_bits(bf16_hi(w.x))), max(abs_bits(bf16_lo(w.y)), abs_bits(bf16_hi(w.y)))));
    m = max(m, max(max(abs_bits(bf16_lo(w.z)), abs_bits(bf16_hi(w.z))), max(abs_bits(bf16_lo(w.w)), abs_bits(bf16_hi(w.w)))));
    const uint32_t lo = pack4<E5>(__fmul_rn(bf16_lo(w.x), sc), __fmul_rn(bf16_hi(w.x), sc),
                                  __fmul_rn(bf16_lo(w.y), sc), __fmul_rn(bf16_hi(w.y), sc));
    const uint32_t hi = pack4<E5>(__fmul_rn(bf16_lo(w.z), sc), __fmul_rn(bf16_hi(w.z), sc),
                                  __fmul_rn(bf16_lo(w.w), sc), __fmul_rn(bf16_hi(w.w), sc));
    uint32_t* dst = reinterpret_cast<uint32_t*>(tile + kk * ROW + d0);
    dst[0] = lo;
    dst[1] = hi;
    if (out_nat && key < S)
      *reinterpret_cast<uint2*>(out_nat + (((size_t)b * S + key) * H + h) * D + d0) = make_uint2(lo, hi);
  }
  block_amax(m, amax_out);
  __syncthreads();
  constexpr int DG = D / 4;  // groups of 4 head dims
  for (int t = threadIdx.x; t < DG * (KT / 16); t += blockDim.x) {
    const int dg = t % DG, kg = t / DG;
    const int key = k0 + kg * 16;
    if (key >= S_pad) continue;
    uint32_t o[4][4];  // o[e][q]: head dim 4*dg+e, keys 4q .. 4q+3 of the group
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint32_t w[4];  // key kg*16 + 4q + r: its codes of head dims 4*dg .. 4*dg+3
#pragma unroll
      for (int r = 0; r < 4; ++r) w[r] = *reinterpret_cast<const uint32_t*>(tile + (kg * 16 + 4 * q + r) * ROW + 4 * dg);
      const uint32_t t0 = __byte_perm(w[0], w[1], 0x5140), t1 = __byte_perm(w[0], w[1], 0x7362);
      const uint32_t t2 = __byte_perm(w[2], w[3], 0x5140), t3 = __byte_perm(w[2], w[3], 0x7362);
      o[0][q] = __byte_perm(t0, t2, 0x5410);
      o[1][q] = __byte_perm(t0, t2, 0x7632);
      o[2][q] = __byte_perm(t1, t3, 0x5410);
      o[3][q] = __byte_perm(t1, t3, 0x7632);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e)
      *reinterpret_cast<uint4*>(out + (((size_t)b * H + h) * D + 4 * dg + e) * S_pad + key) =
          make_uint4(o[e][0], o[e][1], o[e][2], o[e][3]);
  }
}

unsigned grid_for(size_t work) {
  const size_t g = (work + 255) / 256;
  return (unsigned)(g == 0 ? 1 : (g < kGridCap ? g : kGridCap));
}

}  // namespace

int launch_fp8_amax(const __nv_bfloat16* x, size_t n, float* amax, cudaStream_t stream) {
  if (cudaMemsetAsync(amax, 0, sizeof(float), stream) != cudaSuccess) return -1;
  if (n == 0) return 0;
  fp8_amax_kernel<<<grid_for(n / 8), 256, 0, stream>>>(reinterpret_cast<const uint4*>(x), x, n,
                                                       reinterpret_cast<unsigned*>(amax));
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <bool E5>
static int quantize_t(const __nv_bfloat16* x, uint8_t* x8, int B, int S, int H, int d, bool transpose, int S_pad,
                      const float* amax, float* descale, unsigned* ao, cudaStream_t stream, uint8_t* x8_nat) {
  const size_t n = (size_t)B * S * H * d;
  if (!transpose) {
    fp8_quant_kernel<E5><<<grid_for(n / 8), 256, 0, stream>>>(reinterpret_cast<const uint4*>(x), x,
                                                              reinterpret_cast<uint2*>(x8), x8, n, amax, descale, ao);
  } else {
    const long long blocks = (long long)((S_pad + 127) / 128) * H * B;
    if (blocks <= 0 || blocks > 0x7fffffffLL) return -2;
    if (d == 128)
      fp8_quant_t_kernel<128, E5><<<(unsigned)blocks, 256, 0, stream>>>(x, x8, S, H, S_pad, amax, descale, ao, x8_nat);
    else if (d == 64)
      fp8_quant_t_kernel<64, E5><<<(unsigned)blocks, 256, 0, stream>>>(x, x8, S, H, S_pad, amax, descale, ao, x8_nat);
    else
      return -2;
  }
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_fp8_quantize(const __nv_bfloat16* x, uint8_t* x8, int B, int S, int H, int d, bool transpose, int S_pad,
                        const float* amax, float* descale, float* amax_out, cudaStream_t stream, bool e5m2,
                        uint8_t* x8_nat) {
  unsigned* ao = reinterpret_cast<unsigned*>(amax_out);
  if (amax_out && cudaMemsetAsync(amax_out, 0, sizeof(float), stream) != cudaSuccess) return -1;
  if (x8_nat && !transpose) return -2;
  return e5m2 ? quantize_t<true>(x, x8, B, S, H, d, transpose, S_pad, amax, descale, ao, stream, x8_nat)
              : quantize_t<false>(x, x8, B, S, H, d, transpose, S_pad, amax, descale, ao, stream, x8_nat);
}

}  // namespace sdpa
