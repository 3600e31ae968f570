// attn_common.cuh -- index arithmetic shared by the forward and backward kernels:
// which keys a query row sees, which kv tiles a block of query rows touches, and
// which query tiles a block of keys is seen by.
//
// Masking rule (causal with an optional left window, top-left diagonal):
//   key j is visible to query i  iff  i < S_q and j < S_kv and (!causal or j <= i)
//                                     and (window < 0 or j >= i - window).
// In a padded batch S_q and S_kv are the entry's own lengths, so its padded query
// rows see no key and its padded keys are seen by no query.
// ("JAX: Single-GPU Attention with TransformerEngine", sections 1-2: causal
// mask plus sliding window; codelab "Speed up attention on GPU with cuDNN and
// TransformerEngine", step 7: query i sees keys j <= i.)
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

namespace sdpa {

struct MaskSpec {
  int S_q, S_kv, causal, window;
};

// VL: the batch is padded (S_q is the entry's own length and rows past it exist);
// without it every row the kernels look at is below S_q and the row test is dropped.
template <bool VL>
__host__ __device__ __forceinline__ bool key_visible(const MaskSpec& m, int i, int j) {
  return (!VL || i < m.S_q) && j < m.S_kv && (!m.causal || j <= i) && (m.window < 0 || j >= i - m.window);
}

// The keys query row i sees form one interval [*lo, *hi] (empty when lo > hi):
// the same set key_visible<VL> describes, as two bounds a mask loop can compare with.
template <bool VL>
__host__ __device__ __forceinline__ void visible_keys(const MaskSpec& m, int i, int* lo, int* hi) {
  int a = m.window >= 0 ? i - m.window : 0;
  int z = m.causal ? i : m.S_kv - 1;
  if (z > m.S_kv - 1) z = m.S_kv - 1;
  *lo = a < 0 ? 0 : a;
  *hi = (VL && i >= m.S_q) ? -1 : z;
}

// The query rows that see key j form one interval [*lo, *hi] (empty when lo > hi).
template <bool VL>
__host__ __device__ __forceinline__ void visible_rows(const MaskSpec& m, int j, int* lo, int* hi) {
  int a = m.causal ? j : 0;
  int z = m.window >= 0 ? j + m.window : 0x7fffffff - 1;
  if (VL && z > m.S_q - 1) z = m.S_q - 1;
  *lo = a;
  *hi = j < m.S_kv ? z : -1;
}

// Length of batch entry b: lens[b] clamped to [0, S], or S without a length array.
__host__ __device__ __forceinline__ int entry_len(const int* lens, int b, int S) {
  if (!lens) return S;
  const int l = lens[b];
  return l < 0 ? 0 : (l > S ? S : l);
}

// Inclusive range of kv tiles (size bn) touched by query rows [r0, r1]; returns
// false when those rows see no key at all.
__host__ __device__ __forceinline__ bool kv_tile_range(const MaskSpec& m, int r0, int r1, int bn, int* jlo,
                                                       int* jhi) {
  if (r1 > m.S_q - 1) r1 = m.S_q - 1;
  if (r1 < r0) return false;
  int lo = m.window >= 0 ? (r0 - m.window > 0 ? r0 - m.window : 0) : 0;
  int hi = m.causal ? (r1 < m.S_kv - 1 ? r1 : m.S_kv - 1) : m.S_kv - 1;
  if (hi < lo || m.S_kv <= 0) return false;
  *jlo = lo / bn;
  *jhi = hi / bn;
  return true;
}

// Inclusive range of query tiles (size bm) that see at least one key of
// [k0, k1]; returns false when none does.
__host__ __device__ __forceinline__ bool q_tile_range(const MaskSpec& m, int k0, int k1, int bm, int* ilo,
                                                      int* ihi) {
  if (k1 > m.S_kv - 1) k1 = m.S_kv - 1;
  if (k1 < k0) return false;
  int lo = m.causal ? k0 : 0;
  int hi = m.window >= 0 ? k1 + m.window : m.S_q - 1;
  if (hi > m.S_q - 1) hi = m.S_q - 1;
  if (hi < lo || m.S_q <= 0) return false;
  *ilo = lo / bm;
  *ihi = hi / bm;
  return true;
}

// Is the whole (rows [r0, r0+bm), keys [k0, k0+bn)) tile visible?  Then the
// per-element mask can be skipped.  (Without VL, rows past S_q are never stored.)
template <bool VL>
__host__ __device__ __forceinline__ bool tile_fully_visible(const MaskSpec& m, int r0, int bm, int k0, int bn) {
  int r1 = r0 + bm - 1;
  int k1 = k0 + bn - 1;
  if (k1 >= m.S_kv || (VL && r1 >= m.S_q)) return false;
  if (m.causal && k1 > r0) return false;
  if (m.window >= 0 && k0 < r1 - m.window) return false;
  return true;
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~static_cast<uintptr_t>(1023));
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Additive bias ("JAX: Single-GPU Attention with TransformerEngine", section "Other
// attention knobs": `bias` with an `attn_bias_type`): a bf16 [Bb, Hb, S_q, S_kv] tensor
// added to the scaled scores; Bb in {1, B} and Hb in {1, H_q} broadcast, expressed as
// element strides that are 0 along a broadcast dim.
__device__ __forceinline__ float bf16_bits_to_float(unsigned short u) { return __uint_as_float((uint32_t)u << 16); }

// 8 consecutive bias values of one row, starting at key k (0 for keys >= S_kv).  vec:
// S_kv is a multiple of 8 and k of 8, so one 16-byte load covers them (all or none
// below S_kv).
__device__ __forceinline__ void load_bias8(const __nv_bfloat16* row, int k, int S_kv, bool vec, float (&out)[8]) {
  if (vec) {
    uint4 w = make_uint4(0u, 0u, 0u, 0u);
    if (k < S_kv) w = __ldg(reinterpret_cast<const uint4*>(row + k));
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      out[2 * q] = __uint_as_float(ws[q] << 16);
      out[2 * q + 1] = __uint_as_float(ws[q] & 0xFFFF0000u);
    }
  } else {
    const unsigned short* r = reinterpret_cast<const unsigned short*>(row);
#pragma unroll
    for (int e = 0; e < 8; ++e) out[e] = (k + e < S_kv) ? bf16_bits_to_float(__ldg(r + k + e)) : 0.f;
  }
}

}  // namespace sdpa
