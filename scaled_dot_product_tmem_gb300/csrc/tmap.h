// tmap.h -- host-side creation of TMA tensor maps (cuTensorMapEncodeTiled, fetched
// through the runtime's driver entry point so the library needs no -lcuda).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace sdpa {

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline PFN_encodeTiled get_encode_tiled() {
  static PFN_encodeTiled fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(p);
  }
  return fn;
}

// A BSHD bf16 tensor [B, S, H, D] viewed as a 4-D TMA tensor (d, h, s, b) with a
// box of 64 head-dim elements (128 bytes, one swizzle row) x 1 head x `box_rows`
// sequence rows x 1 batch, 128-byte swizzle.  Rows past S read as zeros.
inline bool make_bshd_map(CUtensorMap* m, const void* base, int B, int S, int H, int D, int box_rows) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)S * H * D * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An fp32 BSHD tensor [B, S, H, D] (D <= 256) as a 4-D TMA tensor with a box of
// D x 1 head x `box_rows` rows x 1 batch, no swizzle (used for bulk reductions).
inline bool make_f32_bshd_map(CUtensorMap* m, const void* base, int B, int S, int H, int D, int box_rows) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4, (cuuint64_t)S * H * D * 4};
  cuuint32_t box[4] = {(cuuint32_t)D, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A bf16 additive bias [Bb, Hb, S_q, S_kv] as a 4-D TMA tensor (key, query, head, batch)
// with a box of `box_keys` keys x `box_rows` query rows, no swizzle (rows of the box
// land densely in shared memory).  The row stride must be a multiple of 16 bytes:
// S_kv % 8 == 0.  Rows past S_q and keys past S_kv read as zeros.
inline bool make_bias_map(CUtensorMap* m, const void* base, int Bb, int Hb, int S_q, int S_kv, int box_rows,
                          int box_keys) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc || S_kv % 8 != 0) return false;
  cuuint64_t dims[4] = {(cuuint64_t)S_kv, (cuuint64_t)S_q, (cuuint64_t)Hb, (cuuint64_t)Bb};
  cuuint64_t strides[3] = {(cuuint64_t)S_kv * 2, (cuuint64_t)S_q * S_kv * 2, (cuuint64_t)Hb * S_q * S_kv * 2};
  cuuint32_t box[4] = {(cuuint32_t)box_keys, (cuuint32_t)box_rows, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The same bias as boxes of 64 keys (128 bytes) x 128 query rows with 128-byte swizzle:
// row r's 16-byte chunk c lands at chunk c ^ (r % 8) of its 128-byte row, so a warp that
// reads one chunk of 32 consecutive rows touches every bank once per 8 rows.
inline bool make_bias_map_sw128(CUtensorMap* m, const void* base, int Bb, int Hb, int S_q, int S_kv) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc || S_kv % 8 != 0) return false;
  cuuint64_t dims[4] = {(cuuint64_t)S_kv, (cuuint64_t)S_q, (cuuint64_t)Hb, (cuuint64_t)Bb};
  cuuint64_t strides[3] = {(cuuint64_t)S_kv * 2, (cuuint64_t)S_q * S_kv * 2, (cuuint64_t)Hb * S_q * S_kv * 2};
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// An E4M3 BSHD tensor [B, S, H, D] (D = 64 or 128 bytes per row) as a 4-D TMA
// tensor (d, h, s, b) with a box of the whole head dim x 1 head x `box_rows` rows
// x 1 batch, swizzled by the row length (128-byte or 64-byte swizzle).
inline bool make_bshd_map_e4m3(CUtensorMap* m, const void* base, int B, int S, int H, int D, int box_rows) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc || (D != 64 && D != 128)) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)D, (cuuint64_t)H * D, (cuuint64_t)S * H * D};
  cuuint32_t box[4] = {(cuuint32_t)D, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// A transposed 8-bit tensor [B, H, D, S_pad] (the sequence innermost, rows S_pad bytes
// apart) as (s, d, h, b) with a box of `box_seq` (64 or 128) positions x D rows x 1 x 1,
// swizzled by the box's row length (64- or 128-byte); positions at or past S read as zeros.
inline bool make_t_map_fp8(CUtensorMap* m, const void* base, int B, int S, int S_pad, int H, int D, int box_seq) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc || S_pad % 16 != 0 || S_pad < S || (box_seq != 64 && box_seq != 128)) return false;
  cuuint64_t dims[4] = {(cuuint64_t)S, (cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)S_pad, (cuuint64_t)D * S_pad, (cuuint64_t)H * D * S_pad};
  cuuint32_t box[4] = {(cuuint32_t)box_seq, (cuuint32_t)D, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, box_seq == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// The transposed E4M3 V of the FP8 forward: boxes of 128 keys x D rows.
inline bool make_vt_map_e4m3(CUtensorMap* m, const void* base, int B, int S, int S_pad, int H, int D) {
  return make_t_map_fp8(m, base, B, S, S_pad, H, D, 128);
}

// A row-major bf16 matrix [rows, cols] as a 2-D TMA tensor with a 64 x box_rows
// box and 128-byte swizzle.
inline bool make_2d_map(CUtensorMap* m, const void* base, int rows, int cols, int box_rows) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace sdpa
