// attn_bwd_fp8.cu -- the FP8 backward of fused BSHD attention for sm_103a: E4M3 Q, K, V
// (the forward's tensors) and E5M2 dO (a gradient), the hybrid recipe of "Speed up
// attention on GPU with cuDNN and TransformerEngine", step 10.  Per (b, h) with P_ij =
// exp(scale q_i.k_j - LSE_i) of the dequantised inputs, in this order:
//   P~  = E4M3(2^8 P) / 2^8                 (the operand of the dV product)
//   dP  = dO.v,  D = dO.O (dequantised dO, the forward's bf16 O)
//   dS  = P (dP - D)                        (fp32, from the unrounded P)
//   dS~ = E5M2(s dS) / s,  s = 57344 / ds_amax  (delayed scaling; max |dS| is recorded)
//   dV  = sum_i P~ dO,  dK = scale sum_i dS~ q,  dQ = scale sum_j dS~ k
// Every product is a tcgen05.mma kind::f8f6f4 with K-major operands:
//   kv-stationary kernel (one CTA per (b, kv head, 128 keys), 64 queries per step):
//     S^T = K Q^T and dP^T = V dO^T from the natural codes; P~^T (E4M3) and dS~^T (E5M2)
//     written to TMEM, 4 per column; dV += P~^T dO and dK += dS~^T Q with dO and Q read
//     from their transposed copies [B, H_q, d, S_pad] (queries innermost);
//   query-stationary kernel (one CTA per (b, h, 128 queries), 64 keys per step):
//     S = Q K^T and dP = dO V^T from the natural codes; dS~ (E5M2) in TMEM;
//     dQ += dS~ K with K read from its transposed copy [B, H_kv, d, S_pad].
// The descales of the codes fold into the score scale, into dP and into the epilogues, and
// the two code scales into the per-row values the preprocess stores: with
//   l' = -LSE log2(e) + 8 and D' = -D s / 2^8 (s the dS scale),
// a thread forms 2^8 P = 2^(S scale log2(e) + l') (the E4M3 operand as it stands) and
// s dS = 2^8 P (dP s / 2^8 + D') (the E5M2 operand as it stands) with one fma, one ex2, one
// more fma and one multiply per element, the fmas and multiplies two lanes at a time.
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_kernels.h"
#include "ptx.cuh"

namespace sdpa {

namespace {

constexpr float kPScale = 256.f;  // P~ = E4M3(2^8 P) / 2^8: P <= 1 keeps the codes <= 256 < 448
constexpr int kF8Chunk = 8;       // (b, head) groups per chunk of the block order, as in the bf16 kernels

__device__ __forceinline__ float e5m2_scale_of(const float* amax) {
  const float a = *amax;
  return (a > 0.f && a <= 3.402823466e38f) ? __fdiv_rn(57344.f, a) : 1.f;
}

// E5M2 byte -> float: the byte is the upper half of an fp16 with the same value.
__device__ __forceinline__ float e5m2_to_float(uint32_t byte) {
  return __half2float(__ushort_as_half(static_cast<unsigned short>(byte << 8)));
}

// K-major 8-bit operand with rows of `row` bytes (64 or 128): 64- or 128-byte swizzle.
__device__ __forceinline__ uint64_t desc_rows(uint32_t saddr, int row) {
  return row == 128 ? smem_desc_sw128(saddr, 16, 1024) : smem_desc_sw64(saddr, 16, 512);
}

// Preprocess: D' = -D s / 2^8 with D = descale_do * sum_d E5M2(dO8) O (fp32) and
// l' = -LSE log2(e) + 8 into the padded [B, H_q, S_pad] rows (D' = 0, l' = -inf past S_q),
// one block per 64 rows.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_fp8_kernel(const BwdParams p) {
  constexpr int TPR = D / 8, RPP = 256 / TPR, TILE = 64, NR = TILE / RPP;
  __shared__ float dsum[TILE];
  const int i0 = blockIdx.x * TILE, h = blockIdx.y, b = blockIdx.z;
  const int sub = threadIdx.x % TPR;
  const float dsc = *p.descale_do;
  const float neg_s8 = -e5m2_scale_of(p.ds_amax) * (1.f / kPScale);  // -s / 2^8 (exact)
  uint4 a[NR];
  uint2 g[NR];
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    const int i = i0 + threadIdx.x / TPR + k * RPP;
    a[k] = make_uint4(0u, 0u, 0u, 0u);
    g[k] = make_uint2(0u, 0u);
    if (i < p.S_q) {
      const size_t off = (((size_t)b * p.S_q + i) * p.H_q + h) * D + sub * 8;
      a[k] = __ldcs(reinterpret_cast<const uint4*>(p.o + off));
      g[k] = __ldcs(reinterpret_cast<const uint2*>(p.do8 + off));
    }
  }
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    const int r = threadIdx.x / TPR + k * RPP;
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a[k]);
    const uint32_t gw[2] = {g[k].x, g[k].y};
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 fa = __bfloat1622float2(a2[e]);
      const uint32_t w = gw[e / 2] >> (16 * (e % 2));
      acc = fmaf(fa.x, e5m2_to_float(w & 0xFFu), acc);
      acc = fmaf(fa.y, e5m2_to_float((w >> 8) & 0xFFu), acc);
    }
#pragma unroll
    for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (sub == 0) dsum[r] = (acc * dsc) * neg_s8;
  }
  __syncthreads();
  if (threadIdx.x < TILE) {
    const int i = i0 + threadIdx.x;
    const size_t bh = (size_t)b * p.H_q + h;
    const bool real = i < p.S_q;
    p.Dsum[bh * p.S_pad + i] = real ? dsum[threadIdx.x] : 0.f;
    const float l = real ? p.lse[bh * p.S_q + i] : -INFINITY;
    p.nlse2[bh * p.S_pad + i] = l == -INFINITY ? -INFINITY : fmaf(-l, kLog2e, 8.f);
  }
}

// d offset_h = -sum_{b,i} exp(offset_h - LSE) D = (2^8 / s) sum_{b,i} 2^(c log2(e) + l' - 8) D',
// as in the bf16 backward (fixed order).
__global__ void __launch_bounds__(256) bwd_doffset_fp8_kernel(const BwdParams p) {
  const int h = blockIdx.x;
  const float c2 = fmaf(p.offset[h], kLog2e, -8.f);
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
    p.d_offset[h] = s * __fdiv_rn(kPScale, e5m2_scale_of(p.ds_amax));
  }
}

// The running max |dS| of a thread into *out (bit pattern max of non-negative floats).
__device__ __forceinline__ void record_amax(float m, float* out) {
  if (!out) return;
  const unsigned bits = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<unsigned*>(out), bits);
}

// =============================================================================
// kv-stationary kernel
// =============================================================================
template <int D>
struct KvF8Cfg {
  static constexpr int BN = 128, BQ = 64;
  static constexpr int K_TILE = BN * D;  // K / V codes, 128 keys x d bytes
  static constexpr int Q_TILE = BQ * D;  // Q / dO codes of a step, 64 queries x d bytes
  static constexpr int T_TILE = D * BQ;  // Q^T / dO^T of a step, d rows x 64 queries
  static constexpr int NQ = D == 128 ? 3 : 6;
  static constexpr int OFF_K = 0, OFF_V = K_TILE;
  static constexpr int OFF_Q = 2 * K_TILE;
  static constexpr int OFF_DO = OFF_Q + NQ * Q_TILE;
  static constexpr int OFF_QT = OFF_DO + NQ * Q_TILE;
  static constexpr int OFF_DOT = OFF_QT + NQ * T_TILE;
  static constexpr int OFF_L = OFF_DOT + NQ * T_TILE;  // nlse2[64] + D[64] per stage
  static constexpr int L_STAGE = 2 * BQ * 4;
  static constexpr int STAGE_TX = 2 * Q_TILE + 2 * T_TILE + L_STAGE;
  static constexpr int OFF_BAR = OFF_L + NQ * L_STAGE;
  // kv_full, q_full[NQ], q_empty[NQ], s_ready[2], dp_ready[2], p_ready[2], ds_ready[2], mma_done, dv_done[2],
  // dk_done[2]
  static constexpr int NBAR = 1 + 2 * NQ + 13;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_RAW = OFF_TMEM_SLOT + 16 + 1024;
  static constexpr int SMEM = SMEM_RAW > 117 * 1024 ? SMEM_RAW : 117 * 1024;  // one CTA per SM
  static constexpr int THREADS = 352;
  // S^T and dP^T double-buffered (slot = step & 1); P~^T and dS~^T overwrite them in place
  static constexpr int COL_S0 = 0, COL_S1 = 64, COL_DP0 = 128, COL_DV = 192, COL_DK = 192 + D, COL_DP1 = 192 + 2 * D;
  static_assert(COL_DP1 + 64 <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum KvF8Site { kF8KvFull = 0x60, kF8QFull, kF8QEmpty, kF8S, kF8DP, kF8P, kF8DS, kF8Done, kF8Drain, kF8DvDone, kF8DkDone };

template <int D>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_kv_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                           const __grid_constant__ CUtensorMap tmQT, const __grid_constant__ CUtensorMap tmDOT,
                           const BwdParams p) {
  using C = KvF8Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + C::NQ;
  uint64_t* s_ready = q_empty + C::NQ;  // [2] per slot
  uint64_t* dp_ready = s_ready + 2;     // [2]
  uint64_t* p_ready = s_ready + 4;      // [2]
  uint64_t* ds_ready = s_ready + 6;     // [2]
  uint64_t* mma_done = s_ready + 8;
  uint64_t* dv_done = s_ready + 9;      // [2]
  uint64_t* dk_done = s_ready + 11;     // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // block order of the bf16 kv kernel: (b, kv head) groups in chunks, kv tile by kv tile
  const int n_kv = (p.S_kv + C::BN - 1) / C::BN;
  const int n_gr = p.H_kv * p.B;
  const int per_chunk = kF8Chunk * n_kv;
  const int chunk = (int)blockIdx.x / per_chunk, within = (int)blockIdx.x % per_chunk;
  const int csize = min(kF8Chunk, n_gr - chunk * kF8Chunk);
  const int g = chunk * kF8Chunk + within % csize;
  const int hk = g % p.H_kv, b = g / p.H_kv;
  const int h0 = hk * p.G;
  const int n0 = (within / csize) * C::BN;
  const MaskSpec mask{p.S_q, p.S_kv, p.causal, p.window};
  int ilo = 0, ihi = -1;
  const bool any_q = q_tile_range(mask, n0, n0 + C::BN - 1, C::BQ, &ilo, &ihi);
  const int nq = any_q ? ihi - ilo + 1 : 0;
  const int nsteps = nq * p.G;

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::NQ; ++s) { mbar_init(&q_full[s], 1); mbar_init(&q_empty[s], 1); }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_ready[k], 1);
      mbar_init(&dp_ready[k], 1);
      mbar_init(&p_ready[k], 128);  // one warpgroup per slot
      mbar_init(&ds_ready[k], 128);
      mbar_init(&dv_done[k], 1);
      mbar_init(&dk_done[k], 1);
    }
    mbar_init(mma_done, 2);
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc<512>(tmem_slot);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int* err = p.err;

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0 && nsteps > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmQT);
      tma_prefetch_desc(&tmDOT);
      mbar_arrive_expect_tx(kv_full, 2 * C::K_TILE);
      tma_load_4d(smem + C::OFF_K, &tmK, kv_full, 0, hk, n0, b);
      tma_load_4d(smem + C::OFF_V, &tmV, kv_full, 0, hk, n0, b);
      for (int s = 0; s < nsteps; ++s) {
        const int st = s % C::NQ;
        if (!mbar_wait(&q_empty[st], ((s / C::NQ) & 1) ^ 1, err, kF8QEmpty)) break;
        const int h = h0 + s / nq;
        const int q0 = (ilo + s % nq) * C::BQ;
        mbar_arrive_expect_tx(&q_full[st], C::STAGE_TX);
        tma_load_4d(smem + C::OFF_Q + st * C::Q_TILE, &tmQ, &q_full[st], 0, h, q0, b);
        tma_load_4d(smem + C::OFF_DO + st * C::Q_TILE, &tmDO, &q_full[st], 0, h, q0, b);
        tma_load_4d(smem + C::OFF_QT + st * C::T_TILE, &tmQT, &q_full[st], q0, 0, h, b);
        tma_load_4d(smem + C::OFF_DOT + st * C::T_TILE, &tmDOT, &q_full[st], q0, 0, h, b);
        const size_t row = ((size_t)b * p.H_q + h) * p.S_pad + q0;
        bulk_load(smem + C::OFF_L + st * C::L_STAGE, p.nlse2 + row, C::BQ * 4, &q_full[st]);
        bulk_load(smem + C::OFF_L + st * C::L_STAGE + C::BQ * 4, p.Dsum + row, C::BQ * 4, &q_full[st]);
      }
      mbar_wait(kv_full, 0, err, kF8Drain);
      for (int s = 0; s < C::NQ && s < nsteps; ++s) {
        const int last = s + ((nsteps - 1 - s) / C::NQ) * C::NQ;
        mbar_wait(&q_full[s], (last / C::NQ) & 1, err, kF8Drain);
      }
    }
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    //   A (warp 8):  S^T(s) = K Q_s^T, dP^T(s) = V dO_s^T
    //   B (warp 10): dV += P~^T(s) dO_s, dK += dS~^T(s) Q_s
    if (nsteps > 0) {
      constexpr uint32_t idS = idesc_f8_f32(128, C::BQ, kF8E4M3, kF8E4M3);
      constexpr uint32_t idP = idesc_f8_f32(128, C::BQ, kF8E4M3, kF8E5M2);
      constexpr uint32_t idV = idesc_f8_f32(128, D, kF8E4M3, kF8E5M2);
      constexpr uint32_t idK = idesc_f8_f32(128, D, kF8E5M2, kF8E4M3);
      bool ok = mbar_wait_warp(kv_full, 0, err, kF8KvFull);
      if (warp == 8) {
        const uint64_t dK0 = desc_rows(smem_u32(smem + C::OFF_K), D);
        const uint64_t dV0 = desc_rows(smem_u32(smem + C::OFF_V), D);
        for (int s = 0; s < nsteps && ok; ++s) {
          const int st = s % C::NQ, slot = s & 1;
          ok = mbar_wait_warp(&q_full[st], (s / C::NQ) & 1, err, kF8QFull);
          if (ok && s >= 2) ok = mbar_wait_warp(&dv_done[slot], ((s >> 1) - 1) & 1, err, kF8DvDone);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dq = desc_rows(smem_u32(smem + C::OFF_Q + st * C::Q_TILE), D);
          const uint32_t colS = tmem + (slot ? C::COL_S1 : C::COL_S0);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8_warp(colS, desc_add(dK0, kk * 32), desc_add(dq, kk * 32), idS, kk > 0);
          mma_commit_warp(&s_ready[slot]);
          // dP^T(s) reuses the slot of dP^T(s - 2): dK(s - 2) must have read its dS~^T
          if (s >= 2) ok = mbar_wait_warp(&dk_done[slot], ((s >> 1) - 1) & 1, err, kF8DkDone);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ddo = desc_rows(smem_u32(smem + C::OFF_DO + st * C::Q_TILE), D);
          const uint32_t colP = tmem + (slot ? C::COL_DP1 : C::COL_DP0);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8_warp(colP, desc_add(dV0, kk * 32), desc_add(ddo, kk * 32), idP, kk > 0);
          mma_commit_warp(&dp_ready[slot]);
        }
      } else {
        for (int s = 0; s < nsteps && ok; ++s) {
          const int st = s % C::NQ, slot = s & 1;
          ok = mbar_wait_warp(&q_full[st], (s / C::NQ) & 1, err, kF8QFull) &&
               mbar_wait_warp(&p_ready[slot], (s >> 1) & 1, err, kF8P);
          if (!ok) break;
          tc_fence_after();
          const uint32_t colS = tmem + (slot ? C::COL_S1 : C::COL_S0);
          // dV += P~^T dO: A = P~^T in TMEM (queries 32 kk .. 32 kk + 31 at colS + 8 kk, 4 per
          // column), B = dO^T (d rows x 64 queries, K-major over the queries)
          const uint64_t ddot = desc_rows(smem_u32(smem + C::OFF_DOT + st * C::T_TILE), 64);
#pragma unroll
          for (int kk = 0; kk < C::BQ / 32; ++kk)
            mma_ts_f8_warp(tmem + C::COL_DV, colS + 8 * kk, desc_add(ddot, kk * 32), idV, (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit_warp(&dv_done[slot]);
          ok = mbar_wait_warp(&ds_ready[slot], (s >> 1) & 1, err, kF8DS);
          if (!ok) break;
          tc_fence_after();
          // dK += dS~^T Q: A = dS~^T in TMEM over the slot's first dP columns, B = Q^T
          const uint64_t dqt = desc_rows(smem_u32(smem + C::OFF_QT + st * C::T_TILE), 64);
          const uint32_t colP = tmem + (slot ? C::COL_DP1 : C::COL_DP0);
#pragma unroll
          for (int kk = 0; kk < C::BQ / 32; ++kk)
            mma_ts_f8_warp(tmem + C::COL_DK, colP + 8 * kk, desc_add(dqt, kk * 32), idK, (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit_warp(&dk_done[slot]);
          mma_commit_warp(&q_empty[st]);  // the stage's S / dP products completed before P~ / dS~ existed
        }
      }
      mma_commit_warp(mma_done);
      mbar_wait_warp(mma_done, 0, err, kF8Done);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ P / dS warpgroups (thread = key)
    // Ping-pong: warpgroup w takes the steps s = w, w + 2, ... (TMEM slot w), all 64 queries of
    // each, so one warpgroup computes while the other waits for its products.
    const int w = warp / 4;
    const int r = (warp % 4) * 32 + lane;
    const int key = n0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const uint32_t colS = lane_addr + (w ? C::COL_S1 : C::COL_S0);
    const uint32_t colP = lane_addr + (w ? C::COL_DP1 : C::COL_DP0);
    const float sl2 = p.scale_log2 * (*p.descale_q) * (*p.descale_k);
    const float s_ds = e5m2_scale_of(p.ds_amax);
    const float dsc = (*p.descale_do) * (*p.descale_v) * (s_ds * (1.f / kPScale));  // dP -> dP s / 2^8
    const uint64_t sl2x2 = f2_pack(sl2, sl2), dsc2 = f2_pack(dsc, dsc);
    float am[4] = {0.f, 0.f, 0.f, 0.f};  // max |s dS|, four independent chains
    bool ok = true;
    for (int s = w; s < nsteps && ok; s += 2) {
      const int st = s % C::NQ;
      const int q0 = (ilo + s % nq) * C::BQ;
      const float* l2 = reinterpret_cast<const float*>(smem + C::OFF_L + st * C::L_STAGE);
      const float* dd = l2 + C::BQ;
      const uint32_t ph = (s >> 1) & 1;
      ok = mbar_wait_warp(&s_ready[w], ph, err, kF8S);
      if (!ok) break;
      tc_fence_after();
      float pr[64];  // 2^8 P of the step's 64 queries
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(colS, ra);
        tmem_ld32(colS + 32, rb);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 la = *reinterpret_cast<const float4*>(&l2[c]);
          const float4 lb = *reinterpret_cast<const float4*>(&l2[32 + c]);
          float x[8];
          f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), sl2x2, f2_pack(la.x, la.y)),
                    x[0], x[1]);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[c + 2]), __uint_as_float(ra[c + 3])), sl2x2, f2_pack(la.z, la.w)),
                    x[2], x[3]);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])), sl2x2, f2_pack(lb.x, lb.y)),
                    x[4], x[5]);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(rb[c + 2]), __uint_as_float(rb[c + 3])), sl2x2, f2_pack(lb.z, lb.w)),
                    x[6], x[7]);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            pr[c + e] = ex2(x[e]);
            pr[32 + c + e] = ex2(x[4 + e]);
          }
        }
      }
      if (!tile_fully_visible<false>(mask, q0, C::BQ, n0, C::BN)) {
        int vlo, vhi;
        visible_rows<false>(mask, key, &vlo, &vhi);
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = (q0 + c >= vlo && q0 + c <= vhi) ? pr[c] : 0.f;
      }
      {  // P~^T: E4M3(2^8 P), 4 queries per TMEM column, over the slot's first 16 S^T columns
        uint32_t p8[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) p8[q] = pack_e4m3x4(pr[4 * q], pr[4 * q + 1], pr[4 * q + 2], pr[4 * q + 3]);
        tmem_st16(colS, p8);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&p_ready[w]);
      ok = mbar_wait_warp(&dp_ready[w], ph, err, kF8DP);
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(colP, ra);
        tmem_ld32(colP + 32, rb);
        tmem_ld_wait();
        uint32_t d8[16];  // dS~^T: E5M2(s dS), over the slot's first 16 dP^T columns
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          const float4 da = *reinterpret_cast<const float4*>(&dd[c]);
          const float4 db = *reinterpret_cast<const float4*>(&dd[32 + c]);
          float y[8];  // s dS = 2^8 P (dP s / 2^8 + D')
          const uint64_t t0 = f2_fma(f2_pack(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), dsc2, f2_pack(da.x, da.y));
          const uint64_t t1 = f2_fma(f2_pack(__uint_as_float(ra[c + 2]), __uint_as_float(ra[c + 3])), dsc2, f2_pack(da.z, da.w));
          const uint64_t t2 = f2_fma(f2_pack(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])), dsc2, f2_pack(db.x, db.y));
          const uint64_t t3 = f2_fma(f2_pack(__uint_as_float(rb[c + 2]), __uint_as_float(rb[c + 3])), dsc2, f2_pack(db.z, db.w));
          f2_unpack(f2_mul(f2_pack(pr[c], pr[c + 1]), t0), y[0], y[1]);
          f2_unpack(f2_mul(f2_pack(pr[c + 2], pr[c + 3]), t1), y[2], y[3]);
          f2_unpack(f2_mul(f2_pack(pr[32 + c], pr[33 + c]), t2), y[4], y[5]);
          f2_unpack(f2_mul(f2_pack(pr[34 + c], pr[35 + c]), t3), y[6], y[7]);
          am[0] = fmax3(am[0], fabsf(y[0]), fabsf(y[1]));
          am[1] = fmax3(am[1], fabsf(y[2]), fabsf(y[3]));
          am[2] = fmax3(am[2], fabsf(y[4]), fabsf(y[5]));
          am[3] = fmax3(am[3], fabsf(y[6]), fabsf(y[7]));
          d8[c / 4] = pack_e5m2x4(y[0], y[1], y[2], y[3]);
          d8[8 + c / 4] = pack_e5m2x4(y[4], y[5], y[6], y[7]);
        }
        tmem_st16(colP, d8);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&ds_ready[w]);
    }
    const float amax = fmaxf(fmax3(am[0], am[1], am[2]), am[3]);
    record_amax(__fdiv_rn(amax, s_ds), p.ds_amax_out);
    // ------------------------------------------------------------ epilogue: dV (w = 0), dK (w = 1)
    bool have = false;
    if (ok && nsteps > 0) {
      have = mbar_wait_warp(mma_done, 0, err, kF8Done);
      tc_fence_after();
    }
    {
      const bool row_ok = key < p.S_kv;
      const int krow = row_ok ? key : 0;
      const int col0 = w == 0 ? C::COL_DV : C::COL_DK;
      const float mul = w == 0 ? (*p.descale_do) / kPScale : p.scale * (*p.descale_q) / s_ds;
      const size_t row = ((size_t)b * p.S_kv + krow) * p.H_kv + hk;
      __nv_bfloat16* dst = (w == 0 ? p.dv : p.dk) + row * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t rr[32];
        if (have) {
          tmem_ld32(lane_addr + col0 + c0, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) rr[c] = 0u;
        }
        uint32_t pw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pw[c] = pack_bf16x2(__uint_as_float(rr[2 * c]) * mul, __uint_as_float(rr[2 * c + 1]) * mul);
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

// =============================================================================
// query-stationary dQ kernel
// =============================================================================
template <int D>
struct QF8Cfg {
  static constexpr int BM = 128, BN = 64;
  static constexpr int Q_TILE = BM * D;  // Q / dO codes, 128 rows x d bytes
  static constexpr int K_TILE = BN * D;  // K / V codes (64 keys x d bytes); K^T (d rows x 64 keys)
  static constexpr int NK = 4;
  static constexpr int OFF_Q = 0, OFF_DO = Q_TILE;
  static constexpr int OFF_K = 2 * Q_TILE;
  static constexpr int OFF_V = OFF_K + NK * K_TILE;
  static constexpr int OFF_KT = OFF_V + NK * K_TILE;
  static constexpr int OFF_BAR = OFF_KT + NK * K_TILE;
  // q_full, k_full[NK], k_empty[NK], s_ready[2], dp_ready[2], ds_ready[2], dq_done[2], mma_done
  static constexpr int NBAR = 1 + 2 * NK + 9;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_RAW = OFF_TMEM_SLOT + 16 + 1024;
  static constexpr int SMEM = SMEM_RAW > 117 * 1024 ? SMEM_RAW : 117 * 1024;
  static constexpr int THREADS = 352;
  // S and dP double-buffered (slot = kv tile & 1); dS~ overwrites the slot's first dP columns
  static constexpr int COL_S0 = 0, COL_S1 = 64, COL_DP0 = 128, COL_DP1 = 192, COL_DQ = 256;
  static_assert(COL_DQ + D <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum QF8Site { kF8QQ = 0x70, kF8QKFull, kF8QKEmpty, kF8QS, kF8QDP, kF8QDS, kF8QDone, kF8QDrain, kF8QDqDone };

template <int D>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_q_fp8_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                          const __grid_constant__ CUtensorMap tmKT, const BwdParams p) {
  using C = QF8Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* s_ready = k_empty + C::NK;  // [2] per slot
  uint64_t* dp_ready = s_ready + 2;     // [2]
  uint64_t* ds_ready = s_ready + 4;     // [2]
  uint64_t* dq_done = s_ready + 6;      // [2]
  uint64_t* mma_done = s_ready + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const int n_gr = p.H_q * p.B;
  const int per_chunk = kF8Chunk * n_qt;
  const int chunk = (int)blockIdx.x / per_chunk, within = (int)blockIdx.x % per_chunk;
  const int csize = min(kF8Chunk, n_gr - chunk * kF8Chunk);
  const int g = chunk * kF8Chunk + within % csize;
  const int qt = p.causal ? n_qt - 1 - within / csize : within / csize;
  const int h = g % p.H_q, b = g / p.H_q, hk = h / p.G;
  const int m0 = qt * C::BM;
  const MaskSpec mask{p.S_q, p.S_kv, p.causal, p.window};
  int jlo = 1, jhi = 0;
  const bool active = kv_tile_range(mask, m0, m0 + C::BM - 1, C::BN, &jlo, &jhi);
  const int nj = active ? jhi - jlo + 1 : 0;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NK; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int k = 0; k < 2; ++k) {
      mbar_init(&s_ready[k], 1);
      mbar_init(&dp_ready[k], 1);
      mbar_init(&ds_ready[k], 128);  // one warpgroup per slot
      mbar_init(&dq_done[k], 1);
    }
    mbar_init(mma_done, 2);
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc<512>(tmem_slot);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  int* err = p.err;

  if (warp == 9) {
    if (lane == 0 && nj > 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmDO);
      tma_prefetch_desc(&tmKT);
      mbar_arrive_expect_tx(q_full, 2 * C::Q_TILE);
      tma_load_4d(smem + C::OFF_Q, &tmQ, q_full, 0, h, m0, b);
      tma_load_4d(smem + C::OFF_DO, &tmDO, q_full, 0, h, m0, b);
      for (int n = 0; n < nj; ++n) {
        const int j0 = (jlo + n) * C::BN, sk = n % C::NK;
        if (!mbar_wait(&k_empty[sk], ((n / C::NK) & 1) ^ 1, err, kF8QKEmpty)) break;
        mbar_arrive_expect_tx(&k_full[sk], 3 * C::K_TILE);
        tma_load_4d(smem + C::OFF_K + sk * C::K_TILE, &tmK, &k_full[sk], 0, hk, j0, b);
        tma_load_4d(smem + C::OFF_V + sk * C::K_TILE, &tmV, &k_full[sk], 0, hk, j0, b);
        tma_load_4d(smem + C::OFF_KT + sk * C::K_TILE, &tmKT, &k_full[sk], j0, 0, hk, b);
      }
      mbar_wait(q_full, 0, err, kF8QDrain);
      for (int s = 0; s < C::NK && s < nj; ++s) {
        const int last = s + ((nj - 1 - s) / C::NK) * C::NK;
        mbar_wait(&k_full[s], (last / C::NK) & 1, err, kF8QDrain);
      }
    }
  } else if (warp == 8 || warp == 10) {
    //   A (warp 8):  S(n) = Q K_n^T and dP(n) = dO V_n^T into slot n & 1
    //   B (warp 10): dQ += dS~(n) K_n (K read as K^T, d rows x 64 keys)
    if (nj > 0) {
      constexpr uint32_t idS = idesc_f8_f32(128, C::BN, kF8E4M3, kF8E4M3);
      constexpr uint32_t idP = idesc_f8_f32(128, C::BN, kF8E5M2, kF8E4M3);
      constexpr uint32_t idQ = idesc_f8_f32(128, D, kF8E5M2, kF8E4M3);
      bool ok = mbar_wait_warp(q_full, 0, err, kF8QQ);
      if (warp == 8) {
        const uint64_t dQ0 = desc_rows(smem_u32(smem + C::OFF_Q), D);
        const uint64_t dDO0 = desc_rows(smem_u32(smem + C::OFF_DO), D);
        for (int n = 0; n < nj && ok; ++n) {
          const int sk = n % C::NK, slot = n & 1;
          ok = mbar_wait_warp(&k_full[sk], (n / C::NK) & 1, err, kF8QKFull);
          // the slot's S and dP were last used by tile n - 2, whose dQ product read its dS~
          // after the compute warps had taken S(n - 2) and dP(n - 2) into registers
          if (ok && n >= 2) ok = mbar_wait_warp(&dq_done[slot], ((n >> 1) - 1) & 1, err, kF8QDqDone);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dKa = desc_rows(smem_u32(smem + C::OFF_K + sk * C::K_TILE), D);
          const uint64_t dVa = desc_rows(smem_u32(smem + C::OFF_V + sk * C::K_TILE), D);
          const uint32_t colS = tmem + (slot ? C::COL_S1 : C::COL_S0);
          const uint32_t colP = tmem + (slot ? C::COL_DP1 : C::COL_DP0);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8_warp(colS, desc_add(dQ0, kk * 32), desc_add(dKa, kk * 32), idS, kk > 0);
          mma_commit_warp(&s_ready[slot]);
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk)
            mma_ss_f8_warp(colP, desc_add(dDO0, kk * 32), desc_add(dVa, kk * 32), idP, kk > 0);
          mma_commit_warp(&dp_ready[slot]);
        }
      } else {
        for (int n = 0; n < nj && ok; ++n) {
          const int sk = n % C::NK, slot = n & 1;
          ok = mbar_wait_warp(&k_full[sk], (n / C::NK) & 1, err, kF8QKFull) &&
               mbar_wait_warp(&ds_ready[slot], (n >> 1) & 1, err, kF8QDS);
          if (!ok) break;
          tc_fence_after();
          // dS~ of keys 32 kk .. 32 kk + 31 at the slot's dP column + 8 kk (4 keys per column)
          const uint64_t dKT = desc_rows(smem_u32(smem + C::OFF_KT + sk * C::K_TILE), 64);
          const uint32_t colP = tmem + (slot ? C::COL_DP1 : C::COL_DP0);
#pragma unroll
          for (int kk = 0; kk < C::BN / 32; ++kk)
            mma_ts_f8_warp(tmem + C::COL_DQ, colP + 8 * kk, desc_add(dKT, kk * 32), idQ, (n > 0 || kk > 0) ? 1u : 0u);
          mma_commit_warp(&dq_done[slot]);
          mma_commit_warp(&k_empty[sk]);  // S(n) / dP(n) (issuer A) completed before dS~(n) existed
        }
      }
      mma_commit_warp(mma_done);
      mbar_wait_warp(mma_done, 0, err, kF8QDone);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ dS warpgroups: thread = query row
    // Ping-pong: warpgroup w takes the kv tiles n = w, w + 2, ... (TMEM slot w), all 64 keys of each.
    const int w = warp / 4;
    const int r = (warp % 4) * 32 + lane;
    const int i = m0 + r;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const uint32_t colS = lane_addr + (w ? C::COL_S1 : C::COL_S0);
    const uint32_t colP = lane_addr + (w ? C::COL_DP1 : C::COL_DP0);
    const float sl2 = p.scale_log2 * (*p.descale_q) * (*p.descale_k);
    const float s_ds = e5m2_scale_of(p.ds_amax);
    const float dsc = (*p.descale_do) * (*p.descale_v) * (s_ds * (1.f / kPScale));  // dP -> dP s / 2^8
    float nl2row = -INFINITY, drow = 0.f;  // l' and D' of the row
    if (i < p.S_q) {
      const size_t ri = ((size_t)b * p.H_q + h) * p.S_pad + i;
      nl2row = p.nlse2[ri];
      drow = p.Dsum[ri];
    }
    const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2x2 = f2_pack(nl2row, nl2row);
    const uint64_t dsc2 = f2_pack(dsc, dsc), dr2 = f2_pack(drow, drow);
    bool ok = true;
    for (int n = w; n < nj && ok; n += 2) {
      const int k0 = (jlo + n) * C::BN;
      const uint32_t ph = (n >> 1) & 1;
      ok = mbar_wait_warp(&s_ready[w], ph, err, kF8QS);
      if (!ok) break;
      tc_fence_after();
      float pr[64];  // 2^8 P of the row's 64 keys
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(colS, ra);
        tmem_ld32(colS + 32, rb);
        tmem_ld_wait();
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          float xa, xb, xc, xd;
          f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), sl2x2, nl2x2), xa, xb);
          f2_unpack(f2_fma(f2_pack(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])), sl2x2, nl2x2), xc, xd);
          pr[c] = ex2(xa);
          pr[c + 1] = ex2(xb);
          pr[32 + c] = ex2(xc);
          pr[33 + c] = ex2(xd);
        }
      }
      if (!tile_fully_visible<false>(mask, m0, C::BM, k0, C::BN)) {
        int vlo, vhi;
        visible_keys<false>(mask, i, &vlo, &vhi);
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = (k0 + c >= vlo && k0 + c <= vhi) ? pr[c] : 0.f;
      }
      ok = mbar_wait_warp(&dp_ready[w], ph, err, kF8QDP);
      if (!ok) break;
      tc_fence_after();
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(colP, ra);
        tmem_ld32(colP + 32, rb);
        tmem_ld_wait();
        uint32_t d8[16];  // dS~: E5M2(s dS) of the row's 64 keys, 4 per TMEM column
#pragma unroll
        for (int c = 0; c < 32; c += 4) {
          float y[8];  // s dS = 2^8 P (dP s / 2^8 + D')
          f2_unpack(f2_mul(f2_pack(pr[c], pr[c + 1]),
                           f2_fma(f2_pack(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), dsc2, dr2)), y[0], y[1]);
          f2_unpack(f2_mul(f2_pack(pr[c + 2], pr[c + 3]),
                           f2_fma(f2_pack(__uint_as_float(ra[c + 2]), __uint_as_float(ra[c + 3])), dsc2, dr2)), y[2], y[3]);
          f2_unpack(f2_mul(f2_pack(pr[32 + c], pr[33 + c]),
                           f2_fma(f2_pack(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])), dsc2, dr2)), y[4], y[5]);
          f2_unpack(f2_mul(f2_pack(pr[34 + c], pr[35 + c]),
                           f2_fma(f2_pack(__uint_as_float(rb[c + 2]), __uint_as_float(rb[c + 3])), dsc2, dr2)), y[6], y[7]);
          d8[c / 4] = pack_e5m2x4(y[0], y[1], y[2], y[3]);
          d8[8 + c / 4] = pack_e5m2x4(y[4], y[5], y[6], y[7]);
        }
        tmem_st16(colP, d8);
        tmem_st_wait();
      }
      tc_fence_before();
      mbar_arrive(&ds_ready[w]);
    }
    // epilogue: dQ = scale * descale_k / s * acc; warpgroup w writes head dims [w D/2, (w+1) D/2)
    bool have = false;
    if (ok && nj > 0) {
      have = mbar_wait_warp(mma_done, 0, err, kF8QDone);
      tc_fence_after();
    }
    {
      const bool row_ok = i < p.S_q;
      const float mul = p.scale * (*p.descale_k) / s_ds;
      __nv_bfloat16* dst = p.dq + (((size_t)b * p.S_q + (row_ok ? i : 0)) * p.H_q + h) * D;
      constexpr int HALF = D / 2;
#pragma unroll 1
      for (int c0 = w * HALF; c0 < (w + 1) * HALF; c0 += 32) {
        uint32_t rr[32];
        if (have) {
          tmem_ld32(lane_addr + C::COL_DQ + c0, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) rr[c] = 0u;
        }
        uint32_t pw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pw[c] = pack_bf16x2(__uint_as_float(rr[2 * c]) * mul, __uint_as_float(rr[2 * c + 1]) * mul);
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

template <int D>
int launch_kv_fp8_t(const CUtensorMap& tq8, const CUtensorMap& tk8, const CUtensorMap& tv8, const CUtensorMap& tdo8,
                    const CUtensorMap& tqt8, const CUtensorMap& tdot8, const BwdParams& p, cudaStream_t stream) {
  using C = KvF8Cfg<D>;
  auto kern = attn_bwd_kv_fp8_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -1;
  const long long blocks = (long long)((p.S_kv + C::BN - 1) / C::BN) * p.H_kv * p.B;
  if (blocks <= 0 || blocks > 0x7fffffffLL) return -2;
  kern<<<(unsigned)blocks, C::THREADS, C::SMEM, stream>>>(tq8, tk8, tv8, tdo8, tqt8, tdot8, p);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

template <int D>
int launch_q_fp8_t(const CUtensorMap& tq8, const CUtensorMap& tk8, const CUtensorMap& tv8, const CUtensorMap& tdo8,
                   const CUtensorMap& tkt8, const BwdParams& p, cudaStream_t stream) {
  using C = QF8Cfg<D>;
  auto kern = attn_bwd_q_fp8_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -1;
  const long long blocks = (long long)((p.S_q + C::BM - 1) / C::BM) * p.H_q * p.B;
  if (blocks <= 0 || blocks > 0x7fffffffLL) return -2;
  kern<<<(unsigned)blocks, C::THREADS, C::SMEM, stream>>>(tq8, tk8, tv8, tdo8, tkt8, p);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace

int launch_bwd_preprocess_fp8(int d, const BwdParams& p, cudaStream_t stream) {
  if ((long long)p.B * p.S_q * p.H_q > 0) {
    const dim3 grid(p.S_pad / 64, p.H_q, p.B);
    if (d == 64)
      bwd_preprocess_fp8_kernel<64><<<grid, 256, 0, stream>>>(p);
    else if (d == 128)
      bwd_preprocess_fp8_kernel<128><<<grid, 256, 0, stream>>>(p);
    else
      return -2;
  }
  if (p.softmax_type == 2)
    bwd_doffset_fp8_kernel<<<p.H_q, 256, 0, stream>>>(p);
  else if (p.d_offset)
    cudaMemsetAsync(p.d_offset, 0, sizeof(float) * p.H_q, stream);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

int launch_bwd_kv_fp8(int d, const CUtensorMap& tq8, const CUtensorMap& tk8, const CUtensorMap& tv8,
                      const CUtensorMap& tdo8, const CUtensorMap& tqt8, const CUtensorMap& tdot8, const BwdParams& p,
                      cudaStream_t stream) {
  if (d == 128) return launch_kv_fp8_t<128>(tq8, tk8, tv8, tdo8, tqt8, tdot8, p, stream);
  if (d == 64) return launch_kv_fp8_t<64>(tq8, tk8, tv8, tdo8, tqt8, tdot8, p, stream);
  return -2;
}

int launch_bwd_q_fp8(int d, const CUtensorMap& tq8_128, const CUtensorMap& tk8, const CUtensorMap& tv8,
                     const CUtensorMap& tdo8_128, const CUtensorMap& tkt8, const BwdParams& p, cudaStream_t stream) {
  if (d == 128) return launch_q_fp8_t<128>(tq8_128, tk8, tv8, tdo8_128, tkt8, p, stream);
  if (d == 64) return launch_q_fp8_t<64>(tq8_128, tk8, tv8, tdo8_128, tkt8, p, stream);
  return -2;
}

}  // namespace sdpa
