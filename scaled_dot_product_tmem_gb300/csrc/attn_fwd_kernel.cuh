// attn_fwd_kernel.cuh -- the fused BSHD attention forward kernel for sm_103a
// (template; instantiated by attn_fwd.cu and, for dropout, attn_dropout.cu).
//
// Computes, per (batch b, query head h, kv head h / G):
//   S = scale * Q K^T, masked (causal + left window), softmax with an optional sink
//   logit c (off-by-one: c = 0; learnable: c = offset[h]), O = P V, and
//   LSE = log(e^c + sum_j e^{S_j}) per row.
// Sources: "Speed up attention on GPU with cuDNN and TransformerEngine", section
// "How attention works" and step 7 (causal); "JAX: Single-GPU Attention with
// TransformerEngine", sections 1, 2, 4 and "Other attention knobs" (GQA, sliding
// window, MLA head dims, scale_factor, sink softmax); "[JAX] Add support for sink
// attention in JAX #2225", Greptile sequence diagrams (the three denominators).
//
// A work tile is two 128-row query tiles of one (b, h); its CTA walks the kv tiles
// that either of them can see.  CTAs are persistent (one per SM), each taking every
// gridDim-th work tile, heaviest causal query blocks first, so one tile's output
// epilogue overlaps the next tile's loads and first GEMM.  Warp roles (320 threads):
//   warps 0-3 / 4-7  softmax warpgroup of query tile 0 / 1: thread r owns row r
//                    (TMEM lane r); online softmax in fp32 with the sink folded
//                    into the running max/denominator; writes bf16 P into TMEM
//                    over its own S columns; rescales O in TMEM only when the
//                    running max grows by more than 2^8 (exact: the final
//                    normalisation uses the same stale max); epilogue O/l, LSE.
//   warp 8           one thread issues tcgen05.mma: S_t = Q_t K_j^T (both from
//                    shared memory) and O_t += P_t V_j (P from TMEM, V from
//                    shared memory, MN-major).
//   warp 9           one thread issues the TMA loads: Q once, then K / V rings.
// TMEM (512 columns): S_t / P_t at t*256, O_t at t*256 + 128.
//
// E4M3 instantiation (F8): Q, K and V arrive as per-tensor-scaled E4M3 bytes (V
// transposed to [B, H_kv, d, S], keys innermost, so both GEMMs read K-major
// operands); S and P.V run as tcgen05.mma kind::f8f6f4 (K = 32 per instruction).
// The scores are rescaled by descale_q * descale_k with the softmax scale; P is
// rounded to E4M3 (values <= 2^8 under the lazy rescale, inside E4M3's range)
// while the row sum keeps the fp32 values; O is multiplied by descale_v / l.
// Source for the FP8 forward: "Speed up attention on GPU with cuDNN and
// TransformerEngine", step 10, section "Inspect the FP8 path".
//
// Bias instantiation (BIAS): each softmax thread reads its row of the bf16 bias for
// the 128 keys of a tile and forms t = s * scale * log2(e) + bias * log2(e); the
// chunk maxima are retaken over t, and the exponent is t - max.
//
// Dropout instantiation (DROP): before waiting for a tile's scores, each softmax
// thread regenerates the keep bits of its row's 128 keys (dropout.cuh); a dropped
// probability is written to TMEM as 0 for P.V while the row sum keeps it, and the
// epilogue multiplies O by 65536 / (65536 - t).
#pragma once
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_kernels.h"
#include "dropout.cuh"
#include "ptx.cuh"

namespace sdpa {

// BT: the bias tiles of the two query tiles are staged in shared memory by TMA.
template <int D_QK, int D_V, int NK, int NV, bool F8 = false, bool BT = false>
struct FwdCfg {
  static constexpr int BM = 128, BN = 128;
  // bf16: boxes of 64 head dims (one 128-byte swizzle row each); E4M3: one box of
  // the whole head dim (64 or 128 bytes per row), and V^T boxes of d rows x 128 keys
  static constexpr int QCH = F8 ? 1 : D_QK / 64, VCH = F8 ? 1 : D_V / 64;
  static constexpr int CHUNK = F8 ? 128 * D_QK : 128 * 128;
  static constexpr int Q_TILE = QCH * CHUNK;
  static constexpr int K_STAGE = QCH * CHUNK;
  static constexpr int V_STAGE = F8 ? D_V * 128 : VCH * CHUNK;
  static_assert(!F8 || (D_QK == D_V && (D_QK == 64 || D_QK == 128)), "E4M3 head dims");
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_K = OFF_Q + 2 * Q_TILE;
  static constexpr int OFF_V = OFF_K + NK * K_STAGE;
  // bias tile of one query tile: 128 rows x 128 keys bf16, as two 64-key boxes with
  // 128-byte swizzle (row r's 16-byte chunk c at chunk c ^ (r % 8) of its 128-byte row)
  static constexpr int B_BOX = 128 * 128, B_TILE = 2 * B_BOX;
  static constexpr int OFF_B = OFF_V + NV * V_STAGE;
  static constexpr int OFF_BAR = OFF_B + (BT ? 2 * B_TILE : 0);
  // q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_ready[2], p_ready[2], o_done[2], mma_done,
  // q_empty, then (BT) b_full[2], b_empty[2]
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 8 + (BT ? 4 : 0);
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_USED = OFF_TMEM_SLOT + 16 + 1024;
  // at least 117 KB so that one CTA per SM holds the 512 TMEM columns
  static constexpr int SMEM = SMEM_USED > 117 * 1024 ? SMEM_USED : 117 * 1024;
  static constexpr int THREADS = 320;
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(SMEM > 116 * 1024, "one CTA per SM keeps the 512-column TMEM allocation uncontended");
};

// One work tile: two 128-row query tiles of one (b, h).  For each query tile: does it
// exist (rows < S_q), does it see any key, and which kv tiles [jlo, jhi] it sees;
// [J0, J1] is the union.  Causal work is ordered heaviest query block first.
struct FwdTile {
  int h, b, hk, m0, J0, J1;
  int jlo[2], jhi[2];
  bool exists[2], active[2], any;
  MaskSpec mask;  // with the entry's own lengths
};

template <int BM, int BN, bool VL>
__device__ __forceinline__ FwdTile fwd_tile(const FwdParams& p, int nqb, int wi) {
  FwdTile T;
  const int hb = wi % (p.H_q * p.B);
  const int q = wi / (p.H_q * p.B);
  const int qb = p.causal ? nqb - 1 - q : q;
  T.h = hb % p.H_q;
  T.b = hb / p.H_q;
  T.hk = T.h / p.G;
  T.m0 = qb * 2 * BM;
  T.mask = VL ? MaskSpec{entry_len(p.seq_q, T.b, p.S_q), entry_len(p.seq_kv, T.b, p.S_kv), p.causal, p.window}
              : MaskSpec{p.S_q, p.S_kv, p.causal, p.window};
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = T.m0 + t * BM;
    T.exists[t] = r0 < p.S_q;  // rows of the padded tensor: they get an output either way
    T.active[t] = T.exists[t] && kv_tile_range(T.mask, r0, r0 + BM - 1, BN, &T.jlo[t], &T.jhi[t]);
    if (!T.active[t]) { T.jlo[t] = 1; T.jhi[t] = 0; }
  }
  T.any = T.active[0] || T.active[1];
  T.J0 = T.active[0] ? (T.active[1] ? min(T.jlo[0], T.jlo[1]) : T.jlo[0]) : T.jlo[1];
  T.J1 = T.active[1] ? (T.active[0] ? max(T.jhi[0], T.jhi[1]) : T.jhi[1]) : T.jhi[0];
  return T;
}

enum FwdSite { kSiteQ = 1, kSiteKFull, kSiteKEmpty, kSiteVFull, kSiteVEmpty, kSiteS, kSiteP, kSiteO, kSiteDrain,
               kSiteBFull, kSiteBEmpty };

// Bias tiles staged by TMA for head dims up to 128 (the MLA dims keep the per-row loads).
template <int D_QK, bool BIAS>
constexpr bool fwd_bias_staged() { return BIAS && D_QK <= 128; }

template <int D_QK, int D_V, int NK, int NV, bool VL, bool F8 = false, bool BIAS = false, bool DROP = false>
__global__ void __launch_bounds__(320, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmB,
                    const FwdParams p) {
  constexpr bool BT = fwd_bias_staged<D_QK, BIAS>();
  using C = FwdCfg<D_QK, D_V, NK, NV, F8, BT>;
  static_assert(!DROP || (!F8 && !BIAS && !VL), "dropout: full-length bf16 batches without a bias");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + NK;
  uint64_t* v_full = k_empty + NK;
  uint64_t* v_empty = v_full + NV;
  uint64_t* s_ready = v_empty + NV;
  uint64_t* p_ready = s_ready + 2;
  uint64_t* o_done = p_ready + 2;
  uint64_t* mma_done = o_done + 2;
  uint64_t* q_empty = mma_done + 1;
  [[maybe_unused]] uint64_t* b_full = q_empty + 1;  // [2] (BT)
  [[maybe_unused]] uint64_t* b_empty = b_full + 2;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
  // the bias tiles are staged only when the rows are whole 16-byte units (S_kv % 8 == 0)
  [[maybe_unused]] const bool b_tma = BT && p.bias_tma;

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nqb = (p.S_q + 2 * C::BM - 1) / (2 * C::BM);
  const int n_work = nqb * p.H_q * p.B;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    for (int s = 0; s < NK; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < NV; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&s_ready[t], 1);
      mbar_init(&p_ready[t], C::BM);
      mbar_init(&o_done[t], 1);
    }
    mbar_init(mma_done, 1);
    if constexpr (BT) {
      for (int t = 0; t < 2; ++t) {
        mbar_init(&b_full[t], 1);
        mbar_init(&b_empty[t], C::BM);
      }
    }
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

  // The CTA is persistent: it takes work tiles wi = blockIdx.x, blockIdx.x + gridDim.x,
  // ...; every role walks the same sequence and counts barrier phases across tiles.
  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      if (b_tma) tma_prefetch_desc(&tmB);
      int n = 0, nw = 0;  // kv stages loaded, Q tiles loaded
      [[maybe_unused]] int nb[2] = {0, 0};  // bias tiles loaded per query tile
      bool ok = true;
      for (int wi = blockIdx.x; wi < n_work && ok; wi += gridDim.x) {
        const FwdTile T = fwd_tile<C::BM, C::BN, VL>(p, nqb, wi);
        if (!T.any) continue;
        // Q of the previous tile must have been read by that tile's last S MMAs
        if (nw > 0) ok = mbar_wait(q_empty, (nw - 1) & 1, err, kSiteQ);
        if (!ok) break;
        const uint32_t qbytes = (T.active[0] ? C::Q_TILE : 0) + (T.active[1] ? C::Q_TILE : 0);
        mbar_arrive_expect_tx(q_full, qbytes);
        for (int t = 0; t < 2; ++t)
          if (T.active[t])
            for (int c = 0; c < C::QCH; ++c)
              tma_load_4d(smem + C::OFF_Q + t * C::Q_TILE + c * C::CHUNK, &tmQ, q_full, c * 64, T.h,
                          T.m0 + t * C::BM, T.b);
        ++nw;
        for (int j = T.J0; j <= T.J1 && ok; ++j, ++n) {
          const int sk = n % NK, sv = n % NV;
          ok = mbar_wait(&k_empty[sk], ((n / NK) & 1) ^ 1, err, kSiteKEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(&k_full[sk], C::K_STAGE);
          for (int c = 0; c < C::QCH; ++c)
            tma_load_4d(smem + C::OFF_K + sk * C::K_STAGE + c * C::CHUNK, &tmK, &k_full[sk], c * 64, T.hk,
                        j * C::BN, T.b);
          if constexpr (BT) {
            // each query tile's bias tile for kv tile j, once its softmax has read the last one
            // (ahead of V(j), which is only needed after that softmax); the next one is
            // prefetched into L2 meanwhile
            const int hb = p.bias_sh ? T.h : 0, bb = p.bias_sb ? T.b : 0;
#pragma unroll
            for (int t = 0; t < 2 && b_tma; ++t) {
              if (!T.active[t] || j < T.jlo[t] || j > T.jhi[t]) continue;
              ok = mbar_wait(&b_empty[t], (nb[t] & 1) ^ 1, err, kSiteBEmpty);
              if (!ok) break;
              const int r0 = T.m0 + t * C::BM;
              mbar_arrive_expect_tx(&b_full[t], C::B_TILE);
              for (int hf = 0; hf < 2; ++hf)
                tma_load_4d(smem + C::OFF_B + t * C::B_TILE + hf * C::B_BOX, &tmB, &b_full[t], j * C::BN + 64 * hf,
                            r0, hb, bb);
              if (j < T.jhi[t])
                for (int hf = 0; hf < 2; ++hf) tma_prefetch_l2_4d(&tmB, (j + 1) * C::BN + 64 * hf, r0, hb, bb);
              ++nb[t];
            }
          }
          if (!ok) break;
          ok = mbar_wait(&v_empty[sv], ((n / NV) & 1) ^ 1, err, kSiteVEmpty);
          if (!ok) break;
          mbar_arrive_expect_tx(&v_full[sv], C::V_STAGE);
          if constexpr (F8) {  // V^T: keys innermost
            tma_load_4d(smem + C::OFF_V + sv * C::V_STAGE, &tmV, &v_full[sv], j * C::BN, 0, T.hk, T.b);
          } else {
            for (int c = 0; c < C::VCH; ++c)
              tma_load_4d(smem + C::OFF_V + sv * C::V_STAGE + c * C::CHUNK, &tmV, &v_full[sv], c * 64, T.hk,
                          j * C::BN, T.b);
          }
        }
      }
      // Drain: every load issued must have landed before the CTA can exit.
      if (nw > 0) mbar_wait(q_full, (nw - 1) & 1, err, kSiteDrain);
      for (int s = 0; s < NK && s < n; ++s) {
        const int last = s + ((n - 1 - s) / NK) * NK;
        mbar_wait(&k_full[s], (last / NK) & 1, err, kSiteDrain);
      }
      for (int s = 0; s < NV && s < n; ++s) {
        const int last = s + ((n - 1 - s) / NV) * NV;
        mbar_wait(&v_full[s], (last / NV) & 1, err, kSiteDrain);
      }
      if constexpr (BT)
        for (int t = 0; t < 2; ++t)
          if (nb[t] > 0) mbar_wait(&b_full[t], (nb[t] - 1) & 1, err, kSiteDrain);
    }
  } else if (warp == 8) {
    // ------------------------------------------------------------ MMA issuer
    // One warp issues for both query tiles in the order PV_0(j), S_0(j+1),
    // PV_1(j), S_1(j+1): each tile's softmax overlaps the other tile's GEMMs.  The
    // first S of the next work tile follows the last PV of this one, so it runs
    // while the softmax warps write this tile's output.
    constexpr uint32_t idS = F8 ? idesc_e4m3_f32(128, 128) : idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idO = F8 ? idesc_e4m3_f32(128, D_V) : idesc_bf16_f32(128, D_V, false, true);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q);
    const uint32_t sK = smem_u32(smem + C::OFF_K);
    const uint32_t sV = smem_u32(smem + C::OFF_V);
    auto issue_S = [&](int t, int stage) {
      if constexpr (F8) {
        // rows of D_QK bytes: 128-byte swizzle for d = 128, 64-byte for d = 64
        const uint64_t dq = D_QK == 128 ? smem_desc_sw128(sQ + t * C::Q_TILE, 16, 1024)
                                        : smem_desc_sw64(sQ + t * C::Q_TILE, 16, 512);
        const uint64_t dk = D_QK == 128 ? smem_desc_sw128(sK + stage * C::K_STAGE, 16, 1024)
                                        : smem_desc_sw64(sK + stage * C::K_STAGE, 16, 512);
#pragma unroll
        for (int kk = 0; kk < D_QK / 32; ++kk)
          mma_ss_f8_warp(tmem + t * 256, desc_add(dq, kk * 32), desc_add(dk, kk * 32), idS, kk > 0);
      } else {
        const uint64_t dq = smem_desc_sw128(sQ + t * C::Q_TILE, 16, 1024);
        const uint64_t dk = smem_desc_sw128(sK + stage * C::K_STAGE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < D_QK / 16; ++kk) {
          const uint32_t off = (kk / 4) * C::CHUNK + (kk % 4) * 32;
          mma_ss_warp(tmem + t * 256, desc_add(dq, off), desc_add(dk, off), idS, kk > 0);
        }
      }
    };
    auto issue_PV = [&](int t, int stage, bool acc) {
      if constexpr (F8) {
        // P: 4 E4M3 per TMEM column (32 keys = 8 columns per MMA); V^T: K-major rows of
        // 128 keys
        const uint64_t dv = smem_desc_sw128(sV + stage * C::V_STAGE, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BN / 32; ++kk)
          mma_ts_f8_warp(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, desc_add(dv, kk * 32), idO,
                         (acc || kk > 0) ? 1u : 0u);
      } else {
        const uint64_t dv = smem_desc_sw128(sV + stage * C::V_STAGE, C::CHUNK, 1024);
#pragma unroll
        for (int kk = 0; kk < C::BN / 16; ++kk)
          mma_ts_warp(tmem + t * 256 + 128, tmem + t * 256 + kk * 8, desc_add(dv, kk * 2048), idO,
                      (acc || kk > 0) ? 1u : 0u);
      }
    };
    int n = 0, nw = 0;      // kv stages consumed, Q tiles consumed
    int pc[2] = {0, 0};     // p_ready phases consumed per query tile
    bool ok = true, issued = false;
    for (int wi = blockIdx.x; wi < n_work && ok; wi += gridDim.x) {
      const FwdTile T = fwd_tile<C::BM, C::BN, VL>(p, nqb, wi);
      if (!T.any) continue;
      issued = true;
      ok = mbar_wait_warp(q_full, nw & 1, err, kSiteQ);
      ++nw;
      if (ok) ok = mbar_wait_warp(&k_full[n % NK], (n / NK) & 1, err, kSiteKFull);
      if (!ok) break;
      tc_fence_after();
#pragma unroll
      for (int t = 0; t < 2; ++t)
        if (T.active[t] && T.jlo[t] == T.J0) {
          issue_S(t, n % NK);
          mma_commit_warp(&s_ready[t]);
        }
      mma_commit_warp(&k_empty[n % NK]);
      if (T.J0 == T.J1) mma_commit_warp(q_empty);  // every S of the tile is issued
      for (int j = T.J0; j <= T.J1 && ok; ++j, ++n) {
        const bool need_k = j + 1 <= T.J1;
        ok = mbar_wait_warp(&v_full[n % NV], (n / NV) & 1, err, kSiteVFull);
        if (ok && need_k) ok = mbar_wait_warp(&k_full[(n + 1) % NK], ((n + 1) / NK) & 1, err, kSiteKFull);
        if (!ok) break;
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (ok && T.active[t] && j >= T.jlo[t] && j <= T.jhi[t]) {
            ok = mbar_wait_warp(&p_ready[t], pc[t] & 1, err, kSiteP);
            ++pc[t];
            if (ok) {
              tc_fence_after();
              issue_PV(t, n % NV, j > T.jlo[t]);
              if (j == T.jhi[t]) mma_commit_warp(&o_done[t]);
            }
          }
          if (ok && T.active[t] && j + 1 >= T.jlo[t] && j + 1 <= T.jhi[t]) {
            issue_S(t, (n + 1) % NK);
            mma_commit_warp(&s_ready[t]);
          }
        }
        if (!ok) break;
        mma_commit_warp(&v_empty[n % NV]);
        if (need_k) mma_commit_warp(&k_empty[(n + 1) % NK]);
        if (j + 1 == T.J1) mma_commit_warp(q_empty);  // the tile's last S MMAs were just issued
      }
    }
    // Every MMA must be complete before TMEM is released.
    if (issued) {
      mma_commit_warp(mma_done);
      mbar_wait_warp(mma_done, 0, err, kSiteDrain);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ softmax + epilogue
    const int t = warp / 4;
    const int r = (warp % 4) * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const uint32_t colS = t * 256, colO = t * 256 + 128;
    // E4M3: the MMA sums products of the stored codes; the per-tensor descales
    // bring the scores and O back to the real values
    const float sl2 = F8 ? p.scale_log2 * (*p.descale_q) * (*p.descale_k) : p.scale_log2;
    const float o_mul = F8 ? *p.descale_v : (DROP ? p.drop_scale : 1.f);
    [[maybe_unused]] DropState drop{};
    if constexpr (DROP) drop = DropState{p.rng[0], p.rng[1], p.drop_t};
    // with a bias the scores become s + bias / scale before the max; the max and the
    // exponent then scale them by scale log2(e) as without one
    const float sx = sl2;
    const bool bias_vec = BIAS && (p.S_kv % 8 == 0);
    int sc = 0, od = 0;  // s_ready / o_done phases consumed
    [[maybe_unused]] int nbc = 0;  // bias tiles consumed (BT)
    [[maybe_unused]] const uint8_t* btile = smem + C::OFF_B + t * C::B_TILE + r * 128;  // this row, first box
    bool ok = true;
    for (int wi = blockIdx.x; wi < n_work && ok; wi += gridDim.x) {
      const FwdTile T = fwd_tile<C::BM, C::BN, VL>(p, nqb, wi);
      // this warpgroup's query tile, selected without a run-time index into T (which
      // would move T to local memory)
      const bool my_exists = t ? T.exists[1] : T.exists[0];
      if (!my_exists) continue;
      const int m0 = T.m0, h = T.h, b = T.b;
      const MaskSpec mask = T.mask;
      const bool my_active = t ? T.active[1] : T.active[0];
      const int my_jlo = t ? T.jlo[1] : T.jlo[0], my_jhi = t ? T.jhi[1] : T.jhi[0];
      const int i = m0 + t * C::BM + r;  // query row
      const __nv_bfloat16* brow = nullptr;  // this row of the bias (rows past S_q read row S_q - 1)
      if constexpr (BIAS) brow = p.bias + b * p.bias_sb + h * p.bias_sh + (size_t)min(i, p.S_q - 1) * p.S_kv;
      // running max (in scaled log2 units) and denominator; the sink starts them
      float m_run = -INFINITY, l = 0.f;
      if (p.softmax_type == 1) { m_run = 0.f; l = 1.f; }
      if (p.softmax_type == 2) { m_run = p.offset[h] * kLog2e; l = 1.f; }
      if (my_active) {
        for (int j = my_jlo; j <= my_jhi; ++j) {
          const int it = j - my_jlo;
          // dropout: this row's keep bits of the tile's 128 keys (bit c of keep[q]: key
          // 128 j + 32 q + c), generated while the tile's scores are still being computed
          [[maybe_unused]] uint32_t keep[4] = {0u, 0u, 0u, 0u};
          if constexpr (DROP) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
              keep[q] = dropout_row_span16(drop, b, h, i, j * C::BN + 32 * q) |
                        (dropout_row_span16(drop, b, h, i, j * C::BN + 32 * q + 16) << 16);
          }
          if (BIAS && !b_tma) {
            // this row's bias for the next kv tile (and, on the first, this one) into L2
            // while the scores are computed, so the loads below do not wait on DRAM
            for (int jj = (it == 0 ? j : j + 1); jj <= min(j + 1, my_jhi); ++jj) {
              const int ka = jj * C::BN, kz = min(ka + C::BN, p.S_kv) - 1;
              prefetch_l2(brow + ka);
              prefetch_l2(brow + min(ka + 64, kz));
              prefetch_l2(brow + kz);
            }
          }
          ok = mbar_wait_warp(&s_ready[t], sc & 1, err, kSiteS);
          ++sc;
          if (!ok) break;
          tc_fence_after();
          // The whole 128-key row in one batch of TMEM loads, one wait; each load also
          // yields the max of its 32 columns.  Where a 32-key chunk is only partly visible
          // to this row, the chunk's max is retaken over its visible keys after masking.
          float s[128], cmax[4];
          {
            uint32_t rr[128];
#pragma unroll
            for (int c0 = 0; c0 < 128; c0 += 32)
              tmem_ld32_max(lane_addr + colS + c0, *reinterpret_cast<uint32_t(*)[32]>(&rr[c0]), cmax[c0 / 32]);
            tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(rr[c]);
          }
          const int k0 = j * C::BN;
          if constexpr (BT) {
            if (b_tma) {
              ok = mbar_wait_warp(&b_full[t], nbc & 1, err, kSiteBFull);
              ++nbc;
              if (!ok) break;
            }
          }
          if constexpr (BIAS) {
            const float rsc = kLog2e / sl2;  // 1 / scale
            const uint64_t rs2 = f2_pack(rsc, rsc);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              float m = -INFINITY;
#pragma unroll
              for (int e8 = 0; e8 < 4; ++e8) {
                float bv[8];
                if (b_tma) {  // chunk (32 q + 8 e8) / 8 of the row: box q / 2, chunk 4 (q % 2) + e8 of 8
                  const uint4 w = *reinterpret_cast<const uint4*>(
                      btile + (q / 2) * C::B_BOX + (((4 * (q % 2) + e8) ^ (r & 7)) << 4));
                  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                  for (int u = 0; u < 4; ++u) {
                    bv[2 * u] = __uint_as_float(ws[u] << 16);
                    bv[2 * u + 1] = __uint_as_float(ws[u] & 0xFFFF0000u);
                  }
                } else {
                  load_bias8(brow, k0 + 32 * q + 8 * e8, p.S_kv, bias_vec, bv);
                }
                // y = s + bias / scale (so y scale log2(e) = s scale log2(e) + bias log2(e)),
                // two keys per paired fma
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                  float* x = &s[32 * q + 8 * e8 + e];
                  f2_unpack(f2_fma(f2_pack(bv[e], bv[e + 1]), rs2, f2_pack(x[0], x[1])), x[0], x[1]);
                  m = fmax3(m, x[0], x[1]);
                }
              }
              cmax[q] = m;
            }
            if (b_tma) mbar_arrive(&b_empty[t]);  // the tile's bias is in registers
          }
          if (!tile_fully_visible<VL>(mask, m0 + t * C::BM, C::BM, k0, C::BN)) {
            // the keys this row sees form one interval [vlo, vhi], so a chunk whose two
            // ends are inside it is fully visible
            int vlo, vhi;
            visible_keys<VL>(mask, i, &vlo, &vhi);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int c0 = k0 + 32 * q;
              if (c0 >= vlo && c0 + 31 <= vhi) continue;
              float m = -INFINITY;
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                if (c0 + c < vlo || c0 + c > vhi) s[32 * q + c] = -INFINITY;
                m = fmaxf(m, s[32 * q + c]);
              }
              cmax[q] = m;
            }
          }
          const float mx = fmax3(cmax[0], cmax[1], fmaxf(cmax[2], cmax[3]));
          const float m_tile = mx * sx;
          // Lazy rescale, decided per warp (the TMEM loads/stores are warp-collective):
          // when any row's max grew by more than 2^8, every row of the warp moves to
          // its new max (alpha = 1 for rows whose max did not change).
          if (__any_sync(0xffffffffu, m_tile > m_run + 8.f)) {
            const float m_new = fmaxf(m_run, m_tile);
            const float alpha = (m_new == m_run) ? 1.f : ex2(m_run - m_new);
            l *= alpha;
            if (it > 0) {
#pragma unroll 1
              for (int c0 = 0; c0 < D_V; c0 += 16) {
                uint32_t rr[16];
                tmem_ld16(lane_addr + colO + c0, rr);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 16; ++c) rr[c] = __float_as_uint(__uint_as_float(rr[c]) * alpha);
                tmem_st16(lane_addr + colO + c0, rr);
              }
            }
            m_run = m_new;
          }
          const float m_sub = (m_run == -INFINITY) ? 0.f : m_run;
          // p = 2^(s * scale * log2e - m), paired: one f32x2 FMA per two keys; the row sum
          // is kept in four paired partial sums so no long add chain forms
          const uint64_t sl2x2 = f2_pack(sx, sx), negm2 = f2_pack(-m_sub, -m_sub);
          uint64_t ls2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int c0 = 0; c0 < 128; c0 += 32) {
            uint32_t pk[16];
            float pf[32];
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              float xa, xb;
              f2_unpack(f2_fma(f2_pack(s[c0 + 2 * c], s[c0 + 2 * c + 1]), sl2x2, negm2), xa, xb);
              const float a = ex2(xa), bq = ex2(xb);
              ls2[c % 4] = f2_add(ls2[c % 4], f2_pack(a, bq));
              if constexpr (F8) {
                pf[2 * c] = a;
                pf[2 * c + 1] = bq;
              } else if constexpr (DROP) {  // the row sum keeps a dropped value; P.V does not
                const uint32_t kb = keep[c0 / 32] >> (2 * c);
                pk[c] = pack_bf16x2((kb & 1u) ? a : 0.f, (kb & 2u) ? bq : 0.f);
              } else {
                pk[c] = pack_bf16x2(a, bq);
              }
            }
            if constexpr (F8) {
              uint32_t p8[8];
#pragma unroll
              for (int q = 0; q < 8; ++q) p8[q] = pack_e4m3x4(pf[4 * q], pf[4 * q + 1], pf[4 * q + 2], pf[4 * q + 3]);
              tmem_st8(lane_addr + colS + c0 / 4, p8);
            } else {
              tmem_st16(lane_addr + colS + c0 / 2, pk);
            }
          }
          {
            float s0, s1, s2, s3, s4, s5, s6, s7;
            f2_unpack(ls2[0], s0, s1);
            f2_unpack(ls2[1], s2, s3);
            f2_unpack(ls2[2], s4, s5);
            f2_unpack(ls2[3], s6, s7);
            l += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
          }
          tmem_st_wait();
          tc_fence_before();
          mbar_arrive(&p_ready[t]);
        }
      }
      // ------------------------------------------------------------ epilogue
      bool have_o = false;
      if (my_active && ok) {  // warp-uniform
        have_o = mbar_wait_warp(&o_done[t], od & 1, err, kSiteO);
        ++od;
        tc_fence_after();
      }
      const bool row_ok = i < p.S_q;
      const float inv = l > 0.f ? o_mul / l : 0.f;
      __nv_bfloat16* orow = p.o + (((size_t)b * p.S_q + (row_ok ? i : 0)) * p.H_q + h) * D_V;
#pragma unroll 1
      for (int c0 = 0; c0 < D_V; c0 += 32) {
        uint32_t rr[32];
        if (have_o) {  // all lanes load; only rows < S_q store
          tmem_ld32(lane_addr + colO + c0, rr);
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) rr[c] = 0u;
        }
        uint32_t pw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          pw[c] = pack_bf16x2(__uint_as_float(rr[2 * c]) * inv, __uint_as_float(rr[2 * c + 1]) * inv);
        if (row_ok) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
        }
      }
      if (row_ok) {
        const float m_sub = (m_run == -INFINITY) ? 0.f : m_run;
        p.lse[((size_t)b * p.H_q + h) * p.S_q + i] = l > 0.f ? (m_sub + lg2(l)) * kLn2 : -INFINITY;
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

template <int D_QK, int D_V, int NK, int NV, bool VL, bool F8 = false, bool BIAS = false, bool DROP = false>
inline int launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const FwdParams& p,
                        cudaStream_t stream, const CUtensorMap* tb = nullptr) {
  using C = FwdCfg<D_QK, D_V, NK, NV, F8, fwd_bias_staged<D_QK, BIAS>()>;
  auto kern = attn_fwd_kernel<D_QK, D_V, NK, NV, VL, F8, BIAS, DROP>;
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -1;
    attr_set = true;
  }
  // persistent: one CTA per SM (at most one work tile per CTA when there are fewer)
  static int n_sm = 0;
  if (n_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
      return -1;
  }
  const long long n_work = (long long)((p.S_q + 2 * C::BM - 1) / (2 * C::BM)) * p.H_q * p.B;
  const unsigned grid = (unsigned)(n_work < n_sm ? n_work : n_sm);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tb ? *tb : tq, p);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sdpa
