// attn_bwd_kernels.cuh -- the kv-stationary and query-stationary backward kernels
// of fused BSHD attention for sm_103a (templates; instantiated by attn_bwd.cu and,
// for dropout, attn_dropout.cu).
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
#pragma once
#include <cuda_runtime.h>

#include "attn_common.cuh"
#include "attn_kernels.h"
#include "dropout.cuh"
#include "ptx.cuh"

namespace sdpa {

// =============================================================================
// kv-stationary main kernel
// =============================================================================
template <int D_QK, int D_V, bool FUSE_DQ, bool BIAS = false>
struct KvCfg {
  static constexpr int BN = 128;  // keys per CTA (TMEM lanes)
  static constexpr int BQ = 64;   // query rows per step
  static constexpr int QCH = D_QK / 64, VCH = D_V / 64;
  static constexpr int KCHUNK = 128 * 128;  // 128 rows x 128 bytes
  static constexpr int QCHUNK = 64 * 128;   // 64 rows x 128 bytes
  // Q/dO stages; with a bias each stage also holds the step's bias tile, so there are fewer
  static constexpr int NQ = !BIAS ? ((D_QK == 64 && D_V == 64) ? 6 : 3)
                                  : ((D_QK == 64 && D_V == 64) ? 4 : ((FUSE_DQ || D_QK == 192) ? 2 : 3));
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + QCH * KCHUNK;
  static constexpr int OFF_DS = OFF_V + VCH * KCHUNK;  // 2 x dS^T [128 keys x 64 q] bf16, swizzled
  static constexpr int DS_BUF = 128 * 128;
  static constexpr int DS_BYTES = FUSE_DQ ? 2 * DS_BUF : 0;
  static constexpr int OFF_Q = OFF_DS + DS_BYTES;
  static constexpr int Q_STAGE = QCH * QCHUNK;
  static constexpr int OFF_DO = OFF_Q + NQ * Q_STAGE;
  static constexpr int DO_STAGE = VCH * QCHUNK;
  static constexpr int OFF_L = OFF_DO + NQ * DO_STAGE;  // nlse2[64] + D[64] per stage
  static constexpr int L_STAGE = 2 * BQ * 4;
  static constexpr int OFF_B = OFF_L + NQ * L_STAGE;    // bias tile [64 q][128 keys] bf16 per stage
  static constexpr int B_STAGE = BIAS ? BQ * BN * 2 : 0;
  static constexpr int OFF_DQS = OFF_B + NQ * B_STAGE;  // fp32 dQ tile [64 q][d_qk] staged for the TMA reduce
  static constexpr int DQS_BYTES = FUSE_DQ ? BQ * D_QK * 4 : 0;
  static constexpr int OFF_BAR = OFF_DQS + DQS_BYTES;
  // kv_full, q_full[NQ], q_empty[NQ], s_ready[2], dp_ready, p_ready[2], ds_ready, dq_ready, dq_free,
  // mma_done, dv_done[2], dk_done, kv_empty, acc_free, fin, tile_full[2], tile_empty[2].  Barriers
  // of the double-buffered S slot are per slot: with two slots the P/dS warps can finish step
  // s+1's P before issuer B has waited for step s's, and a single barrier would then complete
  // two phases before B looks.  The tile index ring (two ints) sits beside the TMEM address.
  static constexpr int NBAR = 1 + 2 * NQ + 19;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TMEM_SLOT + 16 + 1024;
  static constexpr int MMA_B_WARP = FUSE_DQ ? 14 : 10;  // second MMA issuer
  static constexpr int THREADS = FUSE_DQ ? 480 : 352;
  // TMEM columns
  // S^T/P^T is double-buffered (slots COL_S0 / COL_S1, step s uses slot s & 1) so the
  // next step's scores can be computed while the current P^T still feeds dV.
  static constexpr int COL_S0 = 0, COL_DP = 64, COL_DV = 128, COL_DK = 128 + D_V, COL_DQ = 128 + D_V + D_QK;
  static constexpr int COL_S1 = COL_DQ + (FUSE_DQ ? 64 : 0);
  static_assert(COL_S1 + 64 <= 512, "TMEM budget");
  // dQ^T = K^T dS^T is issued with M = 128 head-dim rows; with d_qk = 64 its rows 64-127
  // read the next 64 columns of shared memory (the V tile) and are never drained.
  static_assert(!FUSE_DQ || D_QK == 128 || D_QK == 64, "fused dQ for d_qk in {64, 128}");
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(SMEM > 116 * 1024, "one CTA per SM");
};

constexpr int kKvChunk = 8;  // (b, kv head) groups per chunk of the kv kernel's block order

enum KvSite { kKvFull = 0x20, kKvQFull, kKvQEmpty, kKvS, kKvDP, kKvP, kKvDS, kKvDQReady, kKvDQFree, kKvDone, kKvDrain,
              kKvDvDone, kKvDkDone, kKvEmpty, kKvAccFree, kKvTile };

// PERSIST: the CTAs take tiles from a counter in global memory until it runs out; otherwise
// the grid has one CTA per tile and the tile loops below run once (the cross-tile barriers
// compile away).
template <int D_QK, int D_V, bool FUSE_DQ, bool VL, bool BIAS = false, bool DROP = false, bool PERSIST = false>
__global__ void __launch_bounds__(FUSE_DQ ? 480 : 352, 1)
    attn_bwd_kv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                       const __grid_constant__ CUtensorMap tmDQ, const __grid_constant__ CUtensorMap tmB,
                       const BwdParams p) {
  using C = KvCfg<D_QK, D_V, FUSE_DQ, BIAS>;
  static_assert(!DROP || (!BIAS && !VL), "dropout: full-length batches without a bias");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + C::NQ;
  uint64_t* s_ready = q_empty + C::NQ;  // [2], per S slot
  uint64_t* dp_ready = s_ready + 2;
  uint64_t* p_ready = s_ready + 3;      // [2], per S slot
  uint64_t* ds_ready = s_ready + 5;
  uint64_t* dq_ready = s_ready + 6;
  uint64_t* dq_free = s_ready + 7;
  uint64_t* mma_done = s_ready + 8;
  uint64_t* dv_done = s_ready + 9;      // [2], per S slot
  uint64_t* dk_done = s_ready + 11;
  uint64_t* kv_empty = s_ready + 12;    // a tile's K/V readers are done: the next K/V may load
  uint64_t* acc_free = s_ready + 13;    // the epilogue has read dV/dK: the next tile may overwrite them
  uint64_t* fin = s_ready + 14;         // every MMA issued, before TMEM is released
  uint64_t* tile_full = s_ready + 15;   // [2] PERSIST: the producer has published the next tile
  uint64_t* tile_empty = s_ready + 17;  // [2] PERSIST: every role has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_TMEM_SLOT + 8);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Work tiles: (b, kv head, head split) groups in chunks of kKvChunk; within a chunk,
  // kv tile by kv tile (tile 0, the most work when causal, first) and group by group,
  // so a chunk's long tiles start early while its queries stay few enough to be shared
  // in L2.  With a bias broadcast over the batch, b is the innermost group index: the
  // batch entries of one (kv head, kv tile) then run side by side, in step, and their
  // reductions into the same dbias lines meet in L2.  Persistent CTAs (PERSIST, at most one per SM) take the tiles in that order
  // from a counter, as an SM would take blocks, so a tile's K/V load and first products
  // overlap the previous tile's epilogue; the producer takes each index and publishes
  // it to the other roles through a two-slot ring.  Every role walks the same tiles and
  // numbers the steps of all its tiles in one sequence g, which indexes the stages,
  // slots and barrier phases.
  const int n_kv = (p.S_kv + C::BN - 1) / C::BN;
  const int n_gr = p.H_kv * p.B * p.ns;  // group = (b, kv head, head split)
  const int n_tiles = n_kv * n_gr;
  const int per_chunk = kKvChunk * n_kv;
  const int Gs = p.G / p.ns;  // query heads a tile walks
  struct Tile {
    int b, hk, split, h0, n0, ilo, nq, nsteps;
    MaskSpec mask;
  };
  auto tile_of = [&](int ti) {
    Tile t;
    const int chunk = ti / per_chunk, within = ti % per_chunk;
    const int csize = min(kKvChunk, n_gr - chunk * kKvChunk);
    const int g = chunk * kKvChunk + within % csize;
    if (BIAS && p.bias_sb == 0) {
      t.b = g % p.B;
      t.split = (g / p.B) % p.ns;
      t.hk = g / (p.B * p.ns);
    } else {
      t.split = g % p.ns;
      t.hk = (g / p.ns) % p.H_kv;
      t.b = g / (p.ns * p.H_kv);
    }
    t.h0 = t.hk * p.G + t.split * Gs;  // the first query head the tile walks
    t.n0 = (within / csize) * C::BN;
    t.mask = VL ? MaskSpec{entry_len(p.seq_q, t.b, p.S_q), entry_len(p.seq_kv, t.b, p.S_kv), p.causal, p.window}
                : MaskSpec{p.S_q, p.S_kv, p.causal, p.window};
    int ihi = -1;
    t.ilo = 0;
    const bool any_q = q_tile_range(t.mask, t.n0, t.n0 + C::BN - 1, C::BQ, &t.ilo, &ihi);
    t.nq = any_q ? ihi - t.ilo + 1 : 0;
    t.nsteps = t.nq * Gs;
    return t;
  };
  // Tile k of this CTA for the roles other than the producer: without PERSIST the CTA's
  // own tile, then none; with it, slot k % 2 of the ring once the producer has published
  // it.  whole_warp: the warp waits together and its lane 0 arrives for it.
  auto take_tile = [&](int k, bool whole_warp) -> int {
    if constexpr (!PERSIST) {
      return k == 0 ? (int)blockIdx.x : n_tiles;
    } else {
      const int slot = k & 1;
      if (!mbar_wait_warp(&tile_full[slot], (k >> 1) & 1, p.err, kKvTile)) return n_tiles;
      const int ti = ring[slot];
      if (whole_warp) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&tile_empty[slot]);
      } else {
        mbar_arrive(&tile_empty[slot]);
      }
      return ti;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::NQ; ++s) { mbar_init(&q_full[s], 1); mbar_init(&q_empty[s], 1); }
    mbar_init(&s_ready[0], 1);
    mbar_init(&s_ready[1], 1);
    mbar_init(dp_ready, 1);
    mbar_init(&p_ready[0], 256);
    mbar_init(&p_ready[1], 256);
    mbar_init(ds_ready, 256);
    mbar_init(dq_ready, 1);
    mbar_init(dq_free, 128);
    mbar_init(mma_done, 1);  // issuer B, once per tile: it alone writes the dV/dK sums
    mbar_init(&dv_done[0], 1);
    mbar_init(&dv_done[1], 1);
    mbar_init(dk_done, 1);
    mbar_init(kv_empty, FUSE_DQ ? 2 : 1);  // issuer A (S, dP) and, with the fused dQ, issuer B (K^T dS^T)
    mbar_init(acc_free, 256);
    mbar_init(fin, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tile_full[i], 1);
      mbar_init(&tile_empty[i], 2 + 256 + (FUSE_DQ ? 128 : 0));  // the two issuers (one lane each), P/dS and drain threads
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

  if (warp == 9) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const bool btma = BIAS && p.bias_tma;  // each stage also brings the step's bias tile
      bool ok = true, first = true;
      int g0 = 0, ne = 0;  // steps and non-empty tiles so far
      int ti_next = 0;     // PERSIST: the tile taken for the next iteration
      for (int k = 0;; ++k) {
        int ti;
        if constexpr (PERSIST) {  // publish tile k in ring slot k % 2 once every role has read tile k - 2
          const int slot = k & 1;
          if (k >= 2 && !mbar_wait(&tile_empty[slot], ((k >> 1) - 1) & 1, err, kKvTile)) break;
          ti = k == 0 ? atomicAdd(p.tile_counter, 1) : ti_next;
          ring[slot] = ti;
          mbar_arrive(&tile_full[slot]);
        } else {
          ti = k == 0 ? (int)blockIdx.x : n_tiles;
        }
        if (ti >= n_tiles || !ok) break;
        const Tile t = tile_of(ti);
        if (t.nsteps == 0) {
          if constexpr (PERSIST) ti_next = atomicAdd(p.tile_counter, 1);
          continue;
        }
        if (first) {
          tma_prefetch_desc(&tmQ);
          tma_prefetch_desc(&tmK);
          tma_prefetch_desc(&tmV);
          tma_prefetch_desc(&tmDO);
          if (btma) tma_prefetch_desc(&tmB);
          first = false;
        }
        // K/V of this tile replace the previous tile's once its S, dP (and dQ^T) products are done
        if (PERSIST && ne > 0 && !mbar_wait(kv_empty, (ne - 1) & 1, err, kKvEmpty)) break;
        mbar_arrive_expect_tx(kv_full, (C::QCH + C::VCH) * C::KCHUNK);
        for (int c = 0; c < C::QCH; ++c)
          tma_load_4d(smem + C::OFF_K + c * C::KCHUNK, &tmK, kv_full, c * 64, t.hk, t.n0, t.b);
        for (int c = 0; c < C::VCH; ++c)
          tma_load_4d(smem + C::OFF_V + c * C::KCHUNK, &tmV, kv_full, c * 64, t.hk, t.n0, t.b);
        for (int s = 0; s < t.nsteps; ++s) {
          const int g = g0 + s, st = g % C::NQ;
          if (!mbar_wait(&q_empty[st], ((g / C::NQ) & 1) ^ 1, err, kKvQEmpty)) {
            ok = false;
            break;
          }
          const int h = t.h0 + s / t.nq;
          const int q0 = (t.ilo + s % t.nq) * C::BQ;
          mbar_arrive_expect_tx(&q_full[st], C::Q_STAGE + C::DO_STAGE + C::L_STAGE + (btma ? C::B_STAGE : 0));
          if (btma)  // rows past S_q and keys past S_kv come in as zeros
            tma_load_4d(smem + C::OFF_B + st * C::B_STAGE, &tmB, &q_full[st], t.n0, q0, p.bias_sh ? h : 0,
                        p.bias_sb ? t.b : 0);
          for (int c = 0; c < C::QCH; ++c)
            tma_load_4d(smem + C::OFF_Q + st * C::Q_STAGE + c * C::QCHUNK, &tmQ, &q_full[st], c * 64, h, q0, t.b);
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(smem + C::OFF_DO + st * C::DO_STAGE + c * C::QCHUNK, &tmDO, &q_full[st], c * 64, h, q0,
                        t.b);
          const size_t row = ((size_t)t.b * p.H_q + h) * p.S_pad + q0;
          bulk_load(smem + C::OFF_L + st * C::L_STAGE, p.nlse2 + row, C::BQ * 4, &q_full[st]);
          bulk_load(smem + C::OFF_L + st * C::L_STAGE + C::BQ * 4, p.Dsum + row, C::BQ * 4, &q_full[st]);
        }
        // the next tile is taken once this one's loads are issued: late enough that the
        // counter still balances the last tiles, early enough to hide the atomic
        if constexpr (PERSIST) ti_next = atomicAdd(p.tile_counter, 1);
        g0 += t.nsteps;
        ++ne;
      }
      // every copy this warp started must land before the CTA may exit
      if (ne > 0) mbar_wait(kv_full, (ne - 1) & 1, err, kKvDrain);
      for (int st = 0; st < C::NQ && st < g0; ++st) {
        const int last = st + ((g0 - 1 - st) / C::NQ) * C::NQ;
        mbar_wait(&q_full[st], (last / C::NQ) & 1, err, kKvDrain);
      }
    }
  } else if (warp == 8 || warp == C::MMA_B_WARP) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing warps, because one cannot issue tcgen05.mma fast enough to
    // keep the tensor core busy with these 64-wide tiles:
    //   A (warp 8):  S^T(g) = K Q_g^T, dP^T(g) = V dO_g^T
    //   B:           dV += P^T(g) dO_g, dK += dS^T(g) Q_g, [dQ^T(g) = K^T dS^T(g)]
    // MMAs of different warps are not ordered, so A waits for B's dv_done
    // before S(g) overwrites the columns that held P(g-1), and for B's dk_done(g-1)
    // before dP(g) overwrites the columns that held dS(g-1).  Across tiles, B's first
    // dV and dK of a tile wait for the epilogue to have read the previous tile's sums.
    constexpr uint32_t idS = idesc_bf16_f32(128, C::BQ, false, false);
    constexpr uint32_t idDV = idesc_bf16_f32(128, D_V, false, true);
    constexpr uint32_t idDK = idesc_bf16_f32(128, D_QK, false, true);
    constexpr uint32_t idDQ = idesc_bf16_f32(128, C::BQ, true, true);
    const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
    const uint32_t sDS = smem_u32(smem + C::OFF_DS);
    bool ok = true;
    int g0 = 0, ne = 0;
    for (int k = 0;; ++k) {  // whole warp; elect.sync picks the lane
      const int ti = take_tile(k, true);
      if (ti >= n_tiles || !ok) break;
      const Tile t = tile_of(ti);
      if (t.nsteps == 0) continue;
      // K/V of the tile: read by A's products and, with the fused dQ, by B's K^T dS^T.  Only
      // the warps that read them wait (a wait nothing gates could see a later phase complete).
      if (warp == 8 || FUSE_DQ) ok = mbar_wait_warp(kv_full, ne & 1, err, kKvFull);
      if (warp == 8) {
        const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024);  // K as K-major A of S^T
        const uint64_t dV0 = smem_desc_sw128(sV, 16, 1024);  // V as K-major A of dP^T
        for (int s = 0; s < t.nsteps && ok; ++s) {
          const int g = g0 + s, st = g % C::NQ, slot = g & 1;
          ok = mbar_wait_warp(&q_full[st], (g / C::NQ) & 1, err, kKvQFull);
          // slot reuse: P^T(g-2) in this slot must have been read by dV(g-2)
          if (ok && g >= 2) ok = mbar_wait_warp(&dv_done[slot], ((g >> 1) - 1) & 1, err, kKvDvDone);
          if (!ok) break;
          tc_fence_after();
          const uint64_t dq = smem_desc_sw128(sQ + st * C::Q_STAGE, 16, 1024);
          const uint32_t colS = tmem + (slot ? C::COL_S1 : C::COL_S0);
#pragma unroll
          for (int kk = 0; kk < D_QK / 16; ++kk)
            mma_ss_warp(colS, desc_add(dK0, (kk / 4) * C::KCHUNK + (kk % 4) * 32),
                        desc_add(dq, (kk / 4) * C::QCHUNK + (kk % 4) * 32), idS, kk > 0);
          mma_commit_warp(&s_ready[slot]);
          if (g > 0) ok = mbar_wait_warp(dk_done, (g - 1) & 1, err, kKvDkDone);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ddo = smem_desc_sw128(sDO + st * C::DO_STAGE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D_V / 16; ++kk)
            mma_ss_warp(tmem + C::COL_DP, desc_add(dV0, (kk / 4) * C::KCHUNK + (kk % 4) * 32),
                        desc_add(ddo, (kk / 4) * C::QCHUNK + (kk % 4) * 32), idS, kk > 0);
          mma_commit_warp(dp_ready);
        }
        if constexpr (PERSIST) mma_commit_warp(kv_empty);  // the tile's S and dP products have read K and V
      } else {
        const uint64_t dKt0 = smem_desc_sw128(sK, C::KCHUNK, 1024);   // K as MN-major A of dQ^T
        const uint64_t dDS0 = smem_desc_sw128(sDS, C::KCHUNK, 1024);  // dS^T as MN-major B of dQ^T
        for (int s = 0; s < t.nsteps && ok; ++s) {
          const int g = g0 + s, st = g % C::NQ, slot = g & 1;
          const uint64_t ddo_mn = smem_desc_sw128(sDO + st * C::DO_STAGE, C::QCHUNK, 1024);  // dO, MN-major B of dV
          const uint64_t dq_mn = smem_desc_sw128(sQ + st * C::Q_STAGE, C::QCHUNK, 1024);     // Q, MN-major B of dK
          ok = mbar_wait_warp(&q_full[st], (g / C::NQ) & 1, err, kKvQFull) &&
               mbar_wait_warp(&p_ready[slot], (g >> 1) & 1, err, kKvP);
          // the first dV of a tile overwrites the sums the previous tile's epilogue reads
          if (PERSIST && ok && s == 0 && ne > 0) ok = mbar_wait_warp(acc_free, (ne - 1) & 1, err, kKvAccFree);
          if (!ok) break;
          tc_fence_after();
          const uint32_t colS = tmem + (slot ? C::COL_S1 : C::COL_S0);
          // dV += P^T dO   (P^T bf16 in the slot: q 0-31 at cols 0-15, q 32-63 at cols 32-47)
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            mma_ts_warp(tmem + C::COL_DV, colS + (kk / 2) * 32 + (kk % 2) * 8, desc_add(ddo_mn, kk * 2048), idDV,
                        (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit_warp(&dv_done[slot]);
          ok = mbar_wait_warp(ds_ready, g & 1, err, kKvDS);
          if (!ok) break;
          tc_fence_after();
          // dK += dS^T Q
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            mma_ts_warp(tmem + C::COL_DK, tmem + C::COL_DP + (kk / 2) * 32 + (kk % 2) * 8,
                        desc_add(dq_mn, kk * 2048), idDK, (s > 0 || kk > 0) ? 1u : 0u);
          // dS^T(g) in TMEM is consumed once dK(g) completes: issuer A may write dP(g+1).
          // (dQ^T reads dS^T from shared memory, double-buffered, so it does not gate dP.)
          mma_commit_warp(dk_done);
          if constexpr (FUSE_DQ) {
            ok = mbar_wait_warp(dq_free, (g & 1) ^ 1, err, kKvDQFree);
            if (!ok) break;
            tc_fence_after();
            // dQ^T = K^T dS^T: A = K (MN-major, M = d), B = dS^T from shared memory (MN-major, N = q)
            const uint64_t dDS = desc_add(dDS0, slot * C::DS_BUF);
#pragma unroll
            for (int kk = 0; kk < C::BN / 16; ++kk)
              mma_ss_warp(tmem + C::COL_DQ, desc_add(dKt0, kk * 2048), desc_add(dDS, kk * 2048), idDQ, kk > 0);
            mma_commit_warp(dq_ready);
          }
          // The stage's S/dP MMAs (issuer A) completed before P(g)/dS(g) existed.
          mma_commit_warp(&q_empty[st]);
        }
        if constexpr (FUSE_DQ && PERSIST) mma_commit_warp(kv_empty);  // the tile's dQ^T products have read K
      }
      // The tile's dV/dK sums are complete once B's MMAs are; B alone writes them.  (With
      // both issuers arriving, A could finish the next tile's products first and complete
      // the phase early.)
      if (warp == C::MMA_B_WARP) mma_commit_warp(mma_done);
      g0 += t.nsteps;
      ++ne;
    }
    // Every MMA of both issuers must be complete before TMEM is released.
    mma_commit_warp(fin);
    mbar_wait_warp(fin, 0, err, kKvDone);
  } else if (warp < 8) {
    // ------------------------------------------------------------ P / dS warpgroups
    const int w = warp / 4;  // which 32 query columns of the 64
    const int r = (warp % 4) * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const float sl2 = p.scale_log2;
    [[maybe_unused]] DropState drop{};
    if constexpr (DROP) drop = DropState{p.rng[0], p.rng[1], p.drop_t};
    bool ok = true;
    int g0 = 0, ne = 0;
    for (int k = 0;; ++k) {
      const int ti = take_tile(k, false);
      if (ti >= n_tiles) break;
      const Tile t = tile_of(ti);
      const int key = t.n0 + r;
      // bias: this thread's key column of the bias plane (keys past S_kv read key 0; their P is 0)
      [[maybe_unused]] const int bkey = key < p.S_kv ? key : 0;
      for (int s = 0; s < t.nsteps && ok; ++s) {
        const int g = g0 + s, st = g % C::NQ;
        const int q0 = (t.ilo + s % t.nq) * C::BQ;
        [[maybe_unused]] const long long bplane = BIAS ? t.b * p.bias_sb + (t.h0 + s / t.nq) * p.bias_sh : 0;
        const float* l2 = reinterpret_cast<const float*>(smem + C::OFF_L + st * C::L_STAGE) + 32 * w;
        const float* dd = l2 + C::BQ;
        const int slot = g & 1;
        const uint32_t colS = slot ? C::COL_S1 : C::COL_S0;
        // dropout: keep bits of this key for the step's 32 query rows (bit c: row q0 + 32 w + c),
        // generated while the step's scores are still being computed
        [[maybe_unused]] uint32_t keep = 0u;
        if constexpr (DROP)
          keep = dropout_key_span16(drop, t.b, t.h0 + s / t.nq, key, q0 + 32 * w) |
                 (dropout_key_span16(drop, t.b, t.h0 + s / t.nq, key, q0 + 32 * w + 16) << 16);
        ok = mbar_wait_warp(&s_ready[slot], (g >> 1) & 1, err, kKvS);
        if (!ok) break;
        tc_fence_after();
        float pr[32];
        {
          uint32_t rr[32];
          tmem_ld32(lane_addr + colS + 32 * w, rr);
          float lv[32];  // -LSE * log2(e) of the 32 queries
#pragma unroll
          for (int c = 0; c < 32; c += 4) *reinterpret_cast<float4*>(&lv[c]) = *reinterpret_cast<const float4*>(&l2[c]);
          if constexpr (BIAS) {  // + bias * log2(e) (queries past S_q read 0; their P is 0)
            if (p.bias_tma) {  // this thread's key column of the staged tile [64 q][128 keys]
              const unsigned short* bt =
                  reinterpret_cast<const unsigned short*>(smem + C::OFF_B + st * C::B_STAGE) + 32 * w * C::BN + r;
#pragma unroll
              for (int c = 0; c < 32; ++c) lv[c] = fmaf(bf16_bits_to_float(bt[c * C::BN]), kLog2e, lv[c]);
            } else {
              const unsigned short* bcol = reinterpret_cast<const unsigned short*>(p.bias + bplane) + bkey;
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                const int qq = q0 + 32 * w + c;
                const float bv = qq < p.S_q ? bf16_bits_to_float(__ldg(bcol + (size_t)qq * p.S_kv)) : 0.f;
                lv[c] = fmaf(bv, kLog2e, lv[c]);
              }
            }
          }
          tmem_ld_wait();
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float xa, xb;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[c]), __uint_as_float(rr[c + 1])), sl2x2,
                             f2_pack(lv[c], lv[c + 1])),
                      xa, xb);
            pr[c] = ex2(xa);
            pr[c + 1] = ex2(xb);
          }
        }
        if (!tile_fully_visible<VL>(t.mask, q0, C::BQ, t.n0, C::BN)) {
          int vlo, vhi;  // the query rows that see this thread's key
          visible_rows<VL>(t.mask, key, &vlo, &vhi);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int qq = q0 + 32 * w + c;
            pr[c] = (qq >= vlo && qq <= vhi) ? pr[c] : 0.f;
          }
        }
        {
          uint32_t pk[16];  // P^T for dV: dropped entries are 0 (the 1/(1-p) scale is in dV's epilogue)
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if constexpr (DROP)
              pk[c] = pack_bf16x2(((keep >> (2 * c)) & 1u) ? pr[2 * c] : 0.f,
                                  ((keep >> (2 * c)) & 2u) ? pr[2 * c + 1] : 0.f);
            else
              pk[c] = pack_bf16x2(pr[2 * c], pr[2 * c + 1]);
          }
          tmem_st16(lane_addr + colS + 32 * w, pk);
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&p_ready[slot]);
        ok = mbar_wait_warp(dp_ready, g & 1, err, kKvDP);
        if (!ok) break;
        tc_fence_after();
        uint32_t dsk[16];
        {
          uint32_t rr[32];
          tmem_ld32(lane_addr + C::COL_DP + 32 * w, rr);
          float dv4[32];
#pragma unroll
          for (int c = 0; c < 32; c += 4) *reinterpret_cast<float4*>(&dv4[c]) = *reinterpret_cast<const float4*>(&dd[c]);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            // dS = P (dP - D), paired; with dropout dS = P (M dP - D), M = 0 or 1/(1-p)
            float a, bq;
            if constexpr (DROP) {
              const float za = ((keep >> (2 * c)) & 1u) ? p.drop_scale : 0.f;
              const float zb = ((keep >> (2 * c)) & 2u) ? p.drop_scale : 0.f;
              f2_unpack(f2_mul(f2_pack(pr[2 * c], pr[2 * c + 1]),
                               f2_fma(f2_pack(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1])),
                                      f2_pack(za, zb), f2_pack(-dv4[2 * c], -dv4[2 * c + 1]))),
                        a, bq);
            } else {
              f2_unpack(f2_mul(f2_pack(pr[2 * c], pr[2 * c + 1]),
                               f2_sub(f2_pack(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1])),
                                      f2_pack(dv4[2 * c], dv4[2 * c + 1]))),
                        a, bq);
            }
            dsk[c] = pack_bf16x2(a, bq);
            if constexpr (BIAS) {  // dbias = dS, summed with fp32 atomics over the (b, h) sharing it
              if (p.dbias && key < p.S_kv) {
                const int qq = q0 + 32 * w + 2 * c;
                float* dcol = p.dbias + bplane + key;
                if (qq < p.S_q) atomicAdd(dcol + (size_t)qq * p.S_kv, a);
                if (qq + 1 < p.S_q) atomicAdd(dcol + (size_t)(qq + 1) * p.S_kv, bq);
              }
            }
          }
        }
        tmem_st16(lane_addr + C::COL_DP + 32 * w, dsk);
        if constexpr (FUSE_DQ) {
          // dS^T row r, query columns 32w..32w+31 -> 16-byte chunks 4w..4w+3 (128-byte swizzle)
          uint8_t* rowp = smem + C::OFF_DS + slot * C::DS_BUF + r * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int chunk = (4 * w + k) ^ (r & 7);
            *reinterpret_cast<uint4*>(rowp + chunk * 16) =
                make_uint4(dsk[4 * k], dsk[4 * k + 1], dsk[4 * k + 2], dsk[4 * k + 3]);
          }
          fence_proxy_async_smem();
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_ready);
      }
      // ---------------------------------------------------------- epilogue: dV (w = 0), dK (w = 1)
      // A tile no query sees (nsteps = 0) writes zero rows and touches neither TMEM nor a barrier.
      bool have = false;
      if (ok && t.nsteps > 0) {
        have = mbar_wait_warp(mma_done, ne & 1, err, kKvDone);
        tc_fence_after();
      }
      {
        const bool row_ok = key < p.S_kv;  // all lanes load TMEM; only real keys store
        const int krow = row_ok ? key : 0;
        const int ncols = w == 0 ? D_V : D_QK;
        const int col0 = w == 0 ? C::COL_DV : C::COL_DK;
        const float mul = w == 0 ? (DROP ? p.drop_scale : 1.f) : p.scale;
        const size_t row = ((size_t)t.b * p.S_kv + krow) * p.H_kv + t.hk;
        __nv_bfloat16* dst = w == 0 ? p.dv + row * D_V : p.dk + row * D_QK;
        // with head splits this tile's sum is one fp32 partial slice
        float* part = p.ns == 1 ? nullptr
                                : (w == 0 ? p.dv_part + ((size_t)t.split * p.B * p.S_kv * p.H_kv + row) * D_V
                                          : p.dk_part + ((size_t)t.split * p.B * p.S_kv * p.H_kv + row) * D_QK);
#pragma unroll 1
        for (int c0 = 0; c0 < ncols; c0 += 32) {
          uint32_t rr[32];
          if (have) {
            tmem_ld32(lane_addr + col0 + c0, rr);
            tmem_ld_wait();
          } else {
#pragma unroll
            for (int c = 0; c < 32; ++c) rr[c] = 0u;
          }
          if (part) {
            if (row_ok) {
              float4* f4 = reinterpret_cast<float4*>(part + c0);
#pragma unroll
              for (int q = 0; q < 8; ++q)
                f4[q] = make_float4(__uint_as_float(rr[4 * q]) * mul, __uint_as_float(rr[4 * q + 1]) * mul,
                                    __uint_as_float(rr[4 * q + 2]) * mul, __uint_as_float(rr[4 * q + 3]) * mul);
            }
            continue;
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
      if (t.nsteps > 0) {
        // the sums are in registers or stored: issuer B may start the next tile's dV and dK
        if constexpr (PERSIST) {
          tc_fence_before();
          mbar_arrive(acc_free);
        }
        g0 += t.nsteps;
        ++ne;
      }
    }
  } else if (FUSE_DQ && warp >= 10 && warp < 14) {
    // ------------------------------------------------------------ dQ drain: TMEM lane = head-dim index d
    // dQ^T of each step goes TMEM -> registers -> shared memory as [q][d] fp32, and
    // one thread adds the whole 64 x d_qk tile into the fp32 accumulator with a
    // TMA bulk reduction (rows past S_q are skipped by the TMA unit).
    const int d = (warp % 4) * 32 + lane;
    const int tid_d = threadIdx.x - 320;  // 0..127 over the four drain warps
    const uint32_t lane_addr = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    float* stage = reinterpret_cast<float*>(smem + C::OFF_DQS);
    if (tid_d == 0) tma_prefetch_desc(&tmDQ);
    bool ok = true;
    int g0 = 0;
    for (int k = 0;; ++k) {
      const int ti = take_tile(k, false);
      if (ti >= n_tiles || !ok) break;
      const Tile t = tile_of(ti);
      for (int s = 0; s < t.nsteps; ++s) {
        const int g = g0 + s;
        const bool got = mbar_wait(dq_ready, g & 1, err, kKvDQReady);
        ok = bar_red_and(1, 128, got);  // uniform over the 128 drain threads
        if (!ok) break;
        tc_fence_after();
        const int h = t.h0 + s / t.nq;
        const int q0 = (t.ilo + s % t.nq) * C::BQ;
        uint32_t ra[32], rb[32];
        tmem_ld32(lane_addr + C::COL_DQ, ra);
        tmem_ld32(lane_addr + C::COL_DQ + 32, rb);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(dq_free);  // the TMEM columns may be overwritten now
        if (tid_d == 0) bulk_wait_read_all();  // previous tile has left shared memory
        named_bar_sync(1, 128);
        if (d < D_QK) {  // lanes past d_qk hold the unused rows of the M = 128 product
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            stage[c * D_QK + d] = __uint_as_float(ra[c]);
            stage[(32 + c) * D_QK + d] = __uint_as_float(rb[c]);
          }
        }
        fence_proxy_async_smem();
        named_bar_sync(1, 128);
        if (tid_d == 0) {
          tma_reduce_add_4d(&tmDQ, stage, 0, h, q0, t.b);
          bulk_commit_group();
        }
      }
      g0 += t.nsteps;
    }
    if (tid_d == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 8) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc<512>(tmem);
  }
}

// Which instantiation family a launcher picks: the plain kernels (full-length or
// padded batches), the bias ones (full-length or padded), or the dropout ones
// (full-length).  Each family is instantiated by its own translation unit.
enum class KernVariant { kPlain, kBias, kDrop };

template <int D_QK, int D_V, bool FUSE, KernVariant KV = KernVariant::kPlain>
inline int launch_kv_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                       const CUtensorMap& tdq, const CUtensorMap& tb, const BwdParams& p, cudaStream_t stream) {
  using C = KvCfg<D_QK, D_V, FUSE, KV == KernVariant::kBias>;
  const bool vl = p.seq_q || p.seq_kv;  // padded batches: per-entry lengths and row tests
  decltype(&attn_bwd_kv_kernel<D_QK, D_V, FUSE, false>) kern;
  if constexpr (KV == KernVariant::kDrop) {  // dropout: full-length batches without a bias
    if (vl || p.bias) return -2;
    kern = attn_bwd_kv_kernel<D_QK, D_V, FUSE, false, false, true>;
  } else if constexpr (KV == KernVariant::kBias) {
    if (!p.bias) return -2;
    kern = vl ? attn_bwd_kv_kernel<D_QK, D_V, FUSE, true, true> : attn_bwd_kv_kernel<D_QK, D_V, FUSE, false, true>;
  }
  const long long tiles = (long long)((p.S_kv + C::BN - 1) / C::BN) * p.H_kv * p.B * p.ns;
  if (tiles <= 0 || tiles > 0x7fffffffLL) return -2;
  // The plain fused-dQ kernels of full-length batches with d_qk = d_v run persistent
  // CTAs, one per SM, when there are more tiles than SMs and every tile is short (at most
  // 32 steps): a CTA's fixed costs (TMEM allocation, the K/V load, the first products, the
  // dK/dV epilogue) are then a large share of a tile, and persistent CTAs overlap them
  // with the neighbouring tiles' work; the tile counter hands out tiles in the
  // heaviest-first order as SMs free up, as the hardware does with blocks.  With longer
  // tiles the persistent kernel measured about 4 % slower, so those keep one CTA per tile.
  static int n_sm = 0;
  if (n_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
      return -1;
  }
  bool persist = false;
  if constexpr (KV == KernVariant::kPlain) {
    if (p.bias) return -2;
    const long long max_steps = (long long)(p.G / p.ns) * ((p.S_q + C::BQ - 1) / C::BQ);
    if constexpr (D_QK == D_V && FUSE) persist = !vl && p.tile_counter && tiles > n_sm && max_steps <= 32;
    if (persist) {
      if constexpr (D_QK == D_V && FUSE) kern = attn_bwd_kv_kernel<D_QK, D_V, FUSE, false, false, false, true>;
    } else {
      kern = vl ? attn_bwd_kv_kernel<D_QK, D_V, FUSE, true> : attn_bwd_kv_kernel<D_QK, D_V, FUSE, false>;
    }
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -1;
  const unsigned grid = (unsigned)(persist ? n_sm : tiles);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, tdq, tb, p);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

// =============================================================================
// query-stationary deterministic dQ kernel
// =============================================================================
template <int D_QK, int D_V>
struct QCfg {
  static constexpr int BM = 128, BN = 128;
  static constexpr int QCH = D_QK / 64, VCH = D_V / 64;
  static constexpr int CHUNK = 128 * 128;
  static constexpr int NK = 2;
  static constexpr int NV = (D_QK == 192 && D_V == 128) ? 1 : 2;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + QCH * CHUNK;
  static constexpr int OFF_K = OFF_DO + VCH * CHUNK;
  static constexpr int OFF_V = OFF_K + NK * QCH * CHUNK;
  static constexpr int OFF_BAR = OFF_V + NV * VCH * CHUNK;
  // dP^T slots: two where TMEM has room beside dQ (d_qk <= 128), so that dP(n+1) runs
  // while dS(n) is formed and dQ(n) reads it; one at d_qk = 192
  static constexpr int DPB = D_QK <= 128 ? 2 : 1;
  // q_full, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV], s_ready, dp_ready[DPB],
  // ds_ready[DPB], mma_done, s_free, dq_done[DPB], qo_empty, acc_free, fin, tile_full[2],
  // tile_empty[2]; the tile index ring (two ints) sits beside the TMEM address
  static constexpr int NBAR = 1 + 2 * NK + 2 * NV + 3 + 3 * DPB + 7;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_RAW = OFF_TMEM_SLOT + 16 + 1024;
  static constexpr int SMEM = SMEM_RAW > 117 * 1024 ? SMEM_RAW : 117 * 1024;  // one CTA per SM
  static constexpr int THREADS = 352;
  // dS (bf16) is written over the dP columns, so the next S can be computed as soon
  // as the dS warps have loaded the current S.  Tile n uses dP slot n % DPB.
  static constexpr int COL_S = 0, COL_DP = 128, COL_DQ = 256, COL_DP1 = COL_DQ + D_QK;
  static_assert(COL_DQ + D_QK + (DPB - 1) * 128 <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum QSite { kQQ = 0x40, kQKFull, kQKEmpty, kQVFull, kQVEmpty, kQS, kQDP, kQDS, kQDone, kQDrain, kQSFree, kQDqDone,
             kQQEmpty, kQAccFree, kQTile };

// PERSIST: the CTAs (one per SM) take tiles from a counter in global memory, as the
// persistent kv kernels do; otherwise the grid has one CTA per tile and the tile loops
// run once (the cross-tile barriers compile away).
template <int D_QK, int D_V, bool VL, bool BIAS = false, bool DROP = false, bool PERSIST = false>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                      const BwdParams p) {
  using C = QCfg<D_QK, D_V>;
  static_assert(!DROP || (!BIAS && !VL), "dropout: full-length batches without a bias");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + C::NK;
  uint64_t* v_full = k_empty + C::NK;
  uint64_t* v_empty = v_full + C::NV;
  uint64_t* s_ready = v_empty + C::NV;
  uint64_t* dp_ready = s_ready + 1;         // [DPB], per dP slot
  uint64_t* ds_ready = dp_ready + C::DPB;   // [DPB]
  uint64_t* mma_done = ds_ready + C::DPB;
  uint64_t* s_free = mma_done + 1;
  uint64_t* dq_done = s_free + 1;           // [DPB]
  uint64_t* qo_empty = dq_done + C::DPB;    // a tile's Q/dO readers are done: the next Q/dO may load
  uint64_t* acc_free = qo_empty + 1;        // the epilogue has read dQ: the next tile may overwrite it
  uint64_t* fin = acc_free + 1;             // every MMA issued, before TMEM is released
  uint64_t* tile_full = fin + 1;            // [2] PERSIST: the producer has published the next tile
  uint64_t* tile_empty = tile_full + 2;     // [2] PERSIST: every role has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_TMEM_SLOT + 8);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Tiles in the kv kernel's order: (b, head) groups in chunks of kKvChunk (heads of a
  // chunk share K and V in L2), within a chunk query tile by query tile, the tile with
  // the most kv tiles (the last one when causal) first.  Every role walks the same tiles
  // and numbers the kv tiles of all of them in one sequence n (stages, barrier phases).
  const int n_qt = (p.S_q + C::BM - 1) / C::BM;
  const int n_gr = p.H_q * p.B;
  const int n_tiles = n_qt * n_gr;
  const int per_chunk = kKvChunk * n_qt;
  struct Tile {
    int b, h, hk, m0, jlo, nj;
    MaskSpec mask;
  };
  auto tile_of = [&](int ti) {
    Tile t;
    const int chunk = ti / per_chunk, within = ti % per_chunk;
    const int csize = min(kKvChunk, n_gr - chunk * kKvChunk);
    const int g = chunk * kKvChunk + within % csize;
    const int qt = p.causal ? n_qt - 1 - within / csize : within / csize;
    t.h = g % p.H_q;
    t.b = g / p.H_q;
    t.hk = t.h / p.G;
    t.m0 = qt * C::BM;
    t.mask = VL ? MaskSpec{entry_len(p.seq_q, t.b, p.S_q), entry_len(p.seq_kv, t.b, p.S_kv), p.causal, p.window}
                : MaskSpec{p.S_q, p.S_kv, p.causal, p.window};
    int jhi = 0;
    t.jlo = 1;
    const bool active = kv_tile_range(t.mask, t.m0, t.m0 + C::BM - 1, C::BN, &t.jlo, &jhi);
    t.nj = active ? jhi - t.jlo + 1 : 0;
    return t;
  };
  // Tile k of this CTA for the roles other than the producer (see the fused-dQ kv kernel).
  auto take_tile = [&](int k, bool whole_warp) -> int {
    if constexpr (!PERSIST) {
      return k == 0 ? (int)blockIdx.x : n_tiles;
    } else {
      const int slot = k & 1;
      if (!mbar_wait_warp(&tile_full[slot], (k >> 1) & 1, p.err, kQTile)) return n_tiles;
      const int ti = ring[slot];
      if (whole_warp) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) mbar_arrive(&tile_empty[slot]);
      } else {
        mbar_arrive(&tile_empty[slot]);
      }
      return ti;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::NK; ++s) { mbar_init(&k_full[s], 1); mbar_init(&k_empty[s], 1); }
    for (int s = 0; s < C::NV; ++s) { mbar_init(&v_full[s], 1); mbar_init(&v_empty[s], 1); }
    mbar_init(s_ready, 1);
    for (int d = 0; d < C::DPB; ++d) {
      mbar_init(&dp_ready[d], 1);
      mbar_init(&ds_ready[d], 256);
      mbar_init(&dq_done[d], 1);
    }
    mbar_init(mma_done, 1);  // issuer B, once per tile: it alone writes the dQ sum
    mbar_init(s_free, 256);
    mbar_init(qo_empty, 1);   // issuer A's S and dP read Q and dO
    mbar_init(acc_free, 256);
    mbar_init(fin, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tile_full[i], 1);
      mbar_init(&tile_empty[i], 2 + 256);  // the two issuers (one lane each) and the dS threads
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

  if (warp == 9) {
    if (lane == 0) {
      bool ok = true, first = true;
      int n0 = 0, ne = 0, ti_next = 0;  // kv tiles and non-empty tiles so far
      for (int k = 0;; ++k) {
        int ti;
        if constexpr (PERSIST) {  // publish tile k once every role has read tile k - 2
          const int slot = k & 1;
          if (k >= 2 && !mbar_wait(&tile_empty[slot], ((k >> 1) - 1) & 1, err, kQTile)) break;
          ti = k == 0 ? atomicAdd(p.tile_counter_q, 1) : ti_next;
          ring[slot] = ti;
          mbar_arrive(&tile_full[slot]);
        } else {
          ti = k == 0 ? (int)blockIdx.x : n_tiles;
        }
        if (ti >= n_tiles || !ok) break;
        const Tile t = tile_of(ti);
        if (t.nj == 0) {
          if constexpr (PERSIST) ti_next = atomicAdd(p.tile_counter_q, 1);
          continue;
        }
        if (first) {
          tma_prefetch_desc(&tmQ);
          tma_prefetch_desc(&tmK);
          tma_prefetch_desc(&tmV);
          tma_prefetch_desc(&tmDO);
          first = false;
        }
        // Q/dO of this tile replace the previous tile's once its S and dP products are done
        if (PERSIST && ne > 0 && !mbar_wait(qo_empty, (ne - 1) & 1, err, kQQEmpty)) break;
        mbar_arrive_expect_tx(q_full, (C::QCH + C::VCH) * C::CHUNK);
        for (int c = 0; c < C::QCH; ++c)
          tma_load_4d(smem + C::OFF_Q + c * C::CHUNK, &tmQ, q_full, c * 64, t.h, t.m0, t.b);
        for (int c = 0; c < C::VCH; ++c)
          tma_load_4d(smem + C::OFF_DO + c * C::CHUNK, &tmDO, q_full, c * 64, t.h, t.m0, t.b);
        for (int j0 = 0; j0 < t.nj; ++j0) {
          const int n = n0 + j0, j = t.jlo + j0;
          const int sk = n % C::NK, sv = n % C::NV;
          if (!mbar_wait(&k_empty[sk], ((n / C::NK) & 1) ^ 1, err, kQKEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&k_full[sk], C::QCH * C::CHUNK);
          for (int c = 0; c < C::QCH; ++c)
            tma_load_4d(smem + C::OFF_K + (sk * C::QCH + c) * C::CHUNK, &tmK, &k_full[sk], c * 64, t.hk, j * C::BN,
                        t.b);
          if (!mbar_wait(&v_empty[sv], ((n / C::NV) & 1) ^ 1, err, kQVEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&v_full[sv], C::VCH * C::CHUNK);
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(smem + C::OFF_V + (sv * C::VCH + c) * C::CHUNK, &tmV, &v_full[sv], c * 64, t.hk, j * C::BN,
                        t.b);
        }
        if constexpr (PERSIST) ti_next = atomicAdd(p.tile_counter_q, 1);
        n0 += t.nj;
        ++ne;
      }
      // every copy this warp started must land before the CTA may exit
      if (ne > 0) mbar_wait(q_full, (ne - 1) & 1, err, kQDrain);
      for (int s = 0; s < C::NK && s < n0; ++s) {
        const int last = s + ((n0 - 1 - s) / C::NK) * C::NK;
        mbar_wait(&k_full[s], (last / C::NK) & 1, err, kQDrain);
      }
      for (int s = 0; s < C::NV && s < n0; ++s) {
        const int last = s + ((n0 - 1 - s) / C::NV) * C::NV;
        mbar_wait(&v_full[s], (last / C::NV) & 1, err, kQDrain);
      }
    }
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    //   A (warp 8):  S(n) = Q K_n^T, dP(n) = dO V_n^T into dP slot n % DPB
    //   B (warp 10): dQ += dS(n) K_n
    // S(n+1) waits for the dS warps to have loaded S(n) (s_free); dP(n) waits for
    // dQ(n - DPB), which read dS(n - DPB) from the same slot (dq_done of that slot).
    // Every per-slot barrier completes once per use of its slot, and a slot's next use
    // depends on the waiter having seen the previous one, so no phase is skipped.
    {  // whole warp runs the loops; elect.sync picks the issuing lane
      constexpr uint32_t idS = idesc_bf16_f32(128, 128, false, false);
      constexpr uint32_t idDQ = idesc_bf16_f32(128, D_QK, false, true);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
      const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
      bool ok = true;
      int n0 = 0, ne = 0;
      for (int k = 0;; ++k) {
      const int ti = take_tile(k, true);
      if (ti >= n_tiles || !ok) break;
      const Tile t = tile_of(ti);
      if (t.nj == 0) continue;
      if (warp == 8) {
        // Q and dO of the tile: only A's products read them (a wait nothing gates could
        // see a later phase complete)
        ok = mbar_wait_warp(q_full, ne & 1, err, kQQ);
        const uint64_t dQ0 = smem_desc_sw128(sQ, 16, 1024), dDO0 = smem_desc_sw128(sDO, 16, 1024);
        for (int j0 = 0; j0 < t.nj && ok; ++j0) {
          const int n = n0 + j0;
          const int sk = n % C::NK, sv = n % C::NV;
          const uint64_t dKa = smem_desc_sw128(sK + sk * C::QCH * C::CHUNK, 16, 1024);
          const uint64_t dVa = smem_desc_sw128(sV + sv * C::VCH * C::CHUNK, 16, 1024);
          ok = mbar_wait_warp(&k_full[sk], (n / C::NK) & 1, err, kQKFull);
          if (ok && n > 0) ok = mbar_wait_warp(s_free, (n - 1) & 1, err, kQSFree);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < D_QK / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::CHUNK + (kk % 4) * 32;
            mma_ss_warp(tmem + C::COL_S, desc_add(dQ0, off), desc_add(dKa, off), idS, kk > 0);
          }
          mma_commit_warp(s_ready);
          const int ds = n % C::DPB;
          ok = mbar_wait_warp(&v_full[sv], (n / C::NV) & 1, err, kQVFull);
          if (ok && n >= C::DPB) ok = mbar_wait_warp(&dq_done[ds], ((n / C::DPB) - 1) & 1, err, kQDqDone);
          if (!ok) break;
          tc_fence_after();
          const uint32_t colP = tmem + (ds ? C::COL_DP1 : C::COL_DP);
#pragma unroll
          for (int kk = 0; kk < D_V / 16; ++kk) {
            const uint32_t off = (kk / 4) * C::CHUNK + (kk % 4) * 32;
            mma_ss_warp(colP, desc_add(dDO0, off), desc_add(dVa, off), idS, kk > 0);
          }
          mma_commit_warp(&dp_ready[ds]);
          mma_commit_warp(&v_empty[sv]);
        }
        if constexpr (PERSIST) mma_commit_warp(qo_empty);  // the tile's S and dP products have read Q and dO
      } else {
        for (int j0 = 0; j0 < t.nj && ok; ++j0) {
          const int n = n0 + j0;
          const int sk = n % C::NK;
          const uint64_t dKmn = smem_desc_sw128(sK + sk * C::QCH * C::CHUNK, C::CHUNK, 1024);
          const int ds = n % C::DPB;
          ok = mbar_wait_warp(&k_full[sk], (n / C::NK) & 1, err, kQKFull) &&
               mbar_wait_warp(&ds_ready[ds], (n / C::DPB) & 1, err, kQDS);
          // the first dQ of a tile overwrites the sum the previous tile's epilogue reads
          if (PERSIST && ok && j0 == 0 && ne > 0) ok = mbar_wait_warp(acc_free, (ne - 1) & 1, err, kQAccFree);
          if (!ok) break;
          tc_fence_after();
          // dQ += dS K   (dS bf16 over the slot's dP columns: keys 0-63 at cols 0-31, keys 64-127 at cols 64-95)
          const uint32_t colP = tmem + (ds ? C::COL_DP1 : C::COL_DP);
#pragma unroll
          for (int kk = 0; kk < C::BN / 16; ++kk)
            mma_ts_warp(tmem + C::COL_DQ, colP + (kk / 4) * 64 + (kk % 4) * 8, desc_add(dKmn, kk * 2048),
                   idDQ, (j0 > 0 || kk > 0) ? 1u : 0u);
          mma_commit_warp(&dq_done[ds]);
          mma_commit_warp(&k_empty[sk]);  // S(n) (issuer A) completed before dS(n) existed
        }
      }
      // The tile's dQ sum is complete once B's MMAs are; B alone writes it.  (With both
      // issuers arriving, A could finish the next tile's products first and complete the
      // phase early.)
      if (warp == 10) mma_commit_warp(mma_done);
      n0 += t.nj;
      ++ne;
      }
      // Every MMA of both issuers must be complete before TMEM is released.
      mma_commit_warp(fin);
      mbar_wait_warp(fin, 0, err, kQDone);
    }
  } else if (warp < 8) {
    // ------------------------------------------------------------ dS warpgroups: thread = query row
    const int w = warp / 4;  // keys 64w .. 64w+63 of each kv tile
    const int r = (warp % 4) * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const float sl2 = p.scale_log2;
    [[maybe_unused]] const bool bias_vec = BIAS && (p.S_kv % 8 == 0);
    [[maybe_unused]] DropState drop{};
    if constexpr (DROP) drop = DropState{p.rng[0], p.rng[1], p.drop_t};
    bool ok = true;
    int n0 = 0, ne = 0;
    for (int k = 0;; ++k) {
    const int ti = take_tile(k, false);
    if (ti >= n_tiles) break;
    const Tile t = tile_of(ti);
    const int b = t.b, h = t.h;
    const int i = t.m0 + r;
    float nl2row = -INFINITY, drow = 0.f;
    if (i < p.S_q && t.nj > 0) {
      const size_t ri = ((size_t)b * p.H_q + h) * p.S_pad + i;
      nl2row = p.nlse2[ri];
      drow = p.Dsum[ri];
    }
    // bias: this row of the bias plane (rows past S_q read row S_q - 1; their P is 0)
    [[maybe_unused]] const __nv_bfloat16* brow =
        BIAS ? p.bias + b * p.bias_sb + h * p.bias_sh + (size_t)min(i, p.S_q - 1) * p.S_kv : nullptr;
    for (int j0 = 0; j0 < t.nj && ok; ++j0) {
      const int n = n0 + j0;
      const int k0 = (t.jlo + j0) * C::BN + 64 * w;
      // dropout: keep bits of this row for keys k0 .. k0 + 63 (bit c of keep[q]: key k0 + 32 q + c),
      // generated while the tile's scores are still being computed
      [[maybe_unused]] uint32_t keep[2] = {0u, 0u};
      if constexpr (DROP) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
          keep[q] = dropout_row_span16(drop, b, h, i, k0 + 32 * q) |
                    (dropout_row_span16(drop, b, h, i, k0 + 32 * q + 16) << 16);
      }
      ok = mbar_wait_warp(s_ready, n & 1, err, kQS);
      if (!ok) break;
      tc_fence_after();
      const bool full = tile_fully_visible<VL>(t.mask, t.m0, C::BM, (t.jlo + j0) * C::BN, C::BN);
      float pr[64];
      {
        uint32_t ra[32], rb[32];
        tmem_ld32(lane_addr + C::COL_S + 64 * w, ra);
        tmem_ld32(lane_addr + C::COL_S + 64 * w + 32, rb);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(s_free);  // S is in registers: the next S may be written
        // P = exp2(S * scale * log2(e) - LSE * log2(e)), one f32x2 FMA per key pair
        const uint64_t sl2x2 = f2_pack(sl2, sl2), nl2x2 = f2_pack(nl2row, nl2row);
        if constexpr (BIAS) {  // (+ bias * log2(e)): the bias enters through the addend
          const uint64_t l2e2 = f2_pack(kLog2e, kLog2e);
#pragma unroll
          for (int c8 = 0; c8 < 64; c8 += 8) {
            float bv[8];
            load_bias8(brow, k0 + c8, p.S_kv, bias_vec, bv);
            const uint32_t* src = c8 < 32 ? ra : rb;
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
              const int c = (c8 % 32) + e;
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(__uint_as_float(src[c]), __uint_as_float(src[c + 1])), sl2x2,
                               f2_fma(f2_pack(bv[e], bv[e + 1]), l2e2, nl2x2)),
                        x0, x1);
              pr[c8 + e] = ex2(x0);
              pr[c8 + e + 1] = ex2(x1);
            }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float x0, x1, y0, y1;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(ra[c]), __uint_as_float(ra[c + 1])), sl2x2, nl2x2), x0, x1);
            f2_unpack(f2_fma(f2_pack(__uint_as_float(rb[c]), __uint_as_float(rb[c + 1])), sl2x2, nl2x2), y0, y1);
            pr[c] = ex2(x0);
            pr[c + 1] = ex2(x1);
            pr[32 + c] = ex2(y0);
            pr[32 + c + 1] = ex2(y1);
          }
        }
      }
      if (!full) {  // this row sees keys [vlo, vhi]: two compares per key
        int vlo, vhi;
        visible_keys<VL>(t.mask, i, &vlo, &vhi);
#pragma unroll
        for (int c = 0; c < 64; ++c) pr[c] = (k0 + c >= vlo && k0 + c <= vhi) ? pr[c] : 0.f;
      }
      const int ds = n % C::DPB;
      const uint32_t colP = ds ? C::COL_DP1 : C::COL_DP;
      ok = mbar_wait_warp(&dp_ready[ds], (n / C::DPB) & 1, err, kQDP);
      if (!ok) break;
      tc_fence_after();
      const uint64_t drow2 = f2_pack(drow, drow);
#pragma unroll
      for (int c0 = 0; c0 < 64; c0 += 32) {
        uint32_t rr[32];
        tmem_ld32(lane_addr + colP + 64 * w + c0, rr);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {  // dS = P (dP - D), paired; with dropout P (M dP - D)
          float a, bq;
          if constexpr (DROP) {
            const uint32_t kb = keep[c0 / 32] >> (2 * c);
            f2_unpack(f2_mul(f2_pack(pr[c0 + 2 * c], pr[c0 + 2 * c + 1]),
                             f2_fma(f2_pack(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1])),
                                    f2_pack((kb & 1u) ? p.drop_scale : 0.f, (kb & 2u) ? p.drop_scale : 0.f),
                                    f2_pack(-drow, -drow))),
                      a, bq);
          } else {
            f2_unpack(f2_mul(f2_pack(pr[c0 + 2 * c], pr[c0 + 2 * c + 1]),
                             f2_sub(f2_pack(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1])), drow2)),
                      a, bq);
          }
          pk[c] = pack_bf16x2(a, bq);
        }
        tmem_st16(lane_addr + colP + 64 * w + c0 / 2, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&ds_ready[ds]);
    }
    // epilogue: dQ = scale * acc; warpgroup w writes head-dim columns [w*D_QK/2, (w+1)*D_QK/2).
    // A tile whose rows see no key (nj = 0) writes zeros and touches neither TMEM nor a barrier.
    bool have = false;
    if (ok && t.nj > 0) {
      have = mbar_wait_warp(mma_done, ne & 1, err, kQDone);
      tc_fence_after();
    }
    {
      const bool row_ok = i < p.S_q;  // all lanes load TMEM; only real rows store
      __nv_bfloat16* dst = p.dq + (((size_t)b * p.S_q + (row_ok ? i : 0)) * p.H_q + h) * D_QK;
      constexpr int HALF = D_QK / 2;
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
          pw[c] = pack_bf16x2(__uint_as_float(rr[2 * c]) * p.scale, __uint_as_float(rr[2 * c + 1]) * p.scale);
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q) d4[q] = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
        }
      }
    }
    if (t.nj > 0) {
      if constexpr (PERSIST) {  // the sum is read: issuer B may start the next tile's dQ
        tc_fence_before();
        mbar_arrive(acc_free);
      }
      n0 += t.nj;
      ++ne;
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

template <int D_QK, int D_V, KernVariant KV = KernVariant::kPlain>
inline int launch_q_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                      const BwdParams& p, cudaStream_t stream) {
  using C = QCfg<D_QK, D_V>;
  const bool vl = p.seq_q || p.seq_kv;  // padded batches: per-entry lengths and row tests
  decltype(&attn_bwd_q_kernel<D_QK, D_V, false>) kern;
  const long long tiles = (long long)((p.S_q + C::BM - 1) / C::BM) * p.H_q * p.B;
  if (tiles <= 0 || tiles > 0x7fffffffLL) return -2;
  static int n_sm = 0;
  if (n_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
      return -1;
  }
  bool persist = false;
  if constexpr (KV == KernVariant::kDrop) {  // dropout: full-length batches without a bias
    if (vl || p.bias) return -2;
    kern = attn_bwd_q_kernel<D_QK, D_V, false, false, true>;
  } else if constexpr (KV == KernVariant::kBias) {
    if (!p.bias) return -2;
    kern = vl ? attn_bwd_q_kernel<D_QK, D_V, true, true> : attn_bwd_q_kernel<D_QK, D_V, false, true>;
  } else {
    if (p.bias) return -2;
    // Persistent CTAs (one per SM, tiles from the counter) for the plain kernels of
    // full-length batches with d_qk = d_v when every tile has at most 32 kv tiles: a
    // CTA's fixed costs (the Q/dO load, the first products, the dQ epilogue) then
    // overlap the previous tile.  Measured faster up to 32 kv tiles (S <= 4096), level
    // at 64.
    const long long max_kv = (p.S_kv + C::BN - 1) / C::BN;
    if constexpr (D_QK == D_V) persist = !vl && p.tile_counter_q && tiles > n_sm && max_kv <= 32;
    if (persist) {
      if constexpr (D_QK == D_V) kern = attn_bwd_q_kernel<D_QK, D_V, false, false, false, true>;
    } else {
      kern = vl ? attn_bwd_q_kernel<D_QK, D_V, true> : attn_bwd_q_kernel<D_QK, D_V, false>;
    }
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -1;
  const unsigned grid = (unsigned)(persist ? n_sm : tiles);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, p);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

}  // namespace sdpa
