// attn_bwd_wide.cu -- kv-stationary dK/dV kernel with 128-row query steps, for the
// deterministic backward of sm_103a (dQ comes from the query-stationary kernel).
//
// Same quantities as attn_bwd.cu ("Speed up attention on GPU with cuDNN and
// TransformerEngine", section "How attention works", differentiated):
//   dV_j = sum_{h in group} sum_i P_ij dO_i,   dK_j = scale sum_{h in group} sum_i dS_ij q_i,
//   dS_ij = P_ij (dP_ij - D_i),  dP_ij = dO_i.v_j,  P_ij = exp2(scale log2(e) q_i.k_j - LSE_i log2(e)).
//
// Why a second kv kernel.  The tensor core reads both operands of an SS product from
// shared memory at about 128 bytes per cycle.  A 128 x 64 x 16 bf16 instruction reads
// 6 KB for 32 cycles of math and takes 48; a 128 x 128 x 16 one reads 8 KB for 64
// cycles of math and takes 64.  With 64 query rows per step, S^T = K Q^T and
// dP^T = V dO^T are the former; with 128 rows they are the latter, and each query row
// of a step costs a third less tensor time.  TMEM then holds S^T, dP^T (128 columns
// each) and the dV, dK accumulators, which is all of it: S^T and dP^T have one slot
// each, and there is no room for a fused dQ^T.  P^T and dS^T (bf16) are written over
// the first half of their own S^T / dP^T columns and feed dV and dK as TMEM operands.
//
// Roles (352 threads, one CTA per SM):
//   warps 0-7   P / dS: warp w4 = warp / 4 takes query rows 64 w4 .. 64 w4 + 63 of the
//               step, thread = key (TMEM lane); then the dV (w4 = 0) / dK (w4 = 1) epilogue.
//   warp 8      MMA issuer A: S^T of a tile's first step, and dP^T(s) = V dO_s^T once
//               dK(s-1) has read dS^T(s-1).  Also TMEM allocation.
//   warp 9      TMA producer: K, V per tile; Q, dO tiles and the LSE / D rows per step;
//               with persistent CTAs also the tile indices.
//   warp 10     MMA issuer B: dV += P^T(s) dO_s, then S^T(s+1) of the same tile once
//               dV(s) has read P^T(s), then dK += dS^T(s) Q_s.
#include <cuda_runtime.h>

#include "attn_bwd_kernels.cuh"

namespace sdpa {

template <int D_QK, int D_V>
struct KvWCfg {
  static constexpr int BN = 128;  // keys per CTA (TMEM lanes)
  static constexpr int BQ = 128;  // query rows per step
  static constexpr int QCH = D_QK / 64, VCH = D_V / 64;
  static constexpr int KCHUNK = 128 * 128;  // 128 rows x 128 bytes (64 bf16)
  static constexpr int QCHUNK = 128 * 128;
  static constexpr int NQ = 2;  // Q / dO stages
  static constexpr int OFF_K = 0;
  static constexpr int OFF_V = OFF_K + QCH * KCHUNK;
  static constexpr int OFF_Q = OFF_V + VCH * KCHUNK;
  static constexpr int Q_STAGE = QCH * QCHUNK;
  static constexpr int OFF_DO = OFF_Q + NQ * Q_STAGE;
  static constexpr int DO_STAGE = VCH * QCHUNK;
  static constexpr int OFF_L = OFF_DO + NQ * DO_STAGE;  // nlse2[128] + D[128] per stage
  static constexpr int L_STAGE = 2 * BQ * 4;
  static constexpr int OFF_BAR = OFF_L + NQ * L_STAGE;
  // kv_full, q_full[NQ], q_empty[NQ], s_ready, dp_ready, p_ready, ds_ready, dv_done,
  // dk_done, mma_done, kv_empty, acc_free, fin, tile_full[2], tile_empty[2]; the tile
  // index ring (two ints) sits beside the TMEM address
  static constexpr int NBAR = 1 + 2 * NQ + 14;
  static constexpr int OFF_TMEM_SLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM_RAW = OFF_TMEM_SLOT + 16 + 1024;
  static constexpr int SMEM = SMEM_RAW > 117 * 1024 ? SMEM_RAW : 117 * 1024;  // one CTA per SM (all of TMEM)
  static constexpr int THREADS = 352;
  static constexpr int COL_S = 0, COL_DP = 128, COL_DV = 256, COL_DK = 256 + D_V;
  static_assert(COL_DK + D_QK <= 512, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

enum KvWSite { kWFull = 0x80, kWQFull, kWQEmpty, kWS, kWDP, kWP, kWDS, kWDvDone, kWDkDone, kWDone, kWDrain, kWEmpty,
               kWAccFree, kWTile };

// PERSIST: the CTAs (one per SM) take tiles from a counter in global memory, as the
// persistent fused-dQ kernel does; otherwise the grid has one CTA per tile and the tile
// loops run once (the cross-tile barriers compile away).
template <int D_QK, int D_V, bool VL, bool PERSIST = false>
__global__ void __launch_bounds__(352, 1)
    attn_bwd_kvw_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                        const BwdParams p) {
  using C = KvWCfg<D_QK, D_V>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + C::NQ;
  uint64_t* s_ready = q_empty + C::NQ;
  uint64_t* dp_ready = s_ready + 1;
  uint64_t* p_ready = s_ready + 2;
  uint64_t* ds_ready = s_ready + 3;
  uint64_t* dv_done = s_ready + 4;
  uint64_t* dk_done = s_ready + 5;
  uint64_t* mma_done = s_ready + 6;    // a tile's dV/dK sums are complete
  uint64_t* kv_empty = s_ready + 7;    // a tile's K/V readers are done: the next K/V may load
  uint64_t* acc_free = s_ready + 8;    // the epilogue has read dV/dK: the next tile may overwrite them
  uint64_t* fin = s_ready + 9;         // every MMA issued, before TMEM is released
  uint64_t* tile_full = s_ready + 10;  // [2] PERSIST: the producer has published the next tile
  uint64_t* tile_empty = s_ready + 12; // [2] PERSIST: every role has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_TMEM_SLOT);
  volatile int* ring = reinterpret_cast<volatile int*>(smem + C::OFF_TMEM_SLOT + 8);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  // Tiles in the 64-row kernel's order: (b, kv head, head split) groups in chunks of
  // kKvChunk, kv tile by kv tile within a chunk.  Every role walks the same tiles and
  // numbers the steps of all of them in one sequence g (stages, barrier phases).
  const int n_kv = (p.S_kv + C::BN - 1) / C::BN;
  const int n_gr = p.H_kv * p.B * p.ns;
  const int n_tiles = n_kv * n_gr;
  const int per_chunk = kKvChunk * n_kv;
  const int Gs = p.G / p.ns;
  struct Tile {
    int b, hk, split, h0, n0, ilo, nq, nsteps;
    MaskSpec mask;
  };
  auto tile_of = [&](int ti) {
    Tile t;
    const int chunk = ti / per_chunk, within = ti % per_chunk;
    const int csize = min(kKvChunk, n_gr - chunk * kKvChunk);
    const int g = chunk * kKvChunk + within % csize;
    t.split = g % p.ns;
    t.hk = (g / p.ns) % p.H_kv;
    t.b = g / (p.ns * p.H_kv);
    t.h0 = t.hk * p.G + t.split * Gs;
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
  // Tile k of this CTA for the roles other than the producer (see the fused-dQ kernel).
  auto take_tile = [&](int k, bool whole_warp) -> int {
    if constexpr (!PERSIST) {
      return k == 0 ? (int)blockIdx.x : n_tiles;
    } else {
      const int slot = k & 1;
      if (!mbar_wait_warp(&tile_full[slot], (k >> 1) & 1, p.err, kWTile)) return n_tiles;
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
    for (int s = 0; s < C::NQ; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    mbar_init(s_ready, 1);
    mbar_init(dp_ready, 1);
    mbar_init(p_ready, 256);
    mbar_init(ds_ready, 256);
    mbar_init(dv_done, 1);
    mbar_init(dk_done, 1);
    mbar_init(mma_done, 1);  // issuer B, once per tile: it alone writes the dV/dK sums
    mbar_init(kv_empty, 2);  // both issuers read K (S^T) and A reads V (dP^T)
    mbar_init(acc_free, 256);
    mbar_init(fin, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tile_full[i], 1);
      mbar_init(&tile_empty[i], 2 + 256);  // the two issuers (one lane each) and the P/dS threads
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
      bool ok = true, first = true;
      int g0 = 0, ne = 0, ti_next = 0;
      for (int k = 0;; ++k) {
        int ti;
        if constexpr (PERSIST) {  // publish tile k once every role has read tile k - 2
          const int slot = k & 1;
          if (k >= 2 && !mbar_wait(&tile_empty[slot], ((k >> 1) - 1) & 1, err, kWTile)) break;
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
          first = false;
        }
        if (PERSIST && ne > 0 && !mbar_wait(kv_empty, (ne - 1) & 1, err, kWEmpty)) break;
        mbar_arrive_expect_tx(kv_full, (C::QCH + C::VCH) * C::KCHUNK);
        for (int c = 0; c < C::QCH; ++c)
          tma_load_4d(smem + C::OFF_K + c * C::KCHUNK, &tmK, kv_full, c * 64, t.hk, t.n0, t.b);
        for (int c = 0; c < C::VCH; ++c)
          tma_load_4d(smem + C::OFF_V + c * C::KCHUNK, &tmV, kv_full, c * 64, t.hk, t.n0, t.b);
        for (int s = 0; s < t.nsteps; ++s) {
          const int g = g0 + s, st = g % C::NQ;
          if (!mbar_wait(&q_empty[st], ((g / C::NQ) & 1) ^ 1, err, kWQEmpty)) {
            ok = false;
            break;
          }
          const int h = t.h0 + s / t.nq;
          const int q0 = (t.ilo + s % t.nq) * C::BQ;
          mbar_arrive_expect_tx(&q_full[st], C::Q_STAGE + C::DO_STAGE + C::L_STAGE);
          for (int c = 0; c < C::QCH; ++c)
            tma_load_4d(smem + C::OFF_Q + st * C::Q_STAGE + c * C::QCHUNK, &tmQ, &q_full[st], c * 64, h, q0, t.b);
          for (int c = 0; c < C::VCH; ++c)
            tma_load_4d(smem + C::OFF_DO + st * C::DO_STAGE + c * C::QCHUNK, &tmDO, &q_full[st], c * 64, h, q0,
                        t.b);
          // q0 + 128 <= S_pad: the rows are padded to a multiple of 128
          const size_t row = ((size_t)t.b * p.H_q + h) * p.S_pad + q0;
          bulk_load(smem + C::OFF_L + st * C::L_STAGE, p.nlse2 + row, C::BQ * 4, &q_full[st]);
          bulk_load(smem + C::OFF_L + st * C::L_STAGE + C::BQ * 4, p.Dsum + row, C::BQ * 4, &q_full[st]);
        }
        if constexpr (PERSIST) ti_next = atomicAdd(p.tile_counter, 1);
        g0 += t.nsteps;
        ++ne;
      }
      // every copy this warp started must land before the CTA may exit
      if (ne > 0) mbar_wait(kv_full, (ne - 1) & 1, err, kWDrain);
      for (int st = 0; st < C::NQ && st < g0; ++st) {
        const int last = st + ((g0 - 1 - st) / C::NQ) * C::NQ;
        mbar_wait(&q_full[st], (last / C::NQ) & 1, err, kWDrain);
      }
    }
  } else if (warp == 8 || warp == 10) {
    // ------------------------------------------------------------ MMA issuers
    // Tensor-core order per step: dV(g), S^T(g+1), dK(g), dP^T(g+1).  S^T(g+1) goes
    // ahead of dK(g) so that P(g+1) is computed while dK(g) and dP^T(g+1) run.
    //   A (warp 8):  S^T of a tile's first step, once the previous tile's last dV has read
    //                P^T (S^T columns); dP^T(g) once dK(g-1) has read dS^T(g-1) (dP^T columns).
    //   B (warp 10): dV(g) once P(g) is in TMEM; S^T(g+1) within the tile once dV(g) has
    //                read P^T(g); dK(g) once dS(g) is in TMEM.
    // MMAs into different accumulators are not ordered by the hardware, so every TMEM
    // reuse waits for the completion of the MMA that read the columns last.
    constexpr uint32_t idS = idesc_bf16_f32(128, C::BQ, false, false);
    constexpr uint32_t idDV = idesc_bf16_f32(128, D_V, false, true);
    constexpr uint32_t idDK = idesc_bf16_f32(128, D_QK, false, true);
    const uint32_t sK = smem_u32(smem + C::OFF_K), sV = smem_u32(smem + C::OFF_V);
    const uint32_t sQ = smem_u32(smem + C::OFF_Q), sDO = smem_u32(smem + C::OFF_DO);
    const uint64_t dK0 = smem_desc_sw128(sK, 16, 1024);  // K as K-major A of S^T
    // S^T(g) = K Q_g^T into the S^T columns
    auto issue_s = [&](int g) {
      const uint64_t dq = smem_desc_sw128(sQ + (g % C::NQ) * C::Q_STAGE, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D_QK / 16; ++kk)
        mma_ss_warp(tmem + C::COL_S, desc_add(dK0, (kk / 4) * C::KCHUNK + (kk % 4) * 32),
                    desc_add(dq, (kk / 4) * C::QCHUNK + (kk % 4) * 32), idS, kk > 0);
      mma_commit_warp(s_ready);
    };
    bool ok = true;
    int g0 = 0, ne = 0;
    for (int k = 0;; ++k) {  // whole warp; elect.sync picks the issuing lane
      const int ti = take_tile(k, true);
      if (ti >= n_tiles || !ok) break;
      const Tile t = tile_of(ti);
      if (t.nsteps == 0) continue;
      ok = mbar_wait_warp(kv_full, ne & 1, err, kWFull);
      if (warp == 8) {
        const uint64_t dV0 = smem_desc_sw128(sV, 16, 1024);  // V as K-major A of dP^T
        ok = ok && mbar_wait_warp(&q_full[g0 % C::NQ], (g0 / C::NQ) & 1, err, kWQFull);
        // the tile's first S^T overwrites P^T of the previous tile's last step
        if (ok && g0 > 0) ok = mbar_wait_warp(dv_done, (g0 - 1) & 1, err, kWDvDone);
        if (ok) {
          tc_fence_after();
          issue_s(g0);
        }
        for (int s = 0; s < t.nsteps && ok; ++s) {
          const int g = g0 + s, st = g % C::NQ;
          ok = mbar_wait_warp(&q_full[st], (g / C::NQ) & 1, err, kWQFull);
          if (ok && g > 0) ok = mbar_wait_warp(dk_done, (g - 1) & 1, err, kWDkDone);
          if (!ok) break;
          tc_fence_after();
          const uint64_t ddo = smem_desc_sw128(sDO + st * C::DO_STAGE, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < D_V / 16; ++kk)
            mma_ss_warp(tmem + C::COL_DP, desc_add(dV0, (kk / 4) * C::KCHUNK + (kk % 4) * 32),
                        desc_add(ddo, (kk / 4) * C::QCHUNK + (kk % 4) * 32), idS, kk > 0);
          mma_commit_warp(dp_ready);
        }
      } else {
        for (int s = 0; s < t.nsteps && ok; ++s) {
          const int g = g0 + s, st = g % C::NQ;
          // dO and Q as MN-major B operands (N = head dim, 64-wide blocks QCHUNK apart;
          // K = query rows, 16 rows = 2 KB per instruction)
          const uint64_t ddo_mn = smem_desc_sw128(sDO + st * C::DO_STAGE, C::QCHUNK, 1024);
          const uint64_t dq_mn = smem_desc_sw128(sQ + st * C::Q_STAGE, C::QCHUNK, 1024);
          ok = mbar_wait_warp(&q_full[st], (g / C::NQ) & 1, err, kWQFull) &&
               mbar_wait_warp(p_ready, g & 1, err, kWP);
          // the first dV of a tile overwrites the sums the previous tile's epilogue reads
          if (PERSIST && ok && s == 0 && ne > 0) ok = mbar_wait_warp(acc_free, (ne - 1) & 1, err, kWAccFree);
          if (!ok) break;
          tc_fence_after();
          // dV += P^T dO.  P^T (bf16) of query rows 64 w4 + 2j, 64 w4 + 2j + 1 sits in
          // column 64 w4 + j, so K step kk (rows 16 kk ..) starts at 64 (kk / 4) + 8 (kk % 4).
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            mma_ts_warp(tmem + C::COL_DV, tmem + C::COL_S + (kk / 4) * 64 + (kk % 4) * 8,
                        desc_add(ddo_mn, kk * 2048), idDV, (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit_warp(dv_done);
          if (s + 1 < t.nsteps) {
            ok = mbar_wait_warp(&q_full[(g + 1) % C::NQ], ((g + 1) / C::NQ) & 1, err, kWQFull) &&
                 mbar_wait_warp(dv_done, g & 1, err, kWDvDone);
            if (!ok) break;
            tc_fence_after();
            issue_s(g + 1);
          }
          ok = mbar_wait_warp(ds_ready, g & 1, err, kWDS);
          if (!ok) break;
          tc_fence_after();
          // dK += dS^T Q, dS^T laid out like P^T in the dP^T columns
#pragma unroll
          for (int kk = 0; kk < C::BQ / 16; ++kk)
            mma_ts_warp(tmem + C::COL_DK, tmem + C::COL_DP + (kk / 4) * 64 + (kk % 4) * 8,
                        desc_add(dq_mn, kk * 2048), idDK, (s > 0 || kk > 0) ? 1u : 0u);
          mma_commit_warp(dk_done);
          // the stage's S/dP MMAs completed before P(g)/dS(g) existed
          mma_commit_warp(&q_empty[st]);
        }
      }
      if constexpr (PERSIST) mma_commit_warp(kv_empty);  // this issuer's reads of K (and V) are done
      // The tile's dV/dK sums are complete once B's MMAs are; B alone writes them.  (With
      // both issuers arriving, A could finish the next tile's products first and complete
      // the phase early.)
      if (warp == 10) mma_commit_warp(mma_done);
      g0 += t.nsteps;
      ++ne;
    }
    // Every MMA of both issuers must be complete before TMEM is released.
    mma_commit_warp(fin);
    mbar_wait_warp(fin, 0, err, kWDone);
  } else if (warp < 8) {
    // ------------------------------------------------------------ P / dS warpgroups
    const int w = warp / 4;  // which 64 query rows of the 128
    const int r = (warp % 4) * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)((warp % 4) * 32) << 16);
    const uint32_t colS = C::COL_S + 64 * w, colP = C::COL_DP + 64 * w;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int g0 = 0, ne = 0;
    for (int k = 0;; ++k) {
      const int ti = take_tile(k, false);
      if (ti >= n_tiles) break;
      const Tile t = tile_of(ti);
      const int key = t.n0 + r;
      for (int s = 0; s < t.nsteps && ok; ++s) {
        const int g = g0 + s, st = g % C::NQ;
        const int q0 = (t.ilo + s % t.nq) * C::BQ;
        const float* l2 = reinterpret_cast<const float*>(smem + C::OFF_L + st * C::L_STAGE) + 64 * w;
        const float* dd = l2 + C::BQ;
        ok = mbar_wait_warp(s_ready, g & 1, err, kWS);
        if (!ok) break;
        tc_fence_after();
        // P = exp2(S scale log2(e) - LSE log2(e)) for 64 query rows, in two 32-column halves.
        // Half 1's P^T goes to columns 16..31 of this group, which held half 0's S^T
        // (already in registers); half 1's own S^T (columns 32..63) is not overwritten.
        const bool full = tile_fully_visible<VL>(t.mask, q0, C::BQ, t.n0, C::BN);
        int vlo = 0, vhi = 0;
        if (!full) visible_rows<VL>(t.mask, key, &vlo, &vhi);
        float pr[64];
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t rr[32];
          tmem_ld32(lane_addr + colS + 32 * hf, rr);
          float lv[32];
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(&lv[c]) = *reinterpret_cast<const float4*>(&l2[32 * hf + c]);
          tmem_ld_wait();
          const uint64_t sl2x2 = f2_pack(sl2, sl2);
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float xa, xb;
            f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[c]), __uint_as_float(rr[c + 1])), sl2x2,
                             f2_pack(lv[c], lv[c + 1])),
                      xa, xb);
            pr[32 * hf + c] = ex2(xa);
            pr[32 * hf + c + 1] = ex2(xb);
          }
          if (!full) {
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const int qq = q0 + 64 * w + 32 * hf + c;
              pr[32 * hf + c] = (qq >= vlo && qq <= vhi) ? pr[32 * hf + c] : 0.f;
            }
          }
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = pack_bf16x2(pr[32 * hf + 2 * c], pr[32 * hf + 2 * c + 1]);
          tmem_st16(lane_addr + colS + 16 * hf, pk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(p_ready);
        ok = mbar_wait_warp(dp_ready, g & 1, err, kWDP);
        if (!ok) break;
        tc_fence_after();
        // dS = P (dP - D), written as bf16 over the first half of this group's dP^T columns
#pragma unroll
        for (int hf = 0; hf < 2; ++hf) {
          uint32_t rr[32];
          tmem_ld32(lane_addr + colP + 32 * hf, rr);
          float dv4[32];
#pragma unroll
          for (int c = 0; c < 32; c += 4)
            *reinterpret_cast<float4*>(&dv4[c]) = *reinterpret_cast<const float4*>(&dd[32 * hf + c]);
          tmem_ld_wait();
          uint32_t dsk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            float a, bq;
            f2_unpack(f2_mul(f2_pack(pr[32 * hf + 2 * c], pr[32 * hf + 2 * c + 1]),
                             f2_sub(f2_pack(__uint_as_float(rr[2 * c]), __uint_as_float(rr[2 * c + 1])),
                                    f2_pack(dv4[2 * c], dv4[2 * c + 1]))),
                      a, bq);
            dsk[c] = pack_bf16x2(a, bq);
          }
          tmem_st16(lane_addr + colP + 16 * hf, dsk);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(ds_ready);
      }
      // ---------------------------------------------------------- epilogue: dV (w = 0), dK (w = 1)
      // A tile no query sees (nsteps = 0) writes zero rows and touches neither TMEM nor a barrier.
      bool have = false;
      if (ok && t.nsteps > 0) {
        have = mbar_wait_warp(mma_done, ne & 1, err, kWDone);
        tc_fence_after();
      }
      {
        const bool row_ok = key < p.S_kv;  // all lanes load TMEM; only real keys store
        const int krow = row_ok ? key : 0;
        const int ncols = w == 0 ? D_V : D_QK;
        const int col0 = w == 0 ? C::COL_DV : C::COL_DK;
        const float mul = w == 0 ? 1.f : p.scale;
        const size_t row = ((size_t)t.b * p.S_kv + krow) * p.H_kv + t.hk;
        __nv_bfloat16* dst = w == 0 ? p.dv + row * D_V : p.dk + row * D_QK;
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
        if constexpr (PERSIST) {  // the sums are read: issuer B may start the next tile's dV and dK
          tc_fence_before();
          mbar_arrive(acc_free);
        }
        g0 += t.nsteps;
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

template <int D_QK, int D_V>
static int launch_kvw_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tdo,
                        const BwdParams& p, cudaStream_t stream) {
  using C = KvWCfg<D_QK, D_V>;
  const bool vl = p.seq_q || p.seq_kv;
  const long long tiles = (long long)((p.S_kv + C::BN - 1) / C::BN) * p.H_kv * p.B * p.ns;
  if (tiles <= 0 || tiles > 0x7fffffffLL) return -2;
  // Persistent CTAs (one per SM, tiles from the counter) when every tile has at most 32
  // steps of 128 rows: measured faster up to 32 (MHA at S <= 4096), slower at 128 and
  // 256 (GQA at S = 4096 and 8192).
  static int n_sm = 0;
  if (n_sm == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm <= 0)
      return -1;
  }
  const long long max_steps = (long long)(p.G / p.ns) * ((p.S_q + C::BQ - 1) / C::BQ);
  const bool persist = !vl && p.tile_counter && tiles > n_sm && max_steps <= 32;
  auto kern = persist ? attn_bwd_kvw_kernel<D_QK, D_V, false, true>
                      : (vl ? attn_bwd_kvw_kernel<D_QK, D_V, true> : attn_bwd_kvw_kernel<D_QK, D_V, false>);
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) != cudaSuccess) return -1;
  const unsigned grid = (unsigned)(persist ? n_sm : tiles);
  kern<<<grid, C::THREADS, C::SMEM, stream>>>(tq, tk, tv, tdo, p);
  return cudaPeekAtLastError() == cudaSuccess ? 0 : -1;
}

bool bwd_kv_wide_supported(int d_qk, int d_v) { return d_qk == d_v && (d_qk == 128 || d_qk == 64); }

int launch_bwd_kv_wide(int d_qk, int d_v, const CUtensorMap& tq128, const CUtensorMap& tk, const CUtensorMap& tv,
                       const CUtensorMap& tdo128, const BwdParams& p, cudaStream_t stream) {
  if (p.bias || p.drop_t) return -2;
  if (d_qk == 128 && d_v == 128) return launch_kvw_t<128, 128>(tq128, tk, tv, tdo128, p, stream);
  if (d_qk == 64 && d_v == 64) return launch_kvw_t<64, 64>(tq128, tk, tv, tdo128, p, stream);
  return -2;
}

}  // namespace sdpa
