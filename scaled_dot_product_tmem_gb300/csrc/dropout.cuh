// dropout.cuh -- attention dropout decisions on the device: a counter-based
// Philox4x32-10 generator and the exchange of its keep bits within a warp.
//
// Source of the knob: "JAX: Single-GPU Attention with TransformerEngine", section
// "Other attention knobs" (`attention_dropout`); the sequence diagrams of "[JAX] Add
// support for sink attention in JAX #2225" (the fused forward returns an rng_state
// that the fused backward takes, so the backward regenerates the same decisions).
//
// Generator: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11).  Ten rounds on a counter of four 32-bit words; a round
// maps (c0, c1, c2, c3) under the key (k0, k1) to
//   (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
// and the key grows by the Weyl constants (W0, W1) between rounds.
//
// Decisions: rng_state = (seed, offset).  The key is the seed (low 32 bits, high 32
// bits); the pair (query i, key j) of batch b and query head h uses the counter
// (j / 2, i / 4, 65536 b + h, offset mod 2^32): one call covers the 4 x 2 block of pairs
// with the same i / 4 and j / 2.  Pair (i, j) takes output word i % 4 and its 16-bit
// field j % 2, a uniform u in [0, 65536); the pair is kept iff u >= t, the drop
// threshold (t = floor(p 65536 + 1/2)), and a kept probability is multiplied by
// 65536 / (65536 - t).  B and H_q are at most 65535 (the calls' shape limits), so the
// third counter word is one-to-one in (b, h).
//
// Exchange: every lane computes one 4 x 4 block (two calls) and turns it into a 16-bit
// keep mask (bit 4 r + c: row r, key c of the block).  The four lanes of a quad (lanes
// 4k .. 4k+3) hold four blocks that tile a 16 x 4 or 4 x 16 span, and four shuffles
// give each lane the bits it needs: a lane that owns a query row gets 16 consecutive
// keys of its row, a lane that owns a key gets 16 consecutive query rows of its key.
// Lanes of a quad must own four consecutive rows (or keys) starting at a multiple of
// 4; every lane of the warp must call these together.
#pragma once
#include <cstdint>

namespace sdpa {

__device__ __forceinline__ void philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3, uint32_t k0,
                                              uint32_t k1, uint32_t (&out)[4]) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
    const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
    c0 = hi1 ^ c1 ^ k0;
    c1 = lo1;
    c2 = hi0 ^ c3 ^ k1;
    c3 = lo0;
  }
  out[0] = c0;
  out[1] = c1;
  out[2] = c2;
  out[3] = c3;
}

struct DropState {
  uint64_t seed, offset;  // rng_state: the Philox key (seed) and counter word 3 (offset)
  uint32_t t;             // drop threshold: 16-bit uniforms below it are dropped
};

// Keep mask of the block (query rows 4 rb .. 4 rb + 3, keys 4 kb .. 4 kb + 3) of (b, h):
// bit 4 r + c set iff the pair (4 rb + r, 4 kb + c) is kept.  Keys 4 kb, 4 kb + 1 come
// from the call with counter word 2 kb, keys 4 kb + 2, 4 kb + 3 from 2 kb + 1.
__device__ __forceinline__ uint32_t dropout_block_mask(const DropState& d, int b, int h, int rb, int kb) {
  const uint32_t bh = (uint32_t)b * 65536u + (uint32_t)h;
  const uint32_t k0 = (uint32_t)d.seed, k1 = (uint32_t)(d.seed >> 32), off = (uint32_t)d.offset;
  uint32_t w0[4], w1[4];
  philox4x32_10(2u * (uint32_t)kb, (uint32_t)rb, bh, off, k0, k1, w0);
  philox4x32_10(2u * (uint32_t)kb + 1u, (uint32_t)rb, bh, off, k0, k1, w1);
  uint32_t m = 0;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    m |= ((w0[r] & 0xFFFFu) >= d.t ? 1u : 0u) << (4 * r);
    m |= ((w0[r] >> 16) >= d.t ? 1u : 0u) << (4 * r + 1);
    m |= ((w1[r] & 0xFFFFu) >= d.t ? 1u : 0u) << (4 * r + 2);
    m |= ((w1[r] >> 16) >= d.t ? 1u : 0u) << (4 * r + 3);
  }
  return m;
}

// A lane owning query row i (lanes of a quad own rows 4k .. 4k+3): keep bits of keys
// [k, k + 16) of row i (k a multiple of 16), bit c for key k + c.
__device__ __forceinline__ uint32_t dropout_row_span16(const DropState& d, int b, int h, int i, int k) {
  const int lane = threadIdx.x & 31, q = lane & 3, base = lane & ~3;
  const uint32_t mine = dropout_block_mask(d, b, h, i >> 2, (k >> 2) + q);  // key block q of the span
  uint32_t bits = 0;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t blk = __shfl_sync(0xffffffffu, mine, base + m);  // key block m, rows of the quad
    bits |= ((blk >> (4 * q)) & 0xFu) << (4 * m);                  // this lane's row: 4 keys
  }
  return bits;
}

// A lane owning key j (lanes of a quad own keys 4k .. 4k+3): keep bits of query rows
// [i, i + 16) of key j (i a multiple of 16), bit r for row i + r.
__device__ __forceinline__ uint32_t dropout_key_span16(const DropState& d, int b, int h, int j, int i) {
  const int lane = threadIdx.x & 31, c = lane & 3, base = lane & ~3;
  const uint32_t mine = dropout_block_mask(d, b, h, (i >> 2) + c, j >> 2);  // row block c of the span
  uint32_t bits = 0;
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    const uint32_t blk = __shfl_sync(0xffffffffu, mine, base + m);  // row block m, keys of the quad
    uint32_t x = (blk >> c) & 0x1111u;                               // this lane's key: rows at bits 0, 4, 8, 12
    x = (x | (x >> 3) | (x >> 6) | (x >> 9)) & 0xFu;
    bits |= x << (4 * m);
  }
  return bits;
}

}  // namespace sdpa
