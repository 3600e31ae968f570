/*
 * oracle.c -- plain fp64 CPU oracle for fused BSHD scaled-dot-product attention,
 * forward and backward, with grouped-query heads, a causal left window, distinct
 * Q/K and V head dims and the three sink softmax types.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: it exists so that the tests, the smoke check and the CPU baseline of
 * the benchmark can check the CUDA kernels against an independent definition.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * What it computes, and where the definition comes from:
 *   - "Speed up attention on GPU with cuDNN and TransformerEngine", section
 *     "How attention works": Attention(Q,K,V) = softmax(Q K^T / sqrt(d_k)) V in
 *     four steps (score, scale + softmax, attend, output of Q's shape).
 *   - Same codelab, step 4 "Implement attention from scratch": the score matrix
 *     is materialised in full, one (batch, head) at a time.  This file does the
 *     same: every (b, h) gets its own S_q x S_kv score/probability matrix.
 *   - Same codelab, step 7 "Add causal masking": query i sees keys j <= i.
 *   - "JAX: Single-GPU Attention with TransformerEngine", section 1 (GQA + SWA
 *     baseline: K/V heads are repeated for the query heads of a group; the causal
 *     sliding-window mask is applied explicitly) and section "Other attention
 *     knobs" (scale_factor overrides 1/sqrt(head_dim); sink softmax types).
 *   - "[JAX] Add support for sink attention in JAX #2225", Greptile summaries
 *     (sequence diagrams): vanilla exp(S_i)/sum exp(S); off-by-one
 *     exp(S_i)/(1 + sum exp(S)); learnable exp(S_ji)/(exp(alpha_j) + sum_i exp(S_ji))
 *     with one alpha per head, which receives a gradient in the backward.
 *
 * Readings taken where the pages are silent or at odds (each one is listed in the
 * design notes of the repository):
 *   - the sink is an extra logit c with no value vector: c = -inf (vanilla),
 *     c = 0 (off-by-one: the review thread of PR 2225 settles 0, not 1, which
 *     makes "+1" in the denominator), c = offset[h] (learnable, one per query head,
 *     not multiplied by the scale);
 *   - window w >= 0 with causal: query i sees keys i-w <= j <= i (top-left
 *     diagonal); w < 0 means no window;
 *   - kv head of query head h is h / (H_q / H_kv) (contiguous groups);
 *   - LSE = M_i + ln Z_i includes the sink; a row with no visible key and no sink
 *     gives O = 0, LSE = -inf, and contributes nothing to the backward.
 *
 * Additive bias ("JAX: Single-GPU Attention with TransformerEngine", section "Other
 * attention knobs": pass `bias` with an `attn_bias_type`; the sequence diagrams of
 * PR 2225 pass it to the fused kernels and get grad_bias back).  Reading: the bias
 * is added to the scaled scores, s_ij = scale q_i . k_j + bias_ij (post-scale), before
 * the masks; it is a [Bb, Hb, S_q, S_kv] tensor with Bb in {1, B} and Hb in {1, H_q}
 * broadcast over batch / heads; a -inf bias entry removes that key like a mask.
 * dbias_ij = sum over the (b, h) that share the entry of dS_ij.
 *
 * Backward (derived from the definition; the pages only name the outputs
 * dq, dk, dv, d_softmax_offset):
 *   dP_ij = dO_i . v_j,   D_i = dO_i . O_i,   dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i = scale sum_j dS_ij k_j,  dK_j = scale sum_{h in group} sum_i dS_ij q_i,
 *   dV_j = sum_{h in group} sum_i P_ij dO_i,  d offset_h = -sum_{b,i} p_sink_i D_i.
 *
 * Attention dropout ("JAX: Single-GPU Attention with TransformerEngine", section
 * "Other attention knobs": `attention_dropout`; the sequence diagrams of PR 2225: the
 * fused forward returns an rng_state that the fused backward takes).  Reading: each
 * probability P_ij (after the softmax, sink included in the normaliser) is kept with
 * probability 1 - p and scaled by 1/(1 - p), or dropped to 0; the normaliser, LSE and
 * p_sink are those of the undropped softmax.  The keep decisions come from a
 * counter-based generator, so the backward regenerates them from the same state:
 *   - Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 *     as 1, 2, 3", SC'11): ten rounds on a 4 x 32-bit counter with a 2 x 32-bit key;
 *   - the rng_state is (seed, offset), two 64-bit words.  The key is the seed (low
 *     word first); the counter of pair (b, h, i, j) is
 *     (j / 2, i / 4, 65536 b + h, offset mod 2^32), so b and h are below 65536;
 *   - the call yields four 32-bit words; pair (i, j) takes word i % 4 and, within it,
 *     the 16-bit field j % 2 (bits 16 (j % 2) .. 16 (j % 2) + 15), a uniform u in
 *     [0, 65536);
 *   - the drop probability is realised as t / 65536 with t = floor(p * 65536 + 1/2);
 *     the pair is kept iff u >= t, and a kept P is multiplied by 65536 / (65536 - t).
 * With M_ij = keep_ij * 65536 / (65536 - t) the forward is O_i = sum_j P_ij M_ij v_j
 * and the backward is (dP~_ij = dO_i . v_j):
 *   D_i = dO_i . O_i = sum_j P_ij M_ij dP~_ij,   dS_ij = P_ij (M_ij dP~_ij - D_i),
 *   dV_j = sum_{h in group} sum_i P_ij M_ij dO_i,   dQ, dK, d offset as above.
 *
 * All tensors are contiguous BSHD (batch, sequence, head, head-dim) in double,
 * except lse / psink / rowsum / D which are [B, H_q, S_q] and offset [H_q].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_VANILLA 0
#define ORACLE_OFF_BY_ONE 1
#define ORACLE_LEARNABLE 2
#define ORACLE_MAX_D 512 /* largest head dim the oracle accepts */

static size_t bshd(int b, int s, int h, int c, int S, int H, int D) {
    return (((size_t)b * S + s) * H + h) * D + c;
}

/* Is key j visible to query i?  Causal: j <= i.  Window w >= 0: j >= i - w. */
static int visible(int i, int j, int causal, int window) {
    if (causal && j > i) return 0;
    if (window >= 0 && j < i - window) return 0;
    return 1;
}

/* The [S_q, S_kv] bias plane that batch b, query head h reads, or NULL. */
static const double* bias_plane(const double* bias, int Bb, int Hb, int b, int h, int Sq, int Skv) {
    if (!bias) return NULL;
    return bias + ((size_t)(Bb == 1 ? 0 : b) * Hb + (Hb == 1 ? 0 : h)) * Sq * Skv;
}

/*
 * Philox4x32-10 (SC'11 paper cited above).  One round maps the counter
 * (c0, c1, c2, c3) with key (k0, k1) to
 *   (hi(M1 c2) ^ c1 ^ k0, lo(M1 c2), hi(M0 c0) ^ c3 ^ k1, lo(M0 c0)),
 * hi/lo the upper/lower 32 bits of the 64-bit product; between rounds the key is
 * bumped by the Weyl constants (W0, W1).  Ten rounds, the first with the key itself.
 */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3], k0 = key[0], k1 = key[1];
    for (int r = 0; r < 10; r++) {
        if (r > 0) { k0 += W0; k1 += W1; }
        uint64_t p0 = (uint64_t)M0 * c0, p1 = (uint64_t)M1 * c2;
        uint32_t n0 = (uint32_t)(p1 >> 32) ^ c1 ^ k0, n1 = (uint32_t)p1;
        uint32_t n2 = (uint32_t)(p0 >> 32) ^ c3 ^ k1, n3 = (uint32_t)p0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Dropout state: drop threshold t (0: no dropout), the Philox key (seed, offset), and the
 * batch / query-head index of the arrays' first entry / head in the problem they were cut
 * from (0 for a whole problem): the decisions are those of (b + b0, h + h0). */
typedef struct { int t; uint64_t seed, offset; int b0, h0; } dropout_t;

/* The 16-bit uniform of pair (b, h, i, j) (see the header); b, h < 65536. */
static unsigned dropout_u16(const dropout_t* d, int b, int h, int i, int j) {
    uint32_t ctr[4] = {(uint32_t)(j / 2), (uint32_t)(i / 4), (uint32_t)b * 65536u + (uint32_t)h,
                       (uint32_t)d->offset};
    uint32_t key[2] = {(uint32_t)d->seed, (uint32_t)(d->seed >> 32)}, w[4];
    oracle_philox4x32_10(ctr, key, w);
    return (w[i % 4] >> (16 * (j % 2))) & 0xFFFFu;
}

/* M_ij: 65536 / (65536 - t) if the pair is kept, 0 if dropped; 1 without dropout. */
static double dropout_mult(const dropout_t* d, int b, int h, int i, int j) {
    if (!d || d->t == 0) return 1.0;
    return dropout_u16(d, b + d->b0, h + d->h0, i, j) >= (unsigned)d->t ? 65536.0 / (65536.0 - d->t) : 0.0;
}

/* The keep decisions of one (b, h) as bytes [Sq * Skv] (1 kept, 0 dropped), for tests. */
int oracle_dropout_keep(int b, int h, int Sq, int Skv, int t, uint64_t seed, uint64_t offset,
                        unsigned char* keep) {
    if (t < 0 || t > 65535 || b < 0 || b > 65535 || h < 0 || h > 65535) return -1;
    dropout_t d = {t, seed, offset, 0, 0};
#pragma omp parallel for schedule(static)
    for (int i = 0; i < Sq; i++)
        for (int j = 0; j < Skv; j++)
            keep[(size_t)i * Skv + j] = dropout_u16(&d, b, h, i, j) >= (unsigned)t;
    return 0;
}

/* The sink logit c of query head h (see the readings above). */
static double sink_logit(int softmax_type, const double* offset, int h) {
    if (softmax_type == ORACLE_OFF_BY_ONE) return 0.0;
    if (softmax_type == ORACLE_LEARNABLE) return offset[h];
    return -INFINITY;
}

/*
 * Probabilities of one (b, h): P[i*Skv + j] for every visible pair, 0 elsewhere,
 * plus LSE_i and p_sink_i.  Steps "score" and "scale + softmax" of the codelab,
 * with the sink logit joining the max and the denominator.
 */
static void probs_one_head(const double* q, const double* k, int b, int h, int g,
                           int Sq, int Skv, int Hq, int Hkv, int dqk,
                           double scale, int causal, int window, double c, const double* bias,
                           double* P, double* lse, double* psink) {
#pragma omp parallel for schedule(static)
    for (int i = 0; i < Sq; i++) {
        double* row = P + (size_t)i * Skv;
        /* score: s_ij = scale * q_i . k_j, on visible pairs only */
        double m = c; /* running max starts at the sink logit (-inf for vanilla) */
        for (int j = 0; j < Skv; j++) {
            if (!visible(i, j, causal, window)) { row[j] = -INFINITY; continue; }
            double s = 0.0;
            for (int t = 0; t < dqk; t++)
                s += q[bshd(b, i, h, t, Sq, Hq, dqk)] * k[bshd(b, j, g, t, Skv, Hkv, dqk)];
            s *= scale;
            if (bias) s += bias[(size_t)i * Skv + j]; /* this (b, h)'s bias plane, or NULL */
            row[j] = s;
            if (s > m) m = s;
        }
        double z = 0.0;
        if (m == -INFINITY) { /* no visible key (or all biased to -inf) and no sink: empty row */
            for (int j = 0; j < Skv; j++) row[j] = 0.0;
            lse[i] = -INFINITY;
            psink[i] = 0.0;
            continue;
        }
        if (c != -INFINITY) z += exp(c - m);
        for (int j = 0; j < Skv; j++)
            if (row[j] != -INFINITY) z += exp(row[j] - m);
        for (int j = 0; j < Skv; j++)
            row[j] = (row[j] == -INFINITY) ? 0.0 : exp(row[j] - m) / z;
        lse[i] = m + log(z);
        psink[i] = (c == -INFINITY) ? 0.0 : exp(c - lse[i]);
    }
}

/*
 * Forward.  o: [B,Sq,Hq,dv]; lse, psink, rowsum: [B,Hq,Sq] (psink/rowsum may be
 * NULL).  rowsum_i = sum_j P_ij (1 for vanilla, 1 - p_sink for the sink types).
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_fwd(const double* q, const double* k, const double* v,
               int B, int Sq, int Skv, int Hq, int Hkv, int dqk, int dv,
               double scale, int causal, int window, int softmax_type, const double* offset,
               const double* bias, int Bb, int Hb, int drop_t, uint64_t seed, uint64_t offset_rng,
               int drop_b0, int drop_h0,
               double* o, double* lse, double* psink, double* rowsum) {
    if (B < 0 || Sq < 0 || Skv < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return -1;
    if (drop_t < 0 || drop_t > 65535 || drop_b0 < 0 || drop_h0 < 0) return -1;
    if (drop_t > 0 && ((long)drop_b0 + B > 65536 || (long)drop_h0 + Hq > 65536)) return -1;
    dropout_t drop = {drop_t, seed, offset_rng, drop_b0, drop_h0};
    if (bias && ((Bb != 1 && Bb != B) || (Hb != 1 && Hb != Hq))) return -1;
    if (softmax_type == ORACLE_LEARNABLE && !offset) return -1;
    if (dqk > ORACLE_MAX_D || dv > ORACLE_MAX_D) return -1;
    int G = Hq / Hkv;
    double* P = (double*)malloc(sizeof(double) * ((size_t)Sq * Skv + 1));
    double* ps = (double*)malloc(sizeof(double) * ((size_t)Sq + 1));
    if (!P || !ps) { free(P); free(ps); return -1; }
    for (int b = 0; b < B; b++) {
        for (int h = 0; h < Hq; h++) {
            int g = h / G;
            double c = sink_logit(softmax_type, offset, h);
            double* lrow = lse + ((size_t)b * Hq + h) * Sq;
            probs_one_head(q, k, b, h, g, Sq, Skv, Hq, Hkv, dqk, scale, causal, window, c,
                           bias_plane(bias, Bb, Hb, b, h, Sq, Skv), P, lrow, ps);
            /* attend: O_i = sum_j P_ij M_ij v_j  (M = 1 without dropout) */
#pragma omp parallel for schedule(static)
            for (int i = 0; i < Sq; i++) {
                double acc[ORACLE_MAX_D];
                for (int t = 0; t < dv; t++) acc[t] = 0.0;
                for (int j = 0; j < Skv; j++) {
                    double pij = P[(size_t)i * Skv + j];
                    if (pij == 0.0) continue;
                    pij *= dropout_mult(&drop, b, h, i, j);
                    for (int t = 0; t < dv; t++) acc[t] += pij * v[bshd(b, j, g, t, Skv, Hkv, dv)];
                }
                for (int t = 0; t < dv; t++) o[bshd(b, i, h, t, Sq, Hq, dv)] = acc[t];
                if (rowsum) {
                    double r = 0.0;
                    for (int j = 0; j < Skv; j++) r += P[(size_t)i * Skv + j];
                    rowsum[((size_t)b * Hq + h) * Sq + i] = r;
                }
                if (psink) psink[((size_t)b * Hq + h) * Sq + i] = ps[i];
            }
        }
    }
    free(P);
    free(ps);
    return 0;
}

/*
 * Backward.  Inputs q,k,v,dout (BSHD).  Outputs dq [B,Sq,Hq,dqk], dk [B,Skv,Hkv,dqk],
 * dv [B,Skv,Hkv,dv], d_offset [Hq] (may be NULL unless learnable; written for
 * every type, zero for vanilla / off-by-one since they have no parameter),
 * Dout [B,Hq,Sq] = dO_i . O_i (may be NULL).  Recomputes P and O from scratch.
 */
int oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
               int B, int Sq, int Skv, int Hq, int Hkv, int dqk, int dv,
               double scale, int causal, int window, int softmax_type, const double* offset,
               const double* bias, int Bb, int Hb, int drop_t, uint64_t seed, uint64_t offset_rng,
               int drop_b0, int drop_h0,
               double* dq, double* dk, double* dvout, double* d_offset, double* Dout, double* dbias) {
    if (B < 0 || Sq < 0 || Skv < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv) return -1;
    if (drop_t < 0 || drop_t > 65535 || drop_b0 < 0 || drop_h0 < 0) return -1;
    if (drop_t > 0 && ((long)drop_b0 + B > 65536 || (long)drop_h0 + Hq > 65536)) return -1;
    dropout_t drop = {drop_t, seed, offset_rng, drop_b0, drop_h0};
    if (bias && ((Bb != 1 && Bb != B) || (Hb != 1 && Hb != Hq))) return -1;
    if (softmax_type == ORACLE_LEARNABLE && !offset) return -1;
    if (dqk > ORACLE_MAX_D || dv > ORACLE_MAX_D) return -1;
    int G = Hq / Hkv;
    size_t nP = (size_t)Sq * Skv + 1;
    double* P = (double*)malloc(sizeof(double) * nP);
    double* dS = (double*)malloc(sizeof(double) * nP);
    double* Mk = (double*)malloc(sizeof(double) * nP); /* M_ij of the current (b, h) */
    double* O = (double*)malloc(sizeof(double) * ((size_t)Sq * dv + 1));
    double* D = (double*)malloc(sizeof(double) * ((size_t)Sq + 1));
    double* lse = (double*)malloc(sizeof(double) * ((size_t)Sq + 1));
    double* ps = (double*)malloc(sizeof(double) * ((size_t)Sq + 1));
    if (!P || !dS || !Mk || !O || !D || !lse || !ps) {
        free(P); free(dS); free(Mk); free(O); free(D); free(lse); free(ps);
        return -1;
    }
    memset(dk, 0, sizeof(double) * (size_t)B * Skv * Hkv * dqk);
    memset(dvout, 0, sizeof(double) * (size_t)B * Skv * Hkv * dv);
    if (d_offset) for (int h = 0; h < Hq; h++) d_offset[h] = 0.0;
    if (bias && dbias) memset(dbias, 0, sizeof(double) * (size_t)Bb * Hb * Sq * Skv);

    for (int b = 0; b < B; b++) {
        for (int h = 0; h < Hq; h++) {
            int g = h / G;
            double c = sink_logit(softmax_type, offset, h);
            probs_one_head(q, k, b, h, g, Sq, Skv, Hq, Hkv, dqk, scale, causal, window, c,
                           bias_plane(bias, Bb, Hb, b, h, Sq, Skv), P, lse, ps);
#pragma omp parallel for schedule(static)
            for (int i = 0; i < Sq; i++)
                for (int j = 0; j < Skv; j++) Mk[(size_t)i * Skv + j] = dropout_mult(&drop, b, h, i, j);
#pragma omp parallel for schedule(static)
            for (int i = 0; i < Sq; i++) {
                /* O_i = sum_j P_ij M_ij v_j, then D_i = dO_i . O_i */
                double acc[ORACLE_MAX_D];
                for (int t = 0; t < dv; t++) acc[t] = 0.0;
                for (int j = 0; j < Skv; j++) {
                    double pij = P[(size_t)i * Skv + j] * Mk[(size_t)i * Skv + j];
                    if (pij == 0.0) continue;
                    for (int t = 0; t < dv; t++) acc[t] += pij * v[bshd(b, j, g, t, Skv, Hkv, dv)];
                }
                double Di = 0.0;
                for (int t = 0; t < dv; t++) {
                    O[(size_t)i * dv + t] = acc[t];
                    Di += dout[bshd(b, i, h, t, Sq, Hq, dv)] * acc[t];
                }
                D[i] = Di;
                /* dP~_ij = dO_i . v_j ; dS_ij = P_ij (M_ij dP~_ij - D_i) */
                for (int j = 0; j < Skv; j++) {
                    double pij = P[(size_t)i * Skv + j];
                    if (pij == 0.0) { dS[(size_t)i * Skv + j] = 0.0; continue; }
                    double dp = 0.0;
                    for (int t = 0; t < dv; t++)
                        dp += dout[bshd(b, i, h, t, Sq, Hq, dv)] * v[bshd(b, j, g, t, Skv, Hkv, dv)];
                    dS[(size_t)i * Skv + j] = pij * (Mk[(size_t)i * Skv + j] * dp - Di);
                }
                /* dQ_i = scale sum_j dS_ij k_j */
                for (int t = 0; t < dqk; t++) acc[t] = 0.0;
                for (int j = 0; j < Skv; j++) {
                    double dsij = dS[(size_t)i * Skv + j];
                    if (dsij == 0.0) continue;
                    for (int t = 0; t < dqk; t++) acc[t] += dsij * k[bshd(b, j, g, t, Skv, Hkv, dqk)];
                }
                for (int t = 0; t < dqk; t++) dq[bshd(b, i, h, t, Sq, Hq, dqk)] = scale * acc[t];
            }
            /* dK_j += scale sum_i dS_ij q_i ; dV_j += sum_i P_ij M_ij dO_i  (sum over the group) */
#pragma omp parallel for schedule(static)
            for (int j = 0; j < Skv; j++) {
                double ak[ORACLE_MAX_D], av[ORACLE_MAX_D];
                for (int t = 0; t < dqk; t++) ak[t] = 0.0;
                for (int t = 0; t < dv; t++) av[t] = 0.0;
                for (int i = 0; i < Sq; i++) {
                    double dsij = dS[(size_t)i * Skv + j], pij = P[(size_t)i * Skv + j];
                    if (pij == 0.0) continue;
                    double pm = pij * Mk[(size_t)i * Skv + j];
                    for (int t = 0; t < dqk; t++) ak[t] += dsij * q[bshd(b, i, h, t, Sq, Hq, dqk)];
                    for (int t = 0; t < dv; t++) av[t] += pm * dout[bshd(b, i, h, t, Sq, Hq, dv)];
                }
                for (int t = 0; t < dqk; t++) dk[bshd(b, j, g, t, Skv, Hkv, dqk)] += scale * ak[t];
                for (int t = 0; t < dv; t++) dvout[bshd(b, j, g, t, Skv, Hkv, dv)] += av[t];
            }
            /* dbias_ij += dS_ij (the scores' gradient, summed over the (b, h) sharing it) */
            if (bias && dbias) {
                double* plane = (double*)bias_plane(dbias, Bb, Hb, b, h, Sq, Skv);
#pragma omp parallel for schedule(static)
                for (int i = 0; i < Sq; i++)
                    for (int j = 0; j < Skv; j++) plane[(size_t)i * Skv + j] += dS[(size_t)i * Skv + j];
            }
            /* d offset_h = -sum_i p_sink_i D_i  (learnable only; a sum over b too) */
            if (softmax_type == ORACLE_LEARNABLE && d_offset) {
                double acc = 0.0;
                for (int i = 0; i < Sq; i++) acc += ps[i] * D[i];
                d_offset[h] -= acc;
            }
            if (Dout)
                for (int i = 0; i < Sq; i++) Dout[((size_t)b * Hq + h) * Sq + i] = D[i];
        }
    }
    free(P); free(dS); free(Mk); free(O); free(D); free(lse); free(ps);
    return 0;
}

/* Number of OpenMP threads the oracle runs with (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
