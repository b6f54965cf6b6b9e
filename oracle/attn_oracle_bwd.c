/*
 * attn_oracle_bwd.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of the gradients of the attention
 * forward pass (the backward pass the CUDA library computes).  Only the test
 * suite and the benchmark's CPU-baseline leg may load it; the library never
 * does.  It shares no code, header, table or constant with the CUDA path.
 *
 * Forward (per batch b, query head h, query row i; kvh = h / (H_q / H_kv)):
 *   S_ij = scale * q_i . k_j (+ additive mask), -inf where not allowed
 *   P_ij = exp(S_ij - max_j S_ij) / sum_j exp(...)         (the softmax row)
 *   O_i  = sum_j P_ij v_j
 * Given dO = dLoss/dO, the chain rule through O = P V and the softmax gives
 *   dP_ij = dO_i . v_j
 *   dS_ij = P_ij * (dP_ij - sum_k P_ik dP_ik)               (softmax Jacobian)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_{h in group, i} dS_ij q_i            (summed over the
 *   dV_j  =         sum_{h in group, i} P_ij dO_i             GQA group's heads)
 * Rows with no allowed key have P = 0 and contribute nothing.  The mask and
 * the scale receive no gradient.
 *
 * Allowed keys follow the forward's definition: j <= i + q_offset when
 * causal (q_offset 0 = top-left), and with a sliding window (window > 0)
 * j > i + q_offset - window as well.  With a softcap c > 0 the forward's
 * scaled score s becomes t = c tanh(s / c) before any mask, so the chain rule
 * multiplies dS by dt/ds = 1 - tanh(s / c)^2.  With dropout the forward's
 * weights are W_ij = P_ij Z_ij, Z_ij in {0, 1/(1-p)} (the multipliers are an
 * input here, drawn by the forward oracle's generator), so
 *   dV_j  = sum_i P_ij Z_ij dO_i,   D_i = sum_j P_ij Z_ij dP_ij  (= dO_i . O_i),
 *   dS_ij = P_ij (Z_ij dP_ij - D_i).
 *
 * Sources (web pages on the FlashAttention-2 forward and backward):
 *  - forge "flash_attention_mma.metal", section "backward (MMA)": the three
 *    products per block (S = Q K^T, dP = dO V^T, dS = P (dP - D) scale,
 *    dQ += dS K; transposed, dV += P^T dO and dK += dS^T Q), the dK/dV
 *    accumulation private to one K/V block (summed over the query heads that
 *    share it), and the causal bound.
 *  - mlx-native "ops/flash_attn_train.rs", section "Phase 2 -- FA-2 backward
 *    kernel (dQ, dK, dV)": D[b,h,i] = rowsum(O * dO), dQ/dK/dV shapes
 *    [B,H_q,qL,D] / [B,H_kv,kL,D].
 * Here D_i is written as sum_j P_ij dP_ij, its definition from the softmax
 * Jacobian; rowsum(O * dO) is the same number (O_i = sum_j P_ij v_j), which is
 * the identity the GPU path uses.
 *
 * The definition is written out row by row, no blocking: for each (b, kvh)
 * group one thread walks every head of the group and every query row, so the
 * dK/dV sums of a group are owned by one thread.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ORACLE_MUTANT plants one known mistake (tests only build these variants to
 * show that the pins catch each of them).  0 = the oracle as specified. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

typedef struct {
    const double *q, *k, *v, *dO;
    const void *mask;
    int mask_kind;
    double *dq, *dk, *dv;
    long long B, Hq, Hkv, qL, kL, D;
    double scale;
    int causal;
    long long window, q_offset;  /* 0: off / top-left */
    double softcap;              /* <= 0: off */
    const double *keep;          /* [B, Hq, qL, kL] dropout multipliers, or NULL */
    long long g_begin, g_end;   /* this worker's (b, kvh) groups */
    double *S, *P, *dP, *G;     /* kL doubles each (G: dt/ds of the softcap, 1 without) */
} bwd_job;

static void bwd_group(const bwd_job *J, long long grp)
{
    const long long D = J->D, kL = J->kL, qL = J->qL;
    const long long b = grp / J->Hkv, kvh = grp % J->Hkv;
    const long long group = J->Hq / J->Hkv;
    const double *kb = J->k + (b * J->Hkv + kvh) * kL * D;
    const double *vb = J->v + (b * J->Hkv + kvh) * kL * D;
    double *dkb = J->dk + (b * J->Hkv + kvh) * kL * D;
    double *dvb = J->dv + (b * J->Hkv + kvh) * kL * D;
    double *S = J->S, *P = J->P, *dP = J->dP;
    memset(dkb, 0, sizeof(double) * (size_t)(kL * D));
    memset(dvb, 0, sizeof(double) * (size_t)(kL * D));
    for (long long r = 0; r < group; ++r) {
#if ORACLE_MUTANT == 4
        const long long h = kvh + r * J->Hkv;          /* mistake: wrong heads summed into dK/dV */
#else
        const long long h = kvh * group + r;
#endif
        for (long long i = 0; i < qL; ++i) {
            const double *qi = J->q + ((b * J->Hq + h) * qL + i) * D;
            const double *doi = J->dO + ((b * J->Hq + h) * qL + i) * D;
            double *dqi = J->dq + ((b * J->Hq + h) * qL + i) * D;
            /* the score row and its softmax */
            double m = -INFINITY;
            for (long long j = 0; j < kL; ++j) {
                double dot = 0.0;
                for (long long d = 0; d < D; ++d) dot += qi[d] * kb[j * D + d];
                double s = J->scale * dot;
                J->G[j] = 1.0;
                if (J->softcap > 0.0) {
                    const double th = tanh(s / J->softcap);
                    s = J->softcap * th;
                    J->G[j] = 1.0 - th * th;
                }
                const long long diag = i + J->q_offset;   /* the key aligned with row i */
#if ORACLE_MUTANT == 5
                int allowed = !J->causal || j < diag;     /* mistake: causal off by one */
#elif ORACLE_MUTANT == 7
                int allowed = !J->causal || j <= i - J->q_offset;   /* mistake: offset sign */
#else
                int allowed = !J->causal || j <= diag;
#endif
#if ORACLE_MUTANT == 8
                if (J->window > 0) allowed = allowed && (j >= diag - J->window);  /* mistake: one key too wide */
#else
                if (J->window > 0) allowed = allowed && (j > diag - J->window);
#endif
                if (J->mask_kind == 1) {
                    allowed = allowed && ((const uint8_t *)J->mask)[((b * J->Hq + h) * qL + i) * kL + j] != 0;
                } else if (J->mask_kind == 2) {
                    s += ((const double *)J->mask)[((b * J->Hq + h) * qL + i) * kL + j];
                    allowed = allowed && (s != -INFINITY);
                }
                S[j] = allowed ? s : -INFINITY;
                if (S[j] > m) m = S[j];
            }
            for (long long d = 0; d < D; ++d) dqi[d] = 0.0;
            if (m == -INFINITY) continue;              /* no allowed key: no gradient */
            double l = 0.0;
            for (long long j = 0; j < kL; ++j) { P[j] = exp(S[j] - m); l += P[j]; }
            for (long long j = 0; j < kL; ++j) P[j] /= l;
            /* dP_ij = dO_i . v_j and D_i = sum_j P_ij dP_ij */
            const double *zi = J->keep ? J->keep + ((b * J->Hq + h) * qL + i) * kL : NULL;
            double Di = 0.0;
            for (long long j = 0; j < kL; ++j) {
                double dot = 0.0;
                for (long long d = 0; d < D; ++d) dot += doi[d] * vb[j * D + d];
                dP[j] = zi ? zi[j] * dot : dot;      /* dLoss/dP_ij through the dropped weight */
                Di += P[j] * dP[j];
            }
            for (long long j = 0; j < kL; ++j) {
                if (P[j] == 0.0) continue;
#if ORACLE_MUTANT == 2
                const double dS = P[j] * (dP[j] + Di) * J->G[j];   /* mistake: sign of the D term */
#elif ORACLE_MUTANT == 9
                const double dS = P[j] * (dP[j] - Di);             /* mistake: softcap derivative dropped */
#else
                const double dS = P[j] * (dP[j] - Di) * J->G[j];
#endif
                for (long long d = 0; d < D; ++d) {
                    dqi[d] += J->scale * dS * kb[j * D + d];
#if ORACLE_MUTANT == 1
                    dkb[j * D + d] += dS * qi[d];               /* mistake: scale dropped from dK */
#else
                    dkb[j * D + d] += J->scale * dS * qi[d];
#endif
#if ORACLE_MUTANT == 3
                    dvb[j * D + d] += P[j] * qi[d];             /* mistake: q in place of dO */
#elif ORACLE_MUTANT == 10
                    dvb[j * D + d] += P[j] * doi[d];            /* mistake: dropout dropped from dV */
#else
                    dvb[j * D + d] += (zi ? P[j] * zi[j] : P[j]) * doi[d];
#endif
                }
            }
#if ORACLE_MUTANT == 6
            for (long long d = 0; d < D; ++d) dqi[d] = -dqi[d];  /* mistake: dQ sign */
#endif
        }
    }
}

static void *bwd_worker(void *arg)
{
    bwd_job *J = (bwd_job *)arg;
    for (long long g = J->g_begin; g < J->g_end; ++g) bwd_group(J, g);
    return NULL;
}

/*
 * oracle_attention_bwd -- fp64 gradients dQ, dK, dV of the attention forward.
 *
 * q, dO [B,Hq,qL,D]; k, v [B,Hkv,kL,D]; contiguous fp64 holding the exact
 * stored values.  mask: NULL for mask_kind 0, else [B,Hq,qL,kL] contiguous
 * uint8 (kind 1, nonzero keeps) or fp64 (kind 2, added to the scores).
 * dq [B,Hq,qL,D], dk and dv [B,Hkv,kL,D] are written in full.
 * n_threads <= 0 means one thread.  Returns 0, or -1 on a bad argument.
 */
int oracle_attention_bwd_ex(const double *q, const double *k, const double *v, const void *mask, int mask_kind,
                            const double *dO, double *dq, double *dk, double *dv, long long B, long long Hq,
                            long long Hkv, long long qL, long long kL, long long D, double scale, int causal,
                            long long window, long long q_offset, double softcap, const double *keep,
                            int n_threads)
{
    if (!q || !k || !v || !dO || !dq || !dk || !dv) return -1;
    if (window < 0 || !(softcap >= 0.0)) return -1;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || qL <= 0 || kL <= 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if (mask_kind < 0 || mask_kind > 2) return -1;
    if ((mask_kind != 0) != (mask != NULL)) return -1;
    const long long groups = B * Hkv;
    if (n_threads <= 0) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((long long)n_threads > groups) n_threads = (int)groups;
    bwd_job *jobs = (bwd_job *)calloc((size_t)n_threads, sizeof(bwd_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    double *scratch = (double *)malloc(sizeof(double) * 4 * (size_t)kL * (size_t)n_threads);
    if (!jobs || !tids || !scratch) {
        free(jobs); free(tids); free(scratch);
        return -1;
    }
    for (int t = 0; t < n_threads; ++t) {
        bwd_job *J = &jobs[t];
        J->q = q; J->k = k; J->v = v; J->dO = dO; J->mask = mask; J->mask_kind = mask_kind;
        J->dq = dq; J->dk = dk; J->dv = dv;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->qL = qL; J->kL = kL; J->D = D;
        J->scale = scale; J->causal = causal;
        J->window = window; J->q_offset = q_offset; J->softcap = softcap; J->keep = keep;
        J->g_begin = groups * t / n_threads;
        J->g_end = groups * (t + 1) / n_threads;
        J->S = scratch + (size_t)kL * (4 * (size_t)t);
        J->P = J->S + kL;
        J->dP = J->P + kL;
        J->G = J->dP + kL;
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tids[t], NULL, bwd_worker, &jobs[t]) != 0) break;
        started = t;
    }
    bwd_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    for (int t = started + 1; t < n_threads; ++t) bwd_worker(&jobs[t]);
    free(jobs); free(tids); free(scratch);
    return 0;
}

/* The plain gradients: no window, top-left causal, no softcap. */
int oracle_attention_bwd(const double *q, const double *k, const double *v, const void *mask, int mask_kind,
                         const double *dO, double *dq, double *dk, double *dv, long long B, long long Hq,
                         long long Hkv, long long qL, long long kL, long long D, double scale, int causal,
                         int n_threads)
{
    return oracle_attention_bwd_ex(q, k, v, mask, mask_kind, dO, dq, dk, dv, B, Hq, Hkv, qL, kL, D, scale, causal,
                                   0, 0, 0.0, NULL, n_threads);
}

/* Number of the planted mistake this compiled library carries (0 for the real oracle). */
int oracle_bwd_mutant_id(void) { return ORACLE_MUTANT; }
