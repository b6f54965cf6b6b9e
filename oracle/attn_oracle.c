/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of the attention forward pass that the
 * CUDA library computes.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it; the library itself never does.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes (per batch b, query head h, query row i):
 *
 *   kvh      = h / (H_q / H_kv)                         GQA head map
 *   s_ij     = scale * sum_d q[b,h,i,d] * k[b,kvh,j,d]
 *   softcap > 0:  s_ij = softcap * tanh(s_ij / softcap)  (before any mask)
 *   allowed  = (!causal || j <= i + q_offset)            causal; q_offset 0 = top-left
 *   window > 0:   allowed &= (j > i + q_offset - window)  sliding window of `window` keys
 *   dropout p > 0: O_i = sum_j P_ij * keep_ij * v_j with P the softmax row above
 *                  (its l uses every allowed key) and keep_ij = 1 / (1 - p) or 0
 *                  from a counter-based generator (below); L is unchanged.
 *   bool mask:      allowed &= (mask[b,h,i,j] != 0)      nonzero = keep
 *   additive mask:  s_ij += mask[b,h,i,j];  allowed &= (s_ij != -inf)
 *   S_ij     = allowed ? s_ij : -inf                     (the full score row)
 *   m_i      = max_j S_ij
 *   l_i      = sum_j exp(S_ij - m_i)
 *   O_i      = sum_j exp(S_ij - m_i) * v[b,kvh,j,:] / l_i
 *   L_i      = m_i + ln(l_i)                             natural-log logsumexp
 *   no allowed key:  O_i = 0, L_i = -inf
 *
 * Sources (web pages on the FlashAttention-2 forward):
 *  - mlx-native "ops/flash_attn_train.rs", module doc sections "Algorithm"
 *    (O and L = m + ln l, the FA-2 Algorithm 1 logsumexp) and "Buffer
 *    layout" ([B,H_q,qL,D] Q/O, [B,H_kv,kL,D] K/V, [B,H_q,qL,kL] mask,
 *    [B,H_q,qL] L); validate_params (H_q divisible by H_kv).
 *  - forge "flash_attention_mma.metal", header comment (online softmax, only
 *    L = m + log(l) stored), causal bound "only KV blocks up to the last query
 *    row", GQA map hkv = h / (H / HKV), and the epilogue (l == 0 gives O = 0).
 *  - ruDNN "dense_attention.rs", function `forward`: scale applied to the dot
 *    product first, then the mask; mask kind 1 keeps a key iff the mask value
 *    is nonzero, mask kind 2 adds the value and an additive -inf excludes the
 *    key ("matching the public masked_softmax"); causal keeps token <= row.
 *  - oxibonsai "dit_attention_flash.rs", module doc: full-row max-subtracted
 *    softmax is the CPU reference the flash kernel must match.
 *
 * Dropout generator (ruDNN "dense_attention.rs", functions `keep` and
 * `keep_global`): position = ((b*Hq + h)*qL + i)*kL + j; the Philox4x32-10
 * block cipher (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
 * as 1, 2, 3", SC11) with key (seed_lo, seed_hi) and counter (low 64 bits =
 * offset + position / 4, high 64 bits = 0); word position % 4 of its output,
 * u = (word >> 8) * 2^-24; keep iff u >= p (p = 1 drops everything).
 *
 * Readings where the pages are silent (each listed in the design notes):
 *  - a fully masked row has L = -inf (the empty logsumexp); forge writes 0.
 *  - the mask is added after scaling and is not itself scaled.
 *  - window, softcap and q_offset: the pages only name the fields (forge's
 *    `FlashParams.window`, 0 = off; mlx's `softcapping` and `ql_off`); the
 *    definitions above are the plainest readings of those names.
 *
 * This is the definition written out row by row: the full score row S_i. is
 * materialised, then its max, its exp-sum, O and L.  No online softmax, no
 * blocking, no reordering beyond what the definition states.  Rows are split
 * across POSIX threads; each row is computed independently.
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
    const double *q, *k, *v;     /* q [B,Hq,qL,D], k/v [B,Hkv,kL,D], contiguous */
    const void *mask;            /* [B,Hq,qL,kL] contiguous: uint8 (bool) or double (additive) */
    int mask_kind;               /* 0 none, 1 bool, 2 additive */
    double *o, *lse;             /* o [n_rows or B*Hq*qL, D], lse [...] */
    long long B, Hq, Hkv, qL, kL, D;
    double scale;
    int causal;
    long long window;            /* 0: off */
    double softcap;              /* <= 0: off */
    long long q_offset;
    double dropout_p;            /* 0: off */
    uint64_t seed, offset;       /* dropout generator key and counter offset */
    const long long *rows;       /* optional list of flat rows ((b*Hq+h)*qL+i) */
    long long n_rows;
    long long row_begin, row_end;/* this worker's slice of [0, n_rows) */
    double *scratch;             /* kL doubles for the score row */
    int status;
} oracle_job;

/* Philox4x32-10: ten rounds of the published round function (multipliers
 * 0xD2511F53 and 0xCD9E8D57 on words 0 and 2, Weyl key increments 0x9E3779B9
 * and 0xBB67AE85). */
static void philox4x32_10(const uint32_t ctr[4], uint32_t k0, uint32_t k1, uint32_t out[4])
{
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    for (int r = 0; r < 10; ++r) {
        const uint64_t p0 = (uint64_t)0xD2511F53u * x0;
        const uint64_t p2 = (uint64_t)0xCD9E8D57u * x2;
        const uint32_t y0 = (uint32_t)(p2 >> 32) ^ x1 ^ k0;
        const uint32_t y1 = (uint32_t)p2;
        const uint32_t y2 = (uint32_t)(p0 >> 32) ^ x3 ^ k1;
        const uint32_t y3 = (uint32_t)p0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
#if ORACLE_MUTANT != 14   /* mistake 14: the key is not raised between rounds */
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
#endif
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/* The dropout multiplier of one (b, h, i, j) position: 1 / (1 - p) or 0. */
static double dropout_keep(const oracle_job *J, uint64_t position)
{
    if (J->dropout_p >= 1.0) return 0.0;
    const uint64_t ctr64 = J->offset + position / 4;
    const uint32_t ctr[4] = {(uint32_t)ctr64, (uint32_t)(ctr64 >> 32), 0u, 0u};
    uint32_t out[4];
    philox4x32_10(ctr, (uint32_t)J->seed, (uint32_t)(J->seed >> 32), out);
    const double u = (double)(out[position % 4] >> 8) / 16777216.0;
#if ORACLE_MUTANT == 12
    return u < J->dropout_p ? 1.0 / (1.0 - J->dropout_p) : 0.0;   /* mistake: keep test inverted */
#elif ORACLE_MUTANT == 13
    return u >= J->dropout_p ? 1.0 : 0.0;                         /* mistake: kept weights not rescaled */
#else
    return u >= J->dropout_p ? 1.0 / (1.0 - J->dropout_p) : 0.0;
#endif
}

static void oracle_row(const oracle_job *J, long long flat, long long out_index, double *S)
{
    const long long D = J->D, kL = J->kL, qL = J->qL;
    const long long i = flat % qL;
    const long long h = (flat / qL) % J->Hq;
    const long long b = flat / (qL * J->Hq);
    const long long group = J->Hq / J->Hkv;
#if ORACLE_MUTANT == 2
    const long long kvh = h % J->Hkv;             /* mistake: wrong GQA map */
#else
    const long long kvh = h / group;
#endif
    const double *qi = J->q + ((b * J->Hq + h) * qL + i) * D;
    const double *kb = J->k + (b * J->Hkv + kvh) * kL * D;
    const double *vb = J->v + (b * J->Hkv + kvh) * kL * D;
    double *oi = J->o + out_index * D;

    /* 1. the full score row, with -inf where a key is not allowed */
    for (long long j = 0; j < kL; ++j) {
        double dot = 0.0;
        for (long long d = 0; d < D; ++d) {
#if ORACLE_MUTANT == 5
            /* mistake: q and k swap roles (transposed product) */
            dot += J->q[((b * J->Hq + h) * qL + (j < qL ? j : 0)) * D + d] * kb[(i < kL ? i : 0) * D + d];
#else
            dot += qi[d] * kb[j * D + d];
#endif
        }
#if ORACLE_MUTANT == 1
        double s = dot;                           /* mistake: scale dropped */
#else
        double s = J->scale * dot;
#endif
        if (J->softcap > 0.0) {
#if ORACLE_MUTANT == 9
            s = tanh(s / J->softcap);             /* mistake: cap not multiplied back */
#else
            s = J->softcap * tanh(s / J->softcap);
#endif
        }
        const long long diag = i + J->q_offset;   /* the key aligned with row i */
#if ORACLE_MUTANT == 3
        int allowed = !J->causal || j < diag;     /* mistake: causal off by one */
#elif ORACLE_MUTANT == 10
        int allowed = !J->causal || j <= i - J->q_offset;  /* mistake: offset sign */
#else
        int allowed = !J->causal || j <= diag;
#endif
        if (J->window > 0) {
#if ORACLE_MUTANT == 11
            allowed = allowed && (j >= diag - J->window);  /* mistake: window one key too wide */
#else
            allowed = allowed && (j > diag - J->window);
#endif
        }
        if (J->mask_kind == 1) {
            const uint8_t mv = ((const uint8_t *)J->mask)[((b * J->Hq + h) * qL + i) * kL + j];
#if ORACLE_MUTANT == 7
            allowed = allowed && (mv == 0);       /* mistake: bool polarity flipped */
#else
            allowed = allowed && (mv != 0);
#endif
        } else if (J->mask_kind == 2) {
            const double mv = ((const double *)J->mask)[((b * J->Hq + h) * qL + i) * kL + j];
#if ORACLE_MUTANT == 6
            s += J->scale * mv;                   /* mistake: mask scaled with the scores */
#else
            s += mv;
#endif
            allowed = allowed && (s != -INFINITY);
        }
        S[j] = allowed ? s : -INFINITY;
    }

    /* 2. row max */
    double m = -INFINITY;
    for (long long j = 0; j < kL; ++j)
        if (S[j] > m) m = S[j];

    if (m == -INFINITY) {                          /* no allowed key */
        for (long long d = 0; d < D; ++d) oi[d] = 0.0;
        J->lse[out_index] = -INFINITY;
        return;
    }

    /* 3. l = sum exp(S - m); O = sum exp(S - m) v / l; L = m + ln l */
    double l = 0.0;
    for (long long j = 0; j < kL; ++j) l += exp(S[j] - m);
    for (long long d = 0; d < D; ++d) oi[d] = 0.0;
    for (long long j = 0; j < kL; ++j) {
        double p = exp(S[j] - m);
        if (p == 0.0) continue;                    /* exp(-inf) = 0 contributes nothing */
        if (J->dropout_p > 0.0) p *= dropout_keep(J, (uint64_t)(flat * kL + j));
        for (long long d = 0; d < D; ++d) oi[d] += p * vb[j * D + d];
    }
#if ORACLE_MUTANT != 8
    for (long long d = 0; d < D; ++d) oi[d] /= l;  /* mutant 8 omits the division by l */
#endif
#if ORACLE_MUTANT == 4
    J->lse[out_index] = log(l);                    /* mistake: max term dropped from L */
#else
    J->lse[out_index] = m + log(l);
#endif
}

static void *oracle_worker(void *arg)
{
    oracle_job *J = (oracle_job *)arg;
    for (long long r = J->row_begin; r < J->row_end; ++r) {
        const long long flat = J->rows ? J->rows[r] : r;
        oracle_row(J, flat, r, J->scratch);
    }
    return NULL;
}

/*
 * oracle_attention_ex -- fp64 attention forward, O and L.
 *
 * q [B,Hq,qL,D], k and v [B,Hkv,kL,D], contiguous fp64 holding the exact
 * stored input values.  mask: NULL for mask_kind 0, else [B,Hq,qL,kL]
 * contiguous uint8 (mask_kind 1) or fp64 (mask_kind 2).
 * rows == NULL: every row is computed; o is [B*Hq*qL, D] and lse [B*Hq*qL].
 * rows != NULL: only the n_rows listed flat rows ((b*Hq + h)*qL + i) are
 * computed; o is [n_rows, D] and lse [n_rows], in list order.
 * window (0 = off), softcap (<= 0 = off), q_offset and dropout (p = 0 off,
 * seed, offset) as in the header.
 * n_threads <= 0 means one thread.  Returns 0, or -1 on a bad argument.
 */
int oracle_attention_ex(const double *q, const double *k, const double *v,
                        const void *mask, int mask_kind, double *o, double *lse,
                        long long B, long long Hq, long long Hkv, long long qL,
                        long long kL, long long D, double scale, int causal,
                        long long window, double softcap, long long q_offset,
                        double dropout_p, uint64_t seed, uint64_t offset,
                        const long long *rows, long long n_rows, int n_threads)
{
    if (!q || !k || !v || !o || !lse) return -1;
    if (window < 0) return -1;
    if (!(dropout_p >= 0.0 && dropout_p <= 1.0)) return -1;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || qL <= 0 || kL <= 0 || D <= 0) return -1;
    if (Hq % Hkv != 0) return -1;
    if (mask_kind < 0 || mask_kind > 2) return -1;
    if ((mask_kind != 0) != (mask != NULL)) return -1;

    const long long total = rows ? n_rows : B * Hq * qL;
    if (rows) {
        for (long long r = 0; r < n_rows; ++r)
            if (rows[r] < 0 || rows[r] >= B * Hq * qL) return -1;
    }
    if (n_threads <= 0) n_threads = 1;
    if (n_threads > 256) n_threads = 256;
    if ((long long)n_threads > total) n_threads = (int)(total > 0 ? total : 1);

    oracle_job *jobs = (oracle_job *)calloc((size_t)n_threads, sizeof(oracle_job));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    double *scratch = (double *)malloc(sizeof(double) * (size_t)kL * (size_t)n_threads);
    if (!jobs || !tids || !scratch) {
        free(jobs); free(tids); free(scratch);
        return -1;
    }
    for (int t = 0; t < n_threads; ++t) {
        oracle_job *J = &jobs[t];
        J->q = q; J->k = k; J->v = v; J->mask = mask; J->mask_kind = mask_kind;
        J->o = o; J->lse = lse;
        J->B = B; J->Hq = Hq; J->Hkv = Hkv; J->qL = qL; J->kL = kL; J->D = D;
        J->scale = scale; J->causal = causal; J->rows = rows; J->n_rows = total;
        J->window = window; J->softcap = softcap; J->q_offset = q_offset;
        J->dropout_p = dropout_p; J->seed = seed; J->offset = offset;
        J->row_begin = total * t / n_threads;
        J->row_end = total * (t + 1) / n_threads;
        J->scratch = scratch + (size_t)kL * (size_t)t;
    }
    int started = 0;
    for (int t = 1; t < n_threads; ++t) {
        if (pthread_create(&tids[t], NULL, oracle_worker, &jobs[t]) != 0) break;
        started = t;
    }
    oracle_worker(&jobs[0]);
    for (int t = 1; t <= started; ++t) pthread_join(tids[t], NULL);
    /* any slice whose thread failed to start is computed here */
    for (int t = started + 1; t < n_threads; ++t) oracle_worker(&jobs[t]);

    free(jobs); free(tids); free(scratch);
    return 0;
}

/* The plain definition: no window, no softcap, top-left causal. */
int oracle_attention(const double *q, const double *k, const double *v,
                     const void *mask, int mask_kind, double *o, double *lse,
                     long long B, long long Hq, long long Hkv, long long qL,
                     long long kL, long long D, double scale, int causal,
                     const long long *rows, long long n_rows, int n_threads)
{
    return oracle_attention_ex(q, k, v, mask, mask_kind, o, lse, B, Hq, Hkv, qL, kL, D, scale, causal,
                               0, 0.0, 0, 0.0, 0, 0, rows, n_rows, n_threads);
}

/* The dropout multipliers of `n` consecutive positions starting at `first`
 * (for tests of the generator itself). */
int oracle_dropout_keep(double p, uint64_t seed, uint64_t offset, uint64_t first, long long n, double *out)
{
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.dropout_p = p; J.seed = seed; J.offset = offset;
    for (long long t = 0; t < n; ++t) out[t] = dropout_keep(&J, first + (uint64_t)t);
    return 0;
}

/* One Philox4x32-10 block: the four output words of counter `ctr` under the
 * key (k0, k1), for tests of the generator against an independent copy. */
int oracle_philox4x32_10(const uint32_t *ctr, uint32_t k0, uint32_t k1, uint32_t *out)
{
    philox4x32_10(ctr, k0, k1, out);
    return 0;
}

/* Number of the planted mistake this compiled library carries (0 for the real oracle). */
int oracle_mutant_id(void) { return ORACLE_MUTANT; }
