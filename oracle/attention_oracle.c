/*
 * Attention forward ORACLE -- test infrastructure, not part of the product.
 *
 * A plain, slow, float64 CPU statement of what the fused attention forward
 * computes.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may load it.  It shares no code with the CUDA library.
 *
 * What it computes is the standard attention definition (page "把 FlashAttention
 * 搬上昇腾：Triton-Ascend CV Pipeline 优化实战", section 一: S = Q Kᵀ · scale,
 * P = softmax(S), O = P V), with the extensions that the page "Write Triton
 * Attention Kernel" fixes:
 *   - GQA/MQA: query head hq reads key/value head hq / (Hq / Hkv)
 *     ("Required reasoning process", step 1);
 *   - causal masking keeps key j for query i iff i >= j
 *     (step 5c, the top-left convention for Nq != Nkv);
 *   - the saved log-sum-exp is lse = m + log(l), i.e. the natural log of
 *     sum_j exp(s_ij) over the kept keys (step 8).
 * For each requested row (z, hq, i), in float64 on the exactly upcast
 * fp16/bf16 inputs:
 *   1. s_j   = scale * sum_d Q[z,hq,i,d] K[z,hk,j,d]  for every kept key j
 *   2. M     = max_j s_j,   L = sum_j exp(s_j - M)
 *   3. O[d]  = sum_j (exp(s_j - M) / L) V[z,hk,j,d]
 *   4. lse   = M + ln L
 * The whole row of S is materialised; nothing is tiled, fused or reordered.
 *
 * It also states the combination of results computed over disjoint key sets
 * (oracle_lse_merge below): the sum over a union of key sets is the sum of
 * the per-set sums, so with each set's lse_s = log sum_j exp(s_j) and its
 * normalised O_s, lse = log sum_s exp(lse_s) and O = sum_s exp(lse_s - lse) O_s
 * -- the max-shifted rescaling of the page "Write Triton Attention Kernel"
 * (Kernel design rules) applied to whole sets instead of key blocks.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- exact decoding of the 16-bit storage formats -------------------------- */

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
static double decode_binary16(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double mag;
    if (e == 0) mag = ldexp((double)f, -24);                 /* zero / subnormal */
    else if (e == 31) mag = f ? NAN : INFINITY;
    else mag = ldexp((double)(1024 + f), e - 25);           /* 1.f * 2^(e-15) */
    return sign ? -mag : mag;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
static double decode_bfloat16(uint16_t h) {
    int sign = (h >> 15) & 1, e = (h >> 7) & 0xff, f = h & 0x7f;
    double mag;
    if (e == 0) mag = ldexp((double)f, -133);                /* zero / subnormal */
    else if (e == 255) mag = f ? NAN : INFINITY;
    else mag = ldexp((double)(128 + f), e - 134);           /* 1.f * 2^(e-127) */
    return sign ? -mag : mag;
}

/* Exposed so the tests can check the decoder bit pattern by bit pattern. */
double oracle_decode(uint16_t bits, int dtype) {
    return dtype == 0 ? decode_binary16(bits) : decode_bfloat16(bits);
}

/* ---- one row of the definition --------------------------------------------- */

typedef struct {
    const uint16_t* q;   /* (Z, Hq, Nq, D) bits, contiguous */
    const double* k;     /* (Z, Hkv, Nkv, D) upcast, contiguous */
    const double* v;
    const double* table; /* 65536-entry decode table for q */
    int Z, Hq, Hkv, Nq, Nkv, D;
    double scale;
    int causal;
    const int64_t* rows; /* flat row ids (z*Hq + hq)*Nq + i, or NULL for all rows */
    int64_t nrows;
    double* o;           /* (nrows, D) */
    double* lse;         /* (nrows) */
    int64_t begin, end;  /* this worker's slice of [0, nrows) */
    int status;
} oracle_job;

static void attention_row(const oracle_job* J, int64_t r, double* qrow, double* s, double* out, double* out_lse) {
    const int D = J->D;
    const int64_t i = r % J->Nq;
    const int64_t zh = r / J->Nq;
    const int hq = (int)(zh % J->Hq), z = (int)(zh / J->Hq);
    const int hk = hq / (J->Hq / J->Hkv);
    const double* kh = J->k + ((int64_t)z * J->Hkv + hk) * J->Nkv * D;
    const double* vh = J->v + ((int64_t)z * J->Hkv + hk) * J->Nkv * D;
    const uint16_t* qbits = J->q + r * D;
    for (int d = 0; d < D; ++d) qrow[d] = J->table[qbits[d]];

    /* kept keys: all of them, or j <= i under the causal mask */
    int64_t nkept = J->Nkv;
    if (J->causal && i + 1 < nkept) nkept = i + 1;

    /* 1. scores */
    for (int64_t j = 0; j < nkept; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += qrow[d] * kh[j * D + d];
        s[j] = J->scale * acc;
    }
    /* 2. row maximum and normaliser */
    double M = -INFINITY;
    for (int64_t j = 0; j < nkept; ++j) M = s[j] > M ? s[j] : M;
    double L = 0.0;
    for (int64_t j = 0; j < nkept; ++j) L += exp(s[j] - M);
    /* 3. probabilities times values */
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t j = 0; j < nkept; ++j) {
        const double p = exp(s[j] - M) / L;
        for (int d = 0; d < D; ++d) out[d] += p * vh[j * D + d];
    }
    /* 4. log-sum-exp of the scaled scores */
    *out_lse = M + log(L);
}

static void* oracle_worker(void* arg) {
    oracle_job* J = (oracle_job*)arg;
    double* qrow = (double*)malloc(sizeof(double) * (size_t)J->D);
    double* s = (double*)malloc(sizeof(double) * (size_t)J->Nkv);
    if (!qrow || !s) { J->status = -2; free(qrow); free(s); return NULL; }
    for (int64_t t = J->begin; t < J->end; ++t) {
        const int64_t r = J->rows ? J->rows[t] : t;
        attention_row(J, r, qrow, s, J->o + t * J->D, J->lse + t);
    }
    free(qrow);
    free(s);
    return NULL;
}

/*
 * Attention forward for the rows `rows[0..nrows)` (flat ids (z*Hq + hq)*Nq + i),
 * or for every row in (z, hq, i) order when rows == NULL (then nrows must be
 * Z*Hq*Nq).  q/k/v are contiguous BNSD bit arrays of dtype 0 (fp16) or 1 (bf16).
 * Writes o[nrows*D] and lse[nrows] in float64.
 * Returns 0, -1 for invalid arguments, -2 when memory runs out.
 */
int oracle_attention_fwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype,
                         int Z, int Hq, int Hkv, int Nq, int Nkv, int D, double scale, int causal,
                         const int64_t* rows, int64_t nrows, double* o, double* lse, int nthreads) {
    if (dtype < 0 || dtype > 1 || Z < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 1 || D < 1) return -1;
    if (Hq % Hkv != 0 || !isfinite(scale) || nrows < 0) return -1;
    const int64_t total = (int64_t)Z * Hq * Nq;
    if (!rows && nrows != total) return -1;
    for (int64_t t = 0; rows && t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= total) return -1;
    if (nrows == 0) return 0;

    double* table = (double*)malloc(sizeof(double) * 65536);
    const int64_t nk = (int64_t)Z * Hkv * Nkv * D;
    double* kd = (double*)malloc(sizeof(double) * (size_t)nk);
    double* vd = (double*)malloc(sizeof(double) * (size_t)nk);
    if (!table || !kd || !vd) { free(table); free(kd); free(vd); return -2; }
    for (int b = 0; b < 65536; ++b) table[b] = oracle_decode((uint16_t)b, dtype);
    for (int64_t x = 0; x < nk; ++x) { kd[x] = table[k[x]]; vd[x] = table[v[x]]; }

    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads > nrows) nthreads = (int)nrows;
    oracle_job* jobs = (oracle_job*)calloc((size_t)nthreads, sizeof(oracle_job));
    pthread_t* tid = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    int* created = (int*)calloc((size_t)nthreads, sizeof(int));
    if (!jobs || !tid || !created) { free(jobs); free(tid); free(created); free(table); free(kd); free(vd); return -2; }
    const int64_t chunk = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        oracle_job* J = &jobs[t];
        *J = (oracle_job){q, kd, vd, table, Z, Hq, Hkv, Nq, Nkv, D, scale, causal, rows, nrows, o, lse,
                          (int64_t)t * chunk, (int64_t)t * chunk + chunk < nrows ? (int64_t)t * chunk + chunk : nrows, 0};
        if (J->begin >= J->end) continue;
        if (nthreads > 1 && pthread_create(&tid[t], NULL, oracle_worker, J) == 0) created[t] = 1;
        else oracle_worker(J);
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (created[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs); free(tid); free(created); free(table); free(kd); free(vd);
    return status;
}

/*
 * Combination of nparts results over disjoint key sets, row by row, in
 * float64: o_parts is (nparts, rows, D), lse_parts (nparts, rows), natural
 * log.  For each row: M = max_s lse_s; if M = -inf (no key in any set) the
 * row gets O = 0 and lse = -inf; otherwise
 *   w_s = exp(lse_s - M),  L = sum_s w_s,  O = sum_s w_s O_s / L,  lse = M + ln L.
 * Returns 0, or -1 for invalid arguments.
 */
int oracle_lse_merge(int nparts, const double* o_parts, const double* lse_parts, int64_t rows, int D, double* o,
                     double* lse) {
    if (nparts < 1 || rows < 0 || D < 1) return -1;
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int s = 0; s < nparts; ++s) {
            const double x = lse_parts[(int64_t)s * rows + r];
            M = x > M ? x : M;
        }
        double* out = o + r * D;
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double L = 0.0;
        for (int s = 0; s < nparts; ++s) L += exp(lse_parts[(int64_t)s * rows + r] - M);
        for (int s = 0; s < nparts; ++s) {
            const double w = exp(lse_parts[(int64_t)s * rows + r] - M) / L;
            const double* os = o_parts + ((int64_t)s * rows + r) * D;
            for (int d = 0; d < D; ++d) out[d] += w * os[d];
        }
        lse[r] = M + log(L);
    }
    return 0;
}

/* ---- variants: sliding window, ALiBi, variable-length batches --------------
 *
 * The page "Write Triton Attention Kernel" names windowed attention and ALiBi
 * among the variants such a kernel serves ("Use this when"; "Inputs", item 3)
 * and requires, for variable-length (CSR-style) batches, that each sequence's
 * key loop end at its own length and padding never contribute ("Inputs",
 * item 6; "Correctness requirements").  It gives no formulas; the readings
 * taken, for query row i and key j of one sequence (positions from 0, the
 * top-left convention of the causal mask):
 *   - window: key j is kept iff j >= i - window_left (window_left >= 0) and
 *     j <= i + window_right (window_right >= 0); -1 leaves that side open;
 *     with causal, also j <= i;
 *   - ALiBi: the scaled score gets the linear bias -slope[hq] * |i - j|;
 *   - variable length: sequence z holds query rows cu_q[z] .. cu_q[z+1]-1 and
 *     key rows cu_k[z] .. cu_k[z+1]-1 of packed tensors; its rows attend only
 *     to its own keys.
 * A row with no kept key gets O = 0 and lse = -inf.
 */
typedef struct {
    const uint16_t* q;   /* (Z, Hq, Nq, D) bits, or (1, Hq, total_q, D) when varlen */
    const double* k;     /* (Z, Hkv, Nkv, D) upcast, or (1, Hkv, total_k, D) */
    const double* v;
    const double* table;
    int Z, Hq, Hkv, Nq, Nkv, D;
    double scale;
    int causal, window_left, window_right;
    const double* alibi;                 /* (Hq) slopes or NULL */
    const int32_t* cu_q;                 /* (Z + 1) or NULL */
    const int32_t* cu_k;
    const int64_t* rows;
    int64_t nrows;
    double* o;
    double* lse;
    int64_t begin, end;
    int status;
} oracle_ex_job;

static void attention_row_ex(const oracle_ex_job* J, int64_t r, double* qrow, double* s, double* out,
                             double* out_lse) {
    const int D = J->D;
    const int group = J->Hq / J->Hkv;  /* GQA: query heads per key/value head */
    int64_t i, n_keys;
    int hq, z;
    const double *kh, *vh;
    if (J->cu_q) {
        const int64_t g = r % J->Nq;  /* packed query row */
        hq = (int)(r / J->Nq);
        for (z = 0; z < J->Z && !(g >= J->cu_q[z] && g < J->cu_q[z + 1]); ++z) {}
        if (z == J->Z) {  /* a row of no sequence: not part of the result */
            for (int d = 0; d < D; ++d) out[d] = NAN;
            *out_lse = NAN;
            return;
        }
        i = g - J->cu_q[z];
        n_keys = J->cu_k[z + 1] - J->cu_k[z];
        const int kv_head = hq / group;
        kh = J->k + ((int64_t)kv_head * J->Nkv + J->cu_k[z]) * D;
        vh = J->v + ((int64_t)kv_head * J->Nkv + J->cu_k[z]) * D;
    } else {
        i = r % J->Nq;
        const int64_t zh = r / J->Nq;
        hq = (int)(zh % J->Hq);
        z = (int)(zh / J->Hq);
        n_keys = J->Nkv;
        const int kv_head = hq / group;
        kh = J->k + ((int64_t)z * J->Hkv + kv_head) * J->Nkv * D;
        vh = J->v + ((int64_t)z * J->Hkv + kv_head) * J->Nkv * D;
    }
    const uint16_t* qsrc = J->q + r * D;  /* flat row r of the query tensor */
    for (int d = 0; d < D; ++d) qrow[d] = J->table[qsrc[d]];

    /* kept keys: [lo, hi) */
    int64_t lo = 0, hi = n_keys;
    if (J->causal && i + 1 < hi) hi = i + 1;
    if (J->window_right >= 0 && i + J->window_right + 1 < hi) hi = i + J->window_right + 1;
    if (J->window_left >= 0 && i - J->window_left > lo) lo = i - J->window_left;
    if (lo >= hi) {
        for (int d = 0; d < D; ++d) out[d] = 0.0;
        *out_lse = -INFINITY;
        return;
    }
    const double slope = J->alibi ? J->alibi[hq] : 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += qrow[d] * kh[j * D + d];
        const double dist = (double)(i > j ? i - j : j - i);
        s[j - lo] = J->scale * dot - slope * dist;
    }
    const int64_t n = hi - lo;
    double M = -INFINITY;
    for (int64_t t = 0; t < n; ++t) M = s[t] > M ? s[t] : M;
    double L = 0.0;
    for (int64_t t = 0; t < n; ++t) L += exp(s[t] - M);
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    for (int64_t t = 0; t < n; ++t) {
        const double p = exp(s[t] - M) / L;
        for (int d = 0; d < D; ++d) out[d] += p * vh[(lo + t) * D + d];
    }
    *out_lse = log(L) + M;
}

static void* oracle_ex_worker(void* arg) {
    oracle_ex_job* J = (oracle_ex_job*)arg;
    double* qrow = (double*)malloc(sizeof(double) * (size_t)J->D);
    double* s = (double*)malloc(sizeof(double) * (size_t)(J->Nkv > 0 ? J->Nkv : 1));
    if (!qrow || !s) { J->status = -2; free(qrow); free(s); return NULL; }
    for (int64_t t = J->begin; t < J->end; ++t) {
        const int64_t r = J->rows ? J->rows[t] : t;
        attention_row_ex(J, r, qrow, s, J->o + t * J->D, J->lse + t);
    }
    free(qrow);
    free(s);
    return NULL;
}

/*
 * The attention forward with the variants above.  Without cu_q/cu_k the
 * tensors are (Z, H, N, D) as for oracle_attention_fwd and rows are flat ids
 * (z*Hq + hq)*Nq + i; with them, Z is the number of sequences, the tensors
 * are (1, H, total, D) with Nq = total_q and Nkv = total_k, and rows are flat
 * ids hq*total_q + packed row (a row outside every sequence comes back NaN).
 * alibi (Hq slopes) may be NULL; window_left/right are -1 for an open side.
 * Returns 0, -1 for invalid arguments, -2 when memory runs out.
 */
int oracle_attention_fwd_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, int dtype, int Z, int Hq,
                            int Hkv, int Nq, int Nkv, int D, double scale, int causal, int window_left,
                            int window_right, const double* alibi, const int32_t* cu_q, const int32_t* cu_k,
                            const int64_t* rows, int64_t nrows, double* o, double* lse, int nthreads) {
    if (dtype < 0 || dtype > 1 || Z < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 0 || D < 1) return -1;
    if (Hq % Hkv != 0 || !isfinite(scale) || nrows < 0 || window_left < -1 || window_right < -1) return -1;
    if ((cu_q == NULL) != (cu_k == NULL)) return -1;
    if (cu_q) {
        if (cu_q[0] != 0 || cu_k[0] != 0) return -1;
        for (int z = 0; z < Z; ++z)
            if (cu_q[z + 1] < cu_q[z] || cu_k[z + 1] < cu_k[z]) return -1;
        if (cu_q[Z] > Nq || cu_k[Z] > Nkv) return -1;
    }
    const int64_t total = cu_q ? (int64_t)Hq * Nq : (int64_t)Z * Hq * Nq;
    if (!rows && nrows != total) return -1;
    for (int64_t t = 0; rows && t < nrows; ++t)
        if (rows[t] < 0 || rows[t] >= total) return -1;
    if (nrows == 0) return 0;

    double* table = (double*)malloc(sizeof(double) * 65536);
    const int64_t nk = (cu_q ? (int64_t)Hkv * Nkv : (int64_t)Z * Hkv * Nkv) * D;
    double* kd = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(nk > 0 ? nk : 1));
    if (!table || !kd || !vd) { free(table); free(kd); free(vd); return -2; }
    for (int b = 0; b < 65536; ++b) table[b] = oracle_decode((uint16_t)b, dtype);
    for (int64_t x = 0; x < nk; ++x) { kd[x] = table[k[x]]; vd[x] = table[v[x]]; }

    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads > nrows) nthreads = (int)nrows;
    oracle_ex_job* jobs = (oracle_ex_job*)calloc((size_t)nthreads, sizeof(oracle_ex_job));
    pthread_t* tid = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    int* created = (int*)calloc((size_t)nthreads, sizeof(int));
    if (!jobs || !tid || !created) { free(jobs); free(tid); free(created); free(table); free(kd); free(vd); return -2; }
    const int64_t chunk = (nrows + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        oracle_ex_job* J = &jobs[t];
        *J = (oracle_ex_job){q, kd, vd, table, Z, Hq, Hkv, Nq, Nkv, D, scale, causal, window_left, window_right,
                             alibi, cu_q, cu_k, rows, nrows, o, lse, (int64_t)t * chunk,
                             (int64_t)t * chunk + chunk < nrows ? (int64_t)t * chunk + chunk : nrows, 0};
        if (J->begin >= J->end) continue;
        if (nthreads > 1 && pthread_create(&tid[t], NULL, oracle_ex_worker, J) == 0) created[t] = 1;
        else oracle_ex_worker(J);
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (created[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs); free(tid); free(created); free(table); free(kd); free(vd);
    return status;
}

/* ---- backward ---------------------------------------------------------------
 *
 * Gradients of the forward above (GQA and causal as there) for an upstream
 * gradient dO, the pass the blog "把 FlashAttention 搬上昇腾：Triton-Ascend CV
 * Pipeline 优化实战" describes in section 二 and that the saved lse serves
 * ("Write Triton Attention Kernel", step 8).  Stated from the definition of
 * the softmax, row by row, in float64 on the exactly decoded inputs:
 *   P_ij  = exp(s_ij - M_i) / L_i        (s_ij = scale q_i . k_j, kept keys)
 *   dV_j += P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)     (the softmax Jacobian)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j += scale dS_ij q_i
 * with dK and dV of a key/value head summed over the query heads of its group.
 */
typedef struct {
    const double *q, *k, *v, *dO;    /* decoded (Z,Hq,Nq,D), (Z,Hkv,Nkv,D) x2, (Z,Hq,Nq,D) */
    int Z, Hq, Hkv, Nq, Nkv, D;
    double scale;
    int causal;
    double *dq, *dk, *dv;            /* outputs, float64 */
    int64_t begin, end;              /* this worker's (z, kv head) groups */
    int status;
} oracle_bwd_job;

static void* oracle_bwd_worker(void* arg) {
    oracle_bwd_job* J = (oracle_bwd_job*)arg;
    const int D = J->D, g = J->Hq / J->Hkv;
    double* sc = (double*)malloc(sizeof(double) * (size_t)J->Nkv);
    double* dp = (double*)malloc(sizeof(double) * (size_t)J->Nkv);
    if (!sc || !dp) { J->status = -2; free(sc); free(dp); return NULL; }
    for (int64_t grp = J->begin; grp < J->end; ++grp) {
        const int z = (int)(grp / J->Hkv), hk = (int)(grp % J->Hkv);
        const int64_t kvoff = ((int64_t)z * J->Hkv + hk) * J->Nkv * D;
        const double* kh = J->k + kvoff;
        const double* vh = J->v + kvoff;
        double* dkh = J->dk + kvoff;
        double* dvh = J->dv + kvoff;
        for (int64_t x = 0; x < (int64_t)J->Nkv * D; ++x) { dkh[x] = 0.0; dvh[x] = 0.0; }
        for (int hq = hk * g; hq < hk * g + g; ++hq) {
            const int64_t qoff = ((int64_t)z * J->Hq + hq) * J->Nq * D;
            for (int64_t i = 0; i < J->Nq; ++i) {
                const double* qi = J->q + qoff + i * D;
                const double* gi = J->dO + qoff + i * D;
                double* dqi = J->dq + qoff + i * D;
                int64_t n = J->Nkv;
                if (J->causal && i + 1 < n) n = i + 1;
                double Mx = -INFINITY;  /* row maximum and normaliser of the scaled scores */
                for (int64_t j = 0; j < n; ++j) {
                    double qk = 0.0;
                    for (int d = 0; d < D; ++d) qk += qi[d] * kh[j * D + d];
                    sc[j] = J->scale * qk;
                    Mx = sc[j] > Mx ? sc[j] : Mx;
                }
                double Ls = 0.0;
                for (int64_t j = 0; j < n; ++j) Ls += exp(sc[j] - Mx);
                double rowdot = 0.0;  /* sum_k P_ik dP_ik */
                for (int64_t j = 0; j < n; ++j) {
                    const double pj = exp(sc[j] - Mx) / Ls;
                    double acc = 0.0;
                    for (int d = 0; d < D; ++d) acc += gi[d] * vh[j * D + d];
                    dp[j] = acc;
                    rowdot += pj * acc;
                    for (int d = 0; d < D; ++d) dvh[j * D + d] += pj * gi[d];
                }
                for (int d = 0; d < D; ++d) dqi[d] = 0.0;
                for (int64_t j = 0; j < n; ++j) {
                    const double pj = exp(sc[j] - Mx) / Ls;
                    const double dsj = pj * (dp[j] - rowdot);
                    for (int d = 0; d < D; ++d) {
                        dqi[d] += J->scale * dsj * kh[j * D + d];
                        dkh[j * D + d] += J->scale * dsj * qi[d];
                    }
                }
            }
        }
    }
    free(sc);
    free(dp);
    return NULL;
}

/*
 * Backward of the attention forward: q, dO (Z, Hq, Nq, D) and k, v
 * (Z, Hkv, Nkv, D) contiguous bits of dtype 0 (fp16) or 1 (bf16); writes
 * dq (Z, Hq, Nq, D) and dk, dv (Z, Hkv, Nkv, D) in float64.
 * Returns 0, -1 for invalid arguments, -2 when memory runs out.
 */
int oracle_attention_bwd(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO, int dtype,
                         int Z, int Hq, int Hkv, int Nq, int Nkv, int D, double scale, int causal, double* dq,
                         double* dk, double* dv, int nthreads) {
    if (dtype < 0 || dtype > 1 || Z < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 1 || D < 1) return -1;
    if (Hq % Hkv != 0 || !isfinite(scale)) return -1;
    const int64_t nq = (int64_t)Z * Hq * Nq * D, nk = (int64_t)Z * Hkv * Nkv * D;
    if (nk == 0) return 0;
    double* table = (double*)malloc(sizeof(double) * 65536);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(2 * nq + 2 * nk + 1));
    if (!table || !buf) { free(table); free(buf); return -2; }
    for (int b = 0; b < 65536; ++b) table[b] = oracle_decode((uint16_t)b, dtype);
    double *qd = buf, *gd = buf + nq, *kd = buf + 2 * nq, *vd = buf + 2 * nq + nk;
    for (int64_t x = 0; x < nq; ++x) { qd[x] = table[q[x]]; gd[x] = table[dO[x]]; }
    for (int64_t x = 0; x < nk; ++x) { kd[x] = table[k[x]]; vd[x] = table[v[x]]; }

    const int64_t groups = (int64_t)Z * Hkv;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads > groups) nthreads = (int)groups;
    oracle_bwd_job* jobs = (oracle_bwd_job*)calloc((size_t)nthreads, sizeof(oracle_bwd_job));
    pthread_t* tid = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    int* created = (int*)calloc((size_t)nthreads, sizeof(int));
    if (!jobs || !tid || !created) { free(jobs); free(tid); free(created); free(table); free(buf); return -2; }
    const int64_t chunk = (groups + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        oracle_bwd_job* J = &jobs[t];
        *J = (oracle_bwd_job){qd, kd, vd, gd, Z, Hq, Hkv, Nq, Nkv, D, scale, causal, dq, dk, dv,
                              (int64_t)t * chunk, (int64_t)t * chunk + chunk < groups ? (int64_t)t * chunk + chunk : groups,
                              0};
        if (J->begin >= J->end) continue;
        if (nthreads > 1 && pthread_create(&tid[t], NULL, oracle_bwd_worker, J) == 0) created[t] = 1;
        else oracle_bwd_worker(J);
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (created[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs); free(tid); free(created); free(table); free(buf);
    return status;
}


/*
 * Backward of the attention forward with the window and ALiBi variants
 * (oracle_attention_fwd_ex's readings, dense (Z, H, N, D) tensors): the same
 * steps as oracle_attention_bwd, over each row's kept keys [lo, hi) and with
 * the scaled score s_ij = scale q_i . k_j - slope[hq] |i - j|.  The bias is
 * constant in q, k and v, so the softmax Jacobian and the gradient formulas
 * are those of the plain backward; a row with no kept key contributes
 * nothing (its O is 0).
 */
typedef struct {
    const double *q, *k, *v, *dO;
    int Z, Hq, Hkv, Nq, Nkv, D;
    double scale;
    int causal, window_left, window_right;
    const double* alibi;             /* (Hq) slopes or NULL */
    double *dq, *dk, *dv;
    int64_t begin, end;
    int status;
} oracle_bwd_ex_job;

static void* oracle_bwd_ex_worker(void* arg) {
    oracle_bwd_ex_job* J = (oracle_bwd_ex_job*)arg;
    const int D = J->D, g = J->Hq / J->Hkv;
    double* se = (double*)malloc(sizeof(double) * (size_t)J->Nkv);
    double* dpe = (double*)malloc(sizeof(double) * (size_t)J->Nkv);
    if (!se || !dpe) { J->status = -2; free(se); free(dpe); return NULL; }
    for (int64_t grp = J->begin; grp < J->end; ++grp) {
        const int z = (int)(grp / J->Hkv), hk = (int)(grp % J->Hkv);
        const int64_t kvoff = ((int64_t)z * J->Hkv + hk) * J->Nkv * D;
        const double* kb = J->k + kvoff;
        const double* vb = J->v + kvoff;
        double* dkb = J->dk + kvoff;
        double* dvb = J->dv + kvoff;
        for (int64_t x = 0; x < (int64_t)J->Nkv * D; ++x) { dkb[x] = 0.0; dvb[x] = 0.0; }
        for (int hq = hk * g; hq < hk * g + g; ++hq) {
            const int64_t qoff = ((int64_t)z * J->Hq + hq) * J->Nq * D;
            const double slope = J->alibi ? J->alibi[hq] : 0.0;
            for (int64_t i = 0; i < J->Nq; ++i) {
                const double* qr = J->q + qoff + i * D;
                const double* gr = J->dO + qoff + i * D;
                double* dqr = J->dq + qoff + i * D;
                for (int d = 0; d < D; ++d) dqr[d] = 0.0;
                int64_t klo = 0, khi = J->Nkv;  /* kept keys [klo, khi) */
                if (J->causal && i + 1 < khi) khi = i + 1;
                if (J->window_right >= 0 && i + J->window_right + 1 < khi) khi = i + J->window_right + 1;
                if (J->window_left >= 0 && i - J->window_left > klo) klo = i - J->window_left;
                if (klo >= khi) continue;
                double Mr = -INFINITY;
                for (int64_t j = klo; j < khi; ++j) {
                    double dotk = 0.0;
                    for (int d = 0; d < D; ++d) dotk += qr[d] * kb[j * D + d];
                    const double gap = (double)(i > j ? i - j : j - i);
                    se[j] = J->scale * dotk - slope * gap;
                    Mr = se[j] > Mr ? se[j] : Mr;
                }
                double Lr = 0.0;
                for (int64_t j = klo; j < khi; ++j) Lr += exp(se[j] - Mr);
                double rsum = 0.0;  /* sum_k P_ik dP_ik */
                for (int64_t j = klo; j < khi; ++j) {
                    const double pe = exp(se[j] - Mr) / Lr;
                    double dov = 0.0;
                    for (int d = 0; d < D; ++d) dov += gr[d] * vb[j * D + d];
                    dpe[j] = dov;
                    rsum += pe * dov;
                    for (int d = 0; d < D; ++d) dvb[j * D + d] += pe * gr[d];
                }
                for (int64_t j = klo; j < khi; ++j) {
                    const double pe = exp(se[j] - Mr) / Lr;
                    const double dse = pe * (dpe[j] - rsum);
                    for (int d = 0; d < D; ++d) {
                        dqr[d] += J->scale * dse * kb[j * D + d];
                        dkb[j * D + d] += J->scale * dse * qr[d];
                    }
                }
            }
        }
    }
    free(se);
    free(dpe);
    return NULL;
}

/*
 * The backward with window_left/window_right (-1: an open side) and ALiBi
 * slopes (Hq values, or NULL), tensors as for oracle_attention_bwd.
 * Returns 0, -1 for invalid arguments, -2 when memory runs out.
 */
int oracle_attention_bwd_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dO, int dtype,
                            int Z, int Hq, int Hkv, int Nq, int Nkv, int D, double scale, int causal,
                            int window_left, int window_right, const double* alibi, double* dq, double* dk,
                            double* dv, int nthreads) {
    if (dtype < 0 || dtype > 1 || Z < 0 || Hq < 1 || Hkv < 1 || Nq < 0 || Nkv < 1 || D < 1) return -1;
    if (Hq % Hkv != 0 || !isfinite(scale) || window_left < -1 || window_right < -1) return -1;
    const int64_t nq = (int64_t)Z * Hq * Nq * D, nk = (int64_t)Z * Hkv * Nkv * D;
    if (nk == 0) return 0;
    double* table = (double*)malloc(sizeof(double) * 65536);
    double* buf = (double*)malloc(sizeof(double) * (size_t)(2 * nq + 2 * nk + 1));
    if (!table || !buf) { free(table); free(buf); return -2; }
    for (int b = 0; b < 65536; ++b) table[b] = oracle_decode((uint16_t)b, dtype);
    double *qd = buf, *gd = buf + nq, *kd = buf + 2 * nq, *vd = buf + 2 * nq + nk;
    for (int64_t x = 0; x < nq; ++x) { qd[x] = table[q[x]]; gd[x] = table[dO[x]]; }
    for (int64_t x = 0; x < nk; ++x) { kd[x] = table[k[x]]; vd[x] = table[v[x]]; }

    const int64_t groups = (int64_t)Z * Hkv;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (nthreads > groups) nthreads = (int)groups;
    oracle_bwd_ex_job* jobs = (oracle_bwd_ex_job*)calloc((size_t)nthreads, sizeof(oracle_bwd_ex_job));
    pthread_t* tid = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    int* created = (int*)calloc((size_t)nthreads, sizeof(int));
    if (!jobs || !tid || !created) { free(jobs); free(tid); free(created); free(table); free(buf); return -2; }
    const int64_t chunk = (groups + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        oracle_bwd_ex_job* J = &jobs[t];
        *J = (oracle_bwd_ex_job){qd, kd, vd, gd, Z, Hq, Hkv, Nq, Nkv, D, scale, causal, window_left, window_right,
                                 alibi, dq, dk, dv, (int64_t)t * chunk,
                                 (int64_t)t * chunk + chunk < groups ? (int64_t)t * chunk + chunk : groups, 0};
        if (J->begin >= J->end) continue;
        if (nthreads > 1 && pthread_create(&tid[t], NULL, oracle_bwd_ex_worker, J) == 0) created[t] = 1;
        else oracle_bwd_ex_worker(J);
    }
    int status = 0;
    for (int t = 0; t < nthreads; ++t) {
        if (created[t]) pthread_join(tid[t], NULL);
        if (jobs[t].status) status = jobs[t].status;
    }
    free(jobs); free(tid); free(created); free(table); free(buf);
    return status;
}
