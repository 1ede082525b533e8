/*
 * FP64 oracle for one Gated DeltaNet (GDN) speculative / MTP decode step.
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this library.  The CUDA product path never calls,
 * links or includes anything from this directory, and this file includes
 * nothing from the product path.
 *
 * It is a plain, slow, scalar restatement of what the step computes, written
 * from these vLLM pull-request report pages:
 *   [P1] "PR #46090 report: [CPU][Spec Decode] Support DFlash speculative
 *        decoding for GDN models on CPU" -- implementation step 3 (per-token
 *        multi-slot state writes, rewind to the accepted token's slot) and the
 *        fla.cpp listing in "key source snippets" (parallel over
 *        (sequence, v-head), serial over draft tokens, initial slot
 *        spec_indices[i, max(num_accepted-1, 0)], skip when q_len <= 0,
 *        kh = v_head / (H_v / H_k), gate inputs A_log, a, dt_bias, b and a
 *        softplus threshold, in-kernel q/k L2 normalisation).
 *   [P2] "PR #51674 report: [Kernel][Perf] Add fused CUDA post-conv MTP decode
 *        kernel for Qwen3.5 GDN" -- implementation step 1 (rewind, up to 8
 *        draft tokens in order through the gated delta rule, gated RMSNorm
 *        epilogue), step 2 (scale = 128^-0.5, norm_eps = 1e-5), the
 *        _custom_ops.py listing (out = empty_like(output_gate)), and the
 *        review notes (the kernel writes only unpadded rows).
 *   [P3] "PR #52191 report: [CPU] Support FP16/BF16 persisted GDN state on
 *        AMX" -- implementation steps 3 and 4 (arithmetic in wide precision;
 *        only slot reads and writes use the narrow state type, so each write
 *        rounds once).
 *   [P4] "PR #51812 report: [Bugfix] Align Qwen GDN gates with speculative
 *        tokens" -- motivation and implementation steps 1-3 (q/k/v and the
 *        a/b gates of a mixed batch are gathered with one shared
 *        spec_token_indx).
 *
 * Per token the recurrence is, in this order:
 *     g    = -exp(A_log[h]) * softplus(a + dt_bias[h])      beta = sigmoid(b)
 *     k^   = k / sqrt(sum k^2 + qk_eps)      q^ = q / sqrt(sum q^2 + qk_eps) * scale
 *     S    = S * exp(g)                          (decay)
 *     u    = S^T k^ ;  v' = beta * (v - u)       (delta-rule correction)
 *     S    = S + k^ v'^T                         (rank-1 update)
 *     o    = S^T q^                              (readout)
 * with S a K x V matrix held as double.  The pages name the inputs and the
 * steps but do not print the formulas; the forms above are the standard
 * gated delta rule those names denote.  Readings used here: softplus(x) = x
 * above the threshold 20 (beta = 1) and qk_eps = 1e-6 inside the square root
 * (parity unpinned for these two constants, which the pages do not fix; the
 * forms they enter are pinned); state layout
 * [slot, H_v, K, V] with V contiguous; a padded read slot (< 0) skips the
 * sequence; a padded write slot skips only that write; the carried state is
 * never rounded, only the copy written to a slot.
 *
 * Inputs are read as the exact values of their stored bits.  Numbers are
 * encoded to bf16 / fp16 / fp32 by round-to-nearest-even, written here from
 * the IEEE 754 definition of those formats.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------- */
/* number formats                                                            */
/* ------------------------------------------------------------------------- */

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F16 = 2, ORC_F64 = 3 };

static double bf16_value(uint16_t bits)
{
    /* bf16 is the upper half of an IEEE binary32 */
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double f16_value(uint16_t bits)
{
    /* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
    int sign = bits >> 15;
    int e = (bits >> 10) & 31;
    int m = bits & 1023;
    double x;
    if (e == 0)
        x = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        x = m ? NAN : INFINITY;
    else
        x = ldexp((double)(m + 1024), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -x : x;
}

/*
 * Round x to the nearest point of a binary format with `frac_bits` fraction
 * bits and minimum normal exponent `emin` (gradual underflow below it), ties
 * to even.  The grid spacing inside the binade of |x| is 2^(e - frac_bits);
 * x / spacing is exact (power-of-two scaling) and nearbyint() in the default
 * rounding mode rounds it half-to-even.  Overflow is left to the caller.
 */
static double rne_to_grid(double x, int frac_bits, int emin)
{
    if (x == 0.0 || !isfinite(x))
        return x;
    int E;
    frexp(fabs(x), &E);          /* |x| = m 2^E, m in [0.5, 1): binade e = E - 1 */
    int e = E - 1;
    if (e < emin)
        e = emin;
    double spacing = ldexp(1.0, e - frac_bits);
    return nearbyint(x / spacing) * spacing;
}

static uint16_t bf16_bits_rne(double x)
{
    if (isnan(x))
        return 0x7FC0;
    double y = rne_to_grid(x, 7, -126);
    const double maxf = ldexp(255.0, 120);        /* (2 - 2^-7) 2^127 */
    if (fabs(y) > maxf)
        y = copysign(INFINITY, y);
    float f = (float)y;                           /* exact: y is on the bf16 grid */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

static uint16_t f16_bits_rne(double x)
{
    if (isnan(x))
        return 0x7E00;
    double y = rne_to_grid(x, 10, -14);
    uint16_t sign = signbit(y) ? 0x8000 : 0;
    double a = fabs(y);
    if (a > 65504.0)
        return sign | 0x7C00;                     /* overflow to infinity */
    if (a == 0.0)
        return sign;
    int E;
    frexp(a, &E);
    int e = E - 1;
    if (e < -14)                                  /* subnormal: a = m 2^-24 */
        return sign | (uint16_t)ldexp(a, 24);
    uint16_t frac = (uint16_t)((ldexp(a, -e) - 1.0) * 1024.0);
    return sign | (uint16_t)((e + 15) << 10) | frac;
}

static float f32_rne(double x)
{
    if (isnan(x))
        return NAN;
    double y = rne_to_grid(x, 23, -126);
    const double maxf = ldexp(16777215.0, 104);   /* (2 - 2^-23) 2^127 */
    if (fabs(y) > maxf)
        y = copysign(INFINITY, y);
    return (float)y;                              /* exact */
}

/* helpers exported for the format pins in the tests */
void gdn_oracle_round_bf16(const double* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = bf16_bits_rne(x[i]);
}
void gdn_oracle_round_f16(const double* x, uint16_t* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = f16_bits_rne(x[i]);
}
void gdn_oracle_round_f32(const double* x, float* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = f32_rne(x[i]);
}
void gdn_oracle_value_bf16(const uint16_t* x, double* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = bf16_value(x[i]);
}
void gdn_oracle_value_f16(const uint16_t* x, double* y, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) y[i] = f16_value(x[i]);
}

/* ------------------------------------------------------------------------- */
/* problem description                                                       */
/* ------------------------------------------------------------------------- */

typedef struct {
    int64_t batch, num_tokens, H_k, H_v, K, V, spec_stride, num_slots;
    int32_t state_dtype;          /* ORC_F32 / ORC_BF16 / ORC_F16 / ORC_F64 */
    int32_t num_threads;          /* <= 0: one thread */
    double scale, eps, qk_eps, softplus_threshold;
    const uint16_t *q, *k, *v;    /* bf16 bits: [N,H_k,K], [N,H_k,K], [N,H_v,V] */
    const uint16_t *a, *b;        /* bf16 bits: [N,H_v] */
    const uint16_t *z;            /* bf16 bits [N,H_v,V], or NULL: no epilogue */
    const float *A_log;           /* [H_v] */
    const uint16_t *dt_bias;      /* bf16 bits [H_v] */
    const uint16_t *norm_w;       /* bf16 bits [V]; NULL exactly when z is NULL */
    const int32_t *state_indices; /* [batch, spec_stride] */
    const int32_t *num_accepted;  /* [batch] */
    const int32_t *cu_seqlens;    /* [batch + 1] */
    const int32_t *spec_token_indx; /* [cu_seqlens[batch]] or NULL */
    void *pool;                   /* [num_slots, H_v, K, V], updated in place */
    double *out_f64;              /* [N, H_v, V] or NULL */
    uint16_t *out_bf16;           /* [N, H_v, V] or NULL */
    double *states_f64;           /* [batch, H_v, states_T, K, V] or NULL */
    int64_t states_T;
    /* FP64 q, k, v (same layouts as q, k, v), used in their place when set:
       the output of the convolution below */
    const double *q64, *k64, *v64;
} gdn_oracle_problem;

enum {
    ORC_OK = 0,
    ORC_ERR_NULL = -1,
    ORC_ERR_SHAPE = -2,
    ORC_ERR_ACCEPTED = -3,     /* num_accepted > spec_stride                */
    ORC_ERR_QLEN = -4,         /* q_len > spec_stride                       */
    ORC_ERR_SLOT = -5,         /* slot index >= num_slots                   */
    ORC_ERR_ROW = -6,          /* token row outside [0, num_tokens)         */
    ORC_ERR_CONFLICT = -7,     /* slot or row shared between sequences      */
    ORC_ERR_NOMEM = -8,
};

static size_t state_elem_bytes(int32_t dt)
{
    return dt == ORC_F32 ? 4 : dt == ORC_F64 ? 8 : 2;
}

static double pool_get(const gdn_oracle_problem* p, int64_t off)
{
    switch (p->state_dtype) {
    case ORC_F32: return (double)((const float*)p->pool)[off];
    case ORC_BF16: return bf16_value(((const uint16_t*)p->pool)[off]);
    case ORC_F16: return f16_value(((const uint16_t*)p->pool)[off]);
    default: return ((const double*)p->pool)[off];
    }
}

static void pool_put(const gdn_oracle_problem* p, int64_t off, double x)
{
    switch (p->state_dtype) {
    case ORC_F32: ((float*)p->pool)[off] = f32_rne(x); break;
    case ORC_BF16: ((uint16_t*)p->pool)[off] = bf16_bits_rne(x); break;
    case ORC_F16: ((uint16_t*)p->pool)[off] = f16_bits_rne(x); break;
    default: ((double*)p->pool)[off] = x; break;
    }
}

static int64_t token_row(const gdn_oracle_problem* p, int64_t i, int64_t t)
{
    /* [P4]: spec rows are gathered with spec_token_indx when it is given */
    int64_t n = (int64_t)p->cu_seqlens[i] + t;
    return p->spec_token_indx ? (int64_t)p->spec_token_indx[n] : n;
}

static int64_t read_index(const gdn_oracle_problem* p, int64_t i)
{
    /* [P1] fla.cpp listing and review: clamp acc-1 at 0 so that
       num_accepted = 0 never indexes position -1 */
    int64_t acc = (int64_t)p->num_accepted[i];
    int64_t j = acc - 1 > 0 ? acc - 1 : 0;
    return (int64_t)p->state_indices[i * p->spec_stride + j];
}

/*
 * Check the caller contract before touching anything: indices in range,
 * non-negative write slots distinct across the batch, no sequence's read slot
 * written by another sequence, token rows used at most once.
 */
static int check_contract(const gdn_oracle_problem* p)
{
    int64_t B = p->batch, st = p->spec_stride;
    int64_t* slot_owner = (int64_t*)malloc(sizeof(int64_t) * (size_t)p->num_slots);
    int64_t* row_owner = (int64_t*)malloc(sizeof(int64_t) * (size_t)(p->num_tokens + 1));
    if (!slot_owner || !row_owner) {
        free(slot_owner); free(row_owner);
        return ORC_ERR_NOMEM;
    }
    for (int64_t s = 0; s < p->num_slots; ++s) slot_owner[s] = -1;
    for (int64_t r = 0; r <= p->num_tokens; ++r) row_owner[r] = -1;
    int rc = ORC_OK;
    for (int64_t i = 0; i < B && rc == ORC_OK; ++i) {
        int64_t ql = (int64_t)p->cu_seqlens[i + 1] - p->cu_seqlens[i];
        if (ql <= 0) continue;
        if (ql > st) { rc = ORC_ERR_QLEN; break; }
        if (p->num_accepted[i] > st) { rc = ORC_ERR_ACCEPTED; break; }
        int64_t rs = read_index(p, i);
        if (rs < 0) continue;                      /* padded sequence */
        if (rs >= p->num_slots) { rc = ORC_ERR_SLOT; break; }
        if (p->cu_seqlens[i] < 0) { rc = ORC_ERR_ROW; break; }
        for (int64_t t = 0; t < ql; ++t) {
            int64_t r = token_row(p, i, t);
            if (r < 0 || r >= p->num_tokens) { rc = ORC_ERR_ROW; break; }
            if (row_owner[r] != -1) { rc = ORC_ERR_CONFLICT; break; }
            row_owner[r] = i;
            int64_t ws = p->state_indices[i * st + t];
            if (ws < 0) continue;
            if (ws >= p->num_slots) { rc = ORC_ERR_SLOT; break; }
            if (slot_owner[ws] != -1) { rc = ORC_ERR_CONFLICT; break; }
            slot_owner[ws] = i;
        }
    }
    /* a read slot may be written only by its own sequence */
    for (int64_t i = 0; i < B && rc == ORC_OK; ++i) {
        int64_t ql = (int64_t)p->cu_seqlens[i + 1] - p->cu_seqlens[i];
        if (ql <= 0) continue;
        int64_t rs = read_index(p, i);
        if (rs >= 0 && slot_owner[rs] != -1 && slot_owner[rs] != i) rc = ORC_ERR_CONFLICT;
    }
    free(slot_owner);
    free(row_owner);
    return rc;
}

/* ------------------------------------------------------------------------- */
/* the step                                                                  */
/* ------------------------------------------------------------------------- */

/* q, k, v element `off` of their dense layouts, from the FP64 copy when given */
static double in_q(const gdn_oracle_problem* p, int64_t off) { return p->q64 ? p->q64[off] : bf16_value(p->q[off]); }
static double in_k(const gdn_oracle_problem* p, int64_t off) { return p->k64 ? p->k64[off] : bf16_value(p->k[off]); }
static double in_v(const gdn_oracle_problem* p, int64_t off) { return p->v64 ? p->v64[off] : bf16_value(p->v[off]); }

static double softplus(double x, double threshold)
{
    return x > threshold ? x : log1p(exp(x));
}

static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }

/*
 * One draft token of one (sequence, v-head) unit.  S is K x V, row-major
 * (S[i*V + j] is key row i, value column j).  Writes the readout o[V].
 */
static void token_step(const gdn_oracle_problem* p, int64_t r, int64_t h,
                       double* S, double* kn, double* qn, double* o)
{
    const int64_t K = p->K, V = p->V, H_v = p->H_v;
    const int64_t kh = h / (H_v / p->H_k);            /* [P1]: GQA head map */

    /* gates, per (token, v-head) */
    double x = bf16_value(p->a[r * H_v + h]) + bf16_value(p->dt_bias[h]);
    double g = -exp((double)p->A_log[h]) * softplus(x, p->softplus_threshold);
    double beta = sigmoid(bf16_value(p->b[r * H_v + h]));

    /* L2-normalised key and query; the query also takes the scale */
    const int64_t kbase = (r * p->H_k + kh) * K;
    double sk = 0.0, sq = 0.0;
    for (int64_t i = 0; i < K; ++i) {
        double kv = in_k(p, kbase + i), qv = in_q(p, kbase + i);
        sk += kv * kv;
        sq += qv * qv;
    }
    double rk = 1.0 / sqrt(sk + p->qk_eps), rq = 1.0 / sqrt(sq + p->qk_eps);
    for (int64_t i = 0; i < K; ++i) {
        kn[i] = in_k(p, kbase + i) * rk;
        qn[i] = in_q(p, kbase + i) * rq * p->scale;
    }

    /* decay */
    double decay = exp(g);
    for (int64_t i = 0; i < K * V; ++i) S[i] *= decay;

    /* delta rule: v' = beta (v - S^T k^), then S += k^ v'^T */
    const int64_t vbase = (r * H_v + h) * V;
    for (int64_t j = 0; j < V; ++j) {
        double u = 0.0;
        for (int64_t i = 0; i < K; ++i) u += S[i * V + j] * kn[i];
        double vp = beta * (in_v(p, vbase + j) - u);
        for (int64_t i = 0; i < K; ++i) S[i * V + j] += kn[i] * vp;
    }

    /* readout o = S^T q^ */
    for (int64_t j = 0; j < V; ++j) {
        double acc = 0.0;
        for (int64_t i = 0; i < K; ++i) acc += S[i * V + j] * qn[i];
        o[j] = acc;
    }
}

/* [P2] step 1: gated RMSNorm epilogue, o <- o / sqrt(mean(o^2) + eps) * w * silu(z) */
static void epilogue(const gdn_oracle_problem* p, int64_t r, int64_t h, const double* o)
{
    const int64_t V = p->V;
    const int64_t base = (r * p->H_v + h) * V;
    double ms = 0.0;
    if (p->z) {
        for (int64_t j = 0; j < V; ++j) ms += o[j] * o[j];
        ms /= (double)V;
    }
    double rinv = p->z ? 1.0 / sqrt(ms + p->eps) : 1.0;
    for (int64_t j = 0; j < V; ++j) {
        double y;
        if (p->z) {
            double zz = bf16_value(p->z[base + j]);
            double silu = zz / (1.0 + exp(-zz));
            y = o[j] * rinv * bf16_value(p->norm_w[j]) * silu;
        } else {
            y = o[j];
        }
        if (p->out_f64) p->out_f64[base + j] = y;
        if (p->out_bf16) p->out_bf16[base + j] = bf16_bits_rne(y);
    }
}

static void run_unit(const gdn_oracle_problem* p, int64_t i, int64_t h, double* work)
{
    const int64_t K = p->K, V = p->V, H_v = p->H_v;
    int64_t ql = (int64_t)p->cu_seqlens[i + 1] - p->cu_seqlens[i];
    if (ql <= 0) return;                          /* [P1]: q_len <= 0 -> skip */
    int64_t rs = read_index(p, i);
    if (rs < 0) return;                           /* padded sequence: nothing written */

    double* S = work;
    double* kn = S + K * V;
    double* qn = kn + K;
    double* o = qn + K;

    /* the whole initial state is read before any slot is written */
    const int64_t src = (rs * H_v + h) * K * V;
    for (int64_t e = 0; e < K * V; ++e) S[e] = pool_get(p, src + e);

    for (int64_t t = 0; t < ql; ++t) {
        int64_t r = token_row(p, i, t);
        token_step(p, r, h, S, kn, qn, o);

        /* [P1] step 3 / [P3] step 4: the state after token t goes to slot
           state_indices[i, t], rounded once; the carried S stays unrounded */
        int64_t ws = p->state_indices[i * p->spec_stride + t];
        if (ws >= 0) {
            const int64_t dst = (ws * H_v + h) * K * V;
            for (int64_t e = 0; e < K * V; ++e) pool_put(p, dst + e, S[e]);
        }
        if (p->states_f64 && t < p->states_T)
            memcpy(p->states_f64 + ((i * H_v + h) * p->states_T + t) * K * V, S,
                   sizeof(double) * (size_t)(K * V));
        epilogue(p, r, h, o);
    }
}

static int check_problem(const gdn_oracle_problem* p)
{
    if (!p || !(p->q || p->q64) || !(p->k || p->k64) || !(p->v || p->v64) || !p->a || !p->b || !p->A_log || !p->dt_bias ||
        !p->pool || !p->state_indices || !p->num_accepted || !p->cu_seqlens)
        return ORC_ERR_NULL;
    if ((p->z == NULL) != (p->norm_w == NULL)) return ORC_ERR_NULL;
    if (p->batch < 0 || p->num_tokens < 0 || p->H_k <= 0 || p->H_v <= 0 || p->K <= 0 ||
        p->V <= 0 || p->spec_stride <= 0 || p->num_slots <= 0 || p->H_v % p->H_k != 0)
        return ORC_ERR_SHAPE;
    if (p->state_dtype < ORC_F32 || p->state_dtype > ORC_F64) return ORC_ERR_SHAPE;
    return ORC_OK;
}

/*
 * The speculative decode step over a batch.  Returns 0, or a negative
 * ORC_ERR_* code (nothing modified) when the arguments break the contract.
 */
int gdn_oracle_spec_decode(const gdn_oracle_problem* p)
{
    int rc = check_problem(p);
    if (rc != ORC_OK) return rc;
    rc = check_contract(p);
    if (rc != ORC_OK) return rc;
    (void)state_elem_bytes;

    const int64_t units = p->batch * p->H_v;
    const int64_t work_len = p->K * p->V + 2 * p->K + p->V;
    int nthreads = p->num_threads > 0 ? p->num_threads : 1;
    double* work = (double*)malloc(sizeof(double) * (size_t)(work_len * nthreads));
    if (!work) return ORC_ERR_NOMEM;

#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        run_unit(p, u / p->H_v, u % p->H_v, work + (int64_t)tid * work_len);
    }
    free(work);
    return ORC_OK;
}

/*
 * Ordinary (non-speculative) recurrent decode: sequence i has exactly one
 * token, at row i, and updates slot ssm_state_indices[i] in place (skipped
 * when negative).  The gated delta rule and epilogue are the same token step
 * as above.  `p->state_indices` holds one slot per sequence here;
 * `num_accepted`, `cu_seqlens` and `spec_token_indx` are ignored.
 */
int gdn_oracle_decode_nonspec(const gdn_oracle_problem* p)
{
    if (!p || !p->q || !p->k || !p->v || !p->a || !p->b || !p->A_log || !p->dt_bias ||
        !p->pool || !p->state_indices)
        return ORC_ERR_NULL;
    if ((p->z == NULL) != (p->norm_w == NULL)) return ORC_ERR_NULL;
    if (p->batch > p->num_tokens || p->H_v % p->H_k != 0) return ORC_ERR_SHAPE;
    const int64_t K = p->K, V = p->V, H_v = p->H_v;
    double* work = (double*)malloc(sizeof(double) * (size_t)(K * V + 2 * K + V));
    if (!work) return ORC_ERR_NOMEM;
    double* S = work;
    double* kn = S + K * V;
    double* qn = kn + K;
    double* o = qn + K;
    for (int64_t i = 0; i < p->batch; ++i) {
        int64_t slot = p->state_indices[i];
        if (slot < 0) continue;
        if (slot >= p->num_slots) { free(work); return ORC_ERR_SLOT; }
        for (int64_t h = 0; h < H_v; ++h) {
            const int64_t off = (slot * H_v + h) * K * V;
            for (int64_t e = 0; e < K * V; ++e) S[e] = pool_get(p, off + e);
            token_step(p, i, h, S, kn, qn, o);
            for (int64_t e = 0; e < K * V; ++e) pool_put(p, off + e, S[e]);
            epilogue(p, i, h, o);
        }
    }
    free(work);
    return ORC_OK;
}

/*
 * Prefill over whole prompts (PR #52191 report, implementation step 3: the
 * chunked prefill kernel chunk_gated_delta_rule_fwd_inter_kernel_impl carries
 * the state across the prompt in FP32 and writes it back to its slot).
 * Sequence i is tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 (rows in order, no
 * gather).  It starts from slot read_slots[i], or from the zero state when
 * read_slots[i] < 0, runs the same per-token step as the decode path over all
 * of its tokens in order, writes one output row per token, and stores the
 * state after its last token in slot write_slots[i] (skipped when negative),
 * rounded once.  Reading: the pages' CPU chunk kernel also rounds a narrow
 * state at every chunk write-back; here, as on the decode path, only the
 * stored copy is rounded and the carried state stays wide.
 * `p->state_indices`, `num_accepted` and `spec_token_indx` are ignored.
 */
int gdn_oracle_prefill(const gdn_oracle_problem* p, const int32_t* read_slots, const int32_t* write_slots)
{
    if (!p || !p->q || !p->k || !p->v || !p->a || !p->b || !p->A_log || !p->dt_bias || !p->pool ||
        !p->cu_seqlens || !read_slots || !write_slots)
        return ORC_ERR_NULL;
    if ((p->z == NULL) != (p->norm_w == NULL)) return ORC_ERR_NULL;
    if (p->batch < 0 || p->H_k <= 0 || p->H_v <= 0 || p->H_v % p->H_k != 0 || p->num_slots <= 0)
        return ORC_ERR_SHAPE;
    const int64_t K = p->K, V = p->V, H_v = p->H_v;
    /* contract: rows in range, write slots distinct, no read slot written by
       another sequence */
    for (int64_t i = 0; i < p->batch; ++i) {
        if (p->cu_seqlens[i] < 0 || p->cu_seqlens[i + 1] > p->num_tokens) return ORC_ERR_ROW;
        if (read_slots[i] >= p->num_slots || write_slots[i] >= p->num_slots) return ORC_ERR_SLOT;
        for (int64_t j = 0; j < p->batch; ++j) {
            if (j != i && write_slots[j] >= 0 &&
                (write_slots[j] == write_slots[i] || write_slots[j] == read_slots[i]))
                return ORC_ERR_CONFLICT;
        }
    }
    const int64_t work_len = K * V + 2 * K + V;
    const int nthreads = p->num_threads > 0 ? p->num_threads : 1;
    double* work_all = (double*)malloc(sizeof(double) * (size_t)(work_len * nthreads));
    if (!work_all) return ORC_ERR_NOMEM;
    const int64_t units = p->batch * H_v;
#ifdef _OPENMP
#pragma omp parallel for num_threads(nthreads) schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < units; ++u) {
        const int64_t i = u / H_v, h = u % H_v;
        int tid = 0;
#ifdef _OPENMP
        tid = omp_get_thread_num();
#endif
        double* S = work_all + (int64_t)tid * work_len;
        double* kn = S + K * V;
        double* qn = kn + K;
        double* o = qn + K;
        const int64_t bos = p->cu_seqlens[i], eos = p->cu_seqlens[i + 1];
        if (eos <= bos) continue;
        {
            if (read_slots[i] >= 0) {
                const int64_t src = ((int64_t)read_slots[i] * H_v + h) * K * V;
                for (int64_t e = 0; e < K * V; ++e) S[e] = pool_get(p, src + e);
            } else {
                for (int64_t e = 0; e < K * V; ++e) S[e] = 0.0;
            }
            for (int64_t r = bos; r < eos; ++r) {
                token_step(p, r, h, S, kn, qn, o);
                epilogue(p, r, h, o);
            }
            if (write_slots[i] >= 0) {
                const int64_t dst = ((int64_t)write_slots[i] * H_v + h) * K * V;
                for (int64_t e = 0; e < K * V; ++e) pool_put(p, dst + e, S[e]);
            }
            if (p->states_f64 && p->states_T > 0)
                memcpy(p->states_f64 + (i * H_v + h) * p->states_T * K * V, S, sizeof(double) * (size_t)(K * V));
        }
    }
    free(work_all);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* the short causal convolution in front of the step, with rewind           */
/* ------------------------------------------------------------------------- */

/*
 * The projection rows that feed q, k and v pass first through a depthwise
 * causal convolution of width W with a SiLU, whose history lives in a conv
 * state slot ([P1] implementation step 2 and its spec-aware listing: a wide
 * rolling buffer sliced per token, convolved, written back; [P2]
 * implementation step 3: the speculative path runs causal_conv1d_update with
 * rewind before the post-conv decode kernel; BF16 conv state).  The pages
 * print no formula; the readings taken here:
 *   - a conv slot is [state_len][conv_dim] raw inputs (bf16 bits), rows
 *     0 .. W-2 the history before the previous step, rows W-1 .. the previous
 *     step's own inputs;
 *   - rewind: with a = max(num_accepted[i], 1) (the clamp mirrors the state
 *     rewind), the W-1 inputs before this step's first token are slot rows
 *     a .. a + W - 2, i.e. the history up to the previous step's last
 *     accepted token;
 *   - y_t[c] = silu(bias[c] + sum_{w<W} weight[c][w] x_{t-W+1+w}[c]) over the
 *     inputs x (history first, then this step's rows in order);
 *   - the new slot: rows 0 .. W-2 = that history, rows W-1 .. W-2+q_len = this
 *     step's raw inputs, copied bit for bit; later rows are left as they were;
 *   - a sequence reads conv_in[i] (< 0: zero history) and writes conv_out[i]
 *     (< 0: no write), which must differ from every read slot of the call.
 * conv_dim = 2 H_k K + H_v V with the channels in the order q | k | v.
 */
typedef struct {
    int64_t conv_dim, width, state_len, num_conv_slots;
    const uint16_t* x;            /* bf16 bits [num_tokens, conv_dim]: projection rows */
    const uint16_t* weight;       /* bf16 bits [conv_dim, width] */
    const uint16_t* bias;         /* bf16 bits [conv_dim], or NULL */
    uint16_t* conv_pool;          /* bf16 bits [num_conv_slots, state_len, conv_dim] */
    const int32_t* conv_in;       /* [batch] */
    const int32_t* conv_out;      /* [batch] */
} gdn_oracle_conv;

/* does the step process sequence i (a token and an unpadded read slot)? */
static int processed(const gdn_oracle_problem* p, int64_t i)
{
    int64_t ql = (int64_t)p->cu_seqlens[i + 1] - p->cu_seqlens[i];
    return ql > 0 && read_index(p, i) >= 0;
}

/*
 * The convolution for every processed sequence of the step, then the step
 * itself on its output (q, k, v in FP64).  The step's own contract and the
 * conv slot contract are checked first; nothing is modified on error.
 */
int gdn_oracle_spec_decode_conv(const gdn_oracle_problem* pin, const gdn_oracle_conv* c)
{
    if (!pin || !c || !c->x || !c->weight || !c->conv_pool || !c->conv_in || !c->conv_out) return ORC_ERR_NULL;
    gdn_oracle_problem p = *pin;
    const int64_t B = p.batch, N = p.num_tokens, W = c->width, D = c->conv_dim;
    const int64_t QK = p.H_k * p.K;
    if (D != 2 * QK + p.H_v * p.V || W < 1 || c->state_len < W - 1 + p.spec_stride || c->num_conv_slots <= 0)
        return ORC_ERR_SHAPE;
    /* the bf16 q/k/v pointers are not used: stand-ins for the null checks */
    p.q = p.k = p.v = c->x;
    int rc = check_problem(&p);
    if (rc != ORC_OK) return rc;
    rc = check_contract(&p);
    if (rc != ORC_OK) return rc;
    for (int64_t i = 0; i < B; ++i) {
        if (!processed(&p, i)) continue;
        if (c->conv_in[i] >= c->num_conv_slots || c->conv_out[i] >= c->num_conv_slots) return ORC_ERR_SLOT;
        for (int64_t j = 0; j < B; ++j) {
            if (!processed(&p, j) || c->conv_out[j] < 0) continue;
            if (c->conv_out[j] == c->conv_in[i]) return ORC_ERR_CONFLICT;
            if (j != i && c->conv_out[j] == c->conv_out[i]) return ORC_ERR_CONFLICT;
        }
    }
    double* y = (double*)calloc((size_t)(N * D), sizeof(double));
    double* q64 = (double*)calloc((size_t)(N * QK), sizeof(double));
    double* k64 = (double*)calloc((size_t)(N * QK), sizeof(double));
    double* v64 = (double*)calloc((size_t)(N * p.H_v * p.V), sizeof(double));
    double* hist = (double*)malloc(sizeof(double) * (size_t)((W - 1 + p.spec_stride) * D + 1));
    uint16_t* newslot = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(B * (W - 1 + p.spec_stride) * D + 1));
    if (!y || !q64 || !k64 || !v64 || !hist || !newslot) {
        free(y); free(q64); free(k64); free(v64); free(hist); free(newslot);
        return ORC_ERR_NOMEM;
    }
    const int64_t rows_new = W - 1 + p.spec_stride;
    for (int64_t i = 0; i < B; ++i) {
        if (!processed(&p, i)) continue;
        const int64_t ql = (int64_t)p.cu_seqlens[i + 1] - p.cu_seqlens[i];
        const int64_t acc = p.num_accepted[i] > 1 ? p.num_accepted[i] : 1;
        /* inputs in time order: W-1 history rows, then the step's rows */
        for (int64_t m = 0; m < W - 1; ++m)
            for (int64_t ch = 0; ch < D; ++ch) {
                uint16_t bits = 0;
                if (c->conv_in[i] >= 0)
                    bits = c->conv_pool[((int64_t)c->conv_in[i] * c->state_len + acc + m) * D + ch];
                hist[m * D + ch] = bf16_value(bits);
                newslot[(i * rows_new + m) * D + ch] = bits;
            }
        for (int64_t t = 0; t < ql; ++t) {
            const int64_t r = token_row(&p, i, t);
            for (int64_t ch = 0; ch < D; ++ch) {
                hist[(W - 1 + t) * D + ch] = bf16_value(c->x[r * D + ch]);
                newslot[(i * rows_new + W - 1 + t) * D + ch] = c->x[r * D + ch];
            }
        }
        for (int64_t t = 0; t < ql; ++t) {
            const int64_t r = token_row(&p, i, t);
            for (int64_t ch = 0; ch < D; ++ch) {
                double acc_c = c->bias ? bf16_value(c->bias[ch]) : 0.0;
                for (int64_t w = 0; w < W; ++w)
                    acc_c += bf16_value(c->weight[ch * W + w]) * hist[(t + w) * D + ch];
                y[r * D + ch] = acc_c / (1.0 + exp(-acc_c));          /* SiLU */
            }
        }
    }
    /* all reads done: write the new slots */
    for (int64_t i = 0; i < B; ++i) {
        if (!processed(&p, i) || c->conv_out[i] < 0) continue;
        const int64_t ql = (int64_t)p.cu_seqlens[i + 1] - p.cu_seqlens[i];
        for (int64_t m = 0; m < W - 1 + ql; ++m)
            memcpy(c->conv_pool + ((int64_t)c->conv_out[i] * c->state_len + m) * D,
                   newslot + (i * rows_new + m) * D, sizeof(uint16_t) * (size_t)D);
    }
    /* split the conv output into the step's q, k, v layouts */
    for (int64_t r = 0; r < N; ++r) {
        memcpy(q64 + r * QK, y + r * D, sizeof(double) * (size_t)QK);
        memcpy(k64 + r * QK, y + r * D + QK, sizeof(double) * (size_t)QK);
        memcpy(v64 + r * p.H_v * p.V, y + r * D + 2 * QK, sizeof(double) * (size_t)(p.H_v * p.V));
    }
    p.q64 = q64;
    p.k64 = k64;
    p.v64 = v64;
    rc = gdn_oracle_spec_decode(&p);
    free(y); free(q64); free(k64); free(v64); free(hist); free(newslot);
    return rc;
}

int gdn_oracle_abi_version(void) { return 2; }
