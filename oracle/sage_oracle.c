/*
 * Plain, slow CPU oracle of the quantized attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this library.  The CUDA library never
 * calls it and shares no code, header, table or constant with it.
 *
 * Every fp32 step of the quantized program is written as a double-precision
 * operation on fp32 operands followed by an explicit rounding to fp32
 * (FL below).  For +, -, *, / that is the correctly rounded fp32 result
 * (binary64 carries more than 2*24+2 bits), so the code needs no reasoning
 * about compiler evaluation order; it is built with -ffp-contract=off so no
 * multiply-add is fused behind its back.
 *
 * What the pages fix, and where:
 *  - Q/K INT8 per-block quantisation, K smoothing (per-channel mean of K
 *    subtracted), V FP8 quantisation with a transpose: "H3 Performance
 *    Roadmap", section "Measured GB10 Baseline", table "SageAttention 2.2.0
 *    internals", and section "Phase 4: Dense Sage-Compatible Attention",
 *    items 2-3.
 *  - Per-tile order QK -> online-softmax update of (m, d, O) -> accumulate the
 *    denominator -> scores to FP8 -> PV: "Sage2 SM89 Temporal Pair
 *    Experiment", section "Candidate".
 *  - V scale fused into the epilogue: the same page, kernel name
 *    "..._fuse_v_scale_attn_inst_buf".
 *  - Int8 KV-cache prompt attention compared against FP64: "Strata PR #2092",
 *    table "qsa_prompt_attn_parity (int8 KV), ms per chunk and error against
 *    FP64".
 * Readings where the pages are silent are listed beside each function.
 *
 * Parity status: every function below is pinned by the CPU tests (closed
 * forms, brute force, invariants, library conversions); none is unpinned.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define D 128

/* ------------------------------------------------------------------------
 * number formats, written from their definitions
 * --------------------------------------------------------------------- */

/* round to the nearest fp32 (ties to even): the cast does it */
static double FL(double x) { return (double)(float)x; }

/* bf16: 1 sign, 8 exponent (bias 127), 7 mantissa bits */
double orc_bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* nearest multiple of q to x, ties to the even multiple (exact in double
   for the magnitudes used here) */
static double round_to_quantum(double x, double q)
{
    return nearbyint(x / q) * q;
}

/* fp32 -> bf16, round to nearest even.  The quantum of bf16 in the binade
   [2^k, 2^(k+1)) is 2^(k-7); below 2^-126 it is 2^-133. */
uint16_t orc_f32_to_bf16(float xf)
{
    double x = (double)xf;
    double a = fabs(x);
    double r;
    if (a == 0.0) {
        r = 0.0;
    } else {
        int e;
        frexp(a, &e);           /* a = f * 2^e, f in [0.5, 1) -> binade k = e-1 */
        int k = e - 1;
        if (k < -126) k = -126;
        r = round_to_quantum(a, ldexp(1.0, k - 7));
    }
    float rf = (float)r;          /* r is a bf16 value, exact in fp32 */
    uint32_t u;
    memcpy(&u, &rf, 4);
    uint16_t h = (uint16_t)(u >> 16);
    if (signbit(x)) h |= 0x8000u;
    return h;
}

/* fp16 (IEEE binary16): 1 sign, 5 exponent (bias 15), 10 mantissa bits */
double orc_f16_value(uint16_t h)
{
    int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
    double v;
    if (e == 0) v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31) v = m ? NAN : INFINITY;
    else v = ldexp(1.0 + m / 1024.0, e - 15);
    return s ? -v : v;
}

/* fp32 -> fp16, round to nearest even.  Quantum in the binade
   [2^k, 2^(k+1)) is 2^(k-10) for k >= -14 and 2^-24 below; a magnitude that
   rounds beyond the largest finite value 65504 becomes infinity, as IEEE
   round-to-nearest does (the threshold is 65520, halfway to 2^16). */
uint16_t orc_f32_to_f16(float xf)
{
    double x = (double)xf;
    double a = fabs(x);
    uint16_t code = 0;
    if (isnan(x)) {
        code = 0x7E00u;
    } else if (a > 0.0) {
        int e;
        frexp(a, &e);
        int k = e - 1;
        if (k < -14) k = -14;
        double r = round_to_quantum(a, ldexp(1.0, k - 10));
        if (r >= 65536.0 || isinf(a)) {
            code = 0x7C00u;                                     /* infinity */
        } else if (r < ldexp(1.0, -14)) {
            code = (uint16_t)(r / ldexp(1.0, -24));              /* subnormal (or 2^-14 exactly below) */
        } else {
            double f = frexp(r, &e);                            /* r = f*2^e, f in [0.5, 1) */
            int E = (e - 1) + 15;
            int M = (int)((2.0 * f - 1.0) * 1024.0 + 0.5);
            code = (uint16_t)((E << 10) | M);
        }
    }
    if (signbit(x)) code |= 0x8000u;
    return code;
}

/* OCP 8-bit floating point, E4M3 ("FN"): bias 7, 3 mantissa bits, no
   infinities, S.1111.111 is NaN, largest finite 448, subnormals m * 2^-9. */
double orc_e4m3_value(uint8_t c)
{
    int s = (c >> 7) & 1, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0) v = ldexp((double)m, -9);
    else if (e == 15 && m == 7) v = NAN;
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* fp32 -> E4M3, round to nearest even, saturating to +-448 (the
   "satfinite" behaviour: anything beyond the largest finite value becomes
   that value).  Quantum in the binade [2^k, 2^(k+1)) is 2^(k-3) for
   k >= -6, and 2^-9 below 2^-6. */
uint8_t orc_f32_to_e4m3(float xf)
{
    double x = (double)xf;
    double a = fabs(x);
    double r = 0.0;
    if (a > 0.0) {
        int e;
        frexp(a, &e);
        int k = e - 1;
        if (k < -6) k = -6;
        r = round_to_quantum(a, ldexp(1.0, k - 3));
        if (r > 448.0) r = 448.0;
    }
    /* encode r (a representable magnitude) */
    uint8_t code = 0;
    if (r > 0.0) {
        if (r < ldexp(1.0, -6)) {
            code = (uint8_t)(r / ldexp(1.0, -9));               /* subnormal */
        } else {
            int e;
            double f = frexp(r, &e);                           /* r = f*2^e */
            int E = (e - 1) + 7;                                /* biased exponent */
            int M = (int)((2.0 * f - 1.0) * 8.0 + 0.5);
            code = (uint8_t)((E << 3) | M);
        }
    }
    /* the format has a signed zero: a negative input that rounds to zero
       keeps its sign (code 0x80), as round-to-nearest does in IEEE formats */
    if (signbit(x)) code |= 0x80u;
    return code;
}

/* fp32 -> int8 code: round half to even, saturated to [-127, 127] */
static int rni_sat127(double x)
{
    double r = nearbyint(x);
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
    return (int)r;
}

/* ------------------------------------------------------------------------
 * a1: K smoothing mean.
 * Reading (the pages name the step but not its reduction order): each
 * channel's mean over the Nk valid tokens; tokens are summed in ascending
 * order in fp32 inside chunks of 256 tokens, the chunk sums are added in
 * ascending chunk order in fp32, and the total is divided by Nk (fp32
 * division).
 * --------------------------------------------------------------------- */
#define MEAN_CHUNK 256

void orc_k_mean(const uint16_t *k, int Nk, float *mu)
{
    for (int c = 0; c < D; ++c) {
        double total = 0.0;
        for (int t0 = 0; t0 < Nk; t0 += MEAN_CHUNK) {
            double part = 0.0;
            int t1 = t0 + MEAN_CHUNK < Nk ? t0 + MEAN_CHUNK : Nk;
            for (int t = t0; t < t1; ++t) part = FL(part + orc_bf16_value(k[(size_t)t * D + c]));
            total = FL(total + part);
        }
        mu[c] = Nk > 0 ? (float)FL(total / (double)Nk) : 0.0f;
    }
}

/* ------------------------------------------------------------------------
 * a2: symmetric INT8 per-block quantisation of a [n, 128] fp32 matrix.
 * Reading: one scale per block of `blk` tokens (the last block partial);
 * amax = max |x| over the block's valid tokens and all channels;
 * scale = fl(amax / 127); inv = fl(127 / amax) (0 when amax = 0);
 * code = clamp(rint_even(fl(x * inv)), -127, 127).
 * --------------------------------------------------------------------- */
static void quant_blocks_i8(const float *x, int n, int blk, int8_t *codes, float *scales)
{
    int nb = (n + blk - 1) / blk;
    for (int b = 0; b < nb; ++b) {
        int t0 = b * blk, t1 = t0 + blk < n ? t0 + blk : n;
        double amax = 0.0;
        for (int t = t0; t < t1; ++t)
            for (int c = 0; c < D; ++c) {
                double a = fabs((double)x[(size_t)t * D + c]);
                if (a > amax) amax = a;
            }
        double scale = FL(amax / 127.0);
        double inv = amax > 0.0 ? FL(127.0 / amax) : 0.0;
        scales[b] = (float)scale;
        for (int t = t0; t < t1; ++t)
            for (int c = 0; c < D; ++c)
                codes[(size_t)t * D + c] = (int8_t)rni_sat127(FL((double)x[(size_t)t * D + c] * inv));
    }
}

/* Q: [Nq, 128] bf16 -> int8 codes [Nq, 128] and fp32 scales [ceil(Nq/bq)] */
void orc_quant_q(const uint16_t *q, int Nq, int bq, int8_t *codes, float *scales)
{
    float *x = (float *)malloc(sizeof(float) * (size_t)Nq * D + 1);
    for (size_t i = 0; i < (size_t)Nq * D; ++i) x[i] = (float)orc_bf16_value(q[i]);
    quant_blocks_i8(x, Nq, bq, codes, scales);
    free(x);
}

/* K: smoothed first.  Reading: Ks = fl(float(K) - mu) stays fp32 (not
   rounded back to bf16) before quantisation. */
void orc_quant_k(const uint16_t *k, int Nk, int bk, const float *mu, int8_t *codes, float *scales)
{
    float *x = (float *)malloc(sizeof(float) * (size_t)Nk * D + 1);
    for (int t = 0; t < Nk; ++t)
        for (int c = 0; c < D; ++c)
            x[(size_t)t * D + c] = (float)FL(orc_bf16_value(k[(size_t)t * D + c]) - (double)mu[c]);
    quant_blocks_i8(x, Nk, bk, codes, scales);
    free(x);
}

/* ------------------------------------------------------------------------
 * a3: V FP8 E4M3 per-channel quantisation, written transposed.
 * Reading: per channel c, amax_c over all valid tokens; sv_c = fl(amax_c/448);
 * inv = fl(448/amax_c) (0 when amax_c = 0); code = e4m3(fl(v * inv)).
 * Output layout [128, Nk_pad] (channel-major, tokens contiguous), tokens
 * Nk..Nk_pad-1 hold code 0.
 * --------------------------------------------------------------------- */
void orc_quant_v(const uint16_t *v, int Nk, int Nk_pad, uint8_t *codes_t, float *scales)
{
    for (int c = 0; c < D; ++c) {
        double amax = 0.0;
        for (int t = 0; t < Nk; ++t) {
            double a = fabs(orc_bf16_value(v[(size_t)t * D + c]));
            if (a > amax) amax = a;
        }
        double sv = FL(amax / 448.0);
        double inv = amax > 0.0 ? FL(448.0 / amax) : 0.0;
        scales[c] = (float)sv;
        for (int t = 0; t < Nk_pad; ++t) {
            uint8_t code = 0;
            if (t < Nk) code = orc_f32_to_e4m3((float)FL(orc_bf16_value(v[(size_t)t * D + c]) * inv));
            codes_t[(size_t)c * Nk_pad + t] = code;
        }
    }
}

/* ------------------------------------------------------------------------
 * a4-a8: the per-tile online-softmax program, one query row at a time.
 *
 * `quantized` = 1 runs the quantized program (fp32 steps, FP8 P);
 * `quantized` = 0 runs the same loop in plain fp64 with identity
 * quantisers: codes are the raw values, scales are 1, P is not rounded, and
 * the result is softmax(Q K^T * sm_scale) V.  The second mode exists so the
 * tile loop itself can be checked against a brute-force softmax.
 *
 * Per key tile (ascending), for row i (reading of the order QK ->
 * update m/l/O -> accumulate the denominator from fp32 p -> P to FP8 -> PV):
 *   S_ij  = sum_c q_ic k_jc                      (exact: integer codes)
 *   t     = fl(fl(sq_blk(i) * sk_blk(j)) * C),   C = fl(sm_scale * log2 e)
 *   s_ij  = fl(S_ij * t)                         (base-2 logits)
 *   m'    = max(m, max_j s_ij)
 *   alpha = exp2f(fl(m - m'))                    (0 while m = -inf)
 *   p_ij  = exp2f(fl(s_ij - m'))
 *   l     = fl(fl(alpha * l) + rowsum),  rowsum = fp32 sum of p_ij, j ascending
 *   P_ij  = e4m3(fl(448 * p_ij))                 (448: p <= 1 spans the format)
 *   T_c   = sum_j P_ij V_jc   exact (products of two E4M3 values and their
 *           sum fit a double exactly), then rounded once to fp32
 *   O_c   = fl(fl(alpha * O_c) + T_c);  m = m'
 * Epilogue: out_c = fl(fl(O_c / l) * fl(sv_c / 448)).
 * Keys j >= Nk do not exist for the row (their logits are -inf).
 *
 * Causal variant (the pages name it as the next step and fix nothing else):
 * query i sees keys j <= i + (Nk - Nq), the bottom-right alignment under
 * which the last query sees every key (for Nq = Nk: j <= i); the other
 * logits are -inf, so a tile with no visible key leaves m, l and O as they
 * are.  Log-sum-exp of the row, natural base, from the final m and l:
 * lse = ln 2 * (m + log2 l), evaluated in fp64 (l sums p, not 448 p).
 * --------------------------------------------------------------------- */
typedef struct {
    int quantized;
    int tile;
    double C;        /* base-2 logit multiplier */
    double pscale;   /* 448 or 1 */
} orc_prog;

static void program_row(const orc_prog *pg, const double *qrow, double sq,
                        const double *kmat, const double *skey,
                        const double *vmat, const double *sv, int Nk, int nvis,
                        double *S, double *s, double *P, double *out, double *lse)
{
    double m = -INFINITY, l = 0.0;
    double O[D];
    for (int c = 0; c < D; ++c) O[c] = 0.0;
    for (int j0 = 0; j0 < Nk; j0 += pg->tile) {
        int jn = Nk - j0 < pg->tile ? Nk - j0 : pg->tile;
        double mt = -INFINITY;
        for (int j = 0; j < jn; ++j) {
            const double *krow = kmat + (size_t)(j0 + j) * D;
            double acc = 0.0;
            for (int c = 0; c < D; ++c) acc += qrow[c] * krow[c];
            S[j] = acc;
            double t, sj;
            if (pg->quantized) {
                t = FL(FL(sq * skey[j0 + j]) * pg->C);
                sj = FL(S[j] * t);
            } else {
                sj = S[j] * pg->C;
            }
            if (j0 + j >= nvis) sj = -INFINITY;         /* outside the causal window */
            s[j] = sj;
            if (sj > mt) mt = sj;
        }
        double mnew = m > mt ? m : mt;
        double alpha, rowsum = 0.0;
        if (pg->quantized) {
            alpha = (m == -INFINITY) ? 0.0 : (double)exp2f((float)FL(m - mnew));
            for (int j = 0; j < jn; ++j) {
                double p = (double)exp2f((float)FL(s[j] - mnew));
                rowsum = FL(rowsum + p);
                P[j] = orc_e4m3_value(orc_f32_to_e4m3((float)FL(pg->pscale * p)));
            }
            l = FL(FL(alpha * l) + rowsum);
        } else {
            alpha = (m == -INFINITY) ? 0.0 : exp2(m - mnew);
            for (int j = 0; j < jn; ++j) {
                double p = exp2(s[j] - mnew);
                rowsum += p;
                P[j] = p;
            }
            l = alpha * l + rowsum;
        }
        for (int c = 0; c < D; ++c) {
            double T = 0.0;
            for (int j = 0; j < jn; ++j) T += P[j] * vmat[(size_t)(j0 + j) * D + c];
            if (pg->quantized) O[c] = FL(FL(alpha * O[c]) + FL(T));
            else O[c] = alpha * O[c] + T;
        }
        m = mnew;
    }
    for (int c = 0; c < D; ++c) {
        if (pg->quantized) out[c] = FL(FL(O[c] / l) * FL(sv[c] / pg->pscale));
        else out[c] = O[c] / l * sv[c];
    }
    if (lse) *lse = log(2.0) * (m + log2(l));
}

/* visible keys of query row i */
static int visible_keys(int i, int Nq, int Nk, int causal)
{
    if (!causal) return Nk;
    int v = i + (Nk - Nq) + 1;
    return v < 0 ? 0 : (v > Nk ? Nk : v);
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
    return omp_get_max_threads();
#else
    (void)nthreads;
    return 1;
#endif
}

/* The quantized program for selected rows of one (b, h).
 * qc [Nq,128] int8, sq [ceil(Nq/bq)], kc [Nk,128] int8, sk [ceil(Nk/bk)],
 * vct [128, Nk_pad] E4M3 codes (transposed), sv [128].
 * out_f32 [nrows,128] (before the bf16 rounding), out_bf16 [nrows,128].
 * Returns the number of threads used. */
int orc_sage_attn_rows(const int8_t *qc, const float *sq, int bq,
                       const int8_t *kc, const float *sk, int bk,
                       const uint8_t *vct, int Nk_pad, const float *sv,
                       int Nq, int Nk, float sm_scale, int tile,
                       const int *rows, int nrows, float *out_f32, uint16_t *out_bf16,
                       int nthreads, int causal, double *lse)
{
    int used = set_threads(nthreads);
    double *kmat = (double *)malloc(sizeof(double) * (size_t)Nk * D + 8);
    double *vmat = (double *)malloc(sizeof(double) * (size_t)Nk * D + 8);
    double *skey = (double *)malloc(sizeof(double) * (size_t)Nk + 8);
    double svd[D];
    for (size_t i = 0; i < (size_t)Nk * D; ++i) kmat[i] = (double)kc[i];
    for (int t = 0; t < Nk; ++t) {
        skey[t] = (double)sk[t / bk];
        for (int c = 0; c < D; ++c) vmat[(size_t)t * D + c] = orc_e4m3_value(vct[(size_t)c * Nk_pad + t]);
    }
    for (int c = 0; c < D; ++c) svd[c] = (double)sv[c];
    const double log2e_f32 = (double)(float)1.4426950408889634;
    orc_prog pg = {1, tile, FL((double)sm_scale * log2e_f32), 448.0};
#pragma omp parallel
    {
        double *S = (double *)malloc(sizeof(double) * (size_t)tile);
        double *s = (double *)malloc(sizeof(double) * (size_t)tile);
        double *P = (double *)malloc(sizeof(double) * (size_t)tile);
        double qrow[D], out[D];
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < nrows; ++r) {
            int i = rows[r];
            for (int c = 0; c < D; ++c) qrow[c] = (double)qc[(size_t)i * D + c];
            program_row(&pg, qrow, (double)sq[i / bq], kmat, skey, vmat, svd, Nk,
                        visible_keys(i, Nq, Nk, causal), S, s, P, out, lse ? lse + r : NULL);
            for (int c = 0; c < D; ++c) {
                out_f32[(size_t)r * D + c] = (float)out[c];
                out_bf16[(size_t)r * D + c] = orc_f32_to_bf16((float)out[c]);
            }
        }
        free(S); free(s); free(P);
    }
    free(kmat); free(vmat); free(skey);
    return used;
}

/* The same tile loop with quantisation off, in fp64: q,k,v [N,128] doubles. */
void orc_attn_rows_f64(const double *q, const double *k, const double *v,
                       int Nq, int Nk, double sm_scale, int tile,
                       const int *rows, int nrows, double *out, int causal, double *lse)
{
    double *skey = (double *)malloc(sizeof(double) * (size_t)Nk + 8);
    double sv[D];
    for (int t = 0; t < Nk; ++t) skey[t] = 1.0;
    for (int c = 0; c < D; ++c) sv[c] = 1.0;
    orc_prog pg = {0, tile, sm_scale / log(2.0), 1.0};
    double *S = (double *)malloc(sizeof(double) * (size_t)tile);
    double *s = (double *)malloc(sizeof(double) * (size_t)tile);
    double *P = (double *)malloc(sizeof(double) * (size_t)tile);
    for (int r = 0; r < nrows; ++r)
        program_row(&pg, q + (size_t)rows[r] * D, 1.0, k, skey, v, sv, Nk,
                    visible_keys(rows[r], Nq, Nk, causal), S, s, P, out + (size_t)r * D,
                    lse ? lse + r : NULL);
    free(S); free(s); free(P); free(skey);
}

/* ------------------------------------------------------------------------
 * a9: int8 KV-cache prompt attention, the exact program in fp64.
 * Query i (position q_pos0 + i) of query head h reads kv head
 * g = h / (Hq / Hkv) (contiguous groups) and keys j <= q_pos0 + i:
 *   s_ij = sm_scale * ks_j * sum_c q_ic kc_jc
 *   p    = softmax_j(s)                (natural base, fp64)
 *   o_ic = sum_j p_ij * vs_j * vc_jc
 * Layouts: q [Nq, Hq, 128] bf16; kc, vc [Hkv, Nk, 128] int8 (kv head stride
 * Nk*128); ks, vs [Hkv, Nk] fp16; rows/heads select (i, h) pairs;
 * out [n, 128] fp64.
 * --------------------------------------------------------------------- */
int orc_int8kv_rows(const uint16_t *q, const int8_t *kc, const uint16_t *ks,
                    const int8_t *vc, const uint16_t *vs,
                    int Nq, int q_pos0, int Nk, int Hq, int Hkv, double sm_scale,
                    const int *rows, const int *heads, int n, double *out, int nthreads)
{
    (void)Nq;
    int used = set_threads(nthreads);
    int grp = Hq / Hkv;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Nk + 8);
#pragma omp for schedule(dynamic, 1)
        for (int r = 0; r < n; ++r) {
            int i = rows[r], h = heads[r], g = h / grp;
            int last = q_pos0 + i;                  /* keys 0..last are visible */
            if (last > Nk - 1) last = Nk - 1;
            const uint16_t *qrow = q + ((size_t)i * Hq + h) * D;
            double qd[D];
            for (int c = 0; c < D; ++c) qd[c] = orc_bf16_value(qrow[c]);
            double m = -INFINITY;
            for (int j = 0; j <= last; ++j) {
                const int8_t *krow = kc + ((size_t)g * Nk + j) * D;
                double acc = 0.0;
                for (int c = 0; c < D; ++c) acc += qd[c] * (double)krow[c];
                s[j] = sm_scale * orc_f16_value(ks[(size_t)g * Nk + j]) * acc;
                if (s[j] > m) m = s[j];
            }
            double l = 0.0, o[D];
            for (int c = 0; c < D; ++c) o[c] = 0.0;
            for (int j = 0; j <= last; ++j) {
                double p = exp(s[j] - m);
                l += p;
                double w = p * orc_f16_value(vs[(size_t)g * Nk + j]);
                const int8_t *vrow = vc + ((size_t)g * Nk + j) * D;
                for (int c = 0; c < D; ++c) o[c] += w * (double)vrow[c];
            }
            for (int c = 0; c < D; ++c) out[(size_t)r * D + c] = o[c] / l;
        }
        free(s);
    }
    return used;
}

/* ------------------------------------------------------------------------
 * The int8 KV cache itself, per token: "Strata PR #2092" (int8 K/V cache
 * with per-token fp16 scales; the cache is written upstream of the prompt
 * attention).  Reading of the recipe (the page gives the format, not the
 * rounding): per row of 128 channels of one (kv head, token),
 *   amax  = max |x_c|                       (exact)
 *   scale = fp16_rn(fl(amax / 127))         (fp32 division, then fp16)
 *   code  = clamp(rint_even(fl(x_c / float(scale))), -127, 127), and 0
 *           wherever the fp16 scale is 0.
 * x: [nrows][128] fp32; codes [nrows][128]; scales [nrows] fp16 bits.
 * --------------------------------------------------------------------- */
void orc_cache_quantise_rows(const float *x, int64_t nrows, int8_t *codes, uint16_t *scales)
{
    for (int64_t r = 0; r < nrows; ++r) {
        const float *row = x + r * D;
        double amax = 0.0;
        for (int c = 0; c < D; ++c) {
            double a = fabs((double)row[c]);
            if (a > amax) amax = a;
        }
        uint16_t h = orc_f32_to_f16((float)FL(amax / 127.0));
        double s = orc_f16_value(h);
        scales[r] = h;
        for (int c = 0; c < D; ++c)
            codes[r * D + c] = (int8_t)(s > 0.0 ? rni_sat127(FL((double)row[c] / s)) : 0);
    }
}

/* ------------------------------------------------------------------------
 * array forms of the conversions (for exhaustive checks from the tests)
 * --------------------------------------------------------------------- */
void orc_f32_to_bf16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_bf16(x[i]);
}

void orc_f32_to_e4m3_array(const float *x, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_e4m3(x[i]);
}

void orc_e4m3_value_array(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3_value(c[i]);
}

void orc_f16_value_array(const uint16_t *h, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16_value(h[i]);
}

void orc_f32_to_f16_array(const float *x, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f32_to_f16(x[i]);
}

/* the int8 code of a quantised value: round half to even, saturated to
   [-127, 127] (the last step of the Q/K and cache quantisers) */
void orc_f32_to_i8_array(const float *x, int64_t n, int8_t *out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (int8_t)rni_sat127((double)x[i]);
}
