/*
 * oracle.c -- plain, slow, single-threaded CPU oracle for the fused-chain hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's CPU-baseline
 * leg may load this library.  It shares no code, header, table or helper with the CUDA
 * path (epilogue_chains_gb300/csrc); neither side includes or links the other.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no -ffast-math, no FMA contraction), so
 * every float expression below rounds exactly where it is written.
 *
 * Sources (the web pages this library is built from):
 *   [K4]   "K4 walkthrough: the three ledgers of fusion -- bytes, launches, registers"
 *          (AI-compiler drills, hints/k4_fusion)
 *   [C05]  "C-05 Kernel Fusion cost boundary: less write-back vs register pressure and occupancy"
 *   [OFCG] "AIGC fundamentals | operator fusion and CUDA Graph"
 *
 * Every function states the passage it follows.  Where the pages leave a step open, the
 * reading taken is written next to the code.  Each function is pinned by the -m "not gpu"
 * tests against closed forms, invariants, special cases and brute force on tiny inputs.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------------------ */
/* Rounding a double to a narrower IEEE binary format, round-to-nearest-even.            */
/* p = significand bits including the hidden bit, emin = exponent of the smallest normal, */
/* emax = exponent of the largest finite binade.  Used for fp16 (11,-14,15),             */
/* bf16 (8,-126,127) and fp32 (24,-126,127).  Written from the IEEE 754 definition:     */
/* the representable numbers near |v| are the multiples of q = 2^(max(e,emin)-p+1),      */
/* where e is the exponent of v's leading bit; v/q is exact (q is a power of two) and    */
/* nearbyint() in the default rounding mode rounds it half-to-even.                      */
/* ------------------------------------------------------------------------------------ */
static double round_to_format(double v, int p, int emin, int emax)
{
    if (v != v || v == 0.0 || isinf(v)) return v;
    int e2;
    frexp(fabs(v), &e2);          /* |v| = f * 2^e2, f in [0.5, 1) */
    int lead = e2 - 1;            /* exponent of the leading bit */
    if (lead < emin) lead = emin; /* subnormal range: fixed quantum */
    double q = ldexp(1.0, lead - p + 1);
    double r = nearbyint(v / q) * q;
    double maxfin = ldexp(2.0 - ldexp(1.0, 1 - p), emax);
    if (fabs(r) > maxfin) r = copysign(INFINITY, v);
    return r;
}

double orc_round_half(double v) { return round_to_format(v, 11, -14, 15); }
double orc_round_bf16(double v) { return round_to_format(v, 8, -126, 127); }
double orc_round_f32(double v) { return round_to_format(v, 24, -126, 127); }

/* Encode an already-representable value into binary16 / bfloat16 bit patterns. */
static uint16_t encode_small(double r, int p, int emin, int ebias, int ebits)
{
    uint16_t sign = signbit(r) ? (uint16_t)(1u << (p - 1 + ebits)) : 0;
    double a = fabs(r);
    uint16_t expmask = (uint16_t)((1u << ebits) - 1u);
    if (r != r) return (uint16_t)(sign | (expmask << (p - 1)) | (1u << (p - 2)));
    if (isinf(r)) return (uint16_t)(sign | (expmask << (p - 1)));
    if (a == 0.0) return sign;
    int e2;
    frexp(a, &e2);
    int lead = e2 - 1;
    if (lead < emin) { /* subnormal: exponent field 0, mantissa = a / 2^(emin-p+1) */
        uint16_t m = (uint16_t)ldexp(a, -(emin - p + 1));
        return (uint16_t)(sign | m);
    }
    uint16_t m = (uint16_t)(ldexp(a, -(lead - p + 1)) - ldexp(1.0, p - 1));
    uint16_t ef = (uint16_t)(lead + ebias);
    return (uint16_t)(sign | (uint16_t)(ef << (p - 1)) | m);
}

static double decode_small(uint16_t h, int p, int emin, int ebias, int ebits)
{
    int sign = (h >> (p - 1 + ebits)) & 1;
    int ef = (h >> (p - 1)) & ((1 << ebits) - 1);
    int m = h & ((1 << (p - 1)) - 1);
    double v;
    if (ef == (1 << ebits) - 1) v = m ? NAN : INFINITY;
    else if (ef == 0) v = ldexp((double)m, emin - p + 1);
    else v = ldexp((double)(m + (1 << (p - 1))), ef - ebias - p + 1);
    return sign ? -v : v;
}

uint16_t orc_half_bits(double v) { return encode_small(orc_round_half(v), 11, -14, 15, 5); }
uint16_t orc_bf16_bits(double v) { return encode_small(orc_round_bf16(v), 8, -126, 127, 8); }
double orc_half_value(uint16_t h) { return decode_small(h, 11, -14, 15, 5); }
double orc_bf16_value(uint16_t h) { return decode_small(h, 8, -126, 127, 8); }

/* storage types of the pointwise chain (values match the library's dtype codes by definition
 * of the interface: 0 = fp32, 1 = fp16, 2 = bf16) */
static double load_elem(const void* base, int dtype, int64_t i)
{
    if (dtype == 0) return (double)((const float*)base)[i];
    if (dtype == 1) return orc_half_value(((const uint16_t*)base)[i]);
    return orc_bf16_value(((const uint16_t*)base)[i]);
}
static void store_elem(void* base, int dtype, int64_t i, float v)
{
    if (dtype == 0) ((float*)base)[i] = v;
    else if (dtype == 1) ((uint16_t*)base)[i] = orc_half_bits((double)v);
    else ((uint16_t*)base)[i] = orc_bf16_bits((double)v);
}

/* ------------------------------------------------------------------------------------ */
/* O1/O2  pointwise chain.                                                               */
/* [C05] §3 "API / experiment shape": stage s computes y = a_s*y + b_s, ReLU on the even  */
/* stages; the fused kernel loops s = 0..k-1 over that stage op.  [OFCG] §4.1 runs the    */
/* same chain as numpy multiply-then-add (two roundings per stage), which is the          */
/* rounding taken here: t = fl32(fl32(a_s*y) + b_s).                                      */
/* Readings: "even" is 0-based (s = 0, 2, 4, ...); ReLU follows the affine step and is    */
/* ReLU(t) = t if t > 0 else +0 (so -0 and NaN map to +0).  relu[s] != 0 switches ReLU on */
/* for stage s, so the all-affine chain of [OFCG] §4.1 is relu[] = 0.                     */
/* Values are loaded from the storage type exactly, the math is fp32, and the final value */
/* is rounded once to the storage type.                                                   */
/* ------------------------------------------------------------------------------------ */
void orc_chain(const int32_t* relu, const float* a, const float* b, int K,
               const void* x, void* y, int64_t n, int dtype)
{
    for (int64_t i = 0; i < n; ++i) {
        float v = (float)load_elem(x, dtype, i);
        for (int s = 0; s < K; ++s) {
            float prod = a[s] * v;   /* one fp32 rounding */
            float t = prod + b[s];   /* one fp32 rounding */
            if (relu[s]) t = (t > 0.0f) ? t : 0.0f;
            v = t;
        }
        store_elem(y, dtype, i, v);
    }
}

/* [OFCG] §4.1, V3 "algebraic merge": K identical affine stages compose into one affine map,
 * h_K = A^K h_0 + B (A^K - 1)/(A - 1).  Evaluated in double with A, B given as the fp32
 * constants the chain uses (numpy casts the scalar to the array's fp32 type). */
void orc_affine_closed_form(const float* x, double* y, int64_t n, int K, float A, float B)
{
    double Ad = (double)A, Bd = (double)B;
    double Ak = pow(Ad, (double)K);
    double Bk = Bd * (Ak - 1.0) / (Ad - 1.0);
    for (int64_t i = 0; i < n; ++i) y[i] = Ak * (double)x[i] + Bk;
}

/* ------------------------------------------------------------------------------------ */
/* O3  RMSNorm.  [OFCG] §3.2 / fusion_lab [A2] lists the unfused steps as x*x, reduce     */
/* mean, x*r, *g; written out: r_i = 1/sqrt(mean_j x_ij^2 + eps), y_ij = (x_ij*r_i)*w_j.  */
/* Reading: the mean runs over the last (hidden) axis, eps sits inside the square root,  */
/* w is per column.  Sum, mean and both products in double; one rounding to fp32 at the  */
/* end.                                                                                   */
/* ------------------------------------------------------------------------------------ */
void orc_rmsnorm(const float* x, const float* w, float* y, int64_t rows, int64_t hidden,
                 double eps)
{
    for (int64_t i = 0; i < rows; ++i) {
        const float* xr = x + i * hidden;
        double acc = 0.0;
        for (int64_t j = 0; j < hidden; ++j) acc += (double)xr[j] * (double)xr[j];
        double ms = acc / (double)hidden;
        double r = 1.0 / sqrt(ms + eps);
        for (int64_t j = 0; j < hidden; ++j)
            y[i * hidden + j] = (float)(((double)xr[j] * r) * (double)w[j]);
    }
}

/* ------------------------------------------------------------------------------------ */
/* O4  causal attention-score softmax over the last axis of s[BH, S, S] (bf16 storage).  */
/* [OFCG] fusion_lab [E] gives the five steps max -> subtract -> exp -> sum -> divide;   */
/* §3.5 gives the causal rule "query i sees keys up to i".                                */
/* Readings: z_ij = s_ij * scale for j <= i (0-based), masked (j > i) entries are        */
/* excluded and their output is exactly +0; max, exp, sum and the division in double;    */
/* one rounding to the output type (out_dtype 2 = bf16 bits, 0 = fp32).                  */
/* ------------------------------------------------------------------------------------ */
void orc_causal_softmax(const uint16_t* s, void* p, int64_t BH, int64_t S, double scale,
                        int out_dtype)
{
    for (int64_t bh = 0; bh < BH; ++bh) {
        for (int64_t i = 0; i < S; ++i) {
            const uint16_t* row = s + (bh * S + i) * S;
            int64_t base = (bh * S + i) * S;
            double m = -INFINITY;
            for (int64_t j = 0; j <= i; ++j) {
                double z = orc_bf16_value(row[j]) * scale;
                if (z > m) m = z;
            }
            double l = 0.0;
            for (int64_t j = 0; j <= i; ++j) l += exp(orc_bf16_value(row[j]) * scale - m);
            for (int64_t j = 0; j < S; ++j) {
                double v = 0.0;
                if (j <= i) v = exp(orc_bf16_value(row[j]) * scale - m) / l;
                if (out_dtype == 2) ((uint16_t*)p)[base + j] = orc_bf16_bits(v);
                else ((float*)p)[base + j] = (float)v;
            }
        }
    }
}

/* The five-step unfused form with its intermediates stored in bf16 between steps, i.e. the
 * same arithmetic rounded at the points where the unfused kernels write global memory:
 *   m_i  = max_{j<=i} fl32(s_ij*scale)                     (fp32 row statistic)
 *   d_ij = bf16(fl32(fl32(s_ij*scale) - m_i)), -inf where j > i
 *   e_ij = bf16(exp(d_ij))                                 (exp(-inf) = +0)
 *   l_i  = sum_j e_ij                                      (double here)
 *   p_ij = out(e_ij / l_i)
 * Reading: [OFCG] fusion_lab [E] writes each step's result back before the next step; the
 * masked entries are carried as -inf so that no separate mask tensor exists. */
void orc_causal_softmax_unfused(const uint16_t* s, void* p, int64_t BH, int64_t S,
                                double scale, int out_dtype)
{
    float sc = (float)scale;
    for (int64_t bh = 0; bh < BH; ++bh) {
        for (int64_t i = 0; i < S; ++i) {
            const uint16_t* row = s + (bh * S + i) * S;
            int64_t base = (bh * S + i) * S;
            float m = -INFINITY;
            for (int64_t j = 0; j <= i; ++j) {
                float z = (float)orc_bf16_value(row[j]) * sc;
                if (z > m) m = z;
            }
            double l = 0.0;
            for (int64_t j = 0; j <= i; ++j) {
                float z = (float)orc_bf16_value(row[j]) * sc;
                float d = z - m;
                double dq = orc_bf16_value(orc_bf16_bits((double)d));
                double e = orc_bf16_value(orc_bf16_bits(exp(dq)));
                l += e;
            }
            for (int64_t j = 0; j < S; ++j) {
                double v = 0.0;
                if (j <= i) {
                    float z = (float)orc_bf16_value(row[j]) * sc;
                    float d = z - m;
                    double dq = orc_bf16_value(orc_bf16_bits((double)d));
                    double e = orc_bf16_value(orc_bf16_bits(exp(dq)));
                    v = e / l;
                }
                if (out_dtype == 2) ((uint16_t*)p)[base + j] = orc_bf16_bits(v);
                else ((float*)p)[base + j] = (float)v;
            }
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* O5  GEMM + bias + GELU + residual under a cut plan.                                    */
/* [K4] §① chain_mlp_epilogue: stages mm -> +bias -> GELU -> +residual at fp16; a cut    */
/* plan splits the four stages into consecutive kernels, and every cut writes the        */
/* intermediate back as fp16 (the "C, C', C''" round trips of the §① table).             */
/* cut_mask bit i (i = 0, 1, 2) = a kernel boundary after stage i (0 mm, 1 bias, 2 gelu); */
/* plan [1,1,1,1] = 0b111, [1,3] = 0b001, [2,2] = 0b010, [4] = 0.                          */
/* Readings: A [M,K] and B [K,N] row-major fp16, bias [N], R and Y [M,N] fp16; the        */
/* product is summed exactly enough in double; GELU is the erf form                      */
/* g(v) = v/2 (1 + erf(v/sqrt 2)); every cut and the final store round to fp16 (RNE).    */
/* Only the listed rows are computed: Y is [nrows, N], row r of Y is row rows[r] of the  */
/* full result (rows == NULL means all M rows).                                            */
/* ------------------------------------------------------------------------------------ */
static double gelu_erf(double v) { return 0.5 * v * (1.0 + erf(v / sqrt(2.0))); }

/* exported so that the GELU step can be checked on its own */
double orc_gelu(double v) { return gelu_erf(v); }

void orc_gemm_epilogue(const uint16_t* A, const uint16_t* B, const uint16_t* bias,
                       const uint16_t* R, uint16_t* Y, int64_t M, int64_t N, int64_t K,
                       uint32_t cut_mask, const int64_t* rows, int64_t nrows)
{
    if (rows == 0) nrows = M;
    /* Decode the fp16 operands to double once.  B is kept column by column (bt[n*K + k]) so
     * the k-sum reads contiguous memory; the sum still runs k = 0, 1, ..., K-1. */
    double* bt = (double*)malloc((size_t)(N * K) * sizeof(double));
    double* ar = (double*)malloc((size_t)K * sizeof(double));
    if (!bt || !ar) { free(bt); free(ar); return; }
    for (int64_t k = 0; k < K; ++k)
        for (int64_t n = 0; n < N; ++n) bt[n * K + k] = orc_half_value(B[k * N + n]);
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t m = rows ? rows[r] : r;
        for (int64_t k = 0; k < K; ++k) ar[k] = orc_half_value(A[m * K + k]);
        for (int64_t n = 0; n < N; ++n) {
            const double* bc = bt + n * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += ar[k] * bc[k];
            double v = acc;                                  /* stage 0: mm       */
            if (cut_mask & 1u) v = orc_round_half(v);
            v = v + orc_half_value(bias[n]);                 /* stage 1: + bias   */
            if (cut_mask & 2u) v = orc_round_half(v);
            v = gelu_erf(v);                                 /* stage 2: GELU     */
            if (cut_mask & 4u) v = orc_round_half(v);
            v = v + orc_half_value(R[m * N + n]);            /* stage 3: + R      */
            Y[r * N + n] = orc_half_bits(v);
        }
    }
    free(ar);
    free(bt);
}

/* ------------------------------------------------------------------------------------ */
/* Residual add + RMSNorm.  [OFCG] appendix launch_model [F3], the per-layer list after    */
/* fusion: "residual + RMSNorm fused" replaces the residual-add kernel and the four        */
/* RMSNorm kernels of the unfused list ([OFCG] §2: "residual 1, post RMSNorm 4").          */
/* Reading: the residual stream h = x + r (one fp32 rounding) is an output too, since it   */
/* feeds the next residual add; y is RMSNorm of h with the same definition as orc_rmsnorm. */
/* ------------------------------------------------------------------------------------ */
void orc_add_rmsnorm(const float* x, const float* r, const float* w, float* h, float* y,
                     int64_t rows, int64_t hidden, double eps)
{
    for (int64_t i = 0; i < rows * hidden; ++i) {
        float sum = x[i] + r[i];   /* one fp32 rounding */
        h[i] = sum;
    }
    orc_rmsnorm(h, w, y, rows, hidden, eps);
}

/* ------------------------------------------------------------------------------------ */
/* SiLU(gate) * up.  [OFCG] appendix launch_model [F3]: the gate/up projection is one GEMM  */
/* and "SiLU + mul fused" one kernel, where the unfused list has a SiLU kernel and an     */
/* element-wise multiply kernel.  SiLU(v) = v * logistic(v) = v / (1 + e^-v).             */
/* Readings: g and u are rows x cols with a common row stride ld (ld = 2 cols when both   */
/* halves of one merged gate/up output are passed); y is rows x cols, contiguous.  The    */
/* math is in double; the fused form rounds once to the storage type, the unfused form    */
/* also rounds the SiLU tensor it stores between its two kernels.                          */
/* ------------------------------------------------------------------------------------ */
static double silu(double v) { return v / (1.0 + exp(-v)); }
static double round_storage(double v, int dtype)
{
    if (dtype == 0) return (double)(float)v;
    if (dtype == 1) return orc_round_half(v);
    return orc_round_bf16(v);
}
static void store_elem_d(void* base, int dtype, int64_t i, double v)
{
    if (dtype == 0) ((float*)base)[i] = (float)v;
    else if (dtype == 1) ((uint16_t*)base)[i] = orc_half_bits(v);
    else ((uint16_t*)base)[i] = orc_bf16_bits(v);
}
double orc_silu(double v) { return silu(v); }

void orc_silu_mul(const void* g, const void* u, int64_t ld, void* y, int64_t rows, int64_t cols,
                  int dtype, int unfused)
{
    for (int64_t i = 0; i < rows; ++i) {
        for (int64_t j = 0; j < cols; ++j) {
            double gv = load_elem(g, dtype, i * ld + j);
            double uv = load_elem(u, dtype, i * ld + j);
            double s = silu(gv);
            if (unfused) s = round_storage(s, dtype);
            store_elem_d(y, dtype, i * cols + j, s * uv);
        }
    }
}

/* ------------------------------------------------------------------------------------ */
/* Causal attention without the score matrix.  [OFCG] §6.3 and its reading list            */
/* (FlashAttention, arXiv:2205.14135): the fused attention never materialises the S x S    */
/* scores of the softmax row above and normalises online.  What it computes is plain       */
/* causal scaled-dot-product attention, written out here from its definition:              */
/*     s_ij = scale * sum_d q_id k_jd   (j <= i),   p_ij = exp(s_ij - max_j s_ij),          */
/*     o_id = sum_j p_ij v_jd / sum_j p_ij,                                                 */
/* per (batch, head) slice, in double from the bf16 inputs, one rounding of o to bf16.      */
/* Reading: q, k, v, o are bf16 [BH, S, D] with D = d_model / heads (4096 / 16 = 256 for    */
/* the pages' B=8, H=16, S=2048 shape) and scale = 1/sqrt(D); mask j > i, 0-based.          */
/* rows (optional): only these query rows of every slice are computed (o has nrows rows    */
/* per slice then).                                                                         */
/* ------------------------------------------------------------------------------------ */
void orc_attention(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                   int64_t BH, int64_t S, int64_t D, double scale, const int64_t* rows,
                   int64_t nrows)
{
    double* srow = (double*)malloc(sizeof(double) * (size_t)S);
    double* acc = (double*)malloc(sizeof(double) * (size_t)D);
    const int64_t nr = rows ? nrows : S;
    for (int64_t b = 0; b < BH; ++b) {
        const uint16_t* qb = q + b * S * D;
        const uint16_t* kb = k + b * S * D;
        const uint16_t* vb = v + b * S * D;
        for (int64_t t = 0; t < nr; ++t) {
            const int64_t i = rows ? rows[t] : t;
            double m = -INFINITY;
            for (int64_t j = 0; j <= i; ++j) {
                double dot = 0.0;
                for (int64_t d = 0; d < D; ++d)
                    dot += orc_bf16_value(qb[i * D + d]) * orc_bf16_value(kb[j * D + d]);
                srow[j] = scale * dot;
                if (srow[j] > m) m = srow[j];
            }
            double l = 0.0;
            for (int64_t d = 0; d < D; ++d) acc[d] = 0.0;
            for (int64_t j = 0; j <= i; ++j) {
                const double pj = exp(srow[j] - m);
                l += pj;
                for (int64_t d = 0; d < D; ++d) acc[d] += pj * orc_bf16_value(vb[j * D + d]);
            }
            uint16_t* ob = o + (b * nr + t) * D;
            for (int64_t d = 0; d < D; ++d) ob[d] = orc_bf16_bits(acc[d] / l);
        }
    }
    free(srow);
    free(acc);
}

int orc_version(void) { return 1; }
