/*
 * Plain C, fp32, fixed-order fold of split-KV attention states.
 *
 * TEST INFRASTRUCTURE ONLY: this file is part of the CPU oracle.  The CUDA
 * library neither includes nor links it.
 *
 * What it computes (page: "Learning FlashAttention the Hard Way - Part 1"):
 *  - "Associativity is All You Need": split-K writes per-chunk partials to
 *    scratch and folds them in a second pass.
 *  - "The Merge, and the Twist": the merge keeps the larger maximum and
 *    rescales the other side by e^{dm} with dm <= 0; identity (-inf, 0, 0).
 *  - "Alternative Twist: Base 2": states over sigma = s log2(e), so every
 *    exponential is 2^x; the row is read off as o / d at the end.
 * Every row folds chunk 0, 1, ..., S-1 into the identity, left to right, in
 * binary32 with one rounding per operation (fmaf, +, *, /), so a GPU fold
 * that performs the same operation sequence gives the same bits.
 *
 * The two transcendental steps are written here from textbook methods, not
 * taken from any math library:
 *  - 2^x: range reduction x = n + f, n = rint(x), |f| <= 1/2 (exact in
 *    binary32), then the Taylor series of 2^f = sum (f ln2)^k / k!, truncated
 *    after k = 7 (remainder < 6e-9 relative), evaluated by Horner with fmaf,
 *    then multiplied by 2^n built from its exponent bits.  Arguments below
 *    -126 return 0.
 *  - ln(d) for d a positive normal number: d = 2^e x with x in
 *    [sqrt(1/2), sqrt(2)], ln x = 2 atanh(t), t = (x-1)/(x+1), |t| < 0.172,
 *    atanh(t) = t (1 + t^2/3 + t^4/5 + ... + t^10/11).
 * Coefficients are derived from their definitions at run time in double and
 * rounded to binary32 once.
 *
 * Build with -ffp-contract=off (no implicit fused multiply-adds).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static float coef_exp2[8];   /* (ln 2)^k / k!, k = 0..7 */
static float coef_atanh[6];  /* 1/(2j+1), j = 0..5      */
static float ln2_f, sqrt2_f;
static int coef_ready = 0;

static void init_coefficients(void) {
    const double ln2 = 0.693147180559945309417232121458;
    double c = 1.0;
    coef_exp2[0] = 1.0f;
    for (int k = 1; k < 8; ++k) {
        c = c * ln2 / (double)k;
        coef_exp2[k] = (float)c;
    }
    for (int j = 0; j < 6; ++j) coef_atanh[j] = (float)(1.0 / (double)(2 * j + 1));
    ln2_f = (float)ln2;
    sqrt2_f = (float)1.41421356237309504880;
    coef_ready = 1;
}

static float bits_to_float(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }
static uint32_t float_to_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }

float fa_oracle_exp2f(float x) {
    if (!coef_ready) init_coefficients();
    if (x != x) return x;
    if (x < -126.0f) return 0.0f;
    if (x >= 128.0f) return INFINITY;
    float n = rintf(x);
    float f = x - n;
    float p = coef_exp2[7];
    for (int k = 6; k >= 0; --k) p = fmaf(p, f, coef_exp2[k]);
    int ni = (int)n;
    float two_n = bits_to_float((uint32_t)(ni + 127) << 23);
    return p * two_n;
}

/* ln(d) for positive normal d, returned as (e, ln x) with ln d = e ln2 + ln x. */
static void ln_split(float d, int* e_out, float* lnx_out) {
    uint32_t u = float_to_bits(d);
    int e = (int)((u >> 23) & 0xffu) - 127;
    float x = bits_to_float((u & 0x7fffffu) | 0x3f800000u);
    if (x > sqrt2_f) { x = x * 0.5f; e += 1; }
    float t = (x - 1.0f) / (x + 1.0f);
    float w = t * t;
    float p = coef_atanh[5];
    for (int j = 4; j >= 0; --j) p = fmaf(p, w, coef_atanh[j]);
    *e_out = e;
    *lnx_out = (t + t) * p;
}

float fa_oracle_lnf(float d) {
    if (!coef_ready) init_coefficients();
    int e; float lnx;
    ln_split(d, &e, &lnx);
    return fmaf((float)e, ln2_f, lnx);
}

static uint16_t f32_to_bf16_rne(float x) {
    uint32_t u = float_to_bits(x);
    if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/*
 * part_m, part_d: [rows, S]; part_o: [rows, S, D] (row-major, fp32, base-2
 * states).  Writes out_o [rows, D] (fp32, may be NULL), out_o_bf16 [rows, D]
 * (RNE of the same fp32 value, may be NULL) and out_lse [rows] (natural log).
 * A row whose chunks are all empty gives O = 0 and LSE = -inf.
 * Returns 0, or -1 on bad sizes.
 */
int fa_oracle_combine_f32(const float* part_m, const float* part_d,
                          const float* part_o, int rows, int S, int D,
                          float* out_o, uint16_t* out_o_bf16, float* out_lse) {
    if (!coef_ready) init_coefficients();
    if (rows < 0 || S <= 0 || D <= 0 || D > 1024) return -1;
    float o[1024];
    for (int r = 0; r < rows; ++r) {
        float m = -INFINITY, dsum = 0.0f;
        for (int i = 0; i < D; ++i) o[i] = 0.0f;
        for (int c = 0; c < S; ++c) {
            const float mb = part_m[(size_t)r * S + c];
            const float db = part_d[(size_t)r * S + c];
            const float* ob = part_o + ((size_t)r * S + c) * (size_t)D;
            if (mb == -INFINITY) continue;                /* b is the identity */
            if (m == -INFINITY) {                         /* acc is the identity */
                m = mb; dsum = db;
                for (int i = 0; i < D; ++i) o[i] = ob[i];
                continue;
            }
            if (m >= mb) {
                float f = fa_oracle_exp2f(mb - m);
                dsum = fmaf(db, f, dsum);
                for (int i = 0; i < D; ++i) o[i] = fmaf(ob[i], f, o[i]);
            } else {
                float f = fa_oracle_exp2f(m - mb);
                dsum = fmaf(dsum, f, db);
                for (int i = 0; i < D; ++i) o[i] = fmaf(o[i], f, ob[i]);
                m = mb;
            }
        }
        float lse;
        if (dsum == 0.0f) {
            lse = -INFINITY;
            for (int i = 0; i < D; ++i) o[i] = 0.0f;
        } else {
            int e; float lnx;
            ln_split(dsum, &e, &lnx);
            lse = fmaf((float)e + m, ln2_f, lnx);
            for (int i = 0; i < D; ++i) o[i] = o[i] / dsum;
        }
        if (out_lse) out_lse[r] = lse;
        for (int i = 0; i < D; ++i) {
            if (out_o) out_o[(size_t)r * D + i] = o[i];
            if (out_o_bf16) out_o_bf16[(size_t)r * D + i] = f32_to_bf16_rne(o[i]);
        }
    }
    return 0;
}

/*
 * Plain C, fp32, fixed-order fold of Welford states (n, mu, M2), one row at a
 * time (page: "Learning FlashAttention the Hard Way - Part 1", section "The
 * Same Move: Welford's Variance": identity (0, 0, 0), the symmetric merge of
 * two partials over disjoint chunks, and the division of M2 by n at the end).
 * Every row folds chunk 0, 1, ..., S-1 into the identity, left to right:
 *   a (+) b = b if n_a = 0;  a if n_b = 0;  otherwise
 *     n = n_a + n_b,  delta = mu_b - mu_a,  r = n_b / n,
 *     mu = mu_a + delta * r,
 *     M2 = (M2_a + M2_b) + ((delta * delta) * n_a) * r,
 * each operation rounded once in binary32 in this order; then
 * var = M2 / n and rstd = 1 / sqrt(var + eps) (sqrt correctly rounded).
 * rstd may be NULL.  Returns -1 on bad sizes, else 0.
 */
static void welford_merge_f32(float* n, float* mu, float* m2, float nb, float mub, float m2b) {
  if (nb == 0.0f) return;
  if (*n == 0.0f) {
    *n = nb;
    *mu = mub;
    *m2 = m2b;
    return;
  }
  const float na = *n;
  const float nn = na + nb;
  const float delta = mub - *mu;
  const float r = nb / nn;
  const float t = delta * r;
  *mu = *mu + t;
  const float s = *m2 + m2b;
  const float dd = delta * delta;
  const float ddn = dd * na;
  const float cross = ddn * r;
  *m2 = s + cross;
  *n = nn;
}

int fa_oracle_welford_combine_f32(const float* part_n, const float* part_mu,
                                  const float* part_m2, int rows, int S, float eps,
                                  float* mean, float* var, float* rstd) {
  if (rows < 0 || S < 1) return -1;
  for (int r = 0; r < rows; ++r) {
    float n = 0.0f, mu = 0.0f, m2 = 0.0f;
    for (int c = 0; c < S; ++c) {
      const size_t i = (size_t)r * (size_t)S + (size_t)c;
      welford_merge_f32(&n, &mu, &m2, part_n[i], part_mu[i], part_m2[i]);
    }
    const float v = m2 / n;
    mean[r] = mu;
    var[r] = v;
    if (rstd) {
      const float ve = v + eps;
      const float sq = sqrtf(ve);
      rstd[r] = 1.0f / sq;
    }
  }
  return 0;
}
