/*
 * h3fp4_oracle.c -- plain, slow CPU oracle for the modulation-fused NVFP4
 * activation producer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  It shares no
 * code, header, table or helper with the CUDA path under
 * dit_modulate_absmax_gb300/csrc, and the CUDA path never calls it.
 *
 * Every value is computed from its plain definition: each arithmetic step is
 * carried out in IEEE double (exact for every product used here, and
 * correctly rounded for the sums and quotients) and then rounded to its target
 * format by one generic round-to-nearest-even routine, orc_round(), that
 * knows only the format's precision, its smallest normal exponent and its
 * largest finite value.  A double result that is then rounded to a much
 * narrower format (bf16: 8 significand bits, fp32: 24) gives the correctly
 * rounded result of the exact operation, because 53 >= 2p + 2 for both
 * (Figueroa's double-rounding theorem for +, *, /).
 *
 * Sources (page title, section):
 *  - "NVFP4 Modulation Producer Fusion", Exactness Contract: segment-specific
 *    shift/scale selection; (x * (scale + 1)) + shift in that order with BF16
 *    rounding.
 *  - "NVFP4 Streaming Design", Numerical Constraint: one exact global BF16
 *    absolute maximum -> one FP32 tensor scale -> one E4M3 block scale per 16
 *    values -> E2M1 values quantised with both scales.
 *  - "FC2 NVFP4 Library Scheduling", Exact Operation / Current Baseline:
 *    packed E2M1 activation [M,K], E4M3 VEC16 block scales, SwiGLU producer in
 *    exact BF16, 37,810 -> 37,824 zero-row padding.
 * The encoding rule the pages leave open is fixed as:
 *    tensor scale ts = RN_f32(amax / (6 * 448))
 *    block scale  bs = E4M3_RNE_sat(RN_f32(block_amax / RN_f32(6 * ts)))
 *    code         q  = E2M1_RNE_sat(RN_f32(y / RN_f32(dec(bs) * ts)))
 * with the readings: an all-zero block (block_amax == 0) gets bs = 0, and a
 * block whose FP32 scale product is zero gets signed-zero codes.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------------------------------------------------------------------------
 * Threads.  When built with OpenMP the row loops below run their rows on
 * several threads; each row's arithmetic is exactly the same whichever thread
 * runs it, and the only cross-row step (the absolute maximum) is an exact,
 * order-independent max.  Without OpenMP everything runs on one thread.
 * ------------------------------------------------------------------------- */
void orc_set_threads(int n)
{
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}

int orc_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------------------
 * Generic rounding: round finite v to the nearest value of a binary format with
 * p significand bits (implicit bit included) and smallest normal exponent
 * emin (so the subnormal quantum is 2^(emin - p + 1)); ties go to the even
 * significand.  Results above maxv become +-inf (saturate == 0) or +-maxv
 * (saturate != 0).  NaN and infinities pass through unchanged.
 * ------------------------------------------------------------------------- */
double orc_round(double v, int p, int emin, double maxv, int saturate)
{
    if (v != v || isinf(v) || v == 0.0)
        return v;
    double a = fabs(v);
    int e2;
    frexp(a, &e2);               /* a = f * 2^e2, f in [0.5, 1) */
    int lead = e2 - 1;           /* exponent of the leading bit */
    int E = lead > emin ? lead : emin;
    double quantum = ldexp(1.0, E - (p - 1));
    double m = a / quantum;      /* exact: division by a power of two */
    double r = nearbyint(m);     /* default mode: nearest, ties to even */
    double res = r * quantum;
    if (res > maxv)
        res = saturate ? maxv : INFINITY;
    return v < 0 ? -res : res;
}

#define BF16_MAX (ldexp(255.0, 120))          /* (2 - 2^-7) * 2^127 */
#define F32_MAX  (ldexp(16777215.0, 104))     /* (2 - 2^-23) * 2^127 */

double orc_rn_bf16(double v) { return orc_round(v, 8, -126, BF16_MAX, 0); }
double orc_rn_f32(double v)  { return orc_round(v, 24, -126, F32_MAX, 0); }

/* bf16 bit pattern <-> value.  A bf16 is the upper half of an IEEE binary32. */
double orc_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* v must already be a bf16 value (output of orc_rn_bf16) or NaN/inf. */
uint16_t orc_bf16_bits(double v)
{
    float f = (float)v;          /* exact for bf16 values */
    uint32_t u;
    memcpy(&u, &f, 4);
    if (v != v)
        return 0x7FC0;           /* canonical quiet NaN */
    return (uint16_t)(u >> 16);
}

float orc_f32_from_double(double v) { return (float)v; }

/* ---------------------------------------------------------------------------
 * E4M3 (the "fn" variant: bias 7, no infinities, 0x7F / 0xFF are NaN, largest
 * finite 448) and E2M1 (bias 1, values 0, 0.5, 1, 1.5, 2, 3, 4, 6).
 * ------------------------------------------------------------------------- */
double orc_e4m3_decode(uint8_t c)
{
    int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    double v;
    if (e == 0xF && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round to E4M3 with ties to even, saturating to +-448; NaN -> 0x7F. */
uint8_t orc_e4m3_encode(double v)
{
    if (v != v)
        return 0x7F;
    uint8_t s = signbit(v) ? 0x80 : 0x00;
    double r = fabs(orc_round(v, 4, -6, 448.0, 1));
    if (isinf(v))
        r = 448.0;
    if (r == 0.0)
        return s;
    int e2;
    frexp(r, &e2);
    int lead = e2 - 1;
    if (lead < -6)                                  /* subnormal */
        return s | (uint8_t)(r / ldexp(1.0, -9));
    int m = (int)((r / ldexp(1.0, lead) - 1.0) * 8.0);
    return s | (uint8_t)(((lead + 7) << 3) | m);
}

static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(uint8_t c)
{
    double v = E2M1_MAG[c & 7];
    return (c & 8) ? -v : v;
}

/* Round to E2M1 with ties to even, saturating to +-6, keeping the sign of
 * zero (a negative value that rounds to zero gives code 0x8). */
uint8_t orc_e2m1_encode(double v)
{
    uint8_t s = signbit(v) ? 0x8 : 0x0;
    double r = isinf(v) ? 6.0 : fabs(orc_round(v, 2, 0, 6.0, 1));
    for (uint8_t c = 0; c < 8; ++c)
        if (E2M1_MAG[c] == r)
            return s | c;
    return s | 7;   /* NaN input: unspecified by the pages */
}

/* ---------------------------------------------------------------------------
 * AdaLN modulation, "NVFP4 Modulation Producer Fusion", Exactness Contract.
 * Row r belongs to segment s when seg_off[s] <= r < seg_off[s+1]; the
 * segment's shift/scale rows are shift[s*ld_mod .. ], scale[s*ld_mod .. ].
 *   s1 = RN_bf16(scale + 1);  t = RN_bf16(x * s1);  y = RN_bf16(t + shift)
 * ------------------------------------------------------------------------- */
void orc_modulate(const uint16_t *x, int64_t ldx, int64_t m, int64_t d,
                  const uint16_t *shift, const uint16_t *scale, int64_t ld_mod,
                  const int32_t *seg_off, int32_t nseg,
                  uint16_t *y, int64_t ldy)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; ++r) {
        int32_t s = 0;
        while (s + 1 < nseg && r >= seg_off[s + 1])
            ++s;
        for (int64_t j = 0; j < d; ++j) {
            double xv = orc_bf16_value(x[r * ldx + j]);
            double sc = orc_bf16_value(scale[s * ld_mod + j]);
            double sh = orc_bf16_value(shift[s * ld_mod + j]);
            double s1 = orc_rn_bf16(sc + 1.0);
            double t = orc_rn_bf16(xv * s1);
            double yv = orc_rn_bf16(t + sh);
            y[r * ldy + j] = orc_bf16_bits(yv);
        }
    }
}

/* ---------------------------------------------------------------------------
 * Gated residual epilogue, "NVFP4 Streaming Design", P4 (exact epilogue):
 * after the GEMM's BF16 conversion c, the gate multiply and the residual add,
 * each rounded to BF16:
 *   p = RN_bf16(gate_s * c);  out = RN_bf16(res + p)
 * with gate_s the gate row of the row's segment.  A product of two bf16
 * values is exact in double; a sum of two bf16 values is rounded to double
 * only when their exponents differ by more than 45, where that rounding
 * cannot move the bf16 result (53 >= 2 * 8 + 2).
 * ------------------------------------------------------------------------- */
void orc_gated_residual(const uint16_t *c, int64_t ldc, const uint16_t *gate, int64_t ld_gate,
                        const int32_t *seg_off, int32_t nseg, const uint16_t *res, int64_t ldr,
                        int64_t m, int64_t n, uint16_t *out, int64_t ldo)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; ++r) {
        int32_t s = 0;
        while (s + 1 < nseg && r >= seg_off[s + 1])
            ++s;
        for (int64_t j = 0; j < n; ++j) {
            double cv = orc_bf16_value(c[r * ldc + j]);
            double g = orc_bf16_value(gate[s * ld_gate + j]);
            double p = orc_rn_bf16(g * cv);
            double rv = orc_bf16_value(res[r * ldr + j]);
            out[r * ldo + j] = orc_bf16_bits(orc_rn_bf16(rv + p));
        }
    }
}

/* ---------------------------------------------------------------------------
 * SwiGLU producer input, "FC2 NVFP4 Library Scheduling", Exact Operation:
 *   h = RN_bf16(silu_bf16(gate) * up)
 * silu_table[g] is the bf16 pattern of the correctly rounded silu of the bf16
 * pattern g (built by the Python side at high precision).
 * ------------------------------------------------------------------------- */
void orc_swiglu(const uint16_t *g, int64_t ldg, const uint16_t *u, int64_t ldu,
                int64_t m, int64_t f, const uint16_t *silu_table,
                uint16_t *h, int64_t ldh)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; ++r)
        for (int64_t j = 0; j < f; ++j) {
            double sg = orc_bf16_value(silu_table[g[r * ldg + j]]);
            double uv = orc_bf16_value(u[r * ldu + j]);
            h[r * ldh + j] = orc_bf16_bits(orc_rn_bf16(sg * uv));
        }
}

/* ---------------------------------------------------------------------------
 * Global absolute maximum over the logical rows, "NVFP4 Streaming Design",
 * Numerical Constraint item 1.  Returns the bf16 pattern of max |y| (|-0| = 0);
 * any NaN makes the result NaN.
 * ------------------------------------------------------------------------- */
uint16_t orc_absmax(const uint16_t *y, int64_t ldy, int64_t m, int64_t d)
{
    double amax = 0.0;
    int nan = 0;
#pragma omp parallel for schedule(static) reduction(max : amax) reduction(| : nan)
    for (int64_t r = 0; r < m; ++r)
        for (int64_t j = 0; j < d; ++j) {
            double v = orc_bf16_value(y[r * ldy + j]);
            if (v != v)
                nan = 1;
            else if (fabs(v) > amax)
                amax = fabs(v);
        }
    return nan ? 0x7FC0 : orc_bf16_bits(amax);
}

/* Tensor scale from the absmax: RN_f32(amax / (6 * 448)). */
float orc_tensor_scale(uint16_t amax_bits)
{
    double a = orc_bf16_value(amax_bits);
    return (float)orc_rn_f32(a / 2688.0);
}

/* ---------------------------------------------------------------------------
 * NVFP4 pack, "NVFP4 Streaming Design", Numerical Constraint items 3-4.
 * Non-finite inputs (listed as adversarial cases in the Validation Ladder,
 * item 1, with no expected bytes) follow the same formulas in IEEE
 * arithmetic: a NaN in a block makes its maximum NaN, a NaN quotient encodes
 * as the E4M3 NaN code 0x7F (a tensor scale that is NaN, from a NaN anywhere,
 * or infinite, from an infinity, gives such quotients), and a block whose
 * scale product is zero or NaN gets zeros with y's signs.
 * y is [m, d] bf16 (logical rows).  Writes
 *   qdata [m_pad, d/2]: byte (r, j/2) = code(r, j) | code(r, j+1) << 4,
 *   sf    [sf_rows, d/16] (LOGICAL row-major, not swizzled): E4M3 codes,
 * where rows m <= r < m_pad of qdata and rows m <= r < sf_rows of sf are 0.
 * ------------------------------------------------------------------------- */
void orc_pack(const uint16_t *y, int64_t ldy, int64_t m, int64_t m_pad, int64_t d,
              float ts, uint8_t *qdata, uint8_t *sf, int64_t sf_rows)
{
    int64_t nb = d / 16;
    memset(qdata, 0, (size_t)(m_pad * (d / 2)));
    memset(sf, 0, (size_t)(sf_rows * nb));
    double tsd = (double)ts;
    double den = orc_rn_f32(6.0 * tsd);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < m; ++r)
        for (int64_t b = 0; b < nb; ++b) {
            double v[16], bamax = 0.0;
            for (int j = 0; j < 16; ++j) {
                v[j] = orc_bf16_value(y[r * ldy + b * 16 + j]);
                if (v[j] != v[j])
                    bamax = NAN;                    /* a NaN makes the block maximum NaN */
                else if (fabs(v[j]) > bamax)
                    bamax = fabs(v[j]);
            }
            uint8_t bs = 0;                         /* an all-zero block gets scale 0 */
            if (bamax != 0.0)                       /* a NaN quotient encodes as 0x7F */
                bs = orc_e4m3_encode(orc_rn_f32(bamax / den));
            double sc = orc_rn_f32(orc_e4m3_decode(bs) * tsd);
            sf[r * nb + b] = bs;
            for (int j = 0; j < 16; j += 2) {
                uint8_t c[2];
                for (int t = 0; t < 2; ++t) {
                    double yv = v[j + t];
                    if (sc == 0.0 || sc != sc)      /* zero or NaN scale product: signed zeros */
                        c[t] = signbit(yv) ? 0x8 : 0x0;
                    else
                        c[t] = orc_e2m1_encode(orc_rn_f32(yv / sc));
                }
                qdata[r * (d / 2) + (b * 16 + j) / 2] = (uint8_t)(c[0] | (c[1] << 4));
            }
        }
}

/* ---------------------------------------------------------------------------
 * Scale-factor layout consumed by the block-scaled GEMM ("VEC16_UE4M3"
 * swizzled layout named in "FC2 NVFP4 Library Scheduling", Exact Operation):
 * the logical [rows, cols] matrix (rows a multiple of 128, cols a multiple of
 * 4) is cut into 128x4 tiles stored tile-row-major as 512-byte atoms; inside
 * an atom, row r and column c sit at byte (r % 32) * 16 + (r / 32) * 4 + c.
 * ------------------------------------------------------------------------- */
int64_t orc_sf_offset(int64_t r, int64_t c, int64_t cols)
{
    int64_t tile = (r / 128) * (cols / 4) + (c / 4);
    int64_t rr = r % 128;
    return tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (c % 4);
}

void orc_swizzle_sf(const uint8_t *sf, int64_t rows, int64_t cols, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            out[orc_sf_offset(r, c, cols)] = sf[r * cols + c];
}

void orc_unswizzle_sf(const uint8_t *in, int64_t rows, int64_t cols, uint8_t *sf)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c)
            sf[r * cols + c] = in[orc_sf_offset(r, c, cols)];
}

/* Dequantise rows [r0, r1) of a packed operand into doubles:
 * out[(r - r0) * k + j] = e2m1(code(r, j)) * e4m3(sf(r, j/16)) * ts. */
void orc_dequant(const uint8_t *q, const uint8_t *sf, int64_t k, float ts,
                 int64_t r0, int64_t r1, double *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t r = r0; r < r1; ++r)
        for (int64_t j = 0; j < k; ++j) {
            uint8_t byte = q[r * (k / 2) + j / 2];
            uint8_t code = (j & 1) ? (byte >> 4) : (byte & 0xF);
            double s = orc_e4m3_decode(sf[r * (k / 16) + j / 16]);
            out[(r - r0) * k + j] = orc_e2m1_decode(code) * s * (double)ts;
        }
}

/* Array form of orc_round(), for the pins. */
void orc_round_array(const double *in, int64_t n, int p, int emin, double maxv,
                     int saturate, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_round(in[i], p, emin, maxv, saturate);
}

/* Array forms of the two encoders, for the pins. */
void orc_e4m3_encode_array(const double *in, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e4m3_encode(in[i]);
}

void orc_e2m1_encode_array(const double *in, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = orc_e2m1_encode(in[i]);
}
