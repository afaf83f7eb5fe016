/*
 * mxfp8_oracle.c -- plain, slow CPU statement of the MXFP8 cast path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The product path
 * (the CUDA library) shares no code, header, table or constant with it.
 *
 * What it computes, and where each step comes from:
 *
 *  - "Add swiglu + MXFP8 fused CuTe DSL kernel" (torchao fork PR #2),
 *    sections "Summary" and "API": one pass reads gate and up, forms the
 *    SwiGLU activation h = silu(gate) * up, and emits E4M3 data plus one
 *    E8M0 scale per 32-element block, rowwise (1x32), colwise (32x1) or both.
 *    The backward reads grad_h, gate and up and casts dGate and dUp the same
 *    way.  The activation is evaluated at fp32 precision and rounded once to
 *    bf16 before the cast (the oracle evaluates it in double, rounds to fp32,
 *    then rounds to bf16 with ties-to-even).
 *  - Same page, section "Numerics and tests", and its commit message: the
 *    scale rule is RCEIL; a block whose amax is NaN or Inf gets scale byte
 *    255 and all-NaN data; a byte-0 scale descales by 2^127.  RCEIL is
 *    written out as: the scale exponent is the smallest integer e with
 *    amax <= 448 * 2^e (that is ceil(log2(amax/448))), clamped to
 *    [-127, 127]; scale byte = e + 127; an all-zero block gets byte 0.
 *  - E4M3 data: x / 2^e rounded to nearest, ties to even, saturating to the
 *    largest finite magnitude 448; NaN data byte 0x7F; the sign of zero is
 *    kept (-0 and negative values that round to zero give 0x80).
 *  - "[mxfp8 moe training] update 3d quant colwise scaling kernel to use
 *    single input/output TMA descriptors" (pytorch/ao PR #3034), section
 *    "Summary": the 3D quantizer takes (E, N, K) row-major bf16 and writes
 *    each expert's (N, K) slab column-major ("column major per expert"),
 *    blocks of 32 along N, scales (E, N/32, K).
 *  - Other gated activations through the same kernel ("Add swiglu + MXFP8
 *    fused CuTe DSL kernel", section "API": the activation is a
 *    compile-time policy of the one kernel source): GEGLU, h = gelu(g) * u
 *    with the exact GELU g * Phi(g), Phi the standard normal CDF (the erf
 *    form, not the tanh approximation; the pages name no variant, this is
 *    the plainest reading).  Backward: dgate = dh * u * (Phi(g) + g phi(g)),
 *    phi the normal density; dup = dh * gelu(g).
 *  - Scales in the blocked layout the block-scaled tensor-core GEMMs read
 *    ("Add swiglu + MXFP8 fused CuTe DSL kernel", commit message: "the same
 *    blocked tcgen05 layouts as the standalone quantizers"; "[mxfp8 moe
 *    training] add compile support", review thread: scale matrices padded to
 *    multiples of 128 rows and 4 columns).  The order inside a 128 x 4 tile
 *    is not printed there; it is read as the published one for those GEMMs:
 *    32 x 4 x 4, entry (r, c) of a tile at byte (r % 32) * 16 + (r / 32) * 4
 *    + c, tiles row-major over the padded matrix.
 *
 * Every floating-point step is done in IEEE double with no contraction
 * (compile with -ffp-contract=off), no fast-math, and with plain loops in the
 * order the definition states.  Nothing is tiled, fused or reordered.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_ROWWISE 1
#define ORC_COLWISE 2

/* ------------------------------------------------------------------ bf16 */

/* Value of a bf16 bit pattern (exact: bf16 is the top half of an fp32). */
double orc_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Magnitude of a non-negative, non-NaN bf16 pattern on an unbounded exponent
 * scale: 0x7F80 (the pattern after the largest finite value) stands for 2^128,
 * which is where IEEE round-to-nearest overflows to infinity. */
static double bf16_mag_unbounded(uint16_t mag)
{
    if (mag == 0x7F80) return ldexp(1.0, 128);
    return orc_bf16_to_double(mag);
}

/* fp32 -> bf16, round to nearest, ties to even (IEEE 754).  Written as a
 * nearest-neighbour choice between the two bf16 values around |f|. */
uint16_t orc_bf16_round(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000);
    if (isnan(f)) return (uint16_t)(sign | 0x7FC0);
    if (isinf(f)) return (uint16_t)(sign | 0x7F80);
    double a = fabs((double)f);
    uint16_t lo = (uint16_t)((u >> 16) & 0x7FFF); /* truncation: value <= a */
    double vlo = orc_bf16_to_double(lo);
    if (vlo == a) return (uint16_t)(sign | lo);
    uint16_t hi = (uint16_t)(lo + 1);
    double vhi = bf16_mag_unbounded(hi);
    double dlo = a - vlo, dhi = vhi - a; /* both exact in double */
    uint16_t pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = (lo & 1) ? hi : lo; /* tie: even mantissa */
    return (uint16_t)(sign | pick);
}

/* double -> fp32 (IEEE round to nearest even, the C conversion) -> bf16. */
uint16_t orc_bf16_from_double_via_fp32(double x)
{
    return orc_bf16_round((float)x);
}

/* ------------------------------------------------------------------ E8M0 */

/* RCEIL scale byte for a block amax (amax >= 0, or NaN / Inf). */
uint8_t orc_e8m0_rceil(double amax)
{
    if (isnan(amax) || isinf(amax)) return 255;
    if (amax == 0.0) return 0;
    int x;
    frexp(amax, &x);           /* amax = f * 2^x, f in [0.5, 1) */
    int e = x - 10;            /* 448 * 2^(x-10) < 0.5 * 2^x <= amax */
    while (!(amax <= ldexp(448.0, e))) e++;
    if (e < -127) e = -127;
    if (e > 127) e = 127;
    return (uint8_t)(e + 127);
}

/* ------------------------------------------------------------------ E4M3 */

/* Value of an E4M3 (fn) magnitude code 0..126: bias 7, 3 mantissa bits,
 * subnormals m * 2^-9, no infinities, 0x7F is NaN. */
double orc_e4m3_to_double(uint8_t c)
{
    double s = (c & 0x80) ? -1.0 : 1.0;
    int mag = c & 0x7F;
    if (mag == 0x7F) return NAN;
    int e = mag >> 3, m = mag & 7;
    if (e == 0) return s * ldexp((double)m, -9);
    return s * ldexp(1.0 + m / 8.0, e - 7);
}

/* The 127 non-negative finite E4M3 values, by code, filled at load time
 * from the decoding rule above. */
static double e4m3_mag[127];

__attribute__((constructor)) static void orc_fill_e4m3_table(void)
{
    for (int c = 0; c < 127; c++) e4m3_mag[c] = orc_e4m3_to_double((uint8_t)c);
}

/* Round y to the nearest E4M3 value, ties to the even code, saturating. */
uint8_t orc_e4m3_encode(double y)
{
    if (isnan(y)) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs(y);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    /* binary search: largest code lo with e4m3_mag[lo] <= a */
    int lo = 0, hi = 126;
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (e4m3_mag[mid] <= a) lo = mid;
        else hi = mid;
    }
    if (e4m3_mag[lo] == a) return (uint8_t)(sign | lo);
    /* now e4m3_mag[lo] < a < e4m3_mag[lo + 1] */
    hi = lo + 1;
    double dlo = a - e4m3_mag[lo], dhi = e4m3_mag[hi] - a;
    int pick;
    if (dlo < dhi) pick = lo;
    else if (dhi < dlo) pick = hi;
    else pick = (lo & 1) ? hi : lo;
    return (uint8_t)(sign | pick);
}

/* ------------------------------------------------------------ one block */

/* Quantize 32 bf16 values (element i at v[i * vstride]) into 32 E4M3 codes
 * (code i at codes[i * cstride]) and one E8M0 scale byte. */
void orc_quant_block(const uint16_t *v, int64_t vstride, uint8_t *codes,
                     int64_t cstride, uint8_t *scale)
{
    double amax = 0.0;
    int special = 0;
    for (int i = 0; i < 32; i++) {
        double x = orc_bf16_to_double(v[i * vstride]);
        if (isnan(x) || isinf(x)) special = 1;
        else if (fabs(x) > amax) amax = fabs(x);
    }
    if (special) {
        *scale = 255;
        for (int i = 0; i < 32; i++) codes[i * cstride] = 0x7F;
        return;
    }
    uint8_t b = orc_e8m0_rceil(amax);
    int e = (int)b - 127;
    *scale = b;
    for (int i = 0; i < 32; i++) {
        double x = orc_bf16_to_double(v[i * vstride]);
        codes[i * cstride] = orc_e4m3_encode(ldexp(x, -e));
    }
}

/* ------------------------------------------------------- 2D quantizer */

/* x: bf16 (M, N), element (r, c) at x[r * ldx + c].
 * Rowwise: codes q_row[r * ld_qrow + c], scales s_row[r * ld_srow + c/32].
 * Colwise: codes q_col[c * ld_qcol + r] (column-major),
 *          scales s_col[(r/32) * ld_scol + c].
 * Only rows [r_begin, r_end) are processed (the colwise range must be whole
 * 32-row blocks); pass 0 and M for the whole matrix. */
void orc_quant_2d(const uint16_t *x, int64_t ldx, int64_t M, int64_t N, int mode,
                  uint8_t *q_row, int64_t ld_qrow, uint8_t *s_row, int64_t ld_srow,
                  uint8_t *q_col, int64_t ld_qcol, uint8_t *s_col, int64_t ld_scol,
                  int64_t r_begin, int64_t r_end)
{
    (void)M;
    if (mode & ORC_ROWWISE) {
        for (int64_t r = r_begin; r < r_end; r++)
            for (int64_t jb = 0; jb < N / 32; jb++)
                orc_quant_block(x + r * ldx + jb * 32, 1,
                                q_row + r * ld_qrow + jb * 32, 1,
                                s_row + r * ld_srow + jb);
    }
    if (mode & ORC_COLWISE) {
        for (int64_t rb = r_begin / 32; rb < r_end / 32; rb++)
            for (int64_t c = 0; c < N; c++)
                orc_quant_block(x + (rb * 32) * ldx + c, ldx,
                                q_col + c * ld_qcol + rb * 32, 1,
                                s_col + rb * ld_scol + c);
    }
}

/* ------------------------------------------------------- 3D quantizer */

/* x: bf16 (E, N, K) row-major, element (e, n, k) at x[(e*N + n)*K + k].
 * Blocks of 32 along N.  Codes q[e*N*K + k*N + n] (column-major per expert),
 * scales s[e*(N/32)*K + (n/32)*K + k].  Experts [e_begin, e_end). */
void orc_quant_3d_colwise(const uint16_t *x, int64_t E, int64_t N, int64_t K,
                          uint8_t *q, uint8_t *s, int64_t e_begin, int64_t e_end)
{
    (void)E;
    for (int64_t e = e_begin; e < e_end; e++)
        for (int64_t nb = 0; nb < N / 32; nb++)
            for (int64_t k = 0; k < K; k++)
                orc_quant_block(x + (e * N + nb * 32) * K + k, K,
                                q + e * N * K + k * N + nb * 32, 1,
                                s + e * (N / 32) * K + nb * K + k);
}

/* ------------------------------------------------------------- SwiGLU */

/* sigma(g) = 1 / (1 + e^-g) */
double orc_sigmoid(double g)
{
    return 1.0 / (1.0 + exp(-g));
}

/* h = silu(g) * u = (g * sigma(g)) * u, in double (before rounding). */
double orc_swiglu_h_f64(double g, double u)
{
    double s = orc_sigmoid(g);
    return g * s * u;
}

/* dgate = dh * u * sigma(g) * (1 + g * (1 - sigma(g)))   (d h / d g)
 * dup   = dh * g * sigma(g)                            (d h / d u)      */
void orc_swiglu_grads_f64(double dh, double g, double u, double *dgate, double *dup)
{
    double s = orc_sigmoid(g);
    *dgate = dh * u * s * (1.0 + g * (1.0 - s));
    *dup = dh * g * s;
}

/* ------------------------------------------------------------- GEGLU */

/* Phi(g) = P(Z <= g) for a standard normal Z = erfc(-g / sqrt 2) / 2 */
double orc_normal_cdf(double g)
{
    return 0.5 * erfc(-g * 0.70710678118654752440);
}

/* phi(g) = exp(-g^2 / 2) / sqrt(2 pi) */
double orc_normal_pdf(double g)
{
    return exp(-0.5 * g * g) * 0.39894228040143267794;
}

/* h = gelu(g) * u = (g * Phi(g)) * u */
double orc_geglu_h_f64(double g, double u)
{
    return g * orc_normal_cdf(g) * u;
}

/* dgate = dh * u * (Phi(g) + g * phi(g)), dup = dh * g * Phi(g) */
void orc_geglu_grads_f64(double dh, double g, double u, double *dgate, double *dup)
{
    double p = orc_normal_cdf(g);
    *dgate = dh * u * (p + g * orc_normal_pdf(g));
    *dup = dh * g * p;
}

/* ---------------------------------------------- gated forward / backward */

#define ORC_ACT_SILU 0
#define ORC_ACT_GELU 1

/* h (bf16) for rows [r_begin, r_end): h[r * ld_h + c], activation `act`. */
void orc_gated_fwd(int act, const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                   int64_t N, uint16_t *h, int64_t ld_h, int64_t r_begin, int64_t r_end)
{
    for (int64_t r = r_begin; r < r_end; r++)
        for (int64_t c = 0; c < N; c++) {
            double g = orc_bf16_to_double(gate[r * ld_in + c]);
            double u = orc_bf16_to_double(up[r * ld_in + c]);
            double v = act == ORC_ACT_GELU ? orc_geglu_h_f64(g, u) : orc_swiglu_h_f64(g, u);
            h[r * ld_h + c] = orc_bf16_from_double_via_fp32(v);
        }
}

/* dgate, dup (bf16) for rows [r_begin, r_end), activation `act`. */
void orc_gated_bwd(int act, const uint16_t *dh, int64_t ld_dh, const uint16_t *gate,
                   const uint16_t *up, int64_t ld_in, int64_t N,
                   uint16_t *dgate, uint16_t *dup, int64_t ld_out,
                   int64_t r_begin, int64_t r_end)
{
    for (int64_t r = r_begin; r < r_end; r++)
        for (int64_t c = 0; c < N; c++) {
            double d = orc_bf16_to_double(dh[r * ld_dh + c]);
            double g = orc_bf16_to_double(gate[r * ld_in + c]);
            double u = orc_bf16_to_double(up[r * ld_in + c]);
            double dg, du;
            if (act == ORC_ACT_GELU)
                orc_geglu_grads_f64(d, g, u, &dg, &du);
            else
                orc_swiglu_grads_f64(d, g, u, &dg, &du);
            dgate[r * ld_out + c] = orc_bf16_from_double_via_fp32(dg);
            dup[r * ld_out + c] = orc_bf16_from_double_via_fp32(du);
        }
}

/* the SwiGLU entry points of the gated forms */
void orc_swiglu_fwd(const uint16_t *gate, const uint16_t *up, int64_t ld_in,
                    int64_t N, uint16_t *h, int64_t ld_h,
                    int64_t r_begin, int64_t r_end)
{
    orc_gated_fwd(ORC_ACT_SILU, gate, up, ld_in, N, h, ld_h, r_begin, r_end);
}

void orc_swiglu_bwd(const uint16_t *dh, int64_t ld_dh, const uint16_t *gate,
                    const uint16_t *up, int64_t ld_in, int64_t N,
                    uint16_t *dgate, uint16_t *dup, int64_t ld_out,
                    int64_t r_begin, int64_t r_end)
{
    orc_gated_bwd(ORC_ACT_SILU, dh, ld_dh, gate, up, ld_in, N, dgate, dup, ld_out, r_begin, r_end);
}

/* ---------------------------------------------------------- blocked layout */

/* The scale matrix S (R rows x C columns, entry (r, c) at
 * s[r * rs + c * cs]) in the blocked layout: the matrix padded to
 * R' = 128 * ceil(R / 128) rows and C' = 4 * ceil(C / 4) columns, cut into
 * 128 x 4 tiles stored one after another row-major (512 bytes each); inside
 * a tile, entry (r, c) at byte (r % 32) * 16 + (r / 32) * 4 + c.  Padding
 * entries are 0.  `out` holds R' * C' bytes. */
void orc_scales_blocked(const uint8_t *s, int64_t R, int64_t C, int64_t rs, int64_t cs, uint8_t *out)
{
    int64_t Rp = (R + 127) / 128 * 128;
    int64_t Cp = (C + 3) / 4 * 4;
    memset(out, 0, (size_t)(Rp * Cp));
    for (int64_t r = 0; r < R; r++)
        for (int64_t c = 0; c < C; c++) {
            int64_t tile = (r / 128) * (Cp / 4) + (c / 4);
            int64_t in_tile = (r % 32) * 16 + ((r % 128) / 32) * 4 + (c % 4);
            out[tile * 512 + in_tile] = s[r * rs + c * cs];
        }
}

