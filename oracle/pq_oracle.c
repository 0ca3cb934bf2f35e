/*
 * pq_oracle.c -- plain, slow CPU oracle for the ParoQuant (PARO) W4A8
 * rotated-int4 linear layer  y = ((x * channel_scales) R^T) dequant(Q)^T.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.  It shares no code with the CUDA
 * library (w4a8_rotated_int4_gb300/csrc).
 *
 * Sources (web page titles and sections):
 *   [LOG]  "ParoQuant (PARO) W4A8 on gfx1201 -- engineering log"
 *          section "Format" (tensor layouts, nibble order 0,2,4,6,1,3,5,7,
 *          zeros not offset by one, pairs local to each 128 group,
 *          channel_scales pre-inverted), the "Inference identity" paragraph,
 *          "Design" items 1-4 (zero point as a row-sum correction, SZ table,
 *          per-group fp8 scales, fused prologue, records {i|j<<8, cos f16,
 *          sin f16}, software e4m3 encode RNE/OCP/saturating, row-sums of the
 *          decoded codes, partition select) and "Gates passed"
 *          (scale = amax * (1/448.f)).
 *   [CVT]  same page, section "2026-09-15: hardware e4m3 convert in the
 *          producers": the encoder maps a NaN to code zero and a negative
 *          zero to positive zero, saturates magnitudes at 448 and rounds to
 *          nearest even.
 *
 * Readings of points the pages leave open:
 *   R1 pairs: entries 2t and 2t+1 of a layer's 128-group form pair t, and the
 *      angle of pair t is theta[layer][64*g + t].
 *   R2 rotation: x_i' = c*x_i + s*x_j, x_j' = -s*x_i + c*x_j, layers 0..7,
 *      evaluated as separate fp32 multiplies and adds (no fused multiply-add):
 *      x_i' = fl(fl(c*x_i) + fl(s*x_j)), x_j' = fl(fl(c*x_j) - fl(s*x_i)).
 *   R3 record cos/sin: the f16 values nearest (RNE) to cos/sin of the f16
 *      angle evaluated in double precision; record bytes little-endian
 *      uint32 (i | j<<8), uint16 cos, uint16 sin.
 *   R4 scale: asg = fl32(amax * fl32(1/448)); if asg == 0 every code of the
 *      group is 0x00 and its row-sum is 0.
 *   R5 quotient: q = fl32(v / asg) (an IEEE division, not a reciprocal).
 *   R6 encode: NaN -> 0x00; clamp |q| to 448; round to nearest, ties to
 *      even, onto the e4m3 grid (subnormals m*2^-9 included); any result
 *      equal to zero is emitted as 0x00 (0x80 is never produced).
 *   R7 row-sum: rs = fl32(exact sum of the decoded codes of the group).
 *   R8 SZ: zscale = f16_RNE(fl32(sc * (zp - 8))) (the fp32 product is exact).
 *   R9 GEMM: y = sum_g asg * (sc * D - zscale * rs) with
 *      D = sum_{k in g} dec(A[k]) * (c[k] - 8), in fp64, using the f16 table
 *      values ("table-true").
 *   R16 fused producer ([LOG] "2026-09-02/03: rotation stream (fused add +
 *      RMSNorm + rotate + quant producers)": residual add + Gemma RMSNorm +
 *      channel scale + rotation + per-group quant in one pass).  Per row:
 *        s[k]  = bf16_RNE(fl32(x[k] + r[k]))          (the new residual)
 *        ss    = pairwise sum (recursive halving: P(v[0:n]) =
 *                fl32(P(v[0:n/2]) + P(v[n/2:n]))) of the 64 lane sums
 *                S[t] = sum over groups g, in order, in fp32, of
 *                fl32(s[128g+2t]^2 + s[128g+2t+1]^2)  (each square is
 *                exact in fp32)
 *        inv   = fl32(1 / fl32(sqrt(fl32(fl32(ss / K) + eps))))  (correctly
 *                rounded sqrt and division)
 *        h[k]  = bf16_RNE(fl32(fl32(s[k] * inv) * fl32(1 + gamma[k])))
 *      then the pq_rotate_quant semantics on h.  The page fixes the order of
 *      the operations (the serving engine's own: s times the reciprocal root
 *      of mean(s^2) + eps, times 1 + w) but not the reduction order or the
 *      rounding of the reciprocal root; these are the readings.
 *   R17 silu-mul producer ([LOG] "2026-09-03: rotation stream 2 (silu-mul,
 *      ...)", its first mode: silu of the gate rounded to bf16, multiplied by
 *      the up value and rounded to bf16 again, followed by the rotate_quant
 *      body).  The merged gate/up output y holds g in columns
 *      [0, I) and u in [I, 2I).  Per element:
 *        e   = exp32(-g)        (below)
 *        sg  = bf16_RNE(fl32(g / fl32(1 + e)))
 *        act = bf16_RNE(fl32(sg * u))
 *      then the pq_rotate_quant semantics on act (K = I).  exp32 is fixed
 *      here so that both implementations give the same bits: Cody-Waite
 *      reduction n = rint(x * log2(e)), r = fl(fl(x - n*LN2_HI) - n*LN2_LO)
 *      (LN2_HI = 0.693145751953125 has 13 trailing zero bits, so n*LN2_HI is
 *      exact for |n| <= 2^13), the Taylor polynomial of exp of degree 6 in
 *      Horner form with separately rounded steps, and an exact scaling by
 *      2^n (x < -103 gives 0, x > 88 gives +inf).
 *   R18 per-token activation scales ([LOG] "PER-TOKEN PREFILL (v3, BUILT)":
 *      pass A rotates into a bf16 scratch with group amaxes, pass C takes
 *      As = max_g asg, encodes and forms plain row-sums; the PTOK GEMM folds
 *      without the activation scale and applies As in the epilogue).  Per
 *      row and partition:
 *        v      = the pq_rotate_quant rotation of x * cs (fp32)
 *        xr[k]  = bf16_RNE(v[k])                      (the scratch row)
 *        asg_g  = fl32(max_{k in g} |xr[k]| * fl32(1/448));  As = max_g asg_g
 *        a[k]   = e4m3(fl32(xr[k] / As)) (R6 rules; all 0x00 when As == 0)
 *        rs_g   = fl32(exact sum of the decoded codes of group g)
 *      GEMM: y = As * sum_g (sc * D - zscale * rs_g), in fp64 as R9.
 *   R19 int5 weights ([LOG] "2026-09-10: int5 W5A8 ParoQuant": 5-bit codes,
 *      low nibbles in the int4 AWQ words, the fifth bit in [K, N/32] int32
 *      planes; (c - 16) runs -16..15, every value exact in e4m3).  Readings:
 *      bit j of plane word [r][w] is the fifth bit of column 32w + j (plain
 *      bit order; the pages give no permutation for the planes); the zero
 *      point's plane qzeros_hi is [G, N/32] (one row per group, as qzeros);
 *      c = nibble + 16 * bit, zp likewise; zscale = f16_RNE(fl32(sc *
 *      (zp - 16))) (exact product); the GEMM is R9 with
 *      D = sum_{k in g} dec(A[k]) * (c[k] - 16).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_ERR_SHAPE 2
#define ORC_ERR_PAIRS 4

/* ------------------------------------------------------------------ */
/* scalar formats                                                      */
/* ------------------------------------------------------------------ */

/* IEEE binary16 bit pattern -> double (exact). */
double orc_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0x1F)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* double -> IEEE binary16, round to nearest, ties to even, overflow -> inf. */
uint16_t orc_f16_from_double(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x))
        return 0x7E00;
    double a = fabs(x);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                 /* a in [2^(e-1), 2^e) */
    int eb = e - 1;               /* binade of a */
    if (eb < -14)
        eb = -14;                 /* the subnormal range shares the spacing 2^-24 */
    double quantum = ldexp(1.0, eb - 10);
    double n = nearbyint(a / quantum);       /* a/quantum is exact; nearbyint is RNE */
    double v = n * quantum;                  /* rounded magnitude */
    if (v > 65504.0)
        return sign | 0x7C00;
    if (v < ldexp(1.0, -14))
        return sign | (uint16_t)(v / ldexp(1.0, -24));
    frexp(v, &e);
    eb = e - 1;
    uint16_t mant = (uint16_t)(v / ldexp(1.0, eb - 10) - 1024.0);
    return sign | (uint16_t)((eb + 15) << 10) | mant;
}

/* bf16 bit pattern -> float (exact: bf16 is the top half of a binary32). */
float orc_bf16_to_float(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* OCP FP8 E4M3FN code -> value: bias 7, no infinities, 0x7F/0xFF are NaN. */
double orc_e4m3_decode(uint8_t c)
{
    int sign = c >> 7;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                  /* subnormal: m/8 * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);        /* (1 + m/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* float -> OCP FP8 E4M3FN (readings R6): NaN -> 0, saturate at 448,
 * RNE onto the e4m3 grid, zero results always +0. */
uint8_t orc_e4m3_encode(float q)
{
    if (isnan(q))
        return 0x00;
    int neg = signbit(q) ? 1 : 0;
    double a = fabs((double)q);
    if (a > 448.0)
        a = 448.0;
    if (a == 0.0)
        return 0x00;
    int e;
    frexp(a, &e);
    int eb = e - 1;
    if (eb < -6)
        eb = -6;                  /* subnormals: spacing 2^-9 below 2^-6 */
    double quantum = ldexp(1.0, eb - 3);
    double n = nearbyint(a / quantum);
    double v = n * quantum;       /* <= 448 because 448 is on the grid */
    if (v == 0.0)
        return 0x00;
    uint8_t code;
    if (v < ldexp(1.0, -6)) {
        code = (uint8_t)(v / ldexp(1.0, -9));          /* 1..7 */
    } else {
        frexp(v, &e);
        eb = e - 1;                                      /* -6..8 */
        int mant = (int)(v / ldexp(1.0, eb - 3)) - 8;  /* 0..7 */
        code = (uint8_t)(((eb + 7) << 3) | mant);
    }
    return neg ? (uint8_t)(code | 0x80) : code;
}

/* fp32 arithmetic helpers: one IEEE operation each, never contracted
 * (the file is compiled with -ffp-contract=off). */
static float f_mul(float a, float b) { return a * b; }
static float f_add(float a, float b) { return a + b; }
static float f_sub(float a, float b) { return a - b; }
static float f_div(float a, float b) { return a / b; }

/* ------------------------------------------------------------------ */
/* checkpoint format: AWQ nibble order                                 */
/* ------------------------------------------------------------------ */

/* [LOG] Format: word slot i holds column order[i] with order 0,2,4,6,1,3,5,7,
 * so column j sits in slot awq_slot[j]. */
static const int awq_slot[8] = {0, 4, 1, 5, 2, 6, 3, 7};

/* qweight int32 [K, N/8] -> codes uint8 [K, N] (0..15). */
void orc_unpack_awq(int rows, int N, const int32_t *packed, uint8_t *out)
{
    for (int r = 0; r < rows; r++)
        for (int n = 0; n < N; n++) {
            uint32_t w = (uint32_t)packed[(size_t)r * (N / 8) + n / 8];
            out[(size_t)r * N + n] = (uint8_t)((w >> (4 * awq_slot[n % 8])) & 15u);
        }
}

/* R19: fifth-bit plane int32 [rows, N/32] -> bits uint8 [rows, N] (0/1). */
void orc_unpack_plane(int rows, int N, const int32_t *plane, uint8_t *out)
{
    for (int r = 0; r < rows; r++)
        for (int n = 0; n < N; n++) {
            uint32_t w = (uint32_t)plane[(size_t)r * (N / 32) + n / 32];
            out[(size_t)r * N + n] = (uint8_t)((w >> (n % 32)) & 1u);
        }
}

/* R19: 5-bit codes [rows, N] (0..31) from the nibble words and the plane. */
void orc_codes5(int rows, int N, const int32_t *lo, const int32_t *hi, uint8_t *out)
{
    uint8_t *bit = (uint8_t *)malloc((size_t)rows * N);
    orc_unpack_awq(rows, N, lo, out);
    orc_unpack_plane(rows, N, hi, bit);
    for (size_t i = 0; i < (size_t)rows * N; i++)
        out[i] = (uint8_t)(out[i] + 16 * bit[i]);
    free(bit);
}

/* ------------------------------------------------------------------ */
/* load-time tables                                                    */
/* ------------------------------------------------------------------ */

/* Check that every (p, layer, group) row of pairs is a permutation of 0..127. */
int orc_check_pairs(int P, int K, const int16_t *pairs)
{
    int G = K / 128;
    for (int p = 0; p < P; p++)
        for (int r = 0; r < 8; r++)
            for (int g = 0; g < G; g++) {
                int seen[128] = {0};
                for (int t = 0; t < 128; t++) {
                    int v = pairs[((size_t)p * 8 + r) * K + 128 * g + t];
                    if (v < 0 || v > 127 || seen[v])
                        return ORC_ERR_PAIRS;
                    seen[v] = 1;
                }
            }
    return ORC_OK;
}

/* Rotation records [P][8][G][64] x 8 bytes (readings R1, R3). */
int orc_records(int P, int K, const int16_t *pairs, const uint16_t *theta, uint8_t *rec)
{
    if (K <= 0 || K % 128 || P < 1)
        return ORC_ERR_SHAPE;
    if (orc_check_pairs(P, K, pairs) != ORC_OK)
        return ORC_ERR_PAIRS;
    int G = K / 128;
    for (int p = 0; p < P; p++)
        for (int r = 0; r < 8; r++)
            for (int g = 0; g < G; g++)
                for (int t = 0; t < 64; t++) {
                    const int16_t *row = pairs + ((size_t)p * 8 + r) * K + 128 * g;
                    uint32_t i = (uint32_t)row[2 * t], j = (uint32_t)row[2 * t + 1];
                    double th = orc_f16_to_double(theta[((size_t)p * 8 + r) * (K / 2) + 64 * g + t]);
                    uint16_t c16 = orc_f16_from_double(cos(th));
                    uint16_t s16 = orc_f16_from_double(sin(th));
                    uint32_t ij = i | (j << 8);
                    uint8_t *o = rec + ((((size_t)p * 8 + r) * G + g) * 64 + t) * 8;
                    o[0] = ij & 0xFF; o[1] = (ij >> 8) & 0xFF; o[2] = 0; o[3] = 0;
                    o[4] = c16 & 0xFF; o[5] = c16 >> 8;
                    o[6] = s16 & 0xFF; o[7] = s16 >> 8;
                }
    return ORC_OK;
}

/* SZ table [G][N][2] f16: (sc, zscale) with zscale = f16(sc * (zp - 8)) (R8). */
void orc_sz(int G, int N, const uint16_t *scales, const int32_t *qzeros, uint16_t *sz)
{
    uint8_t *zp = (uint8_t *)malloc((size_t)G * N);
    orc_unpack_awq(G, N, qzeros, zp);
    for (int g = 0; g < G; g++)
        for (int n = 0; n < N; n++) {
            uint16_t sc = scales[(size_t)g * N + n];
            float prod = f_mul((float)orc_f16_to_double(sc), (float)(zp[(size_t)g * N + n] - 8));
            sz[((size_t)g * N + n) * 2 + 0] = sc;
            sz[((size_t)g * N + n) * 2 + 1] = orc_f16_from_double((double)prod);
        }
    free(zp);
}

/* R19: SZ table of int5 weights, zscale = f16(sc * (zp - 16)). */
void orc_sz5(int G, int N, const uint16_t *scales, const int32_t *qzeros, const int32_t *qzeros_hi,
             uint16_t *sz)
{
    uint8_t *zp = (uint8_t *)malloc((size_t)G * N);
    orc_codes5(G, N, qzeros, qzeros_hi, zp);
    for (int g = 0; g < G; g++)
        for (int n = 0; n < N; n++) {
            uint16_t sc = scales[(size_t)g * N + n];
            float prod = f_mul((float)orc_f16_to_double(sc), (float)(zp[(size_t)g * N + n] - 16));
            sz[((size_t)g * N + n) * 2 + 0] = sc;
            sz[((size_t)g * N + n) * 2 + 1] = orc_f16_from_double((double)prod);
        }
    free(zp);
}

/* Kernel weight layout w[n][K/2] (this build's choice; the pages fix only the
 * AWQ input): each run of eight codes k = 8t .. 8t+7 of row n fills the four
 * bytes 4t .. 4t+3, byte 4t + b holding code 8t + b in its low nibble and
 * code 8t + b + 4 in its high nibble. */
void orc_repack(int K, int N, const int32_t *qweight, uint8_t *w)
{
    uint8_t *c = (uint8_t *)malloc((size_t)K * N);
    orc_unpack_awq(K, N, qweight, c);
    for (int n = 0; n < N; n++)
        for (int t = 0; t < K / 8; t++)
            for (int b = 0; b < 4; b++)
                w[(size_t)n * (K / 2) + 4 * t + b] =
                    (uint8_t)(c[(size_t)(8 * t + b) * N + n] | (c[(size_t)(8 * t + b + 4) * N + n] << 4));
    free(c);
}

/* Kernel layouts of int5 weights (this build's choice): the low nibbles as
 * orc_repack, and the fifth bits whi[n][K/8] in 4-byte blocks of 32 k: for
 * k = 32t + 16h + 4q + j (h in 0..1, q and j in 0..3) the fifth bit of (k, n)
 * is bit 4h + q of byte 4t + j. */
void orc_repack5(int K, int N, const int32_t *qweight, const int32_t *qweight_hi, uint8_t *w, uint8_t *whi)
{
    orc_repack(K, N, qweight, w);
    uint8_t *bit = (uint8_t *)malloc((size_t)K * N);
    orc_unpack_plane(K, N, qweight_hi, bit);
    memset(whi, 0, (size_t)N * (K / 8));
    for (int n = 0; n < N; n++)
        for (int k = 0; k < K; k++) {
            const int t = k / 32, h = (k % 32) / 16, q = (k % 16) / 4, j = k % 4;
            whi[(size_t)n * (K / 8) + 4 * t + j] |= (uint8_t)(bit[(size_t)k * N + n] << (4 * h + q));
        }
    free(bit);
}

/* ------------------------------------------------------------------ */
/* prologue: channel scale, 8 Givens layers, per-group fp8 quantisation */
/* ------------------------------------------------------------------ */

/* Read record (p, r, g, t). */
static void rec_get(const uint8_t *rec, int G, int p, int r, int g, int t,
                    int *i, int *j, float *c, float *s)
{
    const uint8_t *o = rec + ((((size_t)p * 8 + r) * G + g) * 64 + t) * 8;
    *i = o[0];
    *j = o[1];
    *c = (float)orc_f16_to_double((uint16_t)(o[4] | (o[5] << 8)));
    *s = (float)orc_f16_to_double((uint16_t)(o[6] | (o[7] << 8)));
}

/* Rotate one 128-vector in fp32 with layers 0..7 of (p, g) (reading R2). */
void orc_rotate_group_f32(const uint8_t *rec, int G, int p, int g, float *v)
{
    for (int r = 0; r < 8; r++)
        for (int t = 0; t < 64; t++) {
            int i, j;
            float c, s;
            rec_get(rec, G, p, r, g, t, &i, &j, &c, &s);
            float vi = v[i], vj = v[j];
            v[i] = f_add(f_mul(c, vi), f_mul(s, vj));
            v[j] = f_sub(f_mul(c, vj), f_mul(s, vi));
        }
}

/* fl32(1/448): the scale constant of [LOG] "Gates passed". */
static float inv448(void)
{
    volatile float one = 1.0f, d = 448.0f;
    return f_div(one, d);
}

/*
 * pq_rotate_quant semantics.  x bf16 [M][ldx]; cs f16 [P][K]; rec from
 * orc_records.  Outputs a e4m3 [P][M][K], asg f32 [P][G][M], rs f32 [P][G][M].
 * Optional v_out f32 [P][M][K] receives the rotated, scaled activations.
 */
void orc_rotate_quant(int M, int K, int ldx, int P, const uint16_t *x, const uint16_t *cs,
                      const uint8_t *rec, uint8_t *a, float *asg, float *rs, float *v_out)
{
    int G = K / 128;
    float c448 = inv448();
#pragma omp parallel for collapse(2) schedule(static)
    for (int p = 0; p < P; p++)
        for (int m = 0; m < M; m++)
            for (int g = 0; g < G; g++) {
                float v[128];
                for (int k = 0; k < 128; k++)
                    v[k] = f_mul(orc_bf16_to_float(x[(size_t)m * ldx + 128 * g + k]),
                                 (float)orc_f16_to_double(cs[(size_t)p * K + 128 * g + k]));
                orc_rotate_group_f32(rec, G, p, g, v);
                float amax = 0.0f;
                for (int k = 0; k < 128; k++)
                    if (fabsf(v[k]) > amax)
                        amax = fabsf(v[k]);
                float scale = f_mul(amax, c448);
                int64_t sum512 = 0;             /* exact: sum of dec(code) * 2^9 */
                uint8_t *arow = a + ((size_t)p * M + m) * K + 128 * g;
                for (int k = 0; k < 128; k++) {
                    uint8_t code = 0;
                    if (scale != 0.0f)
                        code = orc_e4m3_encode(f_div(v[k], scale));
                    arow[k] = code;
                    sum512 += (int64_t)llround(orc_e4m3_decode(code) * 512.0);
                }
                asg[((size_t)p * G + g) * M + m] = scale;
                rs[((size_t)p * G + g) * M + m] = (float)((double)sum512 / 512.0);
                if (v_out)
                    memcpy(v_out + ((size_t)p * M + m) * K + 128 * g, v, sizeof v);
            }
}

/* fp32 -> bf16 bit pattern, round to nearest, ties to even (finite input). */
uint16_t orc_bf16_from_float(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    uint32_t lsb = (u >> 16) & 1u;
    return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

/* Pairwise sum of n = 2^j fp32 values (reading R16): the two halves' sums,
 * added in fp32. */
static float pairwise_f32(const float *v, int n)
{
    if (n == 1)
        return v[0];
    return f_add(pairwise_f32(v, n / 2), pairwise_f32(v + n / 2, n / 2));
}

/* Sum of squares of one bf16-valued row of K values (reading R16): lane t
 * of 64 sums its channel pair (2t, 2t+1) over the groups in order, then
 * the 64 lane sums are added pairwise. */
float orc_row_sumsq(int K, const float *s)
{
    float lane[64];
    for (int t = 0; t < 64; t++) {
        float acc = 0.0f;
        for (int g = 0; g < K / 128; g++) {
            const float a = s[128 * g + 2 * t], b = s[128 * g + 2 * t + 1];
            acc = f_add(acc, f_add(f_mul(a, a), f_mul(b, b)));
        }
        lane[t] = acc;
    }
    return pairwise_f32(lane, 64);
}

/*
 * Fused producer (reading R16).  x, res bf16 [M][ldx]; gamma bf16 [K]; the
 * rest as orc_rotate_quant.  Writes res_out bf16 [M][K] (the new residual),
 * h_out bf16 [M][K] (the normed rows) and the rotate_quant outputs of h.
 */
void orc_add_rms_rotate_quant(int M, int K, int ldx, int P, const uint16_t *x, const uint16_t *res,
                              const uint16_t *gamma, float eps, const uint16_t *cs, const uint8_t *rec,
                              uint16_t *res_out, uint16_t *h_out, uint8_t *a, float *asg, float *rs)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++) {
        float *s = (float *)malloc(sizeof(float) * (size_t)K);
        for (int k = 0; k < K; k++) {
            uint16_t sb = orc_bf16_from_float(f_add(orc_bf16_to_float(x[(size_t)m * ldx + k]),
                                                    orc_bf16_to_float(res[(size_t)m * ldx + k])));
            res_out[(size_t)m * K + k] = sb;
            s[k] = orc_bf16_to_float(sb);
        }
        float ss = orc_row_sumsq(K, s);
        float var = f_div(ss, (float)K);
        float inv = f_div(1.0f, sqrtf(f_add(var, eps)));
        for (int k = 0; k < K; k++) {
            float w1 = f_add(1.0f, orc_bf16_to_float(gamma[k]));
            h_out[(size_t)m * K + k] = orc_bf16_from_float(f_mul(f_mul(s[k], inv), w1));
        }
        free(s);
    }
    orc_rotate_quant(M, K, K, P, h_out, cs, rec, a, asg, rs, NULL);
}

/* exp(x) in fp32 by the fixed sequence of reading R17. */
float orc_exp32(float x)
{
    if (x > 88.0f)
        return INFINITY;
    if (x < -103.0f)
        return 0.0f;
    const float log2e = 1.44269502f, ln2_hi = 0.693145751953125f, ln2_lo = 1.42860677e-06f;
    const float n = rintf(f_mul(x, log2e));
    const float r = f_sub(f_sub(x, f_mul(n, ln2_hi)), f_mul(n, ln2_lo));
    /* 1 + r(1 + r(1/2 + r(1/6 + r(1/24 + r(1/120 + r/720))))) */
    float p = f_mul(r, 1.0f / 720.0f);
    p = f_mul(r, f_add(1.0f / 120.0f, p));
    p = f_mul(r, f_add(1.0f / 24.0f, p));
    p = f_mul(r, f_add(1.0f / 6.0f, p));
    p = f_mul(r, f_add(0.5f, p));
    p = f_mul(r, f_add(1.0f, p));
    p = f_add(1.0f, p);
    return ldexpf(p, (int)n);
}

/* silu(g) * u of one element as bf16 bits (reading R17). */
uint16_t orc_silu_mul(uint16_t g, uint16_t u)
{
    const float gf = orc_bf16_to_float(g);
    const float e = orc_exp32(-gf);
    const float sg = orc_bf16_to_float(orc_bf16_from_float(f_div(gf, f_add(1.0f, e))));
    return orc_bf16_from_float(f_mul(sg, orc_bf16_to_float(u)));
}

/*
 * silu-mul producer (reading R17).  y bf16 [M][ldy] with the gate in
 * columns [0, I) and up in [I, 2I); writes act_out bf16 [M][I] and the
 * rotate_quant outputs of act (K = I).
 */
void orc_silu_mul_rotate_quant(int M, int I, int ldy, int P, const uint16_t *y, const uint16_t *cs,
                               const uint8_t *rec, uint16_t *act_out, uint8_t *a, float *asg, float *rs)
{
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; m++)
        for (int k = 0; k < I; k++)
            act_out[(size_t)m * I + k] = orc_silu_mul(y[(size_t)m * ldy + k], y[(size_t)m * ldy + I + k]);
    orc_rotate_quant(M, I, I, P, act_out, cs, rec, a, asg, rs, NULL);
}

/*
 * Per-token prologue (reading R18).  Outputs: xr bf16 [P][M][K] (the scratch
 * row), a e4m3 [P][M][K], As f32 [P][M], rs f32 [P][G][M].
 */
void orc_rotate_tokquant(int M, int K, int ldx, int P, const uint16_t *x, const uint16_t *cs,
                         const uint8_t *rec, uint16_t *xr, uint8_t *a, float *As, float *rs)
{
    int G = K / 128;
    float c448 = inv448();
#pragma omp parallel for collapse(2) schedule(static)
    for (int p = 0; p < P; p++)
        for (int m = 0; m < M; m++) {
            uint16_t *xrow = xr + ((size_t)p * M + m) * K;
            float as = 0.0f;
            for (int g = 0; g < G; g++) {
                float v[128];
                for (int k = 0; k < 128; k++)
                    v[k] = f_mul(orc_bf16_to_float(x[(size_t)m * ldx + 128 * g + k]),
                                 (float)orc_f16_to_double(cs[(size_t)p * K + 128 * g + k]));
                orc_rotate_group_f32(rec, G, p, g, v);
                float amax = 0.0f;
                for (int k = 0; k < 128; k++) {
                    xrow[128 * g + k] = orc_bf16_from_float(v[k]);
                    float q = fabsf(orc_bf16_to_float(xrow[128 * g + k]));
                    if (q > amax)
                        amax = q;
                }
                float sg = f_mul(amax, c448);
                if (sg > as)
                    as = sg;
            }
            As[(size_t)p * M + m] = as;
            uint8_t *arow = a + ((size_t)p * M + m) * K;
            for (int g = 0; g < G; g++) {
                int64_t sum512 = 0;
                for (int k = 0; k < 128; k++) {
                    uint8_t code = 0;
                    if (as != 0.0f)
                        code = orc_e4m3_encode(f_div(orc_bf16_to_float(xrow[128 * g + k]), as));
                    arow[128 * g + k] = code;
                    sum512 += (int64_t)llround(orc_e4m3_decode(code) * 512.0);
                }
                rs[((size_t)p * G + g) * M + m] = (float)((double)sum512 / 512.0);
            }
        }
}

/* ------------------------------------------------------------------ */
/* GEMM in fp64                                                        */
/* ------------------------------------------------------------------ */

static int part_of(int n, int pb1, int pb2) { return (n >= pb1) + (n >= pb2); }

/* one output element, table-true (reading R9); off = 8 for int4 codes,
 * 16 for int5 (R19) */
static double gemm_elem_off(int m, int n, int M, int N, int K, int pb1, int pb2,
                            const uint8_t *a, const float *asg, const float *rs,
                            const uint8_t *codes, const uint16_t *sz, int off)
{
    int G = K / 128;
    int p = part_of(n, pb1, pb2);
    const uint8_t *arow = a + ((size_t)p * M + m) * K;
    double y = 0.0;
    for (int g = 0; g < G; g++) {
        double D = 0.0;             /* exact: products and sums are multiples of 2^-9 below 2^53 */
        for (int k = 128 * g; k < 128 * g + 128; k++)
            D += orc_e4m3_decode(arow[k]) * (double)((int)codes[(size_t)k * N + n] - off);
        double sc = orc_f16_to_double(sz[((size_t)g * N + n) * 2 + 0]);
        double zs = orc_f16_to_double(sz[((size_t)g * N + n) * 2 + 1]);
        double s = asg[((size_t)p * G + g) * M + m];
        double r = rs[((size_t)p * G + g) * M + m];
        y += s * (sc * D - zs * r);
    }
    return y;
}

static double gemm_elem(int m, int n, int M, int N, int K, int pb1, int pb2,
                        const uint8_t *a, const float *asg, const float *rs,
                        const uint8_t *codes, const uint16_t *sz)
{
    return gemm_elem_off(m, n, M, N, K, pb1, pb2, a, asg, rs, codes, sz, 8);
}

/* R19: the GEMM of int5 codes (0..31) with their SZ table, full and sampled. */
void orc_gemm5_f64(int M, int N, int K, int pb1, int pb2, const uint8_t *a, const float *asg,
                   const float *rs, const uint8_t *codes, const uint16_t *sz, double *y)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++)
            y[(size_t)m * N + n] = gemm_elem_off(m, n, M, N, K, pb1, pb2, a, asg, rs, codes, sz, 16);
}

void orc_gemm5_f64_sampled(int count, const int *ms, const int *ns, int M, int N, int K,
                           int pb1, int pb2, const uint8_t *a, const float *asg, const float *rs,
                           const uint8_t *codes, const uint16_t *sz, double *y)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < count; i++)
        y[i] = gemm_elem_off(ms[i], ns[i], M, N, K, pb1, pb2, a, asg, rs, codes, sz, 16);
}

/*
 * Full GEMM: a e4m3 [P][M][K], asg/rs f32 [P][G][M], codes uint8 [K][N]
 * (unpacked qweight), sz [G][N][2] -> y f64 [M][N].
 */
void orc_gemm_f64(int M, int N, int K, int pb1, int pb2, const uint8_t *a, const float *asg,
                  const float *rs, const uint8_t *codes, const uint16_t *sz, double *y)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++)
            y[(size_t)m * N + n] = gemm_elem(m, n, M, N, K, pb1, pb2, a, asg, rs, codes, sz);
}

/* Sampled GEMM: y[i] = element (ms[i], ns[i]). */
/* PTOK GEMM (reading R18): y[m][n] = As[p][m] * sum_g (sc * D - zscale * rs),
 * fp64, table-true as R9.  As f32 [P][M]. */
void orc_gemm_ptok_f64(int M, int N, int K, int pb1, int pb2, const uint8_t *a, const float *As,
                       const float *rs, const uint8_t *codes, const uint16_t *sz, double *y)
{
    int G = K / 128, P = 1 + (pb1 < N) + (pb2 < N);
#pragma omp parallel for collapse(2) schedule(static)
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
            int p = part_of(n, pb1, pb2);
            const uint8_t *arow = a + ((size_t)p * M + m) * K;
            double acc = 0.0;
            for (int g = 0; g < G; g++) {
                double D = 0.0;
                for (int k = 128 * g; k < 128 * (g + 1); k++)
                    D += orc_e4m3_decode(arow[k]) * ((double)codes[(size_t)k * N + n] - 8.0);
                double sc = orc_f16_to_double(sz[((size_t)g * N + n) * 2]);
                double zs = orc_f16_to_double(sz[((size_t)g * N + n) * 2 + 1]);
                acc += sc * D - zs * (double)rs[((size_t)p * G + g) * M + m];
            }
            y[(size_t)m * N + n] = (double)As[(size_t)p * M + m] * acc;
        }
    (void)P;
}

/* the PTOK GEMM at sampled (m, n) pairs */
void orc_gemm_ptok_f64_sampled(int count, const int *ms, const int *ns, int M, int N, int K, int pb1, int pb2,
                               const uint8_t *a, const float *As, const float *rs, const uint8_t *codes,
                               const uint16_t *sz, double *y)
{
    int G = K / 128;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < count; i++) {
        int m = ms[i], n = ns[i], p = part_of(n, pb1, pb2);
        const uint8_t *arow = a + ((size_t)p * M + m) * K;
        double acc = 0.0;
        for (int g = 0; g < G; g++) {
            double D = 0.0;
            for (int k = 128 * g; k < 128 * (g + 1); k++)
                D += orc_e4m3_decode(arow[k]) * ((double)codes[(size_t)k * N + n] - 8.0);
            double sc = orc_f16_to_double(sz[((size_t)g * N + n) * 2]);
            double zs = orc_f16_to_double(sz[((size_t)g * N + n) * 2 + 1]);
            acc += sc * D - zs * (double)rs[((size_t)p * G + g) * M + m];
        }
        y[i] = (double)As[(size_t)p * M + m] * acc;
    }
}

void orc_gemm_f64_sampled(int count, const int *ms, const int *ns, int M, int N, int K,
                          int pb1, int pb2, const uint8_t *a, const float *asg, const float *rs,
                          const uint8_t *codes, const uint16_t *sz, double *y)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < count; i++)
        y[i] = gemm_elem(ms[i], ns[i], M, N, K, pb1, pb2, a, asg, rs, codes, sz);
}

/* "Format-true" diagnostic: sum_k dec(a)*asg * (c - zp)*sc, zero point exact. */
void orc_gemm_format_f64(int M, int N, int K, int pb1, int pb2, const uint8_t *a,
                         const float *asg, const uint8_t *codes, const uint8_t *zp,
                         const uint16_t *scales, double *y)
{
    int G = K / 128;
#pragma omp parallel for schedule(dynamic, 1)
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
            int p = part_of(n, pb1, pb2);
            double acc = 0.0;
            for (int k = 0; k < K; k++) {
                int g = k / 128;
                double av = orc_e4m3_decode(a[((size_t)p * M + m) * K + k]) *
                            (double)asg[((size_t)p * G + g) * M + m];
                double wv = (double)((int)codes[(size_t)k * N + n] - (int)zp[(size_t)g * N + n]) *
                            orc_f16_to_double(scales[(size_t)g * N + n]);
                acc += av * wv;
            }
            y[(size_t)m * N + n] = acc;
        }
}

/* ------------------------------------------------------------------ */
/* fp64 references for the inference identity (no quantisation)       */
/* ------------------------------------------------------------------ */

/* Apply the layers of (p, g) in fp64 to a 128-vector with exact cos/sin of
 * the f16 angles; forward = layers 0..7, transpose = layers 7..0 with the
 * angle negated. */
static void rotate_group_f64(int K, int p, int g, const int16_t *pairs, const uint16_t *theta,
                             double *v, int transpose)
{
    for (int rr = 0; rr < 8; rr++) {
        int r = transpose ? 7 - rr : rr;
        for (int t = 0; t < 64; t++) {
            const int16_t *row = pairs + ((size_t)p * 8 + r) * K + 128 * g;
            int i = row[2 * t], j = row[2 * t + 1];
            double th = orc_f16_to_double(theta[((size_t)p * 8 + r) * (K / 2) + 64 * g + t]);
            if (transpose)
                th = -th;
            double c = cos(th), s = sin(th);
            double vi = v[i], vj = v[j];
            v[i] = c * vi + s * vj;
            v[j] = c * vj - s * vi;
        }
    }
}

/* y = ((x*cs) R^T) W^T with the rotation applied to the activations.
 * W is the dequantised weight f64 [N][K]; x bf16 [M][K]. */
void orc_linear_rotx_f64(int M, int K, int N, int P, int pb1, int pb2, const uint16_t *x,
                         const uint16_t *cs, const int16_t *pairs, const uint16_t *theta,
                         const double *W, double *y)
{
    int G = K / 128;
    double *v = (double *)malloc(sizeof(double) * (size_t)P * K);
    for (int m = 0; m < M; m++) {
        for (int p = 0; p < P; p++)
            for (int g = 0; g < G; g++) {
                double *vg = v + (size_t)p * K + 128 * g;
                for (int k = 0; k < 128; k++)
                    vg[k] = (double)orc_bf16_to_float(x[(size_t)m * K + 128 * g + k]) *
                            orc_f16_to_double(cs[(size_t)p * K + 128 * g + k]);
                rotate_group_f64(K, p, g, pairs, theta, vg, 0);
            }
        for (int n = 0; n < N; n++) {
            const double *vp = v + (size_t)part_of(n, pb1, pb2) * K;
            double acc = 0.0;
            for (int k = 0; k < K; k++)
                acc += vp[k] * W[(size_t)n * K + k];
            y[(size_t)m * N + n] = acc;
        }
    }
    free(v);
}

/* Same y with R^T moved onto the weights: each weight row is rotated by the
 * transposed layers, and the activations are only channel-scaled. */
void orc_linear_rotw_f64(int M, int K, int N, int P, int pb1, int pb2, const uint16_t *x,
                         const uint16_t *cs, const int16_t *pairs, const uint16_t *theta,
                         const double *W, double *y)
{
    (void)P;                      /* the partition of each row comes from pb1/pb2 */
    int G = K / 128;
    double *Wr = (double *)malloc(sizeof(double) * (size_t)N * K);
    memcpy(Wr, W, sizeof(double) * (size_t)N * K);
    for (int n = 0; n < N; n++)
        for (int g = 0; g < G; g++)
            rotate_group_f64(K, part_of(n, pb1, pb2), g, pairs, theta, Wr + (size_t)n * K + 128 * g, 1);
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
            int p = part_of(n, pb1, pb2);
            double acc = 0.0;
            for (int k = 0; k < K; k++)
                acc += (double)orc_bf16_to_float(x[(size_t)m * K + k]) *
                       orc_f16_to_double(cs[(size_t)p * K + k]) * Wr[(size_t)n * K + k];
            y[(size_t)m * N + n] = acc;
        }
    free(Wr);
}

/* ------------------------------------------------------------------ */
/* self-check: the encoder against nearest-value search on all 2^32    */
/* ------------------------------------------------------------------ */

/*
 * For every binary32 bit pattern compare orc_e4m3_encode with the code found
 * by searching the decoded table of the 127 non-negative finite values for the
 * nearest one (ties to the even code, |q| saturated at 448, NaN -> 0, zero
 * results as 0x00).  lo/hi bound the patterns (hi exclusive, up to 2^32).
 * Returns the number of disagreements; *first_bad receives the first one.
 */
long long orc_e4m3_check_range(uint64_t lo, uint64_t hi, uint32_t *first_bad)
{
    double tab[127];
    for (int c = 0; c < 127; c++)
        tab[c] = orc_e4m3_decode((uint8_t)c);      /* increasing in c */
    long long bad = 0;
    unsigned long long first = ~0ull;
#pragma omp parallel for schedule(static) reduction(+ : bad) reduction(min : first)
    for (long long u = (long long)lo; u < (long long)hi; u++) {
        uint32_t bits = (uint32_t)u;
        float q;
        memcpy(&q, &bits, 4);
        uint8_t want;
        if (isnan(q)) {
            want = 0;
        } else {
            double a = fabs((double)q);
            if (a > 448.0)
                a = 448.0;
            int lo_i = 0, hi_i = 126;                 /* tab[lo_i] <= a <= tab[hi_i] */
            while (hi_i - lo_i > 1) {
                int mid = (lo_i + hi_i) / 2;
                if (tab[mid] <= a)
                    lo_i = mid;
                else
                    hi_i = mid;
            }
            double dl = a - tab[lo_i], dh = tab[hi_i] - a;
            int c;
            if (dl < dh)
                c = lo_i;
            else if (dh < dl)
                c = hi_i;
            else
                c = (lo_i % 2 == 0) ? lo_i : hi_i;   /* tie: the code with an even mantissa */
            want = (uint8_t)c;
            if (c != 0 && signbit(q))
                want |= 0x80;
        }
        if (orc_e4m3_encode(q) != want) {
            bad++;
            if ((unsigned long long)bits < first)
                first = bits;
        }
    }
    if (first_bad)
        *first_bad = (uint32_t)first;
    return bad;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* Encode the binary32 patterns [lo, hi) (as floats) into out[0 .. hi-lo). */
void orc_e4m3_encode_range(uint64_t lo, uint64_t hi, uint8_t *out)
{
#pragma omp parallel for schedule(static)
    for (long long u = (long long)lo; u < (long long)hi; u++) {
        uint32_t bits = (uint32_t)u;
        float q;
        memcpy(&q, &bits, 4);
        out[u - (long long)lo] = orc_e4m3_encode(q);
    }
}
