/*
 * CPU oracle for the MoE grouped matmul (GMM) with blockwise FP8 quantization.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant generator
 * with the CUDA library: every definition below is written out again here.
 *
 * It is deliberately plain and slow: straight loops, fp64 sums, no blocking,
 * no reordering beyond what each definition states.  Quantization follows the
 * precision the method fixes (fp32 scale arithmetic, e4m3 codes); every GEMM
 * sums in fp64 and rounds once at the end.
 *
 * Sources (page title, section):
 *  [Q1..Q9]  "GEMM Kernel 性能优化十问" (pengchengneo.github.io), questions 1-9.
 *  [V2 3.3]  "实现差距：GMM Kernel（V1 vs V2）", §3.3 动态 LHS 量化.
 *  [V2 3.4]  same page, §3.4 Sub-byte 类型支持 (int4 / float4_e2m1fn weights,
 *            the blockwise fp32-scale arithmetic otherwise unchanged).
 *  [V2 3.5]  same page, §3.5 激活函数融合 (fused gate/up activation).
 *  [V2 3.6]  same page, §3.6 异步 DMA 置零 (zeroing the uncovered output).
 *  [MoE 1]   "MoE 优化的探索", §1 (SwiGLU expert: z = SiLU(g) * u).
 *  [MoE 3.7.2] same page, §3.7.2 (a grouped GEMM is one independent GEMM per
 *            expert over that expert's contiguous rows; ragged tails allowed).
 *
 * Parity pins: every function here is pinned by the "not gpu" tests in
 * tests/test_oracle_*.py against closed forms, library routines, brute force
 * and invariants.  The fp32 SQNR figures that the oracle reports are not
 * pinned by any printed value (the pages print none): parity unpinned for
 * the absolute SQNR numbers only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_NEGATIVE_GROUP 1
#define OR_ERR_GROUPS_EXCEED_M 2
#define OR_ERR_SHAPE 3

/* ------------------------------------------------------------------------ */
/* bf16 and fp32 helpers                                                     */
/* ------------------------------------------------------------------------ */

/* bf16 is the top half of an IEEE binary32: widening is exact. */
static float bf16_bits_to_float(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Round a binary32 to bf16, round-to-nearest, ties to even.  The 16 bits that
 * are dropped are compared with one half unit of the kept last place. */
static uint16_t float_to_bf16_bits(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u) /* NaN: keep it a (quiet) NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t hi = u >> 16;
    uint32_t lo = u & 0xffffu;
    if (lo > 0x8000u || (lo == 0x8000u && (hi & 1u)))
        hi += 1u; /* a carry into the exponent is the correct result */
    return (uint16_t)hi;
}

/* fp64 -> fp32 (the C cast rounds to nearest even) -> bf16. */
uint16_t oracle_round_to_bf16(double v)
{
    return float_to_bf16_bits((float)v);
}

void oracle_round_to_bf16_array(const double *v, int64_t n, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_round_to_bf16(v[i]);
}

void oracle_bf16_to_double_array(const uint16_t *b, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (double)bf16_bits_to_float(b[i]);
}

/* ------------------------------------------------------------------------ */
/* FP8 E4M3 ("e4m3fn") codec, from the format definition                    */
/*   1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinities;   */
/*   exponent 15 with mantissa 7 is NaN; largest finite 448; exponent 0 is   */
/*   subnormal, value m/8 * 2^-6.                                             */
/* The method casts x * (1/scale) to e4m3 [V2 3.3]; the rounding of that cast */
/* is read as round-to-nearest, ties to even, saturating to +-448.            */
/* ------------------------------------------------------------------------ */

double oracle_e4m3_decode(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ((double)m / 8.0) * ldexp(1.0, -6);
    else
        mag = (1.0 + (double)m / 8.0) * ldexp(1.0, e - 7);
    return sign ? -mag : mag;
}

/* Encode by brute force over the 127 non-negative finite codes: pick the
 * nearest value; on an exact tie pick the code whose last bit is 0 (adjacent
 * codes differ by one, so this is "ties to even" across exponent steps too).
 * Magnitudes above 448 saturate to 448.  table[c] = decode(c) for c < 127. */
static void e4m3_table(double *table)
{
    for (int c = 0; c <= 0x7e; ++c)
        table[c] = oracle_e4m3_decode((uint8_t)c);
}

static uint8_t e4m3_encode_with(const double *table, float v)
{
    if (v != v)
        return 0x7f;
    uint8_t sign = (signbit(v) ? 0x80 : 0x00);
    double a = fabs((double)v);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7e);
    int best = 0;
    double best_err = a; /* distance to code 0 (value 0) */
    for (int c = 1; c <= 0x7e; ++c) {
        double err = fabs(table[c] - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

uint8_t oracle_e4m3_encode(float v)
{
    double table[127];
    e4m3_table(table);
    return e4m3_encode_with(table, v);
}

void oracle_e4m3_encode_array(const float *v, int64_t n, uint8_t *out)
{
    double table[127];
    e4m3_table(table);
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_encode_with(table, v[i]);
}

void oracle_e4m3_decode_array(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e4m3_decode(c[i]);
}

/* ------------------------------------------------------------------------ */
/* Blockwise quantization                                                   */
/* [Q2]: activations (LHS) get one scale per row per 128 elements (1x128    */
/* blocks), weights (RHS) one scale per 128x128 block.                      */
/* [V2 3.3]: per block, absmax = max|x|; scale = absmax / dtype_max;        */
/* inv = 0 where scale == 0 else 1/scale; q = cast_e4m3(x * inv).           */
/* dtype_max is the largest finite e4m3 value, 448.  The scale arithmetic is */
/* read as IEEE binary32 (the scale is stored as fp32).                      */
/* ------------------------------------------------------------------------ */

static void quantize_block_scale(float absmax, float dtype_max, float *scale, float *inv)
{
    volatile float s = absmax / dtype_max; /* volatile: keep it one fp32 divide */
    *scale = s;
    *inv = (s == 0.0f) ? 0.0f : 1.0f / s;
}

/* X: bf16 [M][K] row-major.  xq: e4m3 codes [M][K].  xs: fp32 [M][K/128]. */
int oracle_quantize_lhs(const uint16_t *x, int64_t M, int64_t K, uint8_t *xq, float *xs)
{
    if (M < 0 || K <= 0 || K % 128 != 0)
        return OR_ERR_SHAPE;
    int64_t KB = K / 128;
    double table[127];
    e4m3_table(table);
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            const uint16_t *blk = x + m * K + kb * 128;
            float absmax = 0.0f;
            for (int j = 0; j < 128; ++j) {
                float a = fabsf(bf16_bits_to_float(blk[j]));
                if (a > absmax)
                    absmax = a;
            }
            float s, inv;
            quantize_block_scale(absmax, 448.0f, &s, &inv);
            xs[m * KB + kb] = s;
            for (int j = 0; j < 128; ++j) {
                volatile float prod = bf16_bits_to_float(blk[j]) * inv;
                xq[m * K + kb * 128 + j] = e4m3_encode_with(table, prod);
            }
        }
    }
    return OR_OK;
}

/* W: bf16 [G][K][N] row-major.  wq: e4m3 codes [G][K][N] (same layout).
 * ws: fp32 [G][K/128][N/128]. */
int oracle_quantize_rhs(const uint16_t *w, int64_t G, int64_t K, int64_t N, uint8_t *wq, float *ws)
{
    if (G <= 0 || K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0)
        return OR_ERR_SHAPE;
    int64_t KB = K / 128, NB = N / 128;
    double table[127];
    e4m3_table(table);
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            for (int64_t nb = 0; nb < NB; ++nb) {
                float absmax = 0.0f;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                    for (int64_t n = nb * 128; n < nb * 128 + 128; ++n) {
                        float a = fabsf(bf16_bits_to_float(w[(g * K + k) * N + n]));
                        if (a > absmax)
                            absmax = a;
                    }
                float s, inv;
                quantize_block_scale(absmax, 448.0f, &s, &inv);
                ws[(g * KB + kb) * NB + nb] = s;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                    for (int64_t n = nb * 128; n < nb * 128 + 128; ++n) {
                        volatile float prod = bf16_bits_to_float(w[(g * K + k) * N + n]) * inv;
                        wq[(g * K + k) * N + n] = e4m3_encode_with(table, prod);
                    }
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* FP4 E2M1 codec, from the format definition (OCP MX FP4): 1 sign bit, 2   */
/* exponent bits (bias 1), 1 mantissa bit; no infinities and no NaN; the     */
/* largest magnitude is 6; exponent field 0 is subnormal, value m/2.  A code */
/* is the low 4 bits of a byte.  [V2 3.4] names float4_e2m1fn as a weight   */
/* type; the cast is read as round-to-nearest, ties to even, saturating at 6.*/
/* ------------------------------------------------------------------------ */

double oracle_e2m1_decode(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double mag = (e == 0) ? 0.5 * (double)m : (1.0 + 0.5 * (double)m) * ldexp(1.0, e - 1);
    return sign ? -mag : mag;
}

/* nearest of the 8 magnitudes; an exact tie goes to the even code */
static uint8_t e2m1_encode_value(float v)
{
    uint8_t sign = (signbit(v) ? 0x8 : 0x0);
    double a = fabs((double)v);
    if (a >= 6.0)
        return (uint8_t)(sign | 0x7);
    int best = 0;
    double best_err = a;
    for (int c = 1; c <= 7; ++c) {
        double err = fabs(oracle_e2m1_decode((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

uint8_t oracle_e2m1_encode(float v)
{
    return e2m1_encode_value(v);
}

void oracle_e2m1_encode_array(const float *v, int64_t n, uint8_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = e2m1_encode_value(v[i]);
}

void oracle_e2m1_decode_array(const uint8_t *c, int64_t n, double *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_e2m1_decode(c[i]);
}

/* 4-bit weights [V2 3.4]: the 128x128 block rule of [Q2] with the 4-bit
 * type's largest value as dtype_max: scale = absmax / 6, inv = 0 where scale
 * == 0 else 1/scale, code = e2m1(w * inv).  wq: one code per byte, [G][K][N]
 * (the natural layout, like oracle_quantize_rhs); ws: fp32 [G][K/128][N/128]. */
int oracle_quantize_rhs_e2m1(const uint16_t *w, int64_t G, int64_t K, int64_t N, uint8_t *wq, float *ws)
{
    if (G <= 0 || K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0)
        return OR_ERR_SHAPE;
    int64_t KB = K / 128, NB = N / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t kb = 0; kb < KB; ++kb) {
            for (int64_t nb = 0; nb < NB; ++nb) {
                float absmax = 0.0f;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                    for (int64_t n = nb * 128; n < nb * 128 + 128; ++n) {
                        float a = fabsf(bf16_bits_to_float(w[(g * K + k) * N + n]));
                        if (a > absmax)
                            absmax = a;
                    }
                float s, inv;
                quantize_block_scale(absmax, 6.0f, &s, &inv);
                ws[(g * KB + kb) * NB + nb] = s;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k)
                    for (int64_t n = nb * 128; n < nb * 128 + 128; ++n) {
                        volatile float prod = bf16_bits_to_float(w[(g * K + k) * N + n]) * inv;
                        wq[(g * K + k) * N + n] = e2m1_encode_value(prod);
                    }
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* Group metadata                                                            */
/* [MoE 3.7.2], [Q6]: rows are sorted by expert into G contiguous groups;    */
/* group g owns rows [off_g, off_g + n_g) with off the exclusive prefix sum  */
/* of group_sizes.  A group that does not fill whole row tiles ends in a     */
/* partial tile.  Rows from S = sum(n_g) to M belong to no group.            */
/* ------------------------------------------------------------------------ */

/* offsets: int32 [G+1].  Returns a status; on error offsets are not used. */
int oracle_group_offsets(const int32_t *sizes, int64_t G, int64_t M, int64_t *offsets)
{
    offsets[0] = 0;
    for (int64_t g = 0; g < G; ++g) {
        if (sizes[g] < 0)
            return OR_ERR_NEGATIVE_GROUP;
        offsets[g + 1] = offsets[g] + sizes[g];
    }
    if (offsets[G] > M)
        return OR_ERR_GROUPS_EXCEED_M;
    return OR_OK;
}

/* Tile list: for each group, in order, consecutive tiles of at most bm rows:
 * (g, row0, row1).  tiles must hold ceil(M/bm) + G entries of 3 int64. */
int oracle_group_tiles(const int32_t *sizes, int64_t G, int64_t M, int64_t bm,
                       int64_t *offsets, int64_t *tiles, int64_t *ntiles)
{
    int st = oracle_group_offsets(sizes, G, M, offsets);
    *ntiles = 0;
    if (st != OR_OK)
        return st;
    int64_t t = 0;
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t r = offsets[g]; r < offsets[g + 1]; r += bm) {
            int64_t r1 = r + bm < offsets[g + 1] ? r + bm : offsets[g + 1];
            tiles[3 * t + 0] = g;
            tiles[3 * t + 1] = r;
            tiles[3 * t + 2] = r1;
            ++t;
        }
    }
    *ntiles = t;
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* SiLU, [MoE 1]: SiLU(v) = v * sigmoid(v) = v / (1 + exp(-v)).             */
/* ------------------------------------------------------------------------ */
double oracle_silu(double v)
{
    return v / (1.0 + exp(-v));
}

/* ------------------------------------------------------------------------ */
/* FP8 blockwise GMM forward                                                 */
/* [Q1],[Q3]: for every 128-wide K block ("subchannel") the exact partial     */
/* product is formed and then rescaled by the LHS row scale and the RHS     */
/* block scale, and added to the accumulator:                                 */
/*   y[m,n] = sum_kb ( sum_{k in kb} dec(xq[m,k]) * dec(wq[g][k,n]) )         */
/*                   * xs[m,kb] * ws[g][kb][n/128]                            */
/* with g the group of row m.  [V2 3.3] applies the two scales one after the  */
/* other (partial *= lhs_scale; partial *= rhs_scale); here the same product  */
/* is formed in fp64.  Rows m >= S stay 0 [V2 3.6].                           */
/* Fused activation [V2 3.5]: W has 2N columns, gate = [0,N), up = [N,2N),    */
/* output h[m,n] = SiLU(y_gate[m,n]) * y_up[m,n].                             */
/*                                                                            */
/* xq: e4m3 [M][K]; xs: fp32 [M][K/128]; wq: e4m3 [G][K][Nw]; ws: fp32        */
/* [G][K/128][Nw/128] with Nw = N (or 2N fused); out: fp64 [M][N].            */
/* ------------------------------------------------------------------------ */

static int64_t group_of_row(const int64_t *offsets, int64_t G, int64_t m)
{
    for (int64_t g = 0; g < G; ++g)
        if (m >= offsets[g] && m < offsets[g + 1])
            return g;
    return -1;
}

/* wdec: the value of every weight code byte (e4m3, or e2m1 for 4-bit
 * weights); the activation codes are e4m3. */
static int gmm_blockwise(const uint8_t *xq, const float *xs, const uint8_t *wq, const float *ws,
                         const int32_t *sizes, int64_t G, int64_t M, int64_t K, int64_t N, int fuse,
                         const double *wdec, double *out)
{
    if (G <= 0 || M < 0 || K <= 0 || N <= 0 || K % 128 != 0 || N % 128 != 0)
        return OR_ERR_SHAPE;
    int64_t *offsets = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    int st = oracle_group_offsets(sizes, G, M, offsets);
    if (st != OR_OK) {
        free(offsets);
        return st;
    }
    int64_t Nw = fuse ? 2 * N : N;
    int64_t KB = K / 128, NBw = Nw / 128;
    double dec[256];
    for (int c = 0; c < 256; ++c)
        dec[c] = oracle_e4m3_decode((uint8_t)c);

#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)Nw);
        double *part = (double *)malloc(sizeof(double) * (size_t)Nw);
#pragma omp for schedule(dynamic, 4)
        for (int64_t m = 0; m < M; ++m) {
            int64_t g = group_of_row(offsets, G, m);
            if (g < 0) {
                for (int64_t n = 0; n < N; ++n)
                    out[m * N + n] = 0.0;
                continue;
            }
            for (int64_t n = 0; n < Nw; ++n)
                acc[n] = 0.0;
            for (int64_t kb = 0; kb < KB; ++kb) {
                for (int64_t n = 0; n < Nw; ++n)
                    part[n] = 0.0;
                for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) {
                    double a = dec[xq[m * K + k]];
                    const uint8_t *wrow = wq + (g * K + k) * Nw;
                    for (int64_t n = 0; n < Nw; ++n)
                        part[n] += a * wdec[wrow[n]];
                }
                double sx = (double)xs[m * KB + kb];
                for (int64_t n = 0; n < Nw; ++n) {
                    double sw = (double)ws[(g * KB + kb) * NBw + n / 128];
                    acc[n] += part[n] * sx * sw;
                }
            }
            for (int64_t n = 0; n < N; ++n)
                out[m * N + n] = fuse ? oracle_silu(acc[n]) * acc[N + n] : acc[n];
        }
        free(acc);
        free(part);
    }
    free(offsets);
    return OR_OK;
}

int oracle_gmm_fp8(const uint8_t *xq, const float *xs, const uint8_t *wq, const float *ws,
                   const int32_t *sizes, int64_t G, int64_t M, int64_t K, int64_t N, int fuse,
                   double *out)
{
    double wdec[256];
    for (int c = 0; c < 256; ++c)
        wdec[c] = oracle_e4m3_decode((uint8_t)c);
    return gmm_blockwise(xq, xs, wq, ws, sizes, G, M, K, N, fuse, wdec, out);
}

/* 4-bit weights [V2 3.4]: the same forward with e2m1 weight codes (one code
 * per byte, [G][K][Nw]) and their 128x128 fp32 scales; the activations stay
 * e4m3 in 1x128 blocks. */
int oracle_gmm_fp8_w4(const uint8_t *xq, const float *xs, const uint8_t *wq, const float *ws,
                      const int32_t *sizes, int64_t G, int64_t M, int64_t K, int64_t N, int fuse,
                      double *out)
{
    double wdec[256];
    for (int c = 0; c < 256; ++c)
        wdec[c] = (c < 16) ? oracle_e2m1_decode((uint8_t)c) : NAN;
    return gmm_blockwise(xq, xs, wq, ws, sizes, G, M, K, N, fuse, wdec, out);
}

/* ------------------------------------------------------------------------ */
/* bf16 GMM forward (the unquantized baseline, [Q7],[Q10] step 4), in fp64:  */
/*   y[m,n] = sum_k x[m,k] * w[g][k,n]   (fused: SiLU(gate) * up as above)   */
/* x: bf16 [M][K]; w: bf16 [G][K][Nw]; out: fp64 [M][N].                     */
/* ------------------------------------------------------------------------ */
int oracle_gmm_bf16(const uint16_t *x, const uint16_t *w, const int32_t *sizes, int64_t G,
                    int64_t M, int64_t K, int64_t N, int fuse, double *out)
{
    if (G <= 0 || M < 0 || K <= 0 || N <= 0)
        return OR_ERR_SHAPE;
    int64_t *offsets = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    int st = oracle_group_offsets(sizes, G, M, offsets);
    if (st != OR_OK) {
        free(offsets);
        return st;
    }
    int64_t Nw = fuse ? 2 * N : N;
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)Nw);
#pragma omp for schedule(dynamic, 4)
        for (int64_t m = 0; m < M; ++m) {
            int64_t g = group_of_row(offsets, G, m);
            if (g < 0) {
                for (int64_t n = 0; n < N; ++n)
                    out[m * N + n] = 0.0;
                continue;
            }
            for (int64_t n = 0; n < Nw; ++n)
                acc[n] = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double a = (double)bf16_bits_to_float(x[m * K + k]);
                const uint16_t *wrow = w + (g * K + k) * Nw;
                for (int64_t n = 0; n < Nw; ++n)
                    acc[n] += a * (double)bf16_bits_to_float(wrow[n]);
            }
            for (int64_t n = 0; n < N; ++n)
                out[m * N + n] = fuse ? oracle_silu(acc[n]) * acc[N + n] : acc[n];
        }
        free(acc);
    }
    free(offsets);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* tgmm, the weight gradient ([Q4]: dW[K,N] += X^T[K,M] x dY[M,N], reduced   */
/* over M; [Q5]: the backward pass stays in bf16, unquantized), per group:   */
/*   dw[g][k,n] = sum_{m in group g} x[m,k] * dy[m,n]                         */
/* An empty group has dw[g] = 0.  x: bf16 [M][K]; dy: bf16 [M][N];            */
/* dw: fp64 [G][K][N].                                                        */
/* ------------------------------------------------------------------------ */
int oracle_tgmm_bf16(const uint16_t *x, const uint16_t *dy, const int32_t *sizes, int64_t G,
                     int64_t M, int64_t K, int64_t N, double *dw)
{
    if (G <= 0 || M < 0 || K <= 0 || N <= 0)
        return OR_ERR_SHAPE;
    int64_t *offsets = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    int st = oracle_group_offsets(sizes, G, M, offsets);
    if (st != OR_OK) {
        free(offsets);
        return st;
    }
#pragma omp parallel for collapse(2) schedule(dynamic, 8)
    for (int64_t g = 0; g < G; ++g) {
        for (int64_t k = 0; k < K; ++k) {
            double *row = dw + (g * K + k) * N;
            for (int64_t n = 0; n < N; ++n)
                row[n] = 0.0;
            for (int64_t m = offsets[g]; m < offsets[g + 1]; ++m) {
                double a = (double)bf16_bits_to_float(x[m * K + k]);
                const uint16_t *dyrow = dy + m * N;
                for (int64_t n = 0; n < N; ++n)
                    row[n] += a * (double)bf16_bits_to_float(dyrow[n]);
            }
        }
    }
    free(offsets);
    return OR_OK;
}

/* ------------------------------------------------------------------------ */
/* bf16 dgrad, the activation gradient of the expert GEMM (the "bwd" phase   */
/* of [Q4], kept in bf16 as [Q5] prescribes for the backward pass):           */
/*   dx[m,k] = sum_n dy[m,n] * w[g][k,n]      for m in group g                */
/* rows m >= S are 0.  dy: bf16 [M][N]; w: bf16 [G][K][N]; dx: fp64 [M][K].   */
/* ------------------------------------------------------------------------ */
int oracle_dgrad_bf16(const uint16_t *dy, const uint16_t *w, const int32_t *sizes, int64_t G,
                      int64_t M, int64_t K, int64_t N, double *dx)
{
    if (G <= 0 || M < 0 || K <= 0 || N <= 0)
        return OR_ERR_SHAPE;
    int64_t *offsets = (int64_t *)malloc(sizeof(int64_t) * (size_t)(G + 1));
    int st = oracle_group_offsets(sizes, G, M, offsets);
    if (st != OR_OK) {
        free(offsets);
        return st;
    }
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t m = 0; m < M; ++m) {
        int64_t g = group_of_row(offsets, G, m);
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            if (g >= 0) {
                const uint16_t *wrow = w + (g * K + k) * N;
                for (int64_t n = 0; n < N; ++n)
                    acc += (double)bf16_bits_to_float(dy[m * N + n]) * (double)bf16_bits_to_float(wrow[n]);
            }
            dx[m * K + k] = acc;
        }
    }
    free(offsets);
    return OR_OK;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
#endif
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
