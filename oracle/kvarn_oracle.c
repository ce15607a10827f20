/*
 * kvarn_oracle.c -- plain, slow, fp64 CPU oracle for the KVarN 2-bit KV-cache
 * path (quantize-on-append and decode attention).
 *
 * TEST INFRASTRUCTURE. Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may build, load or call this file. The CUDA
 * library shares no code, header, table or constant with it.
 *
 * Sources (cited by page title and section):
 *   [ABS]  "KVarN: cuantizacion de KV-Cache normalizada por varianza mitiga la
 *          acumulacion de errores en tareas de razonamiento", English abstract:
 *          Hadamard rotation first, then dual-scaling variance normalisation
 *          over both axes of K and V; 2-bit precision; calibration-free.
 *   [AP3]  "KVarN：方差归一化让 2-bit KV 缓存扛住长链推理", section 三:
 *          3.1 randomised Hadamard H with H H^T = I, q rotated by the same H
 *          so Q K^T is unchanged, rotation keeps vector length;
 *          3.2 VarN: token axis to variance 1, then channel axis to variance 1,
 *          repeated 2-3 times (Sinkhorn-Knopp-like); scales are kept and
 *          re-applied at dequantisation; statistics come from the data itself.
 *   [FB2]  "記憶體突圍：KVarN 如何讓推理模型在 2-bit 精度下逼近 FP16 表現",
 *          section 2 (steps one and two).
 *   Where the pages leave a step open, the comment on each function states
 *   the reading taken (R-n labels name the same reading everywhere).
 *
 * Everything is computed in double precision with straight loops, in the
 * order the method states. No FWHT, no blocking, no fusion. The Hadamard
 * matrix is built explicitly by Sylvester doubling and multiplied in full.
 *
 * Packed head-block format (the written contract both paths implement):
 *   B tokens x 128 channels, B in {32, 64}, 4 channel groups of 32, codes of
 *   `bits` in {2, 3, 4} bits (X = 16 B bits bytes of codes):
 *   bytes [0, X)            codes, records of 8*bits bytes (layout per kind)
 *   bytes [X, X+8B)         s  : fp16 [4][B]  (group-major)
 *   bytes [X+8B, X+16B)     z  : fp16 [4][B]
 *   bytes [X+16B, X+18B)    R  : fp16 [B]     (per-token factor)
 *   bytes [X+18B, X+18B+256) C : fp16 [128]   (per-channel factor)
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Thread count of the OpenMP loops over independent units (the timed CPU
 * baseline is reported single-threaded and on all host cores). */
void orc_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int orc_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

#define ORC_D 128
#define ORC_NG 4
#define ORC_GS 32

/* Ablation switches ([AP3] section 五, 消融): the pages compare the full method
 * with Hadamard only (no VarN: iters = 0), VarN only (no rotation: R = I),
 * and VarN along one axis only (token-only, channel-only). */
#define ORC_NO_ROTATION 1u
#define ORC_NO_TOKEN_PASS 2u
#define ORC_NO_CHANNEL_PASS 4u

/* ------------------------------------------------------------------------ */
/* fp16 grid arithmetic, written from the IEEE-754 binary16 definition:      */
/* 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; the spacing of   */
/* representable values in the binade [2^e, 2^(e+1)) is 2^(e-10), and below  */
/* 2^-14 (subnormals) it is 2^-24. Largest finite value 65504.              */
/* ------------------------------------------------------------------------ */

static double f16_spacing(double a) /* a = |v|, finite, > 0 */
{
    int e2;
    frexp(a, &e2);          /* a = f * 2^e2 with f in [0.5, 1) */
    int e = e2 - 1;         /* a lies in [2^e, 2^(e+1)) */
    if (e < -14) e = -14;   /* subnormal spacing */
    return ldexp(1.0, e - 10);
}

/* round to nearest, ties to even; overflow to +-inf as IEEE does */
double orc_f16_rn(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    double q = f16_spacing(fabs(v));
    double r = nearbyint(v / q) * q;    /* v/q is exact: q is a power of two */
    if (fabs(r) > 65504.0) r = copysign(INFINITY, v);
    return r;
}

/* largest fp16 value <= v */
double orc_f16_rd(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    double q = f16_spacing(fabs(v));
    double r = floor(v / q) * q;
    if (r < -65504.0) r = -INFINITY;
    if (r > 65504.0) r = 65504.0;
    return r;
}

/* smallest fp16 value >= v */
double orc_f16_ru(double v)
{
    if (v == 0.0 || !isfinite(v)) return v;
    double q = f16_spacing(fabs(v));
    double r = ceil(v / q) * q;
    if (r > 65504.0) r = INFINITY;
    if (r < -65504.0) r = -65504.0;
    return r;
}

/* next fp16 value below a non-negative fp16 value h (h > 0) */
static double f16_prev_pos(double h)
{
    /* the gap below h: if h is a power of two >= 2^-13 the gap below is the
     * spacing of the binade under it, otherwise the spacing of h's binade */
    double q = f16_spacing(h);
    double below = h - q;
    if (below > 0 && f16_spacing(below) < q) below = h - f16_spacing(below);
    return below;
}

/* next fp16 value above a non-negative fp16 value h */
static double f16_next_pos(double h)
{
    if (h == 0.0) return ldexp(1.0, -24);
    return h + f16_spacing(h);
}

/* encode an fp16-representable value as its 16-bit pattern */
uint16_t orc_f16_bits(double h)
{
    uint16_t sign = signbit(h) ? 0x8000u : 0u;
    double a = fabs(h);
    if (isnan(h)) return 0x7E00u;
    if (isinf(h)) return sign | 0x7C00u;
    if (a == 0.0) return sign;
    if (a < ldexp(1.0, -14)) {                       /* subnormal */
        return sign | (uint16_t)(a / ldexp(1.0, -24));
    }
    int e2;
    frexp(a, &e2);
    int e = e2 - 1;
    double frac = a / ldexp(1.0, e) - 1.0;           /* in [0, 1) */
    return sign | (uint16_t)((e + 15) << 10) | (uint16_t)(frac * 1024.0);
}

/* decode a 16-bit pattern to its value */
double orc_f16_value(uint16_t b)
{
    int s = (b >> 15) & 1, e = (b >> 10) & 31, f = b & 1023;
    double v;
    if (e == 0) v = ldexp((double)f, -24);
    else if (e == 31) v = f ? NAN : INFINITY;
    else v = ldexp(1.0 + f / 1024.0, e - 15);
    return s ? -v : v;
}

/* bf16 pattern to value: the top 16 bits of an fp32 */
double orc_bf16_value(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Rotation  [AP3 3.1]  R = H_128 diag(sigma) / sqrt(128)                    */
/* Reading R-1: sigma_c = -1 where bit c of sign_bits is set, else +1.       */
/* ------------------------------------------------------------------------ */

/* Sylvester doubling: H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]] */
void orc_hadamard(int n, int32_t* H)
{
    H[0] = 1;
    for (int m = 1; m < n; m <<= 1)
        for (int i = 0; i < m; i++)
            for (int j = 0; j < m; j++) {
                int32_t h = H[i * n + j];
                H[i * n + (j + m)] = h;
                H[(i + m) * n + j] = h;
                H[(i + m) * n + (j + m)] = -h;
            }
}

static int32_t g_H[ORC_D * ORC_D];

/* built once when the library loads, before any thread can use it */
__attribute__((constructor)) static void build_hadamard128(void) { orc_hadamard(ORC_D, g_H); }

static const int32_t* hadamard128(void) { return g_H; }

static double sign_of(const uint32_t sign_bits[4], int c)
{
    return ((sign_bits[c >> 5] >> (c & 31)) & 1u) ? -1.0 : 1.0;
}

/* out = H (sigma . x) / sqrt(128) */
void orc_rotate(const double* x, const uint32_t sign_bits[4], double* out)
{
    const int32_t* H = hadamard128();
    double sx[ORC_D];
    for (int j = 0; j < ORC_D; j++) sx[j] = sign_of(sign_bits, j) * x[j];
    double rt = sqrt((double)ORC_D);
    for (int i = 0; i < ORC_D; i++) {
        double acc = 0.0;
        for (int j = 0; j < ORC_D; j++) acc += (double)H[i * ORC_D + j] * sx[j];
        out[i] = acc / rt;
    }
}

/* inverse: x = sigma . (H^T y) / sqrt(128); H is symmetric */
void orc_unrotate(const double* y, const uint32_t sign_bits[4], double* out)
{
    const int32_t* H = hadamard128();
    double rt = sqrt((double)ORC_D);
    for (int j = 0; j < ORC_D; j++) {
        double acc = 0.0;
        for (int i = 0; i < ORC_D; i++) acc += (double)H[i * ORC_D + j] * y[i];
        out[j] = sign_of(sign_bits, j) * acc / rt;
    }
}

/* ------------------------------------------------------------------------ */
/* VarN  [AP3 3.2], [ABS], [FB2 step two]                                    */
/* One iteration = token (row) pass, then channel (column) pass.             */
/* Readings R-2 (population variance, mean kept: scaling only), R-3 (order   */
/* and count), R-4 (one head-block = B tokens x 128 channels), R-5 (v <= 0   */
/* or non-finite leaves that factor unchanged).                              */
/* trace (may be NULL) gets 3 numbers per iteration:                         */
/*   [0] max_t |var_row(t) - 1| right after the row pass                     */
/*   [1] max_c |var_col(c) - 1| right after the column pass                  */
/*   [2] max_t |var_row(t) - 1| right after the column pass                  */
/* ------------------------------------------------------------------------ */

static void row_stats(const double* Y, int t, double* mu, double* var)
{
    double s = 0.0;
    for (int c = 0; c < ORC_D; c++) s += Y[t * ORC_D + c];
    double m = s / ORC_D;
    double v = 0.0;
    for (int c = 0; c < ORC_D; c++) {
        double d = Y[t * ORC_D + c] - m;
        v += d * d;
    }
    *mu = m;
    *var = v / ORC_D;
}

static void col_stats(const double* Y, int B, int c, double* mu, double* var)
{
    double s = 0.0;
    for (int t = 0; t < B; t++) s += Y[t * ORC_D + c];
    double m = s / B;
    double v = 0.0;
    for (int t = 0; t < B; t++) {
        double d = Y[t * ORC_D + c] - m;
        v += d * d;
    }
    *mu = m;
    *var = v / B;
}

static int usable_variance(double v, double mu)
{
    return v > 0.0 && isfinite(v) && v > ldexp(mu * mu, -30);
}

void orc_varn(int B, int iters, uint32_t flags, const double* Xr, double* Y, double* R, double* C,
              double* trace)
{
    memcpy(Y, Xr, sizeof(double) * (size_t)B * ORC_D);
    for (int t = 0; t < B; t++) R[t] = 1.0;
    for (int c = 0; c < ORC_D; c++) C[c] = 1.0;
    for (int it = 0; it < iters; it++) {
        /* token axis: every row to variance 1 (skipped by the channel-only ablation) */
        for (int t = 0; t < B && !(flags & ORC_NO_TOKEN_PASS); t++) {
            double mu, v;
            row_stats(Y, t, &mu, &v);
            if (!usable_variance(v, mu)) continue;
            double r = sqrt(v);
            for (int c = 0; c < ORC_D; c++) Y[t * ORC_D + c] /= r;
            R[t] *= r;
        }
        if (trace) {
            double worst = 0.0;
            for (int t = 0; t < B; t++) {
                double mu, v;
                row_stats(Y, t, &mu, &v);
                if (usable_variance(v, mu) && fabs(v - 1.0) > worst) worst = fabs(v - 1.0);
            }
            trace[3 * it + 0] = worst;
        }
        /* channel axis: every column to variance 1 (skipped by the token-only ablation) */
        for (int c = 0; c < ORC_D && !(flags & ORC_NO_CHANNEL_PASS); c++) {
            double mu, v;
            col_stats(Y, B, c, &mu, &v);
            if (!usable_variance(v, mu)) continue;
            double r = sqrt(v);
            for (int t = 0; t < B; t++) Y[t * ORC_D + c] /= r;
            C[c] *= r;
        }
        if (trace) {
            double wc = 0.0, wr = 0.0;
            for (int c = 0; c < ORC_D; c++) {
                double mu, v;
                col_stats(Y, B, c, &mu, &v);
                if (usable_variance(v, mu) && fabs(v - 1.0) > wc) wc = fabs(v - 1.0);
            }
            for (int t = 0; t < B; t++) {
                double mu, v;
                row_stats(Y, t, &mu, &v);
                if (usable_variance(v, mu) && fabs(v - 1.0) > wr) wr = fabs(v - 1.0);
            }
            trace[3 * it + 1] = wc;
            trace[3 * it + 2] = wr;
        }
    }
}

/* Reading R-6/R-7: factors are clamped to [2^-14, 65504] and rounded to the
 * nearest fp16 before use; normalised values are recomputed from them. */
double orc_round_factor(double f)
{
    double lo = ldexp(1.0, -14), hi = 65504.0;
    if (!(f >= lo)) f = (f > hi) ? hi : lo;  /* also maps NaN to the lower bound */
    if (f > hi) f = hi;
    return orc_f16_rn(f);
}

/* ------------------------------------------------------------------------ */
/* Asymmetric round-to-nearest over 32-channel groups with L = 2^bits - 1     */
/* steps (reading R-8, R-9; L = 3 for the method's 2 bits, 7 / 15 for 3 / 4-bit  */
/* width). For the group's values with minimum m and maximum M:              */
/*   z = largest fp16 <= m (clamped to +-65504)                              */
/*   s = smallest fp16 >= 0 with z + L s >= M (clamped to 65504)             */
/*   code = clamp(round-half-even((y - z) / s), 0, L); all 0 when s = 0      */
/* ------------------------------------------------------------------------ */

/* least fp16 s >= 0 with z16 + L s >= M (clamped to 65504); 0 when z16 >= M */
double orc_step_for(double z16, double M, int levels)
{
    if (z16 >= M) return 0.0;
    const double L = (double)levels;
    double s = orc_f16_ru((M - z16) / L);
    if (s > 65504.0) s = 65504.0;
    /* the division above rounds in fp64: settle the exact minimum by
     * comparing z + L s against M (exact in fp64 for fp16 operands) */
    while (s > 0.0 && s < 65504.0 && z16 + L * s < M) s = f16_next_pos(s);
    while (s > 0.0) {
        double p = f16_prev_pos(s);
        if (z16 + L * p >= M) s = p; else break;
    }
    return s;
}

void orc_group_params(const double* y, int n, int levels, double* z16, double* s16,
                      double* m_out, double* M_out)
{
    double m = y[0], M = y[0];
    for (int i = 1; i < n; i++) {
        if (y[i] < m) m = y[i];
        if (y[i] > M) M = y[i];
    }
    double mc = m < -65504.0 ? -65504.0 : (m > 65504.0 ? 65504.0 : m);
    double z = orc_f16_rd(mc);
    *z16 = z;
    *s16 = orc_step_for(z, M, levels);
    if (m_out) *m_out = m;
    if (M_out) *M_out = M;
}

int orc_code(double y, double z16, double s16, int levels)
{
    if (s16 == 0.0) return 0;
    double u = nearbyint((y - z16) / s16);    /* default mode: ties to even */
    if (u < 0) u = 0;
    if (u > levels) u = levels;
    return (int)u;
}

/* ------------------------------------------------------------------------ */
/* Code positions in the packed head-block (the written format contract).    */
/* Records of 8*bits bytes; record r = 32*sb + l with sb = t / 32 and a lane  */
/* l = 4a + b; each record holds 2*bits little-endian 32-bit words.          */
/* 2 bits:                                                                   */
/*   kind 0 (K): a = (t%32)/4, i = t%4, g = c/32, b = (c%32)/8, e = c%8;      */
/*               word 2i + g/2, bit 2*(4*(g%2) + e/2) + 16*(e%2)             */
/*   kind 1 (V): b = (t%32)/8, d = t%8, g = c/32, a = (c%32)/4, f = c%4;      */
/*               word 2g + f/2, bit 2*(4*(d/4) + 2*((d%4)/2) + f%2)+16*(d%2) */
/* 4 bits (the same lane assignment, one word per (token, group) for K and    */
/* per (group, channel) for V):                                              */
/*   kind 0 (K): word 4i + g, bit 4*(e/2) + 16*(e%2)                         */
/*   kind 1 (V): word 4g + f, bit 4*(d/2) + 16*(d%2)                         */
/* 3 bits: words 0..7 of the record hold the low two bits of each code at    */
/* its 2-bit position (word w2, bit 2j + 16h: pair j, half h, as above);     */
/* words 8..11 hold the high bit at word 8 + w2/2, bit 8*(w2%2) + j + 16h.   */
/* orc_code_position gives the low field's place, orc_code_high_position    */
/* the high bit's.                                                           */
/* ------------------------------------------------------------------------ */

/* 2-bit layout within a record: word w2 (0..7), pair j (0..7), half h. */
static void pair_position(int kind, int t, int c, int* w2, int* j, int* h)
{
    int g = c / ORC_GS;
    if (kind == 0) {
        int i = t % 4, e = c % 8;
        *w2 = 2 * i + g / 2;
        *j = 4 * (g % 2) + e / 2;
        *h = e % 2;
    } else {
        int d = t % 8, f = c % 4;
        *w2 = 2 * g + f / 2;
        *j = 4 * (d / 4) + 2 * ((d % 4) / 2) + f % 2;
        *h = d % 2;
    }
}

static int record_of(int kind, int t, int c)
{
    int sb = t / 32;
    if (kind == 0) return 32 * sb + 4 * ((t % 32) / 4) + (c % 32) / 8;
    return 32 * sb + 4 * ((c % 32) / 4) + (t % 32) / 8;
}

void orc_code_high_position(int kind, int t, int c, int* word_index, int* bit)
{
    int w2, j, h;
    pair_position(kind, t, c, &w2, &j, &h);
    *word_index = record_of(kind, t, c) * 12 + 8 + w2 / 2;
    *bit = 8 * (w2 % 2) + j + 16 * h;
}

void orc_code_position(int kind, int bits, int t, int c, int* word_index, int* bit)
{
    if (bits == 3) {
        int w2, j, h;
        pair_position(kind, t, c, &w2, &j, &h);
        *word_index = record_of(kind, t, c) * 12 + w2;
        *bit = 2 * j + 16 * h;
        return;
    }
    int sb = t / 32, g = c / ORC_GS;
    if (kind == 0) {
        int a = (t % 32) / 4, i = t % 4, b = (c % 32) / 8, e = c % 8;
        int rec = 32 * sb + 4 * a + b;
        if (bits == 4) {
            *word_index = rec * 16 + 4 * i + g;
            *bit = 4 * (e / 2) + 16 * (e % 2);
        } else {
            *word_index = rec * 8 + 2 * i + g / 2;
            *bit = 2 * (4 * (g % 2) + e / 2) + 16 * (e % 2);
        }
    } else {
        int b = (t % 32) / 8, d = t % 8, a = (c % 32) / 4, f = c % 4;
        int rec = 32 * sb + 4 * a + b;
        if (bits == 4) {
            *word_index = rec * 16 + 4 * g + f;
            *bit = 4 * (d / 2) + 16 * (d % 2);
        } else {
            *word_index = rec * 8 + 2 * g + f / 2;
            *bit = 2 * (4 * (d / 4) + 2 * ((d % 4) / 2) + f % 2) + 16 * (d % 2);
        }
    }
}

static size_t codes_bytes(int B, int bits) { return (size_t)16 * B * bits; }
size_t orc_head_block_bytes(int B, int bits) { return codes_bytes(B, bits) + (size_t)18 * B + 256; }

static void put_u16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xFF); p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Write one head-block from its fields. codes: [B][128] ints 0..3;
 * s16, z16: [B][4] fp16-grid values; R16: [B]; C16: [128]. */
void orc_pack(int B, int bits, int kind, const int32_t* codes, const double* s16, const double* z16,
              const double* R16, const double* C16, uint8_t* out)
{
    size_t nbytes = orc_head_block_bytes(B, bits);
    const int nwords = 4 * B * bits;
    const uint32_t mask = (1u << bits) - 1u;
    memset(out, 0, nbytes);
    uint32_t* words = (uint32_t*)malloc(sizeof(uint32_t) * (size_t)nwords);
    memset(words, 0, sizeof(uint32_t) * (size_t)nwords);
    for (int t = 0; t < B; t++)
        for (int c = 0; c < ORC_D; c++) {
            int w, bit;
            const uint32_t code = (uint32_t)codes[t * ORC_D + c] & mask;
            orc_code_position(kind, bits, t, c, &w, &bit);
            if (bits == 3) {
                words[w] |= (code & 3u) << bit;
                orc_code_high_position(kind, t, c, &w, &bit);
                words[w] |= (code >> 2) << bit;
            } else {
                words[w] |= code << bit;
            }
        }
    for (int w = 0; w < nwords; w++) {
        out[4 * w + 0] = (uint8_t)(words[w] & 0xFF);
        out[4 * w + 1] = (uint8_t)((words[w] >> 8) & 0xFF);
        out[4 * w + 2] = (uint8_t)((words[w] >> 16) & 0xFF);
        out[4 * w + 3] = (uint8_t)((words[w] >> 24) & 0xFF);
    }
    free(words);
    uint8_t* sp = out + codes_bytes(B, bits);
    uint8_t* zp = sp + 8 * B;
    uint8_t* rp = zp + 8 * B;
    uint8_t* cp = rp + 2 * B;
    for (int g = 0; g < ORC_NG; g++)
        for (int t = 0; t < B; t++) {
            put_u16(sp + 2 * (g * B + t), orc_f16_bits(s16[t * ORC_NG + g]));
            put_u16(zp + 2 * (g * B + t), orc_f16_bits(z16[t * ORC_NG + g]));
        }
    for (int t = 0; t < B; t++) put_u16(rp + 2 * t, orc_f16_bits(R16[t]));
    for (int c = 0; c < ORC_D; c++) put_u16(cp + 2 * c, orc_f16_bits(C16[c]));
}

/* Read the fields back from a head-block (the inverse of orc_pack). */
void orc_unpack(int B, int bits, int kind, const uint8_t* in, int32_t* codes, double* s16,
                double* z16, double* R16, double* C16)
{
    const uint32_t mask = (1u << bits) - 1u;
    for (int t = 0; t < B; t++)
        for (int c = 0; c < ORC_D; c++) {
            int w, bit;
            orc_code_position(kind, bits, t, c, &w, &bit);
            uint32_t word = (uint32_t)in[4 * w] | ((uint32_t)in[4 * w + 1] << 8) |
                            ((uint32_t)in[4 * w + 2] << 16) | ((uint32_t)in[4 * w + 3] << 24);
            if (bits == 3) {
                uint32_t code = (word >> bit) & 3u;
                orc_code_high_position(kind, t, c, &w, &bit);
                word = (uint32_t)in[4 * w] | ((uint32_t)in[4 * w + 1] << 8) |
                       ((uint32_t)in[4 * w + 2] << 16) | ((uint32_t)in[4 * w + 3] << 24);
                codes[t * ORC_D + c] = (int32_t)(code | (((word >> bit) & 1u) << 2));
            } else {
                codes[t * ORC_D + c] = (int32_t)((word >> bit) & mask);
            }
        }
    const uint8_t* sp = in + codes_bytes(B, bits);
    const uint8_t* zp = sp + 8 * B;
    const uint8_t* rp = zp + 8 * B;
    const uint8_t* cp = rp + 2 * B;
    for (int g = 0; g < ORC_NG; g++)
        for (int t = 0; t < B; t++) {
            s16[t * ORC_NG + g] = orc_f16_value(get_u16(sp + 2 * (g * B + t)));
            z16[t * ORC_NG + g] = orc_f16_value(get_u16(zp + 2 * (g * B + t)));
        }
    for (int t = 0; t < B; t++) R16[t] = orc_f16_value(get_u16(rp + 2 * t));
    for (int c = 0; c < ORC_D; c++) C16[c] = orc_f16_value(get_u16(cp + 2 * c));
}

/* ------------------------------------------------------------------------ */
/* Whole-block quantisation: rotate -> VarN -> round factors -> normalise -> */
/* group quantise -> pack. X: [B][128] input values (already widened to      */
/* fp64). Any of the detail outputs may be NULL.                             */
/* ------------------------------------------------------------------------ */

void orc_quantize_block(int B, int bits, int iters, uint32_t flags, int kind, const uint32_t sign_bits[4],
                        const double* X, uint8_t* out,
                        double* Xr_out, double* R_out, double* C_out,
                        double* R16_out, double* C16_out, double* y_out,
                        double* z16_out, double* s16_out, int32_t* codes_out,
                        double* trace)
{
    size_t n = (size_t)B * ORC_D;
    double* Xr = (double*)calloc(n, sizeof(double));
    double* Y = (double*)malloc(sizeof(double) * n);
    double* y = (double*)malloc(sizeof(double) * n);
    double* R = (double*)malloc(sizeof(double) * B);
    double* R16 = (double*)malloc(sizeof(double) * B);
    double* s16 = (double*)malloc(sizeof(double) * B * ORC_NG);
    double* z16 = (double*)malloc(sizeof(double) * B * ORC_NG);
    int32_t* codes = (int32_t*)malloc(sizeof(int32_t) * n);
    double C[ORC_D], C16[ORC_D];

    for (int t = 0; t < B; t++) {
        if (flags & ORC_NO_ROTATION) memcpy(Xr + (size_t)t * ORC_D, X + (size_t)t * ORC_D, sizeof(double) * ORC_D);
        else orc_rotate(X + (size_t)t * ORC_D, sign_bits, Xr + (size_t)t * ORC_D);
    }
    orc_varn(B, iters, flags, Xr, Y, R, C, trace);
    for (int t = 0; t < B; t++) R16[t] = orc_round_factor(R[t]);
    for (int c = 0; c < ORC_D; c++) C16[c] = orc_round_factor(C[c]);
    for (int t = 0; t < B; t++)
        for (int c = 0; c < ORC_D; c++)
            y[t * ORC_D + c] = Xr[t * ORC_D + c] / (R16[t] * C16[c]);
    for (int t = 0; t < B; t++)
        for (int g = 0; g < ORC_NG; g++) {
            const double* yg = y + t * ORC_D + g * ORC_GS;
            orc_group_params(yg, ORC_GS, (1 << bits) - 1, &z16[t * ORC_NG + g], &s16[t * ORC_NG + g], NULL, NULL);
            for (int k = 0; k < ORC_GS; k++)
                codes[t * ORC_D + g * ORC_GS + k] =
                    orc_code(yg[k], z16[t * ORC_NG + g], s16[t * ORC_NG + g], (1 << bits) - 1);
        }
    if (out) orc_pack(B, bits, kind, codes, s16, z16, R16, C16, out);

    if (Xr_out) memcpy(Xr_out, Xr, sizeof(double) * n);
    if (R_out) memcpy(R_out, R, sizeof(double) * B);
    if (C_out) memcpy(C_out, C, sizeof(double) * ORC_D);
    if (R16_out) memcpy(R16_out, R16, sizeof(double) * B);
    if (C16_out) memcpy(C16_out, C16, sizeof(double) * ORC_D);
    if (y_out) memcpy(y_out, y, sizeof(double) * n);
    if (z16_out) memcpy(z16_out, z16, sizeof(double) * B * ORC_NG);
    if (s16_out) memcpy(s16_out, s16, sizeof(double) * B * ORC_NG);
    if (codes_out) memcpy(codes_out, codes, sizeof(int32_t) * n);
    free(Xr); free(Y); free(y); free(R); free(R16); free(s16); free(z16); free(codes);
}

/* Many independent head-blocks: X [n][B][128] -> out [n][head_block_bytes]. */
void orc_quantize_blocks(int64_t n, int B, int bits, int iters, uint32_t flags, int kind, const uint32_t sign_bits[4],
                         const double* X, uint8_t* out)
{
    size_t hb = orc_head_block_bytes(B, bits);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < n; i++)
        orc_quantize_block(B, bits, iters, flags, kind, sign_bits, X + (size_t)i * B * ORC_D, out + (size_t)i * hb,
                           NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL);
}

/* ------------------------------------------------------------------------ */
/* Dequantisation: y^ = code * s + z;  x^_rot = y^ * R * C;                  */
/* unrotated x^ = R^T x^_rot  [AP3 3.2: the kept scales are re-applied].    */
/* out: [B][128]; rotated != 0 keeps the rotated space.                      */
/* ------------------------------------------------------------------------ */

void orc_decode_block(int B, int bits, uint32_t flags, int kind, const uint32_t sign_bits[4], const uint8_t* in,
                      int rotated, double* out)
{
    size_t n = (size_t)B * ORC_D;
    int32_t* codes = (int32_t*)malloc(sizeof(int32_t) * n);
    double* s16 = (double*)malloc(sizeof(double) * B * ORC_NG);
    double* z16 = (double*)malloc(sizeof(double) * B * ORC_NG);
    double* R16 = (double*)malloc(sizeof(double) * B);
    double C16[ORC_D], xr[ORC_D];
    orc_unpack(B, bits, kind, in, codes, s16, z16, R16, C16);
    for (int t = 0; t < B; t++) {
        for (int c = 0; c < ORC_D; c++) {
            int g = c / ORC_GS;
            double yh = codes[t * ORC_D + c] * s16[t * ORC_NG + g] + z16[t * ORC_NG + g];
            xr[c] = yh * R16[t] * C16[c];
        }
        if (rotated || (flags & ORC_NO_ROTATION)) memcpy(out + (size_t)t * ORC_D, xr, sizeof(xr));
        else orc_unrotate(xr, sign_bits, out + (size_t)t * ORC_D);
    }
    free(codes); free(s16); free(z16); free(R16);
}

void orc_decode_blocks(int64_t n, int B, int bits, uint32_t flags, int kind, const uint32_t sign_bits[4],
                       const uint8_t* in, int rotated, double* out)
{
    size_t hb = orc_head_block_bytes(B, bits);
    #pragma omp parallel for schedule(dynamic, 4)
    for (int64_t i = 0; i < n; i++)
        orc_decode_block(B, bits, flags, kind, sign_bits, in + (size_t)i * hb, rotated, out + (size_t)i * B * ORC_D);
}

/* ------------------------------------------------------------------------ */
/* Attention, the plain definition (reading R-13, R-14): for one query q and  */
/* L keys/values, p = softmax_t(sm_scale * q.k_t) with the maximum taken out, */
/* o = sum_t p_t v_t. Keys and values are given unrotated.                    */
/* ------------------------------------------------------------------------ */

void orc_attention(const double* q, const double* K, const double* V, int64_t L,
                   double sm_scale, double* out)
{
    for (int c = 0; c < ORC_D; c++) out[c] = 0.0;
    if (L <= 0) return;
    double* logit = (double*)malloc(sizeof(double) * (size_t)L);
    double mx = -INFINITY;
    for (int64_t t = 0; t < L; t++) {
        double dot = 0.0;
        for (int c = 0; c < ORC_D; c++) dot += q[c] * K[t * ORC_D + c];
        logit[t] = sm_scale * dot;
        if (logit[t] > mx) mx = logit[t];
    }
    double den = 0.0;
    for (int64_t t = 0; t < L; t++) {
        double p = exp(logit[t] - mx);
        den += p;
        for (int c = 0; c < ORC_D; c++) out[c] += p * V[t * ORC_D + c];
    }
    for (int c = 0; c < ORC_D; c++) out[c] /= den;
    free(logit);
}

/* The rotated route [AP3 3.1]: rotate q and every key and value with R,
 * attend in the rotated space, rotate the output back. Must equal
 * orc_attention on the same inputs (the rotation is orthogonal). */
void orc_attention_rotated(const double* q, const double* K, const double* V, int64_t L,
                           double sm_scale, const uint32_t sign_bits[4], double* out)
{
    double* Kr = (double*)malloc(sizeof(double) * (size_t)L * ORC_D);
    double* Vr = (double*)malloc(sizeof(double) * (size_t)L * ORC_D);
    double qr[ORC_D], orot[ORC_D];
    orc_rotate(q, sign_bits, qr);
    for (int64_t t = 0; t < L; t++) {
        orc_rotate(K + t * ORC_D, sign_bits, Kr + t * ORC_D);
        orc_rotate(V + t * ORC_D, sign_bits, Vr + t * ORC_D);
    }
    orc_attention(qr, Kr, Vr, L, sm_scale, orot);
    orc_unrotate(orot, sign_bits, out);
    free(Kr); free(Vr);
}

/* ------------------------------------------------------------------------ */
/* Decode attention over a paged 2-bit cache (the whole read path).          */
/* For unit (b, h_kv) and each of its G query heads: keys/values of the      */
/* first floor(L/B)*B tokens are the decoded (unrotated) head-blocks found    */
/* through block_table; the remaining L % B tokens are the raw bf16 staging   */
/* rows (reading R-11, R-12). q is given as fp64 [batch][n_q][128].           */
/* pool: head-block of (physical p, head h, kind k) at                       */
/*   pool + p * block_bytes + (2 h + k) * head_block_bytes                   */
/* staging: bf16 patterns [batch][n_kv][2][B][128]                           */
/* out: fp64 [batch][n_q][128]. Units run in parallel (OpenMP).              */
/* ------------------------------------------------------------------------ */

void orc_decode_attention(int B, int bits, uint32_t flags, int n_q, int n_kv, const uint32_t sign_bits[4], double sm_scale,
                          const double* q, const uint8_t* pool, const uint16_t* staging,
                          const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                          int batch, double* out)
{
    size_t hb = orc_head_block_bytes(B, bits);
    size_t block_bytes = (size_t)n_kv * 2 * hb;
    int G = n_q / n_kv;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int unit = 0; unit < batch * n_kv; unit++) {
        int b = unit / n_kv, h = unit % n_kv;
        int64_t L = seq_lens[b];
        int64_t nfull = L / B;
        int64_t tail = L % B;
        double* K = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * ORC_D);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * ORC_D);
        for (int64_t j = 0; j < nfull; j++) {
            int64_t p = block_table[(int64_t)b * max_blocks + j];
            const uint8_t* base = pool + (size_t)p * block_bytes + (size_t)(2 * h) * hb;
            orc_decode_block(B, bits, flags, 0, sign_bits, base, 0, K + (size_t)j * B * ORC_D);
            orc_decode_block(B, bits, flags, 1, sign_bits, base + hb, 0, V + (size_t)j * B * ORC_D);
        }
        for (int64_t r = 0; r < tail; r++) {
            const uint16_t* sk = staging + ((((size_t)b * n_kv + h) * 2 + 0) * B + r) * ORC_D;
            const uint16_t* sv = staging + ((((size_t)b * n_kv + h) * 2 + 1) * B + r) * ORC_D;
            for (int c = 0; c < ORC_D; c++) {
                K[(nfull * B + r) * ORC_D + c] = orc_bf16_value(sk[c]);
                V[(nfull * B + r) * ORC_D + c] = orc_bf16_value(sv[c]);
            }
        }
        for (int j = 0; j < G; j++) {
            int hq = h * G + j;
            orc_attention(q + ((size_t)b * n_q + hq) * ORC_D, K, V, L, sm_scale,
                          out + ((size_t)b * n_q + hq) * ORC_D);
        }
        free(K); free(V);
    }
}

/* ------------------------------------------------------------------------ */
/* Chunked prefill attention over the same paged cache (reading R-24).       */
/* Each sequence b holds L = seq_lens[b] tokens after its last `chunk` tokens  */
/* were appended; query row r of the chunk sits at position p = L - chunk + r */
/* and attends to tokens 0..p, every token read from the cache as it stands  */
/* (complete blocks decoded, the open tail raw bf16). A row with p < 0 sees  */
/* no token and gives zeros. q: fp64 [batch][chunk][n_q][128]; out likewise. */
/* ------------------------------------------------------------------------ */

void orc_prefill_attention(int B, int bits, uint32_t flags, int n_q, int n_kv, const uint32_t sign_bits[4],
                           double sm_scale, const double* q, const uint8_t* pool, const uint16_t* staging,
                           const int32_t* block_table, int max_blocks, const int32_t* seq_lens, int batch,
                           int chunk, double* out)
{
    size_t hb = orc_head_block_bytes(B, bits);
    size_t block_bytes = (size_t)n_kv * 2 * hb;
    int G = n_q / n_kv;
    #pragma omp parallel for schedule(dynamic, 1)
    for (int unit = 0; unit < batch * n_kv; unit++) {
        int b = unit / n_kv, h = unit % n_kv;
        int64_t L = seq_lens[b];
        int64_t nfull = L / B;
        int64_t tail = L % B;
        double* K = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * ORC_D);
        double* V = (double*)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * ORC_D);
        /* the cache as it stands: decoded complete blocks, then the raw tail */
        for (int64_t j = 0; j < nfull; j++) {
            int64_t p = block_table[(int64_t)b * max_blocks + j];
            const uint8_t* base = pool + (size_t)p * block_bytes + (size_t)(2 * h) * hb;
            orc_decode_block(B, bits, flags, 0, sign_bits, base, 0, K + (size_t)j * B * ORC_D);
            orc_decode_block(B, bits, flags, 1, sign_bits, base + hb, 0, V + (size_t)j * B * ORC_D);
        }
        for (int64_t r = 0; r < tail; r++) {
            const uint16_t* sk = staging + ((((size_t)b * n_kv + h) * 2 + 0) * B + r) * ORC_D;
            const uint16_t* sv = staging + ((((size_t)b * n_kv + h) * 2 + 1) * B + r) * ORC_D;
            for (int c = 0; c < ORC_D; c++) {
                K[(nfull * B + r) * ORC_D + c] = orc_bf16_value(sk[c]);
                V[(nfull * B + r) * ORC_D + c] = orc_bf16_value(sv[c]);
            }
        }
        /* causal: row r sees the first p + 1 tokens */
        for (int r = 0; r < chunk; r++) {
            int64_t visible = L - chunk + r + 1;
            for (int j = 0; j < G; j++) {
                int hq = h * G + j;
                size_t row = (((size_t)b * chunk + r) * n_q + hq) * ORC_D;
                orc_attention(q + row, K, V, visible, sm_scale, out + row);   /* zeros when visible <= 0 */
            }
        }
        free(K); free(V);
    }
}

/* ------------------------------------------------------------------------ */
/* Error decomposition  [AP3] section 二: a token vector x and its quantised  */
/* version x^ = x + eps; eps = E_M + E_D with the magnitude part             */
/*   E_M = (|x^| - |x|) x / |x|                                              */
/* and the direction part                                                     */
/*   E_D = |x^| (x^ / |x^| - x / |x|).                                        */
/* out = (|x|, |x^|, |E_M|, |E_D|). Reading: for x = 0 the direction x/|x| is */
/* undefined and all of eps (= x^) is counted as magnitude error; for x^ = 0  */
/* the formula itself gives E_M = -x, E_D = 0.                               */
/* ------------------------------------------------------------------------ */

void orc_error_split(const double* x, const double* xh, double* out)
{
    double nx = 0.0, nh = 0.0;
    for (int c = 0; c < ORC_D; c++) {
        nx += x[c] * x[c];
        nh += xh[c] * xh[c];
    }
    nx = sqrt(nx);
    nh = sqrt(nh);
    out[0] = nx;
    out[1] = nh;
    if (nx == 0.0) {
        out[2] = nh;
        out[3] = 0.0;
        return;
    }
    out[2] = fabs(nh - nx);
    if (nh == 0.0) {
        out[3] = 0.0;
        return;
    }
    double d = 0.0;
    for (int c = 0; c < ORC_D; c++) {
        double u = xh[c] / nh - x[c] / nx;
        d += u * u;
    }
    out[3] = nh * sqrt(d);
}

/* Per token of a head-block: X [B][128] the values before quantisation,
 * packed the head-block's bytes; out [B][4] as orc_error_split. */
void orc_error_decomposition(int B, int bits, uint32_t flags, int kind, const uint32_t sign_bits[4],
                             const double* X, const uint8_t* packed, double* out)
{
    double* xh = (double*)malloc(sizeof(double) * (size_t)B * ORC_D);
    orc_decode_block(B, bits, flags, kind, sign_bits, packed, 0, xh);
    for (int t = 0; t < B; t++)
        orc_error_split(X + (size_t)t * ORC_D, xh + (size_t)t * ORC_D, out + 4 * t);
    free(xh);
}

/* ------------------------------------------------------------------------ */
/* Staged hand-off helpers for parity: each stage is recomputed from the      */
/* other side's already validated rounded values, so one boundary case      */
/* cannot cascade into later stages.                                         */
/* ------------------------------------------------------------------------ */

/* y from the oracle's rotated values and externally supplied fp16 factors */
void orc_normalise(int B, const double* Xr, const double* R16, const double* C16, double* y)
{
    for (int t = 0; t < B; t++)
        for (int c = 0; c < ORC_D; c++)
            y[t * ORC_D + c] = Xr[t * ORC_D + c] / (R16[t] * C16[c]);
}

/* per (token, group): z16, s16 from y, plus the group's min and max */
void orc_group_params_all(int B, int bits, const double* y, double* z16, double* s16, double* m, double* M)
{
    for (int t = 0; t < B; t++)
        for (int g = 0; g < ORC_NG; g++)
            orc_group_params(y + t * ORC_D + g * ORC_GS, ORC_GS, (1 << bits) - 1, &z16[t * ORC_NG + g],
                             &s16[t * ORC_NG + g], &m[t * ORC_NG + g], &M[t * ORC_NG + g]);
}

/* codes from y with given z16, s16; dist[t][c] = distance from y to the
 * nearest decision boundary z + (k + 1/2) s, k = 0..2 (inf when s = 0) */
void orc_codes_given(int B, int bits, const double* y, const double* z16, const double* s16,
                     int32_t* codes, double* dist)
{
    for (int t = 0; t < B; t++)
        for (int c = 0; c < ORC_D; c++) {
            int g = c / ORC_GS;
            double z = z16[t * ORC_NG + g], s = s16[t * ORC_NG + g];
            double yv = y[t * ORC_D + c];
            codes[t * ORC_D + c] = orc_code(yv, z, s, (1 << bits) - 1);
            double best = INFINITY;
            if (s > 0.0)
                for (int k = 0; k < (1 << bits) - 1; k++) {
                    double bd = fabs(yv - (z + (k + 0.5) * s));
                    if (bd < best) best = bd;
                }
            dist[t * ORC_D + c] = best;
        }
}
