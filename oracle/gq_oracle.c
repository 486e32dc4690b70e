/*
 * gq_oracle.c -- plain, slow, obviously-correct CPU reference for the
 * block-quantized matrix-vector / matrix-matrix product.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file: only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, table or constant with
 * the CUDA library; its only inputs are the seeded arrays produced by the
 * synthetic-input module.
 *
 * Compile: gcc -O2 -ffp-contract=off -fno-fast-math -fopenmp -shared -fPIC.
 * Every floating-point step below is a single IEEE fp32 (or fp64) operation
 * written out in source order; there is no FMA contraction and no division
 * replaced by a reciprocal multiply.
 *
 * Sources followed (page title, then section):
 *   [P2] "llama.cpp 推理引擎" (runguoli.com/llm-libs/14-llama-cpp)
 *        §5.1 symmetric quantization, §5.2 asymmetric quantization,
 *        §5.3 Q4_0, §5.4 Q8_0, §5.5 K-quant (Q4_K super-block and its
 *        two-level dequantization), §6.4 the Q4_0 vec_dot pseudocode
 *        (nibble order: low nibble of byte j is element 2j, high nibble is
 *        element 2j+1).
 *   [P4] "llama.cpp：一个人、一个周末、一个改变 AI 推理格局的 C++ 文件"
 *        (tech-blog-56a.pages.dev), 第二层：量化引擎 -- the block
 *        quantization figure and the 256 = 8 x 32 K-quant hierarchy.
 *   The library's format definition fixes what the pages leave open or
 *   print inconsistently: Q8_0 carries an fp16 scale (34 B, where [P2] §5.4
 *   prints fp32), Q4_K carries 6-bit sub-block scales and mins (144 B, where
 *   [P2] §5.5 prints 4-bit fields) and dequantizes as d*sc*q - dmin*m, codes
 *   are rounded half away from zero.  Q8_K (the 256-element activation
 *   block) is not described by any page; its layout is this library's own.
 *
 * Readings taken where the pages are silent (each also listed in the design
 * notes of the repository):
 *   - Q4_0 scale d = max|x| / 7 ([P2] §5.1 worked example); codes c = q + 8
 *     with q = round(x/d) clamped to [-8, 7].
 *   - fp16 scales of Q8_0 / Q4_0 are rounded to nearest-even; the fp16 d and
 *     dmin of Q4_K are rounded toward +infinity so that the 6-bit ceilings
 *     below always cover the sub-block's range.
 *   - Q4_K: non-iterative min/max fit (the asymmetric formula of [P2] §5.2
 *     with the minimum clamped to <= 0 because the min term is subtracted).
 *   - Q6_K (6-bit K blocks, no sub-blocks, as the discosf.com page's §4
 *     describes them): symmetric rule with scale = max|x| / 31, codes
 *     c = q + 32 with q clamped to [-32, 31]; layout this library's own (see
 *     quantize_q6_k_block).  It pairs with Q8_K activations.
 *   - Q5_K (the same page's §4: one bit more than the 4-bit K-quant): the
 *     Q4_K super-block -- fp16 d and dmin, 6-bit sub-block scales and mins,
 *     the same min/max fit -- with 5-bit codes q in [0, 31], whose fifth
 *     bits sit in a bit plane of their own; layout this library's own (see
 *     quantize_q5_k_block).  It pairs with Q8_K activations.
 *   - A zero scale yields zero codes (Q4_0 code 8, Q6_K code 32).
 *   - Non-finite inputs are rejected (return -2).
 *
 * parity pins: every function here is pinned by tests under tests/ that do
 * not call back into this file for their expected values.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Type codes, in the order of the public type enumeration. */
enum { OR_Q4_0 = 0, OR_Q8_0 = 1, OR_Q4_K = 2, OR_Q8_K = 3, OR_Q6_K = 4, OR_Q5_K = 5 };

/* ------------------------------------------------------------------ */
/* Bit-level helpers                                                    */
/* ------------------------------------------------------------------ */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* fp16 -> fp32, exact (every fp16 value is an fp32 value). */
float or_f16_to_f32(uint16_t h)
{
    uint32_t sign = (uint32_t)(h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1fu;
    uint32_t m = h & 0x3ffu;
    if (e == 0x1f) /* inf / nan */
        return bits_f32(sign | 0x7f800000u | (m << 13));
    if (e == 0) {
        /* zero or subnormal: value = m * 2^-24, exact in fp32 */
        float v = (float)m * bits_f32(0x33800000u); /* 2^-24 */
        return sign ? -v : v;
    }
    return bits_f32(sign | ((e + 112u) << 23) | (m << 13));
}

/*
 * fp32 -> fp16 with a selectable rounding rule.
 *   up == 0 : round to nearest, ties to even (IEEE default)
 *   up == 1 : round toward +infinity
 * Works on the magnitude: the fp32 significand (with its hidden bit) is
 * shifted right to the fp16 grid of the target exponent; the bits shifted out
 * decide the rounding.
 */
static uint16_t f32_to_f16(float f, int up)
{
    uint32_t x = f32_bits(f);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t a = x & 0x7fffffffu;
    int neg = sign != 0;

    if (a > 0x7f800000u) /* nan: keep it a quiet nan */
        return (uint16_t)(sign | 0x7e00u);
    if (a == 0x7f800000u)
        return (uint16_t)(sign | 0x7c00u);

    int32_t exp = (int32_t)(a >> 23);           /* biased fp32 exponent */
    uint32_t sig = (a & 0x7fffffu) | (exp ? 0x800000u : 0); /* 24-bit */
    if (exp == 0) exp = 1;                      /* fp32 subnormal */

    /* The fp16 grid unit at this magnitude: normal fp16 numbers with
     * unbiased exponent E >= -14 keep 10 fraction bits, i.e. a unit of
     * 2^(E-10); below 2^-14 the unit is fixed at 2^-24. */
    int32_t e_unb = exp - 127;
    int32_t unit_exp = (e_unb >= -14) ? e_unb - 10 : -24;
    /* sig * 2^(exp-150) expressed in units of 2^unit_exp: shift right by
     * (unit_exp - (exp - 150)). */
    int32_t shift = unit_exp - (exp - 150);
    uint64_t q, rem, half;
    if (shift >= 40) {
        q = 0; rem = sig; half = (uint64_t)1 << 39; /* rem < half always */
    } else {
        q = (uint64_t)sig >> shift;
        rem = (uint64_t)sig & (((uint64_t)1 << shift) - 1);
        half = (uint64_t)1 << (shift - 1);
    }
    /* shift is >= 13 for every finite fp32 input, so half is well defined */
    int round_up;
    if (up)
        round_up = (!neg) && rem != 0; /* toward +inf: magnitudes of
                                          positives grow, of negatives drop */
    else
        round_up = rem > half || (rem == half && (q & 1));
    q += (uint64_t)round_up;

    /* q counts units of 2^unit_exp; rebuild the fp16 encoding. */
    uint32_t h;
    if (unit_exp == -24) {
        /* subnormal range: q < 2^10 is a subnormal, q == 2^10 is the
         * smallest normal 2^-14 -- both encode as the plain value of q. */
        h = (uint32_t)q;
    } else {
        /* normal: q in [2^10, 2^11]; q == 2^11 carries into the exponent */
        int32_t E = e_unb;
        if (q == 2048) { q = 1024; E += 1; }
        if (E > 15) {
            /* overflow: nearest rounds to inf, toward +inf keeps the
             * largest finite negative */
            h = (up && neg) ? 0x7bffu : 0x7c00u;
        } else {
            h = ((uint32_t)(E + 15) << 10) | ((uint32_t)q & 0x3ffu);
        }
    }
    return (uint16_t)(sign | h);
}

uint16_t or_f16_rn(float f) { return f32_to_f16(f, 0); }
uint16_t or_f16_ru(float f) { return f32_to_f16(f, 1); }

void or_f16_rn_array(const float *x, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; i++) h[i] = f32_to_f16(x[i], 0);
}
void or_f16_ru_array(const float *x, uint16_t *h, int64_t n)
{
    for (int64_t i = 0; i < n; i++) h[i] = f32_to_f16(x[i], 1);
}

static void put_u16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
static uint16_t get_u16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void put_f32(uint8_t *p, float f)
{
    uint32_t u = f32_bits(f);
    p[0] = (uint8_t)u; p[1] = (uint8_t)(u >> 8); p[2] = (uint8_t)(u >> 16); p[3] = (uint8_t)(u >> 24);
}
static float get_f32(const uint8_t *p)
{
    return bits_f32((uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24));
}

/* round half away from zero: the code rounding rule of every format */
static float rha(float v) { return roundf(v); }

static float clampf(float v, float lo, float hi) { return v < lo ? lo : (v > hi ? hi : v); }

/* ------------------------------------------------------------------ */
/* Block geometry                                                       */
/* ------------------------------------------------------------------ */

int64_t or_block_elems(int type)
{
    switch (type) {
    case OR_Q4_0: case OR_Q8_0: return 32;
    case OR_Q4_K: case OR_Q8_K: case OR_Q6_K: case OR_Q5_K: return 256;
    }
    return -1;
}

/* Q4_0: fp16 d + 16 bytes of nibbles ([P2] §5.3: 144 bits).
 * Q8_0: fp16 d + 32 int8.
 * Q4_K: fp16 d, fp16 dmin, 12 bytes of 6-bit scales/mins, 128 bytes of
 *       nibbles.
 * Q8_K: fp32 d, 256 int8, eight int16 sub-block sums.
 * Q6_K: fp16 d, 128 bytes holding the low four bits of the 256 codes, 64
 *       bytes holding their top two bits.
 * Q5_K: the Q4_K fields (144 bytes) and 32 bytes holding the fifth bit of
 *       each of the 256 codes. */
int64_t or_block_bytes(int type)
{
    switch (type) {
    case OR_Q4_0: return 2 + 16;
    case OR_Q8_0: return 2 + 32;
    case OR_Q4_K: return 2 + 2 + 12 + 128;
    case OR_Q8_K: return 4 + 256 + 2 * 8;
    case OR_Q6_K: return 2 + 128 + 64;
    case OR_Q5_K: return 2 + 2 + 12 + 128 + 32;
    }
    return -1;
}

static int all_finite(const float *x, int64_t n)
{
    for (int64_t i = 0; i < n; i++)
        if (!isfinite(x[i])) return 0;
    return 1;
}

/* ------------------------------------------------------------------ */
/* Encoders                                                             */
/* ------------------------------------------------------------------ */

/* Q8_0 ([P2] §5.1 with b = 8, §5.4): symmetric, scale = max|x| / 127. */
static void quantize_q8_0_block(const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    uint16_t dh = or_f16_rn(amax / 127.0f);
    float d = or_f16_to_f32(dh);
    put_u16(blk, dh);
    for (int i = 0; i < 32; i++) {
        float q = (d == 0.0f) ? 0.0f : clampf(rha(x[i] / d), -127.0f, 127.0f);
        blk[2 + i] = (uint8_t)(int8_t)q;
    }
}

/* Q4_0 ([P2] §5.1 with b = 4 -- scale = max|x| / 7 -- and §5.3; the code
 * stored is q + 8, and byte j holds element 2j in its low nibble and 2j+1 in
 * its high nibble as in the §6.4 pseudocode). */
static void quantize_q4_0_block(const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    uint16_t dh = or_f16_rn(amax / 7.0f);
    float d = or_f16_to_f32(dh);
    put_u16(blk, dh);
    uint8_t c[32];
    for (int i = 0; i < 32; i++) {
        float q = (d == 0.0f) ? 0.0f : clampf(rha(x[i] / d), -8.0f, 7.0f);
        c[i] = (uint8_t)((int)q + 8);
    }
    for (int j = 0; j < 16; j++)
        blk[2 + j] = (uint8_t)(c[2 * j] | (c[2 * j + 1] << 4));
}

/* Pack sixteen 6-bit fields LSB-first into 12 bytes (a 96-bit little-endian
 * integer): fields 0..7 are the sub-block scales, 8..15 the mins. */
static void pack6(const uint8_t f[16], uint8_t out[12])
{
    memset(out, 0, 12);
    for (int k = 0; k < 16; k++) {
        for (int b = 0; b < 6; b++) {
            int bit = 6 * k + b;
            if ((f[k] >> b) & 1) out[bit / 8] |= (uint8_t)(1u << (bit % 8));
        }
    }
}
static void unpack6(const uint8_t in[12], uint8_t f[16])
{
    for (int k = 0; k < 16; k++) {
        uint8_t v = 0;
        for (int b = 0; b < 6; b++) {
            int bit = 6 * k + b;
            v |= (uint8_t)(((in[bit / 8] >> (bit % 8)) & 1) << b);
        }
        f[k] = v;
    }
}

/* The asymmetric K-quant fit of one 256-element super-block with codes in
 * [0, qmax] ([P2] §5.2 asymmetric fit per 32-element sub-block, §5.5
 * two-level scales; [P4] 256 = 8 x 32 super-block).  For sub-block j:
 *   lo_j = min(0, min x), hi_j = max x
 *   dmin = f16_ru(max_j(-lo_j) / 63),  m_j = min(63, ceil(-lo_j / dmin))
 *   base_j = -(dmin * m_j)                      (exact in fp32)
 *   r_j = hi_j - base_j
 *   d = f16_ru(max_j r_j / (63 qmax)),  sc_j = min(63, ceil(r_j / (qmax d)))
 *   step_j = d * sc_j                           (exact in fp32)
 *   q_i = clamp(round((x_i - base_j) / step_j), 0, qmax)
 * and the element is reconstructed as d*sc_j*q_i - dmin*m_j.  Q4_K takes
 * qmax = 15 (63 qmax = 945), Q5_K qmax = 31 (1953).  Writes the fp16 d and
 * dmin, the sixteen 6-bit fields (sc_0..sc_7, m_0..m_7) and the codes. */
static void k_asym_fit(const float *x, float qmax, uint16_t *dh_out, uint16_t *dminh_out,
                       uint8_t fields[16], uint8_t q[256])
{
    float lo[8], hi[8];
    for (int j = 0; j < 8; j++) {
        float mn = x[32 * j], mx = x[32 * j];
        for (int i = 1; i < 32; i++) {
            float v = x[32 * j + i];
            if (v < mn) mn = v;
            if (v > mx) mx = v;
        }
        lo[j] = mn < 0.0f ? mn : 0.0f;
        hi[j] = mx;
    }
    float neg_lo_max = 0.0f;
    for (int j = 0; j < 8; j++)
        if (-lo[j] > neg_lo_max) neg_lo_max = -lo[j];
    uint16_t dminh = or_f16_ru(neg_lo_max / 63.0f);
    float dmin = or_f16_to_f32(dminh);

    uint8_t m[8], sc[8];
    float base[8], r[8];
    float r_max = 0.0f;
    for (int j = 0; j < 8; j++) {
        float mj = (dmin == 0.0f) ? 0.0f : ceilf(-lo[j] / dmin);
        if (mj > 63.0f) mj = 63.0f;
        m[j] = (uint8_t)mj;
        base[j] = -(dmin * mj);
        r[j] = hi[j] - base[j];
        if (r[j] > r_max) r_max = r[j];
    }
    uint16_t dh = or_f16_ru(r_max / (63.0f * qmax));
    float d = or_f16_to_f32(dh);
    for (int j = 0; j < 8; j++) {
        float s = (d == 0.0f) ? 0.0f : ceilf(r[j] / (qmax * d));
        if (s > 63.0f) s = 63.0f;
        sc[j] = (uint8_t)s;
    }
    for (int j = 0; j < 8; j++) {
        float step = d * (float)sc[j];
        for (int i = 0; i < 32; i++) {
            float v = (step == 0.0f) ? 0.0f
                      : clampf(rha((x[32 * j + i] - base[j]) / step), 0.0f, qmax);
            q[32 * j + i] = (uint8_t)v;
        }
    }
    *dh_out = dh;
    *dminh_out = dminh;
    for (int j = 0; j < 8; j++) { fields[j] = sc[j]; fields[8 + j] = m[j]; }
}

/* Q4_K: the fit with 4-bit codes; layout fp16 d @0, fp16 dmin @2, the
 * sixteen 6-bit fields @4, then byte l of the 128 code bytes holds element
 * 2l in its low nibble and 2l+1 in its high nibble. */
static void quantize_q4_k_block(const float *x, uint8_t *blk)
{
    uint16_t dh, dminh;
    uint8_t fields[16], q[256];
    k_asym_fit(x, 15.0f, &dh, &dminh, fields, q);
    put_u16(blk + 0, dh);
    put_u16(blk + 2, dminh);
    pack6(fields, blk + 4);
    for (int l = 0; l < 128; l++)
        blk[16 + l] = (uint8_t)(q[2 * l] | (q[2 * l + 1] << 4));
}

/* Q5_K: the 5-bit K-quant, one bit more than Q4_K (the discosf.com page
 * "为什么说 llama.cpp 是'裸引擎'——从模型加载的每一行代码说起", §4 量化不是"压缩"，
 * 而是"精度重分配": Q5_K_S carries one bit more than Q4_K_M).  The pages give
 * no layout; the reading taken is the Q4_K super-block and fit with codes
 * in [0, 31].  Layout (this library's own): the Q4_K fields and low four
 * bits of the codes in bytes 0..143 exactly as Q4_K, then 32 bytes @144 with
 * the fifth bits: byte 144 + 4j + i holds, in bit 2t + p, the fifth bit of
 * element 32j + 8t + 2i + p (sub-block j, t = 0..3, i = 0..3, p = 0..1). */
/* Writes a fitted Q5_K super-block: d, dmin, the fields, the low nibbles
 * and the fifth-bit plane. */
static void put_q5_k_block(uint16_t dh, uint16_t dminh, const uint8_t fields[16], const uint8_t q[256],
                           uint8_t *blk)
{
    put_u16(blk + 0, dh);
    put_u16(blk + 2, dminh);
    pack6(fields, blk + 4);
    for (int l = 0; l < 128; l++)
        blk[16 + l] = (uint8_t)((q[2 * l] & 15) | ((q[2 * l + 1] & 15) << 4));
    for (int k = 0; k < 32; k++) blk[144 + k] = 0;
    for (int e = 0; e < 256; e++) {
        int j = e / 32, t = (e % 32) / 8, i = (e % 8) / 2, p = e % 2;
        if (q[e] >> 4) blk[144 + 4 * j + i] |= (uint8_t)(1u << (2 * t + p));
    }
}

static void quantize_q5_k_block(const float *x, uint8_t *blk)
{
    uint16_t dh, dminh;
    uint8_t fields[16], q[256];
    k_asym_fit(x, 31.0f, &dh, &dminh, fields, q);
    put_q5_k_block(dh, dminh, fields, q, blk);
}

/* ------------------------------------------------------------------ */
/* Error-minimizing K-quant fit                                          */
/* ------------------------------------------------------------------ */

/* [P2] §5.5 stores each sub-block's scale and min as small integers under
 * the super-block's d and dmin, and §7.1 (with §3.3.3's llama-quantize
 * --imatrix) recommends a quantizer that chooses them to minimize the
 * weighted reconstruction error; the importance weights need calibration
 * data, so the reading taken here is the uniform-weight case: per sub-block,
 * the (sc, m) pair that minimizes the squared error of the 32 reconstructed
 * values.  Search space (this library's): d and dmin as the min/max fit sets
 * them, sc in [sc0 - 4, sc0 + 4] and m in [m0 - 4, m0 + 4] clipped to
 * [0, 63] around the min/max fit's pair (sc0, m0), each candidate's codes
 * the nearest in [0, qmax] (the fit's rounding rule).  The error of a
 * candidate is computed in fp32 in a fixed order -- element by element
 * within each eight-element group, then (g0 + g1) + (g2 + g3) -- so that any
 * implementation following it makes the same choice.  The first candidate
 * in (sc, m) ascending order whose error is strictly below the best so far
 * wins, starting from the min/max pair, so the result is never worse than
 * the min/max fit in this measure and stays in the same byte format. */
#define EM_WINDOW 4

static float em_sub_error(const float *x, float d, float dmin, int sc, int m, float qmax, uint8_t *q_out)
{
    float step = d * (float)sc;      /* exact */
    float base = -(dmin * (float)m); /* exact */
    float g[4];
    for (int t = 0; t < 4; t++) {
        float acc = 0.0f;
        for (int k = 0; k < 8; k++) {
            int i = 8 * t + k;
            float qv = (step == 0.0f) ? 0.0f : clampf(rha((x[i] - base) / step), 0.0f, qmax);
            float rec = step * qv + base;  /* the decoder's d*sc*q - dmin*m, rounded once */
            float e = x[i] - rec;
            acc = acc + e * e;
            if (q_out) q_out[i] = (uint8_t)qv;
        }
        g[t] = acc;
    }
    return (g[0] + g[1]) + (g[2] + g[3]);
}

/* Re-chooses sc_j, m_j and the codes of every sub-block of a fitted
 * super-block (fields and q as k_asym_fit wrote them) by the search above. */
static void em_refine(const float *x, float qmax, uint16_t dh, uint16_t dminh, uint8_t fields[16],
                      uint8_t q[256])
{
    float d = or_f16_to_f32(dh), dmin = or_f16_to_f32(dminh);
    for (int j = 0; j < 8; j++) {
        const float *xj = x + 32 * j;
        int sc0 = fields[j], m0 = fields[8 + j];
        int best_sc = sc0, best_m = m0;
        float best = em_sub_error(xj, d, dmin, sc0, m0, qmax, NULL);
        for (int sc = sc0 - EM_WINDOW; sc <= sc0 + EM_WINDOW; sc++) {
            if (sc < 0 || sc > 63) continue;
            for (int m = m0 - EM_WINDOW; m <= m0 + EM_WINDOW; m++) {
                if (m < 0 || m > 63) continue;
                float e = em_sub_error(xj, d, dmin, sc, m, qmax, NULL);
                if (e < best) {
                    best = e;
                    best_sc = sc;
                    best_m = m;
                }
            }
        }
        fields[j] = (uint8_t)best_sc;
        fields[8 + j] = (uint8_t)best_m;
        em_sub_error(xj, d, dmin, best_sc, best_m, qmax, q + 32 * j);
    }
}

/* The error-minimizing Q4_K / Q5_K encoders: the min/max fit, refined. */
static void quantize_k_errmin_block(int type, const float *x, uint8_t *blk)
{
    float qmax = (type == OR_Q4_K) ? 15.0f : 31.0f;
    uint16_t dh, dminh;
    uint8_t fields[16], q[256];
    k_asym_fit(x, qmax, &dh, &dminh, fields, q);
    em_refine(x, qmax, dh, dminh, fields, q);
    if (type == OR_Q5_K) {
        put_q5_k_block(dh, dminh, fields, q, blk);
        return;
    }
    put_u16(blk + 0, dh);
    put_u16(blk + 2, dminh);
    pack6(fields, blk + 4);
    for (int l = 0; l < 128; l++)
        blk[16 + l] = (uint8_t)((q[2 * l] & 15) | ((q[2 * l + 1] & 15) << 4));
}

/* Error-minimizing quantization of n elements of Q4_K or Q5_K (-1 for other
 * types or a bad n, -2 for non-finite input). */
int or_quantize_errmin(int type, const float *x, uint8_t *dst, int64_t n)
{
    if (type != OR_Q4_K && type != OR_Q5_K) return -1;
    int64_t bb = or_block_bytes(type);
    if (n < 0 || n % 256) return -1;
    if (!all_finite(x, n)) return -2;
    for (int64_t b = 0; b < n / 256; b++) quantize_k_errmin_block(type, x + b * 256, dst + b * bb);
    return 0;
}

/* The stored code of element e of a Q4_K (0..15) or Q5_K (0..31) block. */
static int k_code(int type, const uint8_t *blk, int e)
{
    int byte = blk[16 + e / 2];
    int q = (e & 1) ? (byte >> 4) : (byte & 0x0f);
    if (type == OR_Q5_K) {
        int j = e / 32, t = (e % 32) / 8, i = (e % 8) / 2, p = e % 2;
        q |= ((blk[144 + 4 * j + i] >> (2 * t + p)) & 1) << 4;
    }
    return q;
}

/* Q8_K: the 256-element activation block.  Same symmetric rule as Q8_0 but
 * the scale stays fp32, and the eight 32-element sums of the codes are
 * stored so that the Q4_K min term needs no second pass over the codes. */
static void quantize_q8_k_block(const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < 256; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    put_f32(blk, d);
    int8_t q[256];
    for (int i = 0; i < 256; i++) {
        float v = (d == 0.0f) ? 0.0f : clampf(rha(x[i] / d), -127.0f, 127.0f);
        q[i] = (int8_t)v;
        blk[4 + i] = (uint8_t)q[i];
    }
    for (int j = 0; j < 8; j++) {
        int s = 0;
        for (int i = 0; i < 32; i++) s += q[32 * j + i];
        put_u16(blk + 260 + 2 * j, (uint16_t)(int16_t)s);
    }
}

/* Q6_K: the 6-bit K-quant as the discosf.com page ("为什么说 llama.cpp
 * 是'裸引擎'——从模型加载的每一行代码说起", §4 量化不是"压缩"，而是"精度重分配")
 * describes it: K blocks only (256 elements, the K-quant block of [P4]
 * 第二层：量化引擎), no sub-blocks, 6-bit main quantization.  The pages give
 * no formula or layout; the reading taken is the symmetric rule of [P2]
 * §5.1 with b = 6 (scale = max|x| / 31, fp16
 * rounded to nearest-even, the same pattern as Q4_0 with b = 4), codes
 * q = round(x / d) clamped to [-32, 31] and stored as c = q + 32 in [0, 63].
 * Packing (this library's own): byte l of the 128-byte low part holds the low
 * four bits of element 2l (low nibble) and 2l+1 (high nibble), the Q4_0 / Q4_K
 * order; byte l of the 64-byte high part holds the top two bits of elements
 * 4l..4l+3, element 4l+k in bits 2k..2k+1.  w = d * (c - 32). */
static void quantize_q6_k_block(const float *x, uint8_t *blk)
{
    float amax = 0.0f;
    for (int i = 0; i < 256; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    uint16_t dh = or_f16_rn(amax / 31.0f);
    float d = or_f16_to_f32(dh);
    put_u16(blk, dh);
    uint8_t c[256];
    for (int i = 0; i < 256; i++) {
        float q = (d == 0.0f) ? 0.0f : clampf(rha(x[i] / d), -32.0f, 31.0f);
        c[i] = (uint8_t)((int)q + 32);
    }
    for (int l = 0; l < 128; l++)
        blk[2 + l] = (uint8_t)((c[2 * l] & 15) | ((c[2 * l + 1] & 15) << 4));
    for (int l = 0; l < 64; l++) {
        int h = 0;
        for (int k = 0; k < 4; k++) h |= (c[4 * l + k] >> 4) << (2 * k);
        blk[130 + l] = (uint8_t)h;
    }
}

/* The stored 6-bit code of element e of a Q6_K block (0..63). */
static int q6_k_code(const uint8_t *blk, int e)
{
    int lo = (e & 1) ? (blk[2 + e / 2] >> 4) : (blk[2 + e / 2] & 15);
    int hi = (blk[130 + e / 4] >> (2 * (e & 3))) & 3;
    return lo | (hi << 4);
}

int or_quantize(int type, const float *x, uint8_t *dst, int64_t n)
{
    int64_t be = or_block_elems(type), bb = or_block_bytes(type);
    if (be <= 0 || n < 0 || n % be) return -1;
    if (!all_finite(x, n)) return -2;
    for (int64_t b = 0; b < n / be; b++) {
        const float *xb = x + b * be;
        uint8_t *ob = dst + b * bb;
        switch (type) {
        case OR_Q4_0: quantize_q4_0_block(xb, ob); break;
        case OR_Q8_0: quantize_q8_0_block(xb, ob); break;
        case OR_Q4_K: quantize_q4_k_block(xb, ob); break;
        case OR_Q8_K: quantize_q8_k_block(xb, ob); break;
        case OR_Q6_K: quantize_q6_k_block(xb, ob); break;
        case OR_Q5_K: quantize_q5_k_block(xb, ob); break;
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ */
/* Decoders                                                             */
/* ------------------------------------------------------------------ */

/* Per-element reconstruction of one block, exact in double:
 *   Q4_0: d * (c - 8)      Q8_0, Q8_K: d * q
 *   Q4_K, Q5_K: d*sc_j*q - dmin*m_j      Q6_K: d * (c - 32)
 * Every product of an fp16 (or fp32) scale with these small integers, and
 * the Q4_K difference, fits in the 53-bit double significand. */
static void decode_block_f64(int type, const uint8_t *blk, double *out)
{
    switch (type) {
    case OR_Q4_0: {
        double d = or_f16_to_f32(get_u16(blk));
        for (int j = 0; j < 16; j++) {
            out[2 * j] = d * (double)((blk[2 + j] & 0x0f) - 8);
            out[2 * j + 1] = d * (double)((blk[2 + j] >> 4) - 8);
        }
        break;
    }
    case OR_Q8_0: {
        double d = or_f16_to_f32(get_u16(blk));
        for (int i = 0; i < 32; i++) out[i] = d * (double)(int8_t)blk[2 + i];
        break;
    }
    case OR_Q4_K: case OR_Q5_K: {
        double d = or_f16_to_f32(get_u16(blk + 0));
        double dmin = or_f16_to_f32(get_u16(blk + 2));
        uint8_t f[16];
        unpack6(blk + 4, f);
        for (int e = 0; e < 256; e++) {
            int j = e / 32;
            int q = k_code(type, blk, e);
            out[e] = d * (double)f[j] * (double)q - dmin * (double)f[8 + j];
        }
        break;
    }
    case OR_Q8_K: {
        double d = get_f32(blk);
        for (int i = 0; i < 256; i++) out[i] = d * (double)(int8_t)blk[4 + i];
        break;
    }
    case OR_Q6_K: {
        double d = or_f16_to_f32(get_u16(blk));
        for (int e = 0; e < 256; e++) out[e] = d * (double)(q6_k_code(blk, e) - 32);
        break;
    }
    }
}

/* The fp32 reconstruction is the exact value rounded once to fp32 (for
 * Q4_0, Q8_0 and Q8_K the exact value is already an fp32 number). */
static void decode_block(int type, const uint8_t *blk, float *out)
{
    double tmp[256];
    decode_block_f64(type, blk, tmp);
    for (int i = 0; i < or_block_elems(type); i++) out[i] = (float)tmp[i];
}

int or_dequantize_f64(int type, const uint8_t *src, double *dst, int64_t n)
{
    int64_t be = or_block_elems(type), bb = or_block_bytes(type);
    if (be <= 0 || n < 0 || n % be) return -1;
    for (int64_t b = 0; b < n / be; b++) decode_block_f64(type, src + b * bb, dst + b * be);
    return 0;
}

int or_dequantize(int type, const uint8_t *src, float *dst, int64_t n)
{
    int64_t be = or_block_elems(type), bb = or_block_bytes(type);
    if (be <= 0 || n < 0 || n % be) return -1;
    for (int64_t b = 0; b < n / be; b++) decode_block(type, src + b * bb, dst + b * be);
    return 0;
}

/* ------------------------------------------------------------------ */
/* The product                                                          */
/* ------------------------------------------------------------------ */

static int pairing_ok(int wtype, int *atype)
{
    switch (wtype) {
    case OR_Q4_0: case OR_Q8_0: *atype = OR_Q8_0; return 1;
    case OR_Q4_K: case OR_Q6_K: case OR_Q5_K: *atype = OR_Q8_K; return 1;
    }
    return 0;
}

/* Integer dot of one weight block against one activation block.
 *   Q4_0 x Q8_0: s = sum_i (c_i - 8) * a_i          ([P2] §6.4)
 *   Q8_0 x Q8_0: s = sum_i w_i * a_i
 *   Q4_K x Q8_K (and Q5_K x Q8_K):
 *                s_j = sum_{i in j} q_i * a_i per sub-block,
 *                S1 = sum_j sc_j * s_j,  S2 = sum_j m_j * t_j
 *                with t_j the activation sub-block sum (stored bsums).
 *   Q6_K x Q8_K: s = sum_i (c_i - 32) * a_i over the 256 elements.
 * out[0] (and out[1] for Q4_K) receive the sums; returns the number written. */
static int block_int_dot(int wtype, const uint8_t *w, const uint8_t *a, int32_t *out)
{
    if (wtype == OR_Q6_K) {
        int32_t s = 0;
        for (int e = 0; e < 256; e++) s += (q6_k_code(w, e) - 32) * (int8_t)a[4 + e];
        out[0] = s;
        return 1;
    }
    if (wtype == OR_Q4_0) {
        int32_t s = 0;
        for (int j = 0; j < 16; j++) {
            int v0 = (w[2 + j] & 0x0f) - 8;
            int v1 = (w[2 + j] >> 4) - 8;
            s += v0 * (int8_t)a[2 + 2 * j] + v1 * (int8_t)a[2 + 2 * j + 1];
        }
        out[0] = s;
        return 1;
    }
    if (wtype == OR_Q8_0) {
        int32_t s = 0;
        for (int i = 0; i < 32; i++) s += (int8_t)w[2 + i] * (int8_t)a[2 + i];
        out[0] = s;
        return 1;
    }
    /* Q4_K / Q5_K x Q8_K */
    uint8_t f[16];
    unpack6(w + 4, f);
    int32_t S1 = 0, S2 = 0;
    for (int j = 0; j < 8; j++) {
        int32_t s = 0;
        for (int i = 0; i < 32; i++) {
            int e = 32 * j + i;
            s += k_code(wtype, w, e) * (int8_t)a[4 + e];
        }
        int16_t t = (int16_t)get_u16(a + 260 + 2 * j);
        S1 += (int32_t)f[j] * s;
        S2 += (int32_t)f[8 + j] * (int32_t)t;
    }
    out[0] = S1;
    out[1] = S2;
    return 2;
}

/* Per-block integer sums of the whole product.
 * Layout: out[b][r][k][c] with k over the weight blocks of a row and
 * c = 1 (Q4_0, Q8_0, Q6_K) or 2 (Q4_K, Q5_K: S1, S2). */
int or_block_sums(int wtype, const uint8_t *W, const uint8_t *xq, int64_t rows,
                  int64_t cols, int64_t batch, int32_t *out)
{
    int atype;
    if (!pairing_ok(wtype, &atype)) return -1;
    int64_t be = or_block_elems(wtype);
    if (rows < 0 || batch < 0 || cols < 0 || cols % be) return -1;
    int64_t nb = cols / be, wbb = or_block_bytes(wtype), abb = or_block_bytes(atype);
    int c = (wtype == OR_Q4_K || wtype == OR_Q5_K) ? 2 : 1;
    for (int64_t b = 0; b < batch; b++)
        for (int64_t r = 0; r < rows; r++)
            for (int64_t k = 0; k < nb; k++)
                block_int_dot(wtype, W + (r * nb + k) * wbb, xq + (b * nb + k) * abb,
                              out + ((b * rows + r) * nb + k) * c);
    return 0;
}

/* Scale terms of one block pair in double:
 *   Q4_0 / Q8_0: d_w * d_x * s      (d_x the fp16 Q8_0 scale)
 *   Q6_K:        d_w * d_x * s      (d_x the fp32 Q8_K scale)
 *   Q4_K, Q5_K:  d_x * d * S1   and   -(d_x * dmin * S2)
 * y accumulates the terms, T their absolute values. */
static void block_terms(int wtype, const uint8_t *w, const uint8_t *a, double *y, double *T)
{
    int32_t s[2];
    block_int_dot(wtype, w, a, s);
    if (wtype == OR_Q4_K || wtype == OR_Q5_K) {
        double dx = get_f32(a);
        double d = or_f16_to_f32(get_u16(w + 0));
        double dmin = or_f16_to_f32(get_u16(w + 2));
        double t1 = dx * d * (double)s[0];
        double t2 = -(dx * dmin * (double)s[1]);
        *y += t1 + t2;
        *T += fabs(t1) + fabs(t2);
    } else if (wtype == OR_Q6_K) {
        double dw = or_f16_to_f32(get_u16(w));
        double dx = get_f32(a);
        double t = dw * dx * (double)s[0];
        *y += t;
        *T += fabs(t);
    } else {
        double dw = or_f16_to_f32(get_u16(w));
        double dx = or_f16_to_f32(get_u16(a));
        double t = dw * dx * (double)s[0];
        *y += t;
        *T += fabs(t);
    }
}

/* y[b][r] = sum over the row's blocks of the scaled block terms, in double;
 * T[b][r] = sum of their magnitudes (the tolerance scale).  nthreads > 0
 * splits the rows across that many OpenMP threads (0 = one thread). */
int or_matmul_ref(int wtype, const uint8_t *W, const uint8_t *xq, int64_t rows,
                  int64_t cols, int64_t batch, double *y, double *T, int nthreads)
{
    int atype;
    if (!pairing_ok(wtype, &atype)) return -1;
    int64_t be = or_block_elems(wtype);
    if (rows < 0 || batch < 0 || cols < 0 || cols % be) return -1;
    int64_t nb = cols / be, wbb = or_block_bytes(wtype), abb = or_block_bytes(atype);
    int nt = nthreads > 0 ? nthreads : 1;
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        for (int64_t b = 0; b < batch; b++) {
            double acc = 0.0, tol = 0.0;
            for (int64_t k = 0; k < nb; k++)
                block_terms(wtype, W + (r * nb + k) * wbb, xq + (b * nb + k) * abb, &acc, &tol);
            y[b * rows + r] = acc;
            if (T) T[b * rows + r] = tol;
        }
    }
    return 0;
}

/* Whole-row quantization across OpenMP threads, for timing the CPU baseline
 * on larger inputs (rows of `cols` elements each). */
int or_quantize_rows_mt(int type, const float *x, uint8_t *dst, int64_t rows, int64_t cols,
                        int nthreads)
{
    int64_t be = or_block_elems(type), bb = or_block_bytes(type);
    if (be <= 0 || rows < 0 || cols % be) return -1;
    int nt = nthreads > 0 ? nthreads : 1;
    int err = 0;
    (void)nt;
#pragma omp parallel for num_threads(nt) schedule(static) reduction(| : err)
    for (int64_t r = 0; r < rows; r++)
        err |= or_quantize(type, x + r * cols, dst + r * (cols / be) * bb, cols) != 0;
    return err ? -1 : 0;
}

int or_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
