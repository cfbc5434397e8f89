/*
 * bq_oracle.c — plain, slow, scalar CPU oracle for block-quantized weight rows.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg; never by the product path. It shares no code
 * with the CUDA library (no headers, helpers, tables or constants).
 *
 * Build: plain C11, no SIMD intrinsics, no fast-math, no FP contraction
 * (see oracle/build.py), so every float operation below is one IEEE
 * binary32 (or binary64 where stated) operation in program order.
 *
 * Sources (pages on llama.cpp; citations give page title and section):
 *   [FMT4] llama.cpp 原理：如何在普通硬件跑本地大模型, §量化：内存真正去哪了 —
 *          Q4_0: groups of 32 weights, one FP16 scale, each weight a 4-bit
 *          integer; 18 bytes per 32 weights, 4.5 bits per weight.
 *   [FMT8] 05. llama.cpp：从 GGUF 文件到本地推理服务, §量化类型：Q4_K_M 到底是什么,
 *          format table — legacy types: one FP16 scale per 32 weights; Q8_0
 *          about 8.5 bits per weight.
 *   [SYM]  lpnh.cn KV-cache article, §kv-mean-center 进阶技巧 / §问题 — Q4_0 is a
 *          symmetric block format, value ≈ scale × q, with no zero point.
 *   [ROOF] 05. llama.cpp…, §性能直觉：带宽决定 Decode，算力决定 Prefill — decode
 *          reads every weight once per token (GEMV); prefill reuses weights
 *          across many tokens (GEMM).
 *   [KVMC] lpnh.cn KV-cache article, §解法 and §适用边界 — a per-(kv-head,
 *          channel) bias is subtracted from K before Q4_0 quantization; any
 *          other K type is rejected.
 *   [DEQ]  xdnf.cn/news/348240, §2.2 — names dequantize_row_q4_0.
 *   [FA]   05. llama.cpp…, §KV Cache 类型与 Flash Attention, and the lpnh.cn
 *          KV-cache article, §量化 KV Cache 的一键配置方法 — K and V caches take
 *          q8_0 / q4_0; a quantized V cache is read by flash attention, which
 *          computes attention in one pass without the intermediate matrix.
 *   [SHIFT] lpnh.cn KV-cache article, §解法 — q·k_i = q·(k_i − k̄) + q·k̄, and
 *          softmax is unchanged by a constant added to a whole row.
 *   [LEG]  05. llama.cpp…, §量化类型, format table — legacy formats (Q4_0,
 *          Q5_1, Q8_0) group 32 weights with one FP16 scale, and the "_1"
 *          types add a minimum; §KV Cache 类型与 Flash Attention lists q4_1,
 *          q5_0 and q5_1 among the K/V cache types.
 *   [KQ]   05. llama.cpp…, §量化类型, format table — k-quants use super-blocks
 *          of 256 weights holding 8 sub-blocks of 32, whose scales are
 *          themselves quantized with 6 bits; the Llama-3-8B table prints Q8_0
 *          7.96 GiB and Q6_K 6.14 GiB for the same model.
 *   [ROT]  lpnh.cn KV-cache article, §三步上手 (third step) — a quantized K
 *          cache whose head dimension is a multiple of 64 is Hadamard-rotated;
 *          the mean-centering bias must be measured in the same basis as the
 *          cache, the calibration records its basis, and a mismatch fails
 *          fast instead of degrading quietly.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   R1 scale first, little-endian fp16, then the codes;
 *   R2 Q4_0 nibble order: low nibbles hold elements 0..15, high nibbles 16..31,
 *      stored unsigned as q + 8;
 *   R3 scale d = amax / 7 (Q4_0) or amax / 127 (Q8_0), fp32 IEEE division,
 *      rounded to fp16 ties-to-even;
 *   R4 codes q = clamp(round_half_even(x / d16), -8, 7) (Q4_0) or
 *      clamp(..., -127, 127) (Q8_0), dividing by the *stored* fp16 scale;
 *      d16 == 0 gives all codes 0;
 *   R5 activations are quantized to Q8_0 with R3/R4 before the integer dot;
 *   R6 float results are the fp64 sum of exact per-block terms, rounded once
 *      to fp32;
 *   R11 attention is scaled dot-product attention over the dequantized cache,
 *      o_h = sum_t softmax_t(scale q_h . k_t) v_t, query head h reading kv head
 *      h / (n_heads / n_kv_heads); the scale is the caller's;
 *   R12 q . k_t is the block dot of R5/R6: q quantized to Q8_0 per block of
 *      32 channels, the integer dot with K's codes times dk dq.
 *   R14 the rotation is orthonormal and block diagonal: every group of 64
 *      consecutive channels of a head is replaced by H64 x / 8, H64 the
 *      Sylvester-ordered Walsh-Hadamard matrix, H64[i][j] = (-1)^popcount(i&j)
 *      (the pages require head_dim % 64 == 0 and name no size or scaling).
 *      Only K is rotated; q is rotated the same way, so q.k is unchanged.
 *   R16 legacy layouts (the pages give none): Q4_1 = {fp16 d, fp16 m,
 *      16 nibble bytes} (20 bytes), Q5_0 = {fp16 d, 32-bit qh, 16 nibble
 *      bytes} (22), Q5_1 = {fp16 d, fp16 m, qh, 16 nibble bytes} (24); all
 *      little endian; the low 4 bits of code j sit as in R2 (byte j % 16,
 *      low nibble for j < 16), bit 4 of code j is bit j of qh; codes are
 *      stored unsigned u (Q5_0: u = q + 16).
 *   R17 Q5_0 is symmetric like Q4_0: d = amax / 15, q = clamp(round_half_even
 *      (x / d16), -16, 15); value d16 * q.
 *   R18 the "_1" types are affine: m = min_j x_j, d = (max_j x_j - m) /
 *      (2^bits - 1) in fp32, both stored as fp16; u = clamp(round_half_even(
 *      (x - m16) / d16), 0, 2^bits - 1) with one fp32 subtraction and one
 *      fp32 division by the stored values; d16 == 0 gives u = 0; value
 *      d16 * u + m16 (fp32 product, then fp32 sum).
 *   R19 the dot of an affine weight block with a Q8_0 block is
 *      d_w d_x sum_j u_j qx_j + m_w d_x sum_j qx_j, summed in fp64 (R6).
 *   R20 Q4_K layout (PARITY UNPINNED beyond its size): 144 bytes per 256
 *      weights = { fp16 d, fp16 dmin, 12 bytes holding 6-bit sub-block
 *      scales sc[0..7] then 6-bit sub-block minimums mn[0..7] as one
 *      little-endian 96-bit stream (value k at bits 6k..6k+5), 128 bytes of
 *      4-bit codes: sub-block j in bytes 16j..16j+15, Q4_0's nibble order };
 *      value (d sc_j) u - (dmin mn_j), the two sub-block factors rounded to
 *      fp32, then the fp32 product and the fp32 difference.
 *   R21 Q4_K quantizer (PARITY UNPINNED; the pages give no algorithm): per
 *      sub-block m_j = max(0, -min x), s_j = (max x + m_j) / 15; d = max_j s_j
 *      / 63, dmin = max_j m_j / 63 (fp32, stored fp16); sc_j = clamp(rn(s_j
 *      / d16), 0, 63), mn_j = clamp(rn(m_j / dmin16), 0, 63); S_j = fp32(d16
 *      sc_j), M_j = fp32(dmin16 mn_j); u = clamp(rn((x + M_j) / S_j), 0,
 *      15), one fp32 sum and one fp32 division (S_j = 0 gives u = 0).
 *   R22 Q6_K layout (size pinned by the Llama-3-8B table): 210 bytes per
 *      256 weights = { 128 bytes ql: byte i holds the low 4 bits of code i
 *      (low nibble) and of code i + 128 (high nibble); 64 bytes qh: byte i
 *      holds the top 2 bits of codes i, i+64, i+128, i+192 at bits 0-1, 2-3,
 *      4-5, 6-7; int8 scales sc[0..15] of the 16 sub-blocks of 16; fp16 d };
 *      value fp32(d sc_k) * (u - 32), u in 0..63.
 *   R23 Q6_K quantizer (PARITY UNPINNED): per sub-block of 16 s_k = amax /
 *      31; d = max_k s_k / 127; sc_k = clamp(rn(s_k / d16), -128, 127);
 *      S_k = fp32(d16 sc_k); u = clamp(rn(x / S_k), -32, 31) + 32.
 *   R24 k-quant GEMV: x quantized to Q8_0 as always (R5); a super-block
 *      meets the 8 x blocks under it; the terms d_x S sum(u qx) (and
 *      - d_x M sum(qx) for Q4_K; Q6_K: S per half of an x block, codes u - 32)
 *      are exact and summed in fp64 (R6).
 *   R15 the rotated values decide integer codes, so they are computed in the
 *      kernel's precision: the fast Walsh-Hadamard butterflies in fp32,
 *      stages of span 1, 2, 4, 8, 16, 32, each pair (a, b) -> (a + b, a - b),
 *      then the exact scaling by 1/8 (pinned against the fp64 matrix
 *      product of the definition). The calibrated bias is the fp64 mean over
 *      the tokens, in token order, of the rotated fp32 rows, stored as fp32.
 *
 * Parity pins (tests/test_oracle_pins.py): block sizes; hand-worked blocks
 * (tests/golden/); fp16 conversion against numpy's binary16; ties; the
 * round-trip bound |x - x_hat| <= d16/2 (1 + 2^-18); brute-force fp64 dot
 * products of dequantized operands; integer block dots against an int64 loop;
 * bias subtraction against numpy subtraction; softmax shift invariance; the
 * rotation against the fp64 matrix product of H64's definition, its columns,
 * norm preservation and self-inverse; calibration against numpy means and
 * against the rotation of the plain mean (linearity).
 */
#include "bq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define QK 32

static int is_kquant(int type) { return type == ORACLE_TYPE_Q4_K || type == ORACLE_TYPE_Q6_K; }

int64_t oracle_block_values(int type)
{
    if (is_kquant(type)) return 256; /* [KQ] super-blocks of 256 weights */
    return oracle_block_bytes(type) ? QK : 0;
}

int64_t oracle_block_bytes(int type)
{
    if (type == ORACLE_TYPE_Q4_K) return 2 + 2 + 12 + 128; /* R20 */
    if (type == ORACLE_TYPE_Q6_K) return 128 + 64 + 16 + 2; /* R22 */
    /* [FMT4] 18 bytes per 32 Q4_0 weights; [FMT8] 2-byte scale + 32 int8. */
    if (type == ORACLE_TYPE_Q4_0) return 2 + QK / 2;
    if (type == ORACLE_TYPE_Q8_0) return 2 + QK;
    /* [LEG] + R16: scale, (minimum,) (high bits,) nibbles */
    if (type == ORACLE_TYPE_Q4_1) return 2 + 2 + QK / 2;
    if (type == ORACLE_TYPE_Q5_0) return 2 + 4 + QK / 2;
    if (type == ORACLE_TYPE_Q5_1) return 2 + 2 + 4 + QK / 2;
    return 0;
}

/* ---- IEEE binary16 conversion, written from the format definition ---- */

uint16_t oracle_f32_to_f16(float f)
{
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    uint16_t sign = (uint16_t)((x >> 16) & 0x8000u);
    uint32_t ex = (x >> 23) & 0xFFu;
    uint32_t man = x & 0x7FFFFFu;

    if (ex == 0xFFu) /* inf stays inf, NaN stays a quiet NaN */
        return (uint16_t)(sign | 0x7C00u | (man ? 0x0200u : 0u));
    if (ex == 0u) /* binary32 subnormals are below half the smallest binary16 subnormal */
        return sign;

    /* value = sig * 2^(ex - 150), sig has 24 significant bits */
    uint32_t sig = man | 0x800000u;
    int32_t e16 = (int32_t)ex - 127 + 15; /* biased binary16 exponent if normal */
    if (e16 >= 31)
        return (uint16_t)(sign | 0x7C00u);

    /* normal: keep 11 significant bits; subnormal: value / 2^-24 */
    uint32_t shift = (e16 >= 1) ? 13u : (uint32_t)(13 + 1 - e16);
    if (shift >= 25u) /* below half of 2^-24 (ties included, they go to even 0) */
        return sign;

    uint32_t q = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1u);
    if (rem > half || (rem == half && (q & 1u)))
        q++;

    if (e16 >= 1) {
        uint32_t e = (uint32_t)e16;
        if (q == 0x800u) { /* rounding carried into the next binade */
            q = 0x400u;
            e++;
        }
        if (e >= 31u)
            return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | (e << 10) | (q & 0x3FFu));
    }
    /* subnormal result; q == 0x400 is exactly the smallest normal, encoded as is */
    return (uint16_t)(sign | q);
}

float oracle_f16_to_f32(uint16_t h)
{
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = ((uint32_t)h >> 10) & 0x1Fu;
    uint32_t m = (uint32_t)h & 0x3FFu;
    uint32_t x;
    if (e == 0u) {
        /* subnormal (or zero): m * 2^-24, exact in binary32 */
        float v = (float)m * 5.9604644775390625e-08f;
        return sign ? -v : v;
    }
    if (e == 31u)
        x = sign | 0x7F800000u | (m << 13);
    else
        x = sign | ((e + 112u) << 23) | (m << 13);
    float f;
    memcpy(&f, &x, sizeof f);
    return f;
}

float oracle_round_half_even(float v)
{
    /* nearbyintf rounds in the current mode, which is the default
     * round-to-nearest-even: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2, -0.5 -> -0. */
    return nearbyintf(v);
}

/* ---- one block of a legacy type: R16, R17, R18 ---- */

static int legacy_bits(int type) { return type == ORACLE_TYPE_Q4_1 ? 4 : 5; }
static int legacy_affine(int type) { return type != ORACLE_TYPE_Q5_0; }
static int is_legacy(int type)
{
    return type == ORACLE_TYPE_Q4_1 || type == ORACLE_TYPE_Q5_0 || type == ORACLE_TYPE_Q5_1;
}

static void put_u16(uint8_t *p, uint16_t v)
{
    p[0] = (uint8_t)(v & 0xFFu);
    p[1] = (uint8_t)(v >> 8);
}

static void quantize_block_legacy(int type, const float *x, uint8_t *out)
{
    const int umax = (1 << legacy_bits(type)) - 1;
    int u[QK];
    uint16_t d16, m16 = 0;
    if (legacy_affine(type)) {
        float mn = x[0], mx = x[0];
        for (int j = 1; j < QK; j++) {
            if (x[j] < mn) mn = x[j];
            if (x[j] > mx) mx = x[j];
        }
        float d = (mx - mn) / (float)umax; /* R18 */
        d16 = oracle_f32_to_f16(d);
        m16 = oracle_f32_to_f16(mn);
        float ds = oracle_f16_to_f32(d16), ms = oracle_f16_to_f32(m16);
        for (int j = 0; j < QK; j++) {
            int v = 0;
            if (ds != 0.0f)
                v = (int)oracle_round_half_even((x[j] - ms) / ds);
            if (v > umax) v = umax;
            if (v < 0) v = 0;
            u[j] = v;
        }
    } else {
        float amax = 0.0f;
        for (int j = 0; j < QK; j++)
            if (fabsf(x[j]) > amax) amax = fabsf(x[j]);
        float d = amax / 15.0f; /* R17 */
        d16 = oracle_f32_to_f16(d);
        float ds = oracle_f16_to_f32(d16);
        for (int j = 0; j < QK; j++) {
            int v = 0;
            if (ds != 0.0f)
                v = (int)oracle_round_half_even(x[j] / ds);
            if (v > 15) v = 15;
            if (v < -16) v = -16;
            u[j] = v + 16;
        }
    }
    int o = 2;
    put_u16(out, d16);
    if (legacy_affine(type)) {
        put_u16(out + 2, m16);
        o = 4;
    }
    if (legacy_bits(type) == 5) {
        uint32_t qh = 0;
        for (int j = 0; j < QK; j++)
            qh |= (uint32_t)((u[j] >> 4) & 1) << j;
        for (int k = 0; k < 4; k++)
            out[o + k] = (uint8_t)(qh >> (8 * k));
        o += 4;
    }
    for (int j = 0; j < QK / 2; j++)
        out[o + j] = (uint8_t)((unsigned)(u[j] & 15) | ((unsigned)(u[j + QK / 2] & 15) << 4));
}

/* ---- one block: R3 + R4 ---- */

static void quantize_block(int type, const float *x, uint8_t *out)
{
    if (is_legacy(type)) {
        quantize_block_legacy(type, x, out);
        return;
    }
    const int qmax = (type == ORACLE_TYPE_Q4_0) ? 7 : 127;
    const int qmin = (type == ORACLE_TYPE_Q4_0) ? -8 : -127;

    float amax = 0.0f;
    for (int j = 0; j < QK; j++) {
        float a = fabsf(x[j]);
        if (a > amax)
            amax = a;
    }
    float d = amax / (float)qmax;           /* R3: one IEEE binary32 division */
    uint16_t d16 = oracle_f32_to_f16(d);    /* R3: stored scale */
    float ds = oracle_f16_to_f32(d16);      /* R4: quantize with the stored scale */

    int q[QK];
    for (int j = 0; j < QK; j++) {
        if (ds == 0.0f) {
            q[j] = 0;
            continue;
        }
        float r = oracle_round_half_even(x[j] / ds);
        int v = (int)r;
        if (v > qmax) v = qmax;
        if (v < qmin) v = qmin;
        q[j] = v;
    }

    out[0] = (uint8_t)(d16 & 0xFFu); /* R1: little-endian scale first */
    out[1] = (uint8_t)(d16 >> 8);
    if (type == ORACLE_TYPE_Q4_0) {
        for (int j = 0; j < QK / 2; j++) /* R2 */
            out[2 + j] = (uint8_t)((unsigned)(q[j] + 8) | ((unsigned)(q[j + QK / 2] + 8) << 4));
    } else {
        for (int j = 0; j < QK; j++)
            out[2 + j] = (uint8_t)(int8_t)q[j];
    }
}

static float block_scale(const uint8_t *blk)
{
    uint16_t d16 = (uint16_t)(blk[0] | ((uint16_t)blk[1] << 8));
    return oracle_f16_to_f32(d16);
}

/* the stored minimum of an affine block (R18), 0 for the symmetric types */
static float block_min(int type, const uint8_t *blk)
{
    if (!is_legacy(type) || !legacy_affine(type))
        return 0.0f;
    return oracle_f16_to_f32((uint16_t)(blk[2] | ((uint16_t)blk[3] << 8)));
}

/* codes of one block as plain ints, R2 inverted; affine types give u,
 * Q5_0 gives u - 16 (R16-R18) */
static void block_codes(int type, const uint8_t *blk, int *q)
{
    if (is_legacy(type)) {
        int o = legacy_affine(type) ? 4 : 2;
        uint32_t qh = 0;
        if (legacy_bits(type) == 5) {
            qh = (uint32_t)blk[o] | ((uint32_t)blk[o + 1] << 8) | ((uint32_t)blk[o + 2] << 16) |
                 ((uint32_t)blk[o + 3] << 24);
            o += 4;
        }
        for (int j = 0; j < QK; j++) {
            unsigned lo = (j < QK / 2) ? (blk[o + j] & 0x0Fu) : (unsigned)(blk[o + j - QK / 2] >> 4);
            int u = (int)(lo | (((qh >> j) & 1u) << 4));
            q[j] = legacy_affine(type) ? u : u - 16;
        }
        return;
    }
    if (type == ORACLE_TYPE_Q4_0) {
        for (int j = 0; j < QK / 2; j++) {
            q[j] = (int)(blk[2 + j] & 0x0Fu) - 8;
            q[j + QK / 2] = (int)(blk[2 + j] >> 4) - 8;
        }
    } else {
        for (int j = 0; j < QK; j++)
            q[j] = (int)(int8_t)blk[2 + j];
    }
}

/* ---- k-quant super-blocks: R20-R24 ---- */

static int clampi(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

static void q4k_get(const uint8_t *blk, int *sc, int *mn)
{
    uint64_t lo = 0, hi = 0; /* the 96-bit stream in bytes 4..15 */
    for (int k = 0; k < 8; k++) lo |= (uint64_t)blk[4 + k] << (8 * k);
    for (int k = 0; k < 4; k++) hi |= (uint64_t)blk[12 + k] << (8 * k);
    for (int k = 0; k < 16; k++) {
        int bit = 6 * k, v;
        if (bit + 6 <= 64) v = (int)((lo >> bit) & 63u);
        else if (bit >= 64) v = (int)((hi >> (bit - 64)) & 63u);
        else v = (int)(((lo >> bit) | (hi << (64 - bit))) & 63u);
        if (k < 8) sc[k] = v; else mn[k - 8] = v;
    }
}

static void q4k_put(uint8_t *blk, const int *sc, const int *mn)
{
    uint64_t lo = 0, hi = 0;
    for (int k = 0; k < 16; k++) {
        uint64_t v = (uint64_t)(k < 8 ? sc[k] : mn[k - 8]);
        int bit = 6 * k;
        if (bit + 6 <= 64) lo |= v << bit;
        else if (bit >= 64) hi |= v << (bit - 64);
        else { lo |= v << bit; hi |= v >> (64 - bit); }
    }
    for (int k = 0; k < 8; k++) blk[4 + k] = (uint8_t)(lo >> (8 * k));
    for (int k = 0; k < 4; k++) blk[12 + k] = (uint8_t)(hi >> (8 * k));
}

/* sub-block factors of a Q4_K super-block, as the fp32 values R20 uses */
static void q4k_factors(const uint8_t *blk, float *S, float *M)
{
    int sc[8], mn[8];
    q4k_get(blk, sc, mn);
    float d = oracle_f16_to_f32((uint16_t)(blk[0] | (blk[1] << 8)));
    float dm = oracle_f16_to_f32((uint16_t)(blk[2] | (blk[3] << 8)));
    for (int j = 0; j < 8; j++) {
        S[j] = d * (float)sc[j];
        M[j] = dm * (float)mn[j];
    }
}

static void quantize_q4k(const float *x, uint8_t *out)
{
    float s[8], m[8], smax = 0.0f, mmax = 0.0f;
    for (int j = 0; j < 8; j++) {
        float lo = x[32 * j], hi = x[32 * j];
        for (int i = 1; i < 32; i++) {
            if (x[32 * j + i] < lo) lo = x[32 * j + i];
            if (x[32 * j + i] > hi) hi = x[32 * j + i];
        }
        m[j] = lo < 0.0f ? -lo : 0.0f;
        s[j] = (hi + m[j]) / 15.0f;
        if (s[j] > smax) smax = s[j];
        if (m[j] > mmax) mmax = m[j];
    }
    uint16_t d16 = oracle_f32_to_f16(smax / 63.0f), dm16 = oracle_f32_to_f16(mmax / 63.0f);
    float d = oracle_f16_to_f32(d16), dm = oracle_f16_to_f32(dm16);
    int sc[8], mn[8];
    for (int j = 0; j < 8; j++) {
        sc[j] = d == 0.0f ? 0 : clampi((int)oracle_round_half_even(s[j] / d), 0, 63);
        mn[j] = dm == 0.0f ? 0 : clampi((int)oracle_round_half_even(m[j] / dm), 0, 63);
    }
    put_u16(out, d16);
    put_u16(out + 2, dm16);
    q4k_put(out, sc, mn);
    for (int j = 0; j < 8; j++) {
        float S = d * (float)sc[j], M = dm * (float)mn[j];
        int u[32];
        for (int i = 0; i < 32; i++)
            u[i] = S == 0.0f ? 0 : clampi((int)oracle_round_half_even((x[32 * j + i] + M) / S), 0, 15);
        for (int i = 0; i < 16; i++)
            out[16 + 16 * j + i] = (uint8_t)((unsigned)u[i] | ((unsigned)u[i + 16] << 4));
    }
}

static void q4k_codes(const uint8_t *blk, int *u) /* 256 codes, R20 */
{
    for (int j = 0; j < 8; j++)
        for (int i = 0; i < 16; i++) {
            u[32 * j + i] = blk[16 + 16 * j + i] & 15;
            u[32 * j + i + 16] = blk[16 + 16 * j + i] >> 4;
        }
}

static float q6k_scale(const uint8_t *blk) { return oracle_f16_to_f32((uint16_t)(blk[208] | (blk[209] << 8))); }

static void q6k_codes(const uint8_t *blk, int *u) /* 256 codes 0..63, R22 */
{
    for (int i = 0; i < 256; i++) {
        int lo = (i < 128) ? (blk[i] & 15) : (blk[i - 128] >> 4);
        int hi = (blk[128 + (i & 63)] >> (2 * (i >> 6))) & 3;
        u[i] = lo | (hi << 4);
    }
}

static void quantize_q6k(const float *x, uint8_t *out)
{
    float s[16], smax = 0.0f;
    for (int k = 0; k < 16; k++) {
        float amax = 0.0f;
        for (int i = 0; i < 16; i++)
            if (fabsf(x[16 * k + i]) > amax) amax = fabsf(x[16 * k + i]);
        s[k] = amax / 31.0f;
        if (s[k] > smax) smax = s[k];
    }
    uint16_t d16 = oracle_f32_to_f16(smax / 127.0f);
    float d = oracle_f16_to_f32(d16);
    int u[256];
    memset(out, 0, 210);
    for (int k = 0; k < 16; k++) {
        int sc = d == 0.0f ? 0 : clampi((int)oracle_round_half_even(s[k] / d), -128, 127);
        out[192 + k] = (uint8_t)(int8_t)sc;
        float S = d * (float)sc;
        for (int i = 0; i < 16; i++)
            u[16 * k + i] = (S == 0.0f ? 0 : clampi((int)oracle_round_half_even(x[16 * k + i] / S), -32, 31)) + 32;
    }
    for (int i = 0; i < 128; i++)
        out[i] = (uint8_t)((unsigned)(u[i] & 15) | ((unsigned)(u[i + 128] & 15) << 4));
    for (int i = 0; i < 256; i++)
        out[128 + (i & 63)] |= (uint8_t)(((unsigned)u[i] >> 4) << (2 * (i >> 6)));
    put_u16(out + 208, d16);
}

static void dequantize_kquant(int type, const uint8_t *blk, float *dst)
{
    int u[256];
    if (type == ORACLE_TYPE_Q4_K) {
        float S[8], M[8];
        q4k_factors(blk, S, M);
        q4k_codes(blk, u);
        for (int i = 0; i < 256; i++)
            dst[i] = S[i / 32] * (float)u[i] - M[i / 32]; /* R20: fp32 product, then difference */
    } else {
        float d = q6k_scale(blk);
        q6k_codes(blk, u);
        for (int i = 0; i < 256; i++)
            dst[i] = (d * (float)(int8_t)blk[192 + i / 16]) * (float)(u[i] - 32); /* R22 */
    }
}

/* R24: one super-block against the 8 Q8_0 blocks of x under it */
static void kquant_dot(int type, const uint8_t *wb, const uint8_t *xb8, double *acc, double *macc)
{
    int u[256], qx[QK];
    int64_t bx = oracle_block_bytes(ORACLE_TYPE_Q8_0);
    if (type == ORACLE_TYPE_Q4_K) {
        float S[8], M[8];
        q4k_factors(wb, S, M);
        q4k_codes(wb, u);
        for (int j = 0; j < 8; j++) {
            const uint8_t *xb = xb8 + j * bx;
            block_codes(ORACLE_TYPE_Q8_0, xb, qx);
            int64_t su = 0, sx = 0;
            for (int i = 0; i < 32; i++) {
                su += (int64_t)u[32 * j + i] * qx[i];
                sx += qx[i];
            }
            double dx = (double)block_scale(xb);
            double t1 = dx * (double)S[j] * (double)su, t2 = -dx * (double)M[j] * (double)sx;
            *acc += t1 + t2;
            *macc += fabs(t1) + fabs(t2);
        }
    } else {
        float d = q6k_scale(wb);
        q6k_codes(wb, u);
        for (int j = 0; j < 8; j++) {
            const uint8_t *xb = xb8 + j * bx;
            block_codes(ORACLE_TYPE_Q8_0, xb, qx);
            double dx = (double)block_scale(xb);
            for (int h = 0; h < 2; h++) {
                int k = 2 * j + h;
                int64_t si = 0;
                for (int i = 0; i < 16; i++)
                    si += (int64_t)(u[16 * k + i] - 32) * qx[16 * h + i];
                double t = dx * (double)(d * (float)(int8_t)wb[192 + k]) * (double)si;
                *acc += t;
                *macc += fabs(t);
            }
        }
    }
}

int oracle_quantize_rows(int type, const float *src, uint8_t *dst,
                         int64_t n_rows, int64_t n_cols)
{
    int64_t bb = oracle_block_bytes(type);
    if (is_kquant(type)) {
        if (n_cols % 256 != 0 || n_rows < 0 || n_cols < 0)
            return -1;
        int64_t ns = n_cols / 256;
        for (int64_t r = 0; r < n_rows; r++)
            for (int64_t b = 0; b < ns; b++) {
                if (type == ORACLE_TYPE_Q4_K)
                    quantize_q4k(src + r * n_cols + b * 256, dst + (r * ns + b) * bb);
                else
                    quantize_q6k(src + r * n_cols + b * 256, dst + (r * ns + b) * bb);
            }
        return 0;
    }
    if (bb == 0 || n_cols % QK != 0 || n_rows < 0 || n_cols < 0)
        return -1;
    int64_t nb = n_cols / QK;
    for (int64_t r = 0; r < n_rows; r++)
        for (int64_t b = 0; b < nb; b++)
            quantize_block(type, src + r * n_cols + b * QK, dst + (r * nb + b) * bb);
    return 0;
}

int oracle_dequantize_rows(int type, const uint8_t *blocks, float *dst,
                           int64_t n_rows, int64_t n_cols)
{
    int64_t bb = oracle_block_bytes(type);
    if (is_kquant(type)) {
        if (n_cols % 256 != 0 || n_rows < 0 || n_cols < 0)
            return -1;
        int64_t ns = n_cols / 256;
        for (int64_t r = 0; r < n_rows; r++)
            for (int64_t b = 0; b < ns; b++)
                dequantize_kquant(type, blocks + (r * ns + b) * bb, dst + r * n_cols + b * 256);
        return 0;
    }
    if (bb == 0 || n_cols % QK != 0 || n_rows < 0 || n_cols < 0)
        return -1;
    int64_t nb = n_cols / QK;
    int q[QK];
    for (int64_t r = 0; r < n_rows; r++)
        for (int64_t b = 0; b < nb; b++) {
            const uint8_t *blk = blocks + (r * nb + b) * bb;
            float d = block_scale(blk), mn = block_min(type, blk);
            block_codes(type, blk, q);
            for (int j = 0; j < QK; j++) {
                float v = d * (float)q[j]; /* [SYM] value = scale * q */
                if (is_legacy(type) && legacy_affine(type))
                    v = v + mn; /* R18: then the minimum, a second fp32 operation */
                dst[r * n_cols + b * QK + j] = v;
            }
        }
    return 0;
}

static int32_t block_dot(int w_type, const uint8_t *wblk, const uint8_t *xblk)
{
    int qw[QK], qx[QK];
    block_codes(w_type, wblk, qw);
    block_codes(ORACLE_TYPE_Q8_0, xblk, qx);
    int32_t s = 0;
    for (int j = 0; j < QK; j++)
        s += qw[j] * qx[j];
    return s;
}

int oracle_block_dots(int w_type, const uint8_t *w_blocks, const uint8_t *xq_blocks,
                      int32_t *out, int64_t M, int64_t K)
{
    int64_t bw = oracle_block_bytes(w_type);
    int64_t bx = oracle_block_bytes(ORACLE_TYPE_Q8_0);
    if (bw == 0 || is_kquant(w_type) || K % QK != 0 || M < 0 || K < 0)
        return -1;
    int64_t nb = K / QK;
    for (int64_t m = 0; m < M; m++)
        for (int64_t b = 0; b < nb; b++)
            out[m * nb + b] = block_dot(w_type, w_blocks + (m * nb + b) * bw, xq_blocks + b * bx);
    return 0;
}

/* one output: R6 (fp64 sum of exact terms, one rounding to fp32) */
static void dot_row(int w_type, const uint8_t *wrow, const uint8_t *xrow, int64_t nb,
                    float *y, double *mag)
{
    int64_t bw = oracle_block_bytes(w_type);
    int64_t bx = oracle_block_bytes(ORACLE_TYPE_Q8_0);
    double acc = 0.0, macc = 0.0;
    if (is_kquant(w_type)) { /* nb counts 32-blocks of x; a super-block spans 8 */
        for (int64_t b = 0; b < nb / 8; b++)
            kquant_dot(w_type, wrow + b * bw, xrow + 8 * b * bx, &acc, &macc);
        *y = (float)acc;
        if (mag)
            *mag = macc;
        return;
    }
    for (int64_t b = 0; b < nb; b++) {
        const uint8_t *wb = wrow + b * bw;
        const uint8_t *xb = xrow + b * bx;
        int32_t sumi = block_dot(w_type, wb, xb);
        double term = (double)block_scale(wb) * (double)block_scale(xb) * (double)sumi;
        acc += term;
        macc += fabs(term);
        if (is_legacy(w_type) && legacy_affine(w_type)) { /* R19: the minimum times the x block's code sum */
            int qx[QK];
            block_codes(ORACLE_TYPE_Q8_0, xb, qx);
            int32_t xs = 0;
            for (int j = 0; j < QK; j++)
                xs += qx[j];
            double mterm = (double)block_min(w_type, wb) * (double)block_scale(xb) * (double)xs;
            acc += mterm;
            macc += fabs(mterm);
        }
    }
    *y = (float)acc;
    if (mag)
        *mag = macc;
}

int oracle_gemv(int w_type, const uint8_t *w_blocks, const float *x, float *y,
                double *mag, int64_t M, int64_t K)
{
    int64_t bw = oracle_block_bytes(w_type), bv = oracle_block_values(w_type);
    if (bw == 0 || K % bv != 0 || M < 0 || K < 0)
        return -1;
    int64_t nb = K / QK, row_bytes = K / bv * bw;
    uint8_t *xq = (uint8_t *)malloc((size_t)(nb * oracle_block_bytes(ORACLE_TYPE_Q8_0)) + 1);
    if (!xq)
        return -3;
    oracle_quantize_rows(ORACLE_TYPE_Q8_0, x, xq, 1, K); /* R5 */
    /* rows are independent: a build with OpenMP may run them on several
       threads (same per-row arithmetic, same results) */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int64_t m = 0; m < M; m++)
        dot_row(w_type, w_blocks + m * row_bytes, xq, nb, y + m, mag ? mag + m : NULL);
    free(xq);
    return 0;
}

int oracle_gemm(int w_type, const uint8_t *w_blocks, const float *X, float *Y,
                double *mag, int64_t M, int64_t N, int64_t K)
{
    int64_t bw = oracle_block_bytes(w_type), bv = oracle_block_values(w_type);
    int64_t bx = oracle_block_bytes(ORACLE_TYPE_Q8_0);
    if (bw == 0 || K % bv != 0 || M < 0 || N < 0 || K < 0)
        return -1;
    int64_t nb = K / QK, row_bytes = K / bv * bw;
    uint8_t *xq = (uint8_t *)malloc((size_t)(N * nb * bx) + 1);
    if (!xq)
        return -3;
    oracle_quantize_rows(ORACLE_TYPE_Q8_0, X, xq, N, K); /* R5, row by row */
    for (int64_t n = 0; n < N; n++)
        for (int64_t m = 0; m < M; m++)
            dot_row(w_type, w_blocks + m * row_bytes, xq + n * nb * bx, nb,
                    Y + n * M + m, mag ? mag + n * M + m : NULL);
    free(xq);
    return 0;
}

/* ---- Hadamard rotation: [ROT], R14, R15 ---- */

int oracle_hadamard64(float *x, int64_t n)
{
    if (n < 0 || n % 64 != 0)
        return -1;
    for (int64_t g = 0; g < n; g += 64) {
        float *v = x + g;
        for (int h = 1; h < 64; h *= 2) /* R15: spans 1, 2, 4, 8, 16, 32 in turn */
            for (int j = 0; j < 64; j++)
                if ((j & h) == 0) {
                    float a = v[j], b = v[j + h];
                    v[j] = a + b;
                    v[j + h] = a - b;
                }
        for (int j = 0; j < 64; j++)
            v[j] = v[j] * 0.125f; /* R14: orthonormal, 1/sqrt(64); exact */
    }
    return 0;
}

int oracle_kv_quantize_basis(int type, const float *rows, const float *bias, int bias_basis, int basis,
                             uint8_t *dst, int64_t n_tokens, int64_t n_kv_heads, int64_t head_dim)
{
    int64_t bb = oracle_block_bytes(type);
    if (bb == 0 || is_kquant(type) || head_dim % QK != 0 || n_tokens < 0 || n_kv_heads < 0 || head_dim < 0)
        return -1;
    if (basis != ORACLE_BASIS_PLAIN && basis != ORACLE_BASIS_HADAMARD64)
        return -1;
    if (basis == ORACLE_BASIS_HADAMARD64 && head_dim % 64 != 0) /* [ROT] head_dim a multiple of 64 */
        return -1;
    if (bias && type != ORACLE_TYPE_Q4_0) /* [KVMC] mean-centering needs a Q4_0 K cache */
        return -2;
    if (bias && bias_basis != basis) /* [ROT] the bias must be in the cache's basis: fail fast */
        return -4;
    int64_t nb = head_dim / QK;
    float *row = (float *)malloc((size_t)(head_dim > 0 ? head_dim : 1) * sizeof(float));
    if (!row)
        return -3;
    float tmp[QK];
    for (int64_t t = 0; t < n_tokens; t++)
        for (int64_t h = 0; h < n_kv_heads; h++) {
            memcpy(row, rows + (t * n_kv_heads + h) * head_dim, (size_t)head_dim * sizeof(float));
            if (basis == ORACLE_BASIS_HADAMARD64) /* R14: rotate first, then center */
                oracle_hadamard64(row, head_dim);
            uint8_t *out = dst + (t * n_kv_heads + h) * nb * bb;
            for (int64_t b = 0; b < nb; b++) {
                for (int j = 0; j < QK; j++) {
                    float v = row[b * QK + j];
                    if (bias) /* [KVMC] K' = K - bias[h][c], one fp32 subtraction */
                        v = v - bias[h * head_dim + b * QK + j];
                    tmp[j] = v;
                }
                quantize_block(type, tmp, out + b * bb);
            }
        }
    free(row);
    return 0;
}

int oracle_kv_quantize(int type, const float *rows, const float *bias, uint8_t *dst,
                       int64_t n_tokens, int64_t n_kv_heads, int64_t head_dim)
{
    return oracle_kv_quantize_basis(type, rows, bias, ORACLE_BASIS_PLAIN, ORACLE_BASIS_PLAIN, dst, n_tokens,
                                    n_kv_heads, head_dim);
}

int oracle_kv_bias(const float *rows, int basis, float *bias, int64_t n_tokens, int64_t n_kv_heads,
                   int64_t head_dim)
{
    if (n_tokens < 1 || n_kv_heads < 0 || head_dim < 0 || head_dim % QK != 0)
        return -1;
    if (basis != ORACLE_BASIS_PLAIN && basis != ORACLE_BASIS_HADAMARD64)
        return -1;
    if (basis == ORACLE_BASIS_HADAMARD64 && head_dim % 64 != 0)
        return -1;
    int64_t n = n_kv_heads * head_dim;
    double *sum = (double *)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
    float *row = (float *)malloc((size_t)(head_dim > 0 ? head_dim : 1) * sizeof(float));
    if (!sum || !row) {
        free(sum); free(row);
        return -3;
    }
    for (int64_t t = 0; t < n_tokens; t++) /* R15: token order, fp64 */
        for (int64_t h = 0; h < n_kv_heads; h++) {
            memcpy(row, rows + (t * n_kv_heads + h) * head_dim, (size_t)head_dim * sizeof(float));
            if (basis == ORACLE_BASIS_HADAMARD64) /* [ROT] measured in the cache's basis */
                oracle_hadamard64(row, head_dim);
            for (int64_t c = 0; c < head_dim; c++)
                sum[h * head_dim + c] += (double)row[c];
        }
    for (int64_t i = 0; i < n; i++)
        bias[i] = (float)(sum[i] / (double)n_tokens);
    free(sum); free(row);
    return 0;
}

/* ---- decode attention: R11, R12; [FA], [SHIFT] ---- */

int oracle_attn_decode_basis(int k_type, int v_type, int k_basis, const float *q, const uint8_t *K,
                             const uint8_t *V, float *o, double *mag, double *smax, int64_t n_tokens,
                             int64_t n_heads, int64_t n_kv_heads, int64_t head_dim, float scale)
{
    int64_t bk = oracle_block_bytes(k_type), bv = oracle_block_bytes(v_type);
    if (bk == 0 || bv == 0 || head_dim <= 0 || head_dim % QK != 0 || n_tokens < 1 || n_kv_heads < 1 ||
        n_heads < n_kv_heads || n_heads % n_kv_heads != 0)
        return -1;
    if (is_legacy(k_type) || is_legacy(v_type) || is_kquant(k_type) || is_kquant(v_type)) /* Q4_0 / Q8_0 caches */
        return -1;
    if (k_basis != ORACLE_BASIS_PLAIN && (k_basis != ORACLE_BASIS_HADAMARD64 || head_dim % 64 != 0))
        return -1;
    if (k_basis == ORACLE_BASIS_HADAMARD64) {
        /* R14: q in the K cache's basis, (Hq).(Hk) = q.k */
        float *qr = (float *)malloc((size_t)(n_heads * head_dim) * sizeof(float));
        if (!qr)
            return -3;
        memcpy(qr, q, (size_t)(n_heads * head_dim) * sizeof(float));
        oracle_hadamard64(qr, n_heads * head_dim);
        int rc = oracle_attn_decode_basis(k_type, v_type, ORACLE_BASIS_PLAIN, qr, K, V, o, mag, smax, n_tokens,
                                          n_heads, n_kv_heads, head_dim, scale);
        free(qr);
        return rc;
    }
    int64_t nb = head_dim / QK, group = n_heads / n_kv_heads;
    int64_t bq = oracle_block_bytes(ORACLE_TYPE_Q8_0);
    uint8_t *qq = (uint8_t *)malloc((size_t)(n_heads * nb * bq));
    double *s = (double *)malloc((size_t)n_tokens * sizeof(double));
    float *vrow = (float *)malloc((size_t)head_dim * sizeof(float));
    if (!qq || !s || !vrow) {
        free(qq); free(s); free(vrow);
        return -3;
    }
    oracle_quantize_rows(ORACLE_TYPE_Q8_0, q, qq, n_heads, head_dim); /* R12: per head, per 32 channels */
    for (int64_t h = 0; h < n_heads; h++) {
        int64_t kvh = h / group; /* R11: grouped query heads share a kv head */
        const uint8_t *qh = qq + h * nb * bq;
        /* scores: scale * sum_b dk dq sumi, exact terms summed in fp64 */
        double smx = -INFINITY, sabs = 0.0;
        for (int64_t t = 0; t < n_tokens; t++) {
            const uint8_t *kt = K + (t * n_kv_heads + kvh) * nb * bk;
            double acc = 0.0;
            for (int64_t b = 0; b < nb; b++) {
                int32_t sumi = block_dot(k_type, kt + b * bk, qh + b * bq);
                acc += (double)block_scale(kt + b * bk) * (double)block_scale(qh + b * bq) * (double)sumi;
            }
            s[t] = (double)scale * acc;
            if (s[t] > smx) smx = s[t];
            if (fabs(s[t]) > sabs) sabs = fabs(s[t]);
        }
        /* softmax over the tokens, after subtracting the row maximum ([SHIFT]) */
        double l = 0.0;
        for (int64_t t = 0; t < n_tokens; t++) {
            s[t] = exp(s[t] - smx);
            l += s[t];
        }
        double *acc = (double *)calloc((size_t)(2 * head_dim), sizeof(double));
        if (!acc) {
            free(qq); free(s); free(vrow);
            return -3;
        }
        for (int64_t t = 0; t < n_tokens; t++) {
            double w = s[t] / l;
            oracle_dequantize_rows(v_type, V + (t * n_kv_heads + kvh) * nb * bv, vrow, 1, head_dim);
            for (int64_t d = 0; d < head_dim; d++) {
                acc[d] += w * (double)vrow[d];
                acc[head_dim + d] += w * fabs((double)vrow[d]);
            }
        }
        for (int64_t d = 0; d < head_dim; d++) {
            o[h * head_dim + d] = (float)acc[d];
            if (mag) mag[h * head_dim + d] = acc[head_dim + d];
        }
        if (smax) smax[h] = sabs;
        free(acc);
    }
    free(qq); free(s); free(vrow);
    return 0;
}

int oracle_attn_decode(int k_type, int v_type, const float *q, const uint8_t *K, const uint8_t *V,
                       float *o, double *mag, double *smax, int64_t n_tokens, int64_t n_heads,
                       int64_t n_kv_heads, int64_t head_dim, float scale)
{
    return oracle_attn_decode_basis(k_type, v_type, ORACLE_BASIS_PLAIN, q, K, V, o, mag, smax, n_tokens, n_heads,
                                    n_kv_heads, head_dim, scale);
}
