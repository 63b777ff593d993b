/*
 * kv4_oracle.c — plain CPU oracle for the KV4-RL rollout decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load it; the product path never does.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math [-fopenmp] -shared -fPIC.
 * Contraction is off so every float expression below rounds exactly as written;
 * fused multiply-adds appear only where fmaf() is spelled out.
 *
 * Pages cited (title, then section):
 *   [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速"
 *   [ko] "INT4 KV 캐시로 비동기 RLVR 롤아웃을 1.8배 가속한다"
 *
 * What each step follows:
 *   Hadamard rotation of post-RoPE keys and of the query, QH(HK)^T = QK^T
 *       [zh] 前置知识 › 分组仿射 KV 量化; 核心方法; 方法步骤详情 step 2.
 *   Group-affine quantizer x^ = Δc + m, one group per 128-dim token-head vector,
 *   FP16 Δ and m computed online, 4 bits (main cache) or 8 bits (side cache)
 *       [zh] 分组仿射 KV 量化; 方法步骤详情 steps 2-3; [ko] 전제와 한계.
 *   INT8 query; integer QK with the scale and offset applied after the dot
 *       [zh] 分组仿射 KV 量化 (scale/offset deferred past the dot product);
 *       [ko] 전제와 한계; [zh] 方法步骤详情 step 4.
 *   Integer PV over the INT4 region; protected path over sink + recent with
 *   INT8 keys and BF16-dequantized values, FP32 accumulation
 *       [ko] 전제와 한계; [zh] 核心方法, 方法步骤详情 steps 3-4.
 *   Disjoint regions, each giving a local output and log-normaliser, merged by
 *   an exact softmax (log-sum-exp) merge
 *       [ko] 전제와 한계; [zh] 核心方法 (third difference).
 *
 * Readings where the pages leave a step open:
 *   R1 V is not rotated; only K (post-RoPE) and q are.
 *   R2 Δ and m use directed rounding: m = fp16_down(min x) (a zero minimum as +0),
 *      Δ = fp16_up(up((max x − m) / n)), so m ≤ min x and m + nΔ ≥ max x.
 *      Codes are c = clamp(rint((x − m) · fl(1/Δ)), 0, n); Δ = 0 gives c = 0.
 *   R3 The query is symmetric INT8 per q head: s_q = max|q'|/127,
 *      q8 = rint(q' · fl(127/max|q'|)).
 *   R4 Regions: protected = [0, min(s,L)) ∪ [max(s, L−w), L); INT4 = [s, L−w).
 *   R5 Integer PV: per page ∩ INT4 region, p' = 2^(σ − M_page) with the exp2
 *      below, w = p'·Δ^V, and u8 weights with one power-of-two scale per page:
 *      e = floor(log2(max w)), ŵ = min(rint(w · 2^(7−e)), 255) in 0..255 (the
 *      largest weight lands in 128..255), acc_j = Σ ŵ c^V_j, page output
 *      s_w·acc_j + Σ p'·m^V with s_w = 2^(e−7). A page whose max w is not above
 *      2^-64 keeps only its offsets (ŵ = 0).
 *   R6 Scores are log2-domain: σ = fl(fl(u · s_q) · C), u = fmaf(Δ, dot, fl(m · Σq8)),
 *      C = fl(sm_scale · log2 e).
 *   R7 Protected PV ("BF16 PV, FP32 accumulation"): the protected positions are
 *      taken in position order, grouped by their 16-position page of the paged
 *      cache (the unit R5 uses for the INT4 weights; a page may hold both sink and
 *      window positions, or only part of either). In each page
 *      p = exp2(σ − M_page) with the exp2 below and the max over the page's
 *      protected positions; the product uses p and v = bf16(fmaf(Δ8, c, m8)) both
 *      rounded to BF16 and sums in FP32; pages are combined by 2^(M_page − M) like
 *      INT4 pages; the normaliser sums the unrounded p. Float mode keeps p
 *      unrounded. Where a side row sits in the side buffer plays no part.
 *   R10 KV8, the 8-bit whole-cache configuration the pages compare KV4 against
 *      ([zh] 核心发现 (2), (3); 实验结果, decode-forward replay): every position holds
 *      the 8-bit affine codes of the side cache (rotated K, unrotated V, the R2
 *      quantizer with n = 255), and decode applies the protected path of R6 and R7
 *      to every position, in groups of 16 consecutive positions (one page) in
 *      position order.
 *   R11 RoPE, when the caller supplies its table: keys are rotated by RoPE at their
 *      position and then by the Hadamard transform, queries the same at position
 *      L − 1 ([zh] 核心方法: the Hadamard rotation follows RoPE; 方法步骤详情 step 2:
 *      the query takes the same rotations). Pairing (i, i + 64) ("rotate half"), with
 *      a = x_i, b = x_{i+64}: x'_i = fmaf(a, cos, −fl(b·sin)),
 *      x'_{i+64} = fmaf(b, cos, fl(a·sin)); cos and sin are the caller's FP32 table.
 *   R12 NVFP4, the 4-bit floating-point KV format the pages compare against ([zh]
 *      技术新颖性: an appendix compares NVFP4/MXFP4; 未来方向: a KV4 variant on native
 *      FP4 hardware): the public NVFP4 layout with the method's online per-vector
 *      scaling. Each 128-value token-head vector (rotated K, unrotated V) has an FP32
 *      scale g = amax / (6·448) and, per block of 16, an E4M3 scale
 *      s_b = e4m3(amax_b / fl(6g)); each value is e2m1(x · fl(1/fl(s_b g))), nearest
 *      with ties to even. The whole cache is NVFP4 (no protected region). Decode keeps the
 *      INT8 query: the score is ((Σ_b fma-chained s_b·dot_b)·g·s_q)·C with each block dot
 *      exact. PV runs per page (16 consecutive positions) with the page's own max as in
 *      R7, but the value scales move to the weights: the E2M1 values enter exactly, and
 *      position i of head h weighs w_ib = fp16(fp16(fl(p_i·g_i)·2^-k)·s_ib) in block b,
 *      where 2^k is the power of two just above the largest V vector scale g of the
 *      page's positions (2^-126 below the normal range), and the page's sum is scaled
 *      by 2^k. 2^k is a property of the stored values alone, like the block scales:
 *      p ≤ 1 and g < 2^k put every fp16 weight before the block scale at or below 1,
 *      so it neither overflows nor loses the largest value's precision to a scale
 *      that depends on the softmax. The normaliser sums the plain p.
 *   R13 MXFP4, the other 4-bit floating-point format the pages name beside NVFP4
 *      ([zh] 技术新颖性, 未来方向), as the public OCP microscaling format defines it:
 *      per block of 32 values one shared E8M0 scale X = 2^s with
 *      s = floor(log2 max|x|) − 2 (2 being the largest E2M1 exponent), held in
 *      [−127, 127], and each value e2m1(x / X), nearest with ties to even, held at ±6;
 *      an all-zero block takes s = −127 and zero codes. No per-vector scale. Decode
 *      keeps the INT8 query: the score is fl(fl(acc·s_q)·C) with acc the fma chain
 *      fmaf(2^s_b, dot_b, acc) over the four blocks of exact block dots; PV as R12, with
 *      weights w_ib = fp16(fp16(p_i)·2^(s_ib − k)), 2^k the largest block scale of the
 *      page's positions, exact E2M1 values and the page's sum scaled by 2^k.
 * Everything after the integer decisions (page outputs, region merges,
 * the protected path, the final normalisation) is carried in double here.
 */
#include "kv4_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Number formats                                                            */
/* ------------------------------------------------------------------------ */

double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* Encode a double that is exactly an fp16 value (or ±inf). */
static uint16_t f16_encode_exact(double v, int neg)
{
    uint16_t s = neg ? 0x8000 : 0;
    double a = fabs(v);
    if (isinf(a)) return s | 0x7c00;
    if (a == 0.0) return s;
    if (a < ldexp(1.0, -14))                      /* subnormal: a = f * 2^-24 */
        return s | (uint16_t)(a * ldexp(1.0, 24));
    int e;
    double m = frexp(a, &e);                      /* a = m * 2^e, m in [0.5, 1) */
    int E = e - 1;                                /* a = (2m) * 2^E */
    int frac = (int)(m * 2048.0) - 1024;          /* exact: a has ≤ 11 significant bits */
    return s | (uint16_t)(((E + 15) << 10) | frac);
}

/*
 * float -> fp16 in round-to-nearest-even, toward −inf or toward +inf.
 * Written from the definition: pick the fp16 quantum of the binade, scale the
 * value onto an integer grid (exact, the quantum is a power of two), round the
 * grid coordinate with the requested rule, then scale back and handle overflow.
 */
uint16_t orc_f32_to_f16(float xf, int mode)
{
    double x = (double)xf;
    int neg = signbit(xf) != 0;
    if (isnan(x)) return (uint16_t)((neg ? 0x8000 : 0) | 0x7e00);
    if (isinf(x)) return (uint16_t)((neg ? 0x8000 : 0) | 0x7c00);
    if (x == 0.0) return (uint16_t)(neg ? 0x8000 : 0);
    int e;
    frexp(fabs(x), &e);
    int E = e - 1;                    /* 2^E ≤ |x| < 2^(E+1) */
    if (E < -14) E = -14;             /* below the normal range the quantum is 2^-24 */
    double q = ldexp(1.0, E - 10);
    double t = x / q;                 /* exact */
    double r;
    if (mode == ORC_RD)
        r = floor(t);
    else if (mode == ORC_RU)
        r = ceil(t);
    else
        r = nearbyint(t);             /* default rounding mode: nearest, ties to even */
    double v = r * q;
    if (v > 65504.0) return (mode == ORC_RD) ? 0x7bff : 0x7c00;
    if (v < -65504.0) return (mode == ORC_RU) ? 0xfbff : 0xfc00;
    return f16_encode_exact(v, neg);
}

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

uint16_t orc_f32_to_bf16_rn(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN: keep sign, force quiet */
        return (uint16_t)((u >> 16) | 0x40);
    /* round the low 16 bits away, ties to the even upper half */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/*
 * exp2 for the PV weights. Written from the textbook range reduction
 * 2^x = 2^n · 2^f with n = rint(x), f = x − n in [−1/2, 1/2], and the Taylor
 * series 2^f = Σ_k (f ln 2)^k / k!, truncated after k = 7 and evaluated by
 * Horner's rule with fused multiply-adds. Coefficients are (ln 2)^k / k!
 * computed in double and rounded once to float. Defined for x ≤ 0 (the only
 * use); x < −125 returns 0 so every nonzero result is a normal float.
 */
static float exp2_coef[8];

__attribute__((constructor)) static void exp2_init(void)
{
    double fact = 1.0, lnp = 1.0;
    for (int k = 0; k < 8; k++) {
        if (k > 0) { fact *= (double)k; lnp *= 0.69314718055994530942; }
        exp2_coef[k] = (float)(lnp / fact);
    }
}

float orc_exp2f(float x)
{
    if (!(x >= -125.0f)) return 0.0f;
    float n = rintf(x);
    float f = x - n;                                 /* exact */
    float p = exp2_coef[7];
    for (int k = 6; k >= 0; k--) p = fmaf(p, f, exp2_coef[k]);
    return ldexpf(p, (int)n);
}

/* Directed float subtraction a − b rounded toward +inf: the round-to-nearest
   result plus the exact error term (Knuth's TwoSum) decide the direction. */
static float fsub_up(float a, float b)
{
    float nb = -b;
    float s = a + nb;
    float bb = s - a;
    float err = (a - (s - bb)) + (nb - bb);
    return (err > 0.0f) ? nextafterf(s, INFINITY) : s;
}

/* Directed float division a / n rounded toward +inf, for a ≥ 0 and n > 0:
   the remainder a − q·n of the nearest quotient q is exact in one fmaf. */
static float fdiv_up(float a, float n)
{
    float q = a / n;
    float rem = fmaf(-q, n, a);
    return (rem > 0.0f) ? nextafterf(q, INFINITY) : q;
}

/* ------------------------------------------------------------------------ */
/* Steps                                                                     */
/* ------------------------------------------------------------------------ */

/* 128-point fast Walsh–Hadamard transform, normalised to H/√128 (orthonormal,
   symmetric). Butterfly stages h = 1, 2, …, 64 in that order, then one scale.
   [zh] 分组仿射 KV 量化; 方法步骤详情 step 2 (same rotation for K and q). */
void orc_fwht128(const float *in, float *out)
{
    float x[ORC_D];
    memcpy(x, in, sizeof x);
    for (int h = 1; h < ORC_D; h <<= 1)
        for (int i = 0; i < ORC_D; i++)
            if ((i & h) == 0) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
    const float scale = (float)(1.0 / sqrt(128.0));
    for (int i = 0; i < ORC_D; i++) out[i] = x[i] * scale;
}

/* RoPE of one 128-dim vector with one row of the caller's table (reading R11): dims i
   and i + 64 rotate together by the angle whose cos and sin are row[i] and row[64 + i]. */
void orc_rope128(const float *in, const float *cs, float *out)
{
    for (int i = 0; i < ORC_D / 2; i++) {
        const float a = in[i], b = in[i + ORC_D / 2];
        const float c = cs[i], s = cs[ORC_D / 2 + i];
        out[i] = fmaf(a, c, -(b * s));
        out[i + ORC_D / 2] = fmaf(b, c, a * s);
    }
}

/* Group-affine quantizer x^ = Δc + m over one group of n values, levels = 2^b − 1.
   [zh] 分组仿射 KV 量化; 方法步骤详情 step 2 (FP16 Δ and m computed online).
   Rounding directions: reading R2 in the file header. */
void orc_quant_affine(const float *x, int n, int levels,
                      uint8_t *code, uint16_t *delta_h, uint16_t *min_h)
{
    float lo = x[0], hi = x[0];
    for (int i = 1; i < n; i++) {
        if (x[i] < lo) lo = x[i];
        if (x[i] > hi) hi = x[i];
    }
    lo = lo + 0.0f;                       /* a zero minimum carries no sign: −0 becomes +0 */
    uint16_t mh = orc_f32_to_f16(lo, ORC_RD);
    float m = (float)orc_f16_to_f64(mh);
    float r = fsub_up(hi, m);
    float d = fdiv_up(r, (float)levels);
    uint16_t dh = orc_f32_to_f16(d, ORC_RU);
    float delta = (float)orc_f16_to_f64(dh);
    *delta_h = dh;
    *min_h = mh;
    if (delta == 0.0f) {
        memset(code, 0, (size_t)n);
        return;
    }
    float inv = 1.0f / delta;
    for (int i = 0; i < n; i++) {
        float t = (x[i] - m) * inv;
        float c = rintf(t);
        if (c < 0.0f) c = 0.0f;
        if (c > (float)levels) c = (float)levels;
        code[i] = (uint8_t)c;
    }
}

/* Symmetric INT8 query, one scale per q head (reading R3).
   [ko] 전제와 한계 (the rotated query is quantized to INT8 and serves both paths). */
void orc_quant_query(const float *q_rot, int8_t *q8, float *q_scale, int32_t *q_sum)
{
    float a = 0.0f;
    for (int i = 0; i < ORC_D; i++) {
        float v = fabsf(q_rot[i]);
        if (v > a) a = v;
    }
    int32_t sum = 0;
    if (a == 0.0f) {
        memset(q8, 0, ORC_D);
        *q_scale = 0.0f;
        *q_sum = 0;
        return;
    }
    float inv = 127.0f / a;
    for (int i = 0; i < ORC_D; i++) {
        int v = (int)rintf(q_rot[i] * inv);
        q8[i] = (int8_t)v;
        sum += v;
    }
    *q_scale = a / 127.0f;
    *q_sum = sum;
}

/* ---- NVFP4 (reading R12): E2M1 elements, E4M3 block scales, an FP32 vector scale ---- */

/* E4M3 (bias 7, no infinities, largest finite 448): t >= 0 rounded to the nearest
   representable value, ties to even mantissa, values above 448 held at 448. The
   subnormal quantum is 2^-9; normal values of exponent e have quantum 2^(e-3). */
uint8_t orc_e4m3_rn(float t)
{
    if (!(t > 0.0f)) return 0;
    if (t >= 448.0f) return 0x7E;
    int e;
    frexpf(t, &e);                                /* t = f 2^e, f in [0.5, 1) */
    e -= 1;                                       /* floor(log2 t) */
    if (e < -6) e = -6;                           /* subnormal range shares the 2^-9 quantum */
    const float q = ldexpf(1.0f, e - 3);
    float m = rintf(t / q);                       /* exact division by a power of two; rint: ties even */
    float v = m * q;
    if (v >= 448.0f) return 0x7E;
    if (v == 0.0f) return 0;
    if (v < 0x1p-6f) return (uint8_t)(v / 0x1p-9f);            /* subnormal: mantissa only */
    frexpf(v, &e);
    e -= 1;
    const int mant = (int)(v / ldexpf(1.0f, e - 3)) - 8;        /* 0..7 */
    return (uint8_t)(((e + 7) << 3) | mant);
}

float orc_e4m3_value(uint8_t bits)
{
    const int E = (bits >> 3) & 15, m = bits & 7;
    const float mag = E == 0 ? ldexpf((float)m, -9) : ldexpf(1.0f + (float)m / 8.0f, E - 7);
    return (bits & 0x80) ? -mag : mag;
}

/* E2M1 magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6 (codes 0..7), sign in bit 3. v rounded to the
   nearest, ties to the even code, held at 6; a zero magnitude is code 0. */
static const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

uint8_t orc_e2m1_rn(float v)
{
    const float a = fabsf(v);
    int best = 7;
    if (a < 6.0f) {
        for (int k = 0; k < 7; k++) {
            const float mid = 0.5f * (kE2M1[k] + kE2M1[k + 1]);        /* exact */
            if (a < mid || (a == mid && (k & 1) == 0)) { best = k; break; }
        }
    }
    if (best == 0) return 0;
    return (uint8_t)(best | (v < 0.0f ? 8 : 0));
}

float orc_e2m1_value(uint8_t code)
{
    const float mag = kE2M1[code & 7];
    return (code & 8) ? -mag : mag;
}

/* One 128-value vector to NVFP4: g = amax / (6 * 448); block b of 16 values takes the
   E4M3 scale s_b = e4m3(amax_b / fl(6 g)); each value x becomes e2m1(x * fl(1 / fl(s_b g))).
   A zero vector (or block) has zero scales and zero codes. */
void orc_quant_nvfp4(const float *x, uint8_t *codes, uint8_t *bscale, float *gscale)
{
    float amax = 0.0f;
    for (int i = 0; i < ORC_D; i++) amax = fmaxf(amax, fabsf(x[i]));
    const float g = amax / 2688.0f;
    *gscale = g;
    const float d = g * 6.0f;
    for (int b = 0; b < ORC_D / 16; b++) {
        float ab = 0.0f;
        for (int i = 0; i < 16; i++) ab = fmaxf(ab, fabsf(x[16 * b + i]));
        const uint8_t sb = d > 0.0f ? orc_e4m3_rn(ab / d) : 0;
        bscale[b] = sb;
        const float scale = orc_e4m3_value(sb) * g;
        const float inv = scale > 0.0f ? 1.0f / scale : 0.0f;
        for (int i = 0; i < 16; i++)
            codes[16 * b + i] = scale > 0.0f ? orc_e2m1_rn(x[16 * b + i] * inv) : 0;
    }
}

/* R12 score of an NVFP4 key: the exact dot of each block with the INT8 query, scaled by
   the block's E4M3 scale in an fma chain over the blocks in order, then by g, s_q and C. */
static float score_nvfp4(const uint8_t *codes, const uint8_t *bscale, float g, const int8_t *q8,
                         float q_scale, float C)
{
    float acc = 0.0f;
    for (int b = 0; b < ORC_D / 16; b++) {
        double db = 0.0;
        for (int i = 0; i < 16; i++) db += (double)orc_e2m1_value(codes[16 * b + i]) * (double)q8[16 * b + i];
        acc = fmaf(orc_e4m3_value(bscale[b]), (float)db, acc);
    }
    return ((acc * g) * q_scale) * C;
}

/* ---- MXFP4 (reading R13): E2M1 elements, one E8M0 scale per 32 values ---- */

/* One 128-value vector to MXFP4: per block b of 32 values the shared exponent
   s = floor(log2 amax_b) − 2, held in [−127, 127] (stored biased, s + 127), and the codes
   e2m1(x · 2^−s); an all-zero block stores s = −127 and zero codes. */
void orc_quant_mxfp4(const float *x, uint8_t *codes, uint8_t *escale)
{
    for (int b = 0; b < ORC_D / 32; b++) {
        float amax = 0.0f;
        for (int i = 0; i < 32; i++) amax = fmaxf(amax, fabsf(x[32 * b + i]));
        int sx = -127;
        if (amax > 0.0f) {
            int k;
            frexpf(amax, &k);                   /* amax in [2^(k-1), 2^k): floor(log2) = k - 1 */
            sx = k - 1 - 2;
            if (sx < -127) sx = -127;
            if (sx > 127) sx = 127;
        }
        escale[b] = (uint8_t)(sx + 127);
        for (int i = 0; i < 32; i++)
            codes[32 * b + i] = amax > 0.0f ? orc_e2m1_rn(ldexpf(x[32 * b + i], -sx)) : 0;
    }
}

/* R13 score of an MXFP4 key: the exact dot of each 32-value block with the INT8 query,
   scaled by the block's power of two in an fma chain over the blocks in order, then by
   s_q and C. */
static float score_mxfp4(const uint8_t *codes, const uint8_t *escale, const int8_t *q8,
                         float q_scale, float C)
{
    float acc = 0.0f;
    for (int b = 0; b < ORC_D / 32; b++) {
        double db = 0.0;
        for (int i = 0; i < 32; i++) db += (double)orc_e2m1_value(codes[32 * b + i]) * (double)q8[32 * b + i];
        acc = fmaf(ldexpf(1.0f, (int)escale[b] - 127), (float)db, acc);
    }
    return (acc * q_scale) * C;
}

/* ------------------------------------------------------------------------ */
/* Cache state                                                               */
/* ------------------------------------------------------------------------ */

static size_t idx_main(const orc_cache *c, int slot, int pos, int head)
{
    return ((size_t)slot * c->max_len + pos) * c->num_heads + head;
}

static size_t idx_side(const orc_cache *c, int slot, int sidx, int head)
{
    return ((size_t)slot * (c->sink + c->window) + sidx) * c->num_heads + head;
}

static void load_bf16_row(const uint16_t *src, float *dst)
{
    for (int i = 0; i < ORC_D; i++) dst[i] = orc_bf16_to_f32(src[i]);
}

/* Write one token-head into both caches. */
static void append_one(orc_cache *c, int slot, int pos, int head,
                       const float *k_rot, const float *v)
{
    size_t mi = idx_main(c, slot, pos, head);
    if (c->format == ORC_FMT_MXFP4) {               /* R13: MXFP4 codes and scales */
        orc_quant_mxfp4(k_rot, c->k4_code + mi * ORC_D, c->k_bscale + mi * 8);
        orc_quant_mxfp4(v, c->v4_code + mi * ORC_D, c->v_bscale + mi * 8);
        return;
    }
    if (c->format == ORC_FMT_NVFP4) {               /* R12: NVFP4 codes and scales */
        orc_quant_nvfp4(k_rot, c->k4_code + mi * ORC_D, c->k_bscale + mi * 8, c->k_gscale + mi);
        orc_quant_nvfp4(v, c->v4_code + mi * ORC_D, c->v_bscale + mi * 8, c->v_gscale + mi);
        return;
    }
    const int levels = c->format == ORC_FMT_KV8 ? 255 : 15;   /* R10: KV8 keeps 8-bit codes */
    orc_quant_affine(k_rot, ORC_D, levels, c->k4_code + mi * ORC_D, c->k4_delta + mi, c->k4_min + mi);
    orc_quant_affine(v, ORC_D, levels, c->v4_code + mi * ORC_D, c->v4_delta + mi, c->v4_min + mi);
    if (c->format == ORC_FMT_KV8) return;

    /* Side buffer: an INT8 copy of a sink position and of the position in the
       recent ring. [ko] 전제와 한계; [zh] 方法步骤详情 step 3. */
    int s = c->sink, w = c->window;
    int targets[2], nt = 0;
    if (pos < s) targets[nt++] = pos;
    if (w > 0) targets[nt++] = s + (pos % w);
    for (int k = 0; k < nt; k++) {
        size_t si = idx_side(c, slot, targets[k], head);
        orc_quant_affine(k_rot, ORC_D, 255, c->k8_code + si * ORC_D, c->k8_delta + si, c->k8_min + si);
        orc_quant_affine(v, ORC_D, 255, c->v8_code + si * ORC_D, c->v8_delta + si, c->v8_min + si);
    }
}

/* Append T tokens at positions start … start+T−1, one token at a time in order
   (sequential semantics: the ring ends up holding the last w positions). */
int orc_append(orc_cache *c, int slot, int start, int T,
               const uint16_t *k_bf16, const uint16_t *v_bf16)
{
    if (slot < 0 || slot >= c->num_slots || start < 0 || T < 0 || start + T > c->max_len)
        return -1;
    if (c->format != ORC_FMT_HYBRID && (c->sink != 0 || c->window != 0)) return -1;
    if (c->rope && start + T > c->rope_max_pos) return -1;
    float kx[ORC_D], kp[ORC_D], kr[ORC_D], vx[ORC_D];
    for (int t = 0; t < T; t++) {
        for (int h = 0; h < c->num_heads; h++) {
            size_t off = ((size_t)t * c->num_heads + h) * ORC_D;
            load_bf16_row(k_bf16 + off, kx);
            load_bf16_row(v_bf16 + off, vx);
            if (c->rope) {                          /* R11: RoPE, then the Hadamard rotation */
                orc_rope128(kx, c->rope + (size_t)(start + t) * ORC_D, kp);
                memcpy(kx, kp, sizeof kx);
            }
            orc_fwht128(kx, kr);
            append_one(c, slot, start + t, h, kr, vx);
        }
        c->length[slot] = start + t + 1;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Decode attention for one sequence                                         */
/* ------------------------------------------------------------------------ */

static float log2e_scale(float sm_scale)
{
    return (float)((double)sm_scale * 1.4426950408889634074);
}

/* σ from an integer dot, the code group's FP16 (Δ, m) and the query's (s_q, Σq8).
   [zh] 分组仿射 KV 量化: the scale and offset are applied after the dot product. */
static float score_from_dot(int32_t dot, uint16_t dh, uint16_t mh,
                            float q_scale, int32_t q_sum, float C)
{
    float delta = (float)orc_f16_to_f64(dh);
    float m = (float)orc_f16_to_f64(mh);
    float u = fmaf(delta, (float)dot, m * (float)q_sum);
    return (u * q_scale) * C;
}

static int32_t dot_s8_u8(const int8_t *a, const uint8_t *b)
{
    int32_t s = 0;
    for (int i = 0; i < ORC_D; i++) s += (int32_t)a[i] * (int32_t)b[i];
    return s;
}

/* Side row that holds protected position t (R4): sink row t for t < s, ring row
   s + t mod w otherwise (a ring row keeps the latest position with its residue,
   which for a protected t >= max(s, L - w) is t itself). */
static int side_row_of(int t, int s, int w)
{
    return (t < s) ? t : s + t % w;
}

/* One q head against one sequence. Returns output (normalised) and lse (natural log). */
static void decode_head(const orc_cache *c, int slot, int L, int head,
                        const int8_t *q8, float q_scale, int32_t q_sum, float C,
                        int pv_mode, double *out, double *lse,
                        int32_t *dbg_qk, float *dbg_sigma, uint8_t *dbg_w, uint16_t *dbg_p)
{
    const int s = c->sink, w = c->window, P = 16;
    /* Regions, reading R4 (R10: no INT4 region in KV8). */
    int r4_lo = s, r4_hi = L - w;
    if (r4_hi < r4_lo || c->format != ORC_FMT_HYBRID) r4_hi = r4_lo;   /* empty */

    /* ---- INT4 region: integer QK, page-local integer PV (reading R5) ---- */
    double M4 = -INFINITY, l4 = 0.0;
    double o4[ORC_D];
    for (int j = 0; j < ORC_D; j++) o4[j] = 0.0;
    if (r4_hi > r4_lo) {
        int p_first = r4_lo / P, p_last = (r4_hi - 1) / P;
        float sig_buf[16];
        for (int pg = p_first; pg <= p_last; pg++) {
            int t0 = pg * P, t1 = t0 + P;
            if (t0 < r4_lo) t0 = r4_lo;
            if (t1 > r4_hi) t1 = r4_hi;
            int n = t1 - t0;
            float Mp = -INFINITY;
            for (int i = 0; i < n; i++) {
                int t = t0 + i;
                size_t mi = idx_main(c, slot, t, head);
                int32_t dot = dot_s8_u8(q8, c->k4_code + mi * ORC_D);
                float sg = score_from_dot(dot, c->k4_delta[mi], c->k4_min[mi], q_scale, q_sum, C);
                sig_buf[i] = sg;
                if (dbg_qk) dbg_qk[t] = dot;
                if (dbg_sigma) dbg_sigma[t] = sg;
                if (sg > Mp) Mp = sg;
            }
            float pp[16], wv[16];
            float wmax = 0.0f;
            double lp = 0.0, bias = 0.0;
            for (int i = 0; i < n; i++) {
                size_t mi = idx_main(c, slot, t0 + i, head);
                pp[i] = orc_exp2f(sig_buf[i] - Mp);
                float dv = (float)orc_f16_to_f64(c->v4_delta[mi]);
                float mv = (float)orc_f16_to_f64(c->v4_min[mi]);
                wv[i] = pp[i] * dv;
                if (wv[i] > wmax) wmax = wv[i];
                lp += (double)pp[i];
                bias += (double)pp[i] * (double)mv;
            }
            double op[ORC_D];
            if (pv_mode == ORC_PV_FLOAT) {
                for (int j = 0; j < ORC_D; j++) op[j] = 0.0;
                for (int i = 0; i < n; i++) {
                    size_t mi = idx_main(c, slot, t0 + i, head);
                    double dv = orc_f16_to_f64(c->v4_delta[mi]);
                    double mv = orc_f16_to_f64(c->v4_min[mi]);
                    const uint8_t *vc = c->v4_code + mi * ORC_D;
                    for (int j = 0; j < ORC_D; j++) op[j] += (double)pp[i] * (dv * vc[j] + mv);
                }
            } else {
                /* u8 weights sharing the page's power-of-two scale; pages whose
                   largest weight is below 2^-64 contribute their offsets only */
                uint8_t wh[16];
                int quantize = wmax > 0x1p-64f;
                int e = 0;
                if (quantize) frexpf(wmax, &e);      /* wmax = f·2^e, f in [0.5, 1) */
                e -= 1;                              /* floor(log2(wmax)) */
                for (int i = 0; i < n; i++) {
                    float r = quantize ? rintf(ldexpf(wv[i], 7 - e)) : 0.0f;
                    if (r > 255.0f) r = 255.0f;
                    wh[i] = (uint8_t)r;
                    if (dbg_w) dbg_w[t0 + i] = wh[i];
                }
                double sw = quantize ? ldexp(1.0, e - 7) : 0.0;
                for (int j = 0; j < ORC_D; j++) {
                    int32_t acc = 0;
                    for (int i = 0; i < n; i++) {
                        size_t mi = idx_main(c, slot, t0 + i, head);
                        acc += (int32_t)wh[i] * (int32_t)c->v4_code[mi * ORC_D + j];
                    }
                    op[j] = sw * (double)acc + bias;
                }
            }
            /* fold the page into the region total, relative to the running max */
            double Mn = (Mp > M4) ? Mp : M4;
            double a = (M4 == -INFINITY) ? 0.0 : exp2(M4 - Mn);
            double b = exp2(Mp - Mn);
            for (int j = 0; j < ORC_D; j++) o4[j] = o4[j] * a + op[j] * b;
            l4 = l4 * a + lp * b;
            M4 = Mn;
        }
    }

    /* ---- protected region (R7): the protected positions in position order, taken
       by their 16-position page of the paged cache (the unit of R5's INT4 weights);
       INT8 side keys and BF16 values, p against the page's own max over its
       protected positions; the product takes p rounded to BF16 (integer mode) or
       unrounded (float mode); the normaliser sums the unrounded p. KV8, NVFP4 and
       MXFP4 (R10, R12, R13): every position is protected, codes from the main
       arrays, so a group is a whole page. ---- */
    const int is8 = c->format != ORC_FMT_HYBRID;     /* KV8 and NVFP4: every position, in pages */
    const int isf4 = c->format == ORC_FMT_NVFP4;
    const int ismx = c->format == ORC_FMT_MXFP4;
    const uint8_t *k8c = is8 ? c->k4_code : c->k8_code;
    const uint8_t *v8c = is8 ? c->v4_code : c->v8_code;
    const uint16_t *k8d = is8 ? c->k4_delta : c->k8_delta;
    const uint16_t *k8m = is8 ? c->k4_min : c->k8_min;
    const uint16_t *v8d = is8 ? c->v4_delta : c->v8_delta;
    const uint16_t *v8m = is8 ? c->v4_min : c->v8_min;
    float Mr = -INFINITY;
    double lp_ = 0.0;
    double opr[ORC_D];
    for (int j = 0; j < ORC_D; j++) opr[j] = 0.0;
    /* R4: protected = [0, min(s, L)) ∪ [max(s, L − w), L); whole-cache formats: [0, L) */
    const int win_lo = is8 ? 0 : ((L - w > s) ? L - w : s);
    for (int g0 = 0; g0 < L; g0 += P) {
        const int n = (L - g0 < P) ? L - g0 : P;
        int pos[16];
        size_t rix[16];
        float sg[16];
        float Mg = -INFINITY;
        for (int i = 0; i < n; i++) {
            const int t = g0 + i;
            pos[i] = (is8 || t < s || t >= win_lo) ? t : -1;
            if (pos[i] < 0) continue;
            const size_t si = is8 ? idx_main(c, slot, t, head) : idx_side(c, slot, side_row_of(t, s, w), head);
            rix[i] = si;
            if (ismx) {                              /* R13 */
                sg[i] = score_mxfp4(k8c + si * ORC_D, c->k_bscale + si * 8, q8, q_scale, C);
                if (dbg_sigma) dbg_sigma[pos[i]] = sg[i];
                if (sg[i] > Mg) Mg = sg[i];
                continue;
            }
            if (isf4) {                              /* R12 */
                sg[i] = score_nvfp4(k8c + si * ORC_D, c->k_bscale + si * 8, c->k_gscale[si], q8,
                                    q_scale, C);
                if (dbg_sigma) dbg_sigma[pos[i]] = sg[i];
                if (sg[i] > Mg) Mg = sg[i];
                continue;
            }
            int32_t dot = dot_s8_u8(q8, k8c + si * ORC_D);
            sg[i] = score_from_dot(dot, k8d[si], k8m[si], q_scale, q_sum, C);
            if (dbg_qk) dbg_qk[pos[i]] = dot;
            if (dbg_sigma) dbg_sigma[pos[i]] = sg[i];
            if (sg[i] > Mg) Mg = sg[i];
        }
        if (Mg == -INFINITY) continue;               /* no protected position in this page */
        /* the page's output relative to its own max, then folded into the region
           total relative to the running max */
        double og[ORC_D];
        double lg = 0.0;
        for (int j = 0; j < ORC_D; j++) og[j] = 0.0;
        /* R13: 2^mxk, the largest block scale of the page's positions */
        int mxk = -127;
        if (ismx) {
            for (int i = 0; i < n; i++) {
                if (pos[i] < 0) continue;
                for (int bb = 0; bb < ORC_D / 32; bb++)
                    if ((int)c->v_bscale[rix[i] * 8 + bb] - 127 > mxk) mxk = (int)c->v_bscale[rix[i] * 8 + bb] - 127;
            }
        }
        /* R12: the power of two 2^k just above the largest V vector scale of the page */
        int f4k = -126;
        if (isf4) {
            float mx = 0.0f;
            for (int i = 0; i < n; i++) {
                if (pos[i] < 0) continue;
                if (c->v_gscale[rix[i]] > mx) mx = c->v_gscale[rix[i]];
            }
            if (mx >= FLT_MIN) {
                int k;
                frexpf(mx, &k);                      /* mx in [2^(k-1), 2^k) */
                f4k = k;
            }
        }
        for (int i = 0; i < n; i++) {
            if (pos[i] < 0) continue;
            const size_t si = rix[i];
            const float p = orc_exp2f(sg[i] - Mg);
            const double pw = (pv_mode == ORC_PV_FLOAT)
                                  ? (double)p
                                  : (double)orc_bf16_to_f32(orc_f32_to_bf16_rn(p));
            const uint8_t *vc = v8c + si * ORC_D;
            if (dbg_p) dbg_p[pos[i]] = orc_f32_to_bf16_rn(p);
            if (ismx) {                              /* R13 */
                const float p16 = (float)orc_f16_to_f64(orc_f32_to_f16(p, ORC_RN));
                if (dbg_p) dbg_p[pos[i]] = orc_f32_to_f16(p, ORC_RN);
                for (int bb = 0; bb < ORC_D / 32; bb++) {
                    const int sb = (int)c->v_bscale[si * 8 + bb] - 127;
                    const double wb = (pv_mode == ORC_PV_FLOAT)
                                          ? ldexp((double)p, sb)
                                          : orc_f16_to_f64(orc_f32_to_f16(ldexpf(p16, sb - mxk), ORC_RN));
                    for (int j = 32 * bb; j < 32 * bb + 32; j++)
                        og[j] += wb * (double)orc_e2m1_value(vc[j]);
                }
            } else if (isf4) {                       /* R12 */
                const float gi = c->v_gscale[si];
                if (pv_mode == ORC_PV_FLOAT) {       /* exact values, unrounded p */
                    for (int j = 0; j < ORC_D; j++)
                        og[j] += (double)p * (double)orc_e2m1_value(vc[j]) *
                                 (double)orc_e4m3_value(c->v_bscale[si * 8 + j / 16]) * (double)gi;
                } else {                             /* fp16 weights carrying the value scales */
                    const float wn = ldexpf(p * gi, -f4k);
                    const float w1 = (float)orc_f16_to_f64(orc_f32_to_f16(wn, ORC_RN));
                    if (dbg_p) dbg_p[pos[i]] = orc_f32_to_f16(wn, ORC_RN);
                    for (int bb = 0; bb < ORC_D / 16; bb++) {
                        const float sb = orc_e4m3_value(c->v_bscale[si * 8 + bb]);
                        const double wb = orc_f16_to_f64(orc_f32_to_f16(w1 * sb, ORC_RN));
                        for (int j = 16 * bb; j < 16 * bb + 16; j++)
                            og[j] += wb * (double)orc_e2m1_value(vc[j]);
                    }
                }
            } else {
                float dv = (float)orc_f16_to_f64(v8d[si]);
                float mv = (float)orc_f16_to_f64(v8m[si]);
                for (int j = 0; j < ORC_D; j++) {
                    float v = orc_bf16_to_f32(orc_f32_to_bf16_rn(fmaf(dv, (float)vc[j], mv)));
                    og[j] += pw * (double)v;
                }
            }
            lg += (double)p;
        }
        if (isf4 && pv_mode != ORC_PV_FLOAT)
            for (int j = 0; j < ORC_D; j++) og[j] = ldexp(og[j], f4k);
        if (ismx && pv_mode != ORC_PV_FLOAT)
            for (int j = 0; j < ORC_D; j++) og[j] = ldexp(og[j], mxk);
        const float Mn = (Mg > Mr) ? Mg : Mr;
        const double a = (Mr == -INFINITY) ? 0.0 : exp2((double)Mr - (double)Mn);
        const double bsc = exp2((double)Mg - (double)Mn);
        for (int j = 0; j < ORC_D; j++) opr[j] = opr[j] * a + og[j] * bsc;
        lp_ = lp_ * a + lg * bsc;
        Mr = Mn;
    }
    const double Mp_ = (double)Mr;

    /* ---- exact log-sum-exp merge of the two regions ---- */
    double Ms = (M4 > Mp_) ? M4 : Mp_;
    if (Ms == -INFINITY) {                          /* L == 0 */
        for (int j = 0; j < ORC_D; j++) out[j] = 0.0;
        *lse = -INFINITY;
        return;
    }
    double a4 = (M4 == -INFINITY) ? 0.0 : exp2(M4 - Ms);
    double ap = (Mp_ == -INFINITY) ? 0.0 : exp2(Mp_ - Ms);
    double den = a4 * l4 + ap * lp_;
    for (int j = 0; j < ORC_D; j++) out[j] = (a4 * o4[j] + ap * opr[j]) / den;
    *lse = (Ms + log2(den)) * 0.69314718055994530942;
}

/* R11: the query of a decode step sits at position L − 1 */
static void query_rope(const orc_cache *c, int L, float *qx)
{
    if (!c->rope || L <= 0) return;
    float qp[ORC_D];
    orc_rope128(qx, c->rope + (size_t)(L - 1) * ORC_D, qp);
    memcpy(qx, qp, sizeof qp);
}

int orc_decode(const orc_cache *c, int slot, int L, int G, const uint16_t *q_bf16,
               float sm_scale, int pv_mode, double *out, double *lse, orc_debug *dbg)
{
    if (slot < 0 || slot >= c->num_slots || L < 0 || L > c->max_len || G <= 0)
        return -1;
    if (c->sink + c->window > 256) return -1;
    if (c->format != ORC_FMT_HYBRID && (c->sink != 0 || c->window != 0)) return -1;
    if (c->rope && L > c->rope_max_pos) return -1;
    const float C = log2e_scale(sm_scale);
    const int HG = c->num_heads * G;
    for (int hq = 0; hq < HG; hq++) {
        float qx[ORC_D], qr[ORC_D];
        int8_t q8[ORC_D];
        float q_scale;
        int32_t q_sum;
        load_bf16_row(q_bf16 + (size_t)hq * ORC_D, qx);
        query_rope(c, L, qx);
        orc_fwht128(qx, qr);
        orc_quant_query(qr, q8, &q_scale, &q_sum);
        if (dbg) {
            if (dbg->q8) memcpy(dbg->q8 + (size_t)hq * ORC_D, q8, ORC_D);
            if (dbg->q_scale) dbg->q_scale[hq] = q_scale;
            if (dbg->q_sum) dbg->q_sum[hq] = q_sum;
        }
        decode_head(c, slot, L, hq / G, q8, q_scale, q_sum, C, pv_mode,
                    out + (size_t)hq * ORC_D, lse + hq,
                    dbg && dbg->qk ? dbg->qk + (size_t)hq * L : NULL,
                    dbg && dbg->sigma ? dbg->sigma + (size_t)hq * L : NULL,
                    dbg && dbg->w_hat ? dbg->w_hat + (size_t)hq * L : NULL,
                    dbg && dbg->p_bits ? dbg->p_bits + (size_t)hq * L : NULL);
    }
    return 0;
}

/* One q head of one sequence (the unit the batch entry spreads over threads). */
static int decode_one_head(const orc_cache *c, int slot, int L, int G, int hq,
                           const uint16_t *q_row, float C, int pv_mode, double *out, double *lse)
{
    float qx[ORC_D], qr[ORC_D];
    int8_t q8[ORC_D];
    float q_scale;
    int32_t q_sum;
    load_bf16_row(q_row, qx);
    query_rope(c, L, qx);
    orc_fwht128(qx, qr);
    orc_quant_query(qr, q8, &q_scale, &q_sum);
    decode_head(c, slot, L, hq / G, q8, q_scale, q_sum, C, pv_mode, out, lse, NULL, NULL, NULL, NULL);
    return 0;
}

/* A batch of sequences, spread over host threads by (sequence, q head) (CPU baseline). */
int orc_decode_batch(const orc_cache *c, int B, const int32_t *slots, const int32_t *lens,
                     int G, const uint16_t *q_bf16, float sm_scale, int pv_mode,
                     double *out, double *lse, int num_threads)
{
    const int HG = c->num_heads * G;
    const float C = log2e_scale(sm_scale);
    for (int b = 0; b < B; b++)
        if (slots[b] < 0 || slots[b] >= c->num_slots || lens[b] < 0 || lens[b] > c->max_len ||
            (c->rope && lens[b] > c->rope_max_pos))
            return -1;
    if (G <= 0 || c->sink + c->window > 256) return -1;
    if (c->format != ORC_FMT_HYBRID && (c->sink != 0 || c->window != 0)) return -1;
    const long n = (long)B * HG;
#ifdef _OPENMP
    if (num_threads > 0) omp_set_num_threads(num_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long i = 0; i < n; i++) {
        int b = (int)(i / HG), hq = (int)(i % HG);
        decode_one_head(c, slots[b], lens[b], G, hq, q_bf16 + ((size_t)b * HG + hq) * ORC_D, C,
                        pv_mode, out + ((size_t)b * HG + hq) * ORC_D, lse + (size_t)b * HG + hq);
    }
    (void)num_threads;
    return 0;
}

/* Array forms of the scalar conversions, for the tests' bulk checks. */
void orc_f32_to_f16_array(const float *x, uint16_t *out, int64_t n, int mode)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_f32_to_f16(x[i], mode);
}

void orc_f32_to_bf16_array(const float *x, uint16_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_f32_to_bf16_rn(x[i]);
}

void orc_exp2f_array(const float *x, float *out, int64_t n)
{
    for (int64_t i = 0; i < n; i++) out[i] = orc_exp2f(x[i]);
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
