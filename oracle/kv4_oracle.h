/*
 * kv4_oracle.h — plain CPU oracle for the KV4-RL rollout decode hot path.
 *
 * TEST INFRASTRUCTURE ONLY. The test suite, the smoke check and the CPU-baseline
 * leg of the benchmark are the only users of this library. The product path
 * (libkv4 and its Python binding) never loads it, and the two share no code.
 *
 * Pages cited (title, then section):
 *   [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速"
 *        (paper.rainbus.top/paper/2610.14448)
 *   [ko] "INT4 KV 캐시로 비동기 RLVR 롤아웃을 1.8배 가속한다" (onedev.kr/papers/984)
 *
 * The state is LOGICAL, not paged: codes are held one byte per element, in
 * [slot][position][kv_head][128] order, with FP16 metadata beside them. The
 * GPU path's paged layout is decoded back to this form by the tests.
 */
#ifndef KV4_ORACLE_H
#define KV4_ORACLE_H
#include <stdint.h>

#define ORC_D 128

#ifdef __cplusplus
extern "C" {
#endif

/* FP16 rounding modes for orc_f32_to_f16. */
enum { ORC_RN = 0, ORC_RD = 1, ORC_RU = 2 };
/* Cache formats. */
enum { ORC_FMT_HYBRID = 0, ORC_FMT_KV8 = 1, ORC_FMT_NVFP4 = 2, ORC_FMT_MXFP4 = 3 };
/* PV modes for the INT4 region of orc_decode. */
enum { ORC_PV_INTEGER = 0, ORC_PV_FLOAT = 1 };

typedef struct {
    int32_t num_heads;   /* H_kv */
    int32_t sink;        /* s */
    int32_t window;      /* w */
    int32_t max_len;     /* positions per slot */
    int32_t num_slots;
    int32_t format;      /* ORC_FMT_HYBRID: INT4 main cache + INT8 side buffer; ORC_FMT_KV8:
                            whole-cache INT8 (the main arrays hold 8-bit codes); ORC_FMT_NVFP4:
                            whole-cache NVFP4 (E2M1 codes in the main arrays, block and vector
                            scales below); ORC_FMT_MXFP4: whole-cache MXFP4 (E2M1 codes in the
                            main arrays, E8M0 scales of the four 32-value blocks in the first
                            four block-scale bytes); the last three have sink = window = 0 */
    /* INT4 main cache: codes [slot][pos][head][128] in 0..15 (0..255 in KV8), meta
       [slot][pos][head] fp16 bits */
    uint8_t  *k4_code, *v4_code;
    uint16_t *k4_delta, *k4_min, *v4_delta, *v4_min;
    /* INT8 side cache: codes [slot][s+w][head][128] in 0..255, meta [slot][s+w][head] fp16 bits.
       Side index of position p: p for a sink position, s + (p mod w) for a ring position. */
    uint8_t  *k8_code, *v8_code;
    uint16_t *k8_delta, *k8_min, *v8_delta, *v8_min;
    int32_t  *length;    /* [slot] positions appended so far */
    /* RoPE (reading R11), or NULL: keys given to orc_append and queries given to decode
       are then pre-RoPE. Table [rope_max_pos][128]: cos of the angle of pair i at [p][i],
       its sin at [p][64 + i] (i < 64). */
    const float *rope;
    int32_t  rope_max_pos;
    /* NVFP4 scales (reading R12): E4M3 bits of the 8 block scales [slot][pos][head][8] and
       the FP32 vector scale [slot][pos][head], for K and V */
    uint8_t  *k_bscale, *v_bscale;
    float    *k_gscale, *v_gscale;
} orc_cache;

/* Optional per-call debug record of orc_decode (any pointer may be NULL).
   Rows are q heads hq = h*G + g; columns of the [HG][L] arrays are positions. */
typedef struct {
    int8_t  *q8;        /* [HG][128] */
    float   *q_scale;   /* [HG] s_q */
    int32_t *q_sum;     /* [HG] sum of q8 */
    int32_t *qk;        /* [HG][L] integer QK accumulator of the region that owns the position */
    float   *sigma;     /* [HG][L] log2-domain score */
    uint8_t *w_hat;     /* [HG][L] u8 PV weight (INT4 region only; 0 elsewhere) */
    uint16_t *p_bits;   /* [HG][L] bits of each protected position's PV weight as the
                           product takes it: BF16 p (hybrid protected region, KV8), fp16
                           fl(p·g)·2^-k (NVFP4, before the block scale), fp16 p (MXFP4);
                           0 in the INT4 region */
} orc_debug;

/* number formats */
double   orc_f16_to_f64(uint16_t h);
uint16_t orc_f32_to_f16(float x, int mode);
float    orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16_rn(float x);
float    orc_exp2f(float x);

/* steps */
void orc_fwht128(const float *in, float *out);
void orc_rope128(const float *in, const float *cos_sin_row, float *out);
void orc_quant_affine(const float *x, int n, int levels,
                      uint8_t *code, uint16_t *delta_h, uint16_t *min_h);
void orc_quant_query(const float *q_rot, int8_t *q8, float *q_scale, int32_t *q_sum);
uint8_t orc_e4m3_rn(float t);               /* t >= 0, round to nearest even, saturating at 448 */
float   orc_e4m3_value(uint8_t bits);
uint8_t orc_e2m1_rn(float v);               /* sign | magnitude code, nearest even, saturating at 6 */
float   orc_e2m1_value(uint8_t code);
void    orc_quant_nvfp4(const float *x, uint8_t *codes, uint8_t *bscale, float *gscale);
void    orc_quant_mxfp4(const float *x, uint8_t *codes, uint8_t *escale);

/* whole path */
int orc_append(orc_cache *c, int slot, int start, int T,
               const uint16_t *k_bf16, const uint16_t *v_bf16);
int orc_decode(const orc_cache *c, int slot, int L, int G, const uint16_t *q_bf16,
               float sm_scale, int pv_mode, double *out, double *lse, orc_debug *dbg);
int orc_decode_batch(const orc_cache *c, int B, const int32_t *slots, const int32_t *lens,
                     int G, const uint16_t *q_bf16, float sm_scale, int pv_mode,
                     double *out, double *lse, int num_threads);
int orc_num_threads(void);

void orc_f32_to_f16_array(const float *x, uint16_t *out, int64_t n, int mode);
void orc_f32_to_bf16_array(const float *x, uint16_t *out, int64_t n);
void orc_exp2f_array(const float *x, float *out, int64_t n);

#ifdef __cplusplus
}
#endif
#endif
