/*
 * kv4.h — C ABI of libkv4: the KV4-RL rollout decode hot path on GB300 (sm_103a).
 *
 * A paged INT4 KV cache holds every position; a fixed-size INT8 side buffer
 * holds s sink positions and the w most recent positions of each sequence.
 * Decode attention reads the two regions disjointly and merges them exactly.
 *
 * Pages cited (title, then section):
 *   [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速"
 *        (paper.rainbus.top/paper/2610.14448)
 *   [ko] "INT4 KV 캐시로 비동기 RLVR 롤아웃을 1.8배 가속한다" (onedev.kr/papers/984)
 *
 * Conventions for every call
 *   - Pointers named *_dev are device pointers; the caller owns them. The cache
 *     owns its pools and its decode workspace.
 *   - Calls are asynchronous on the caller's CUDA stream (`stream`, a
 *     cudaStream_t passed as void*; NULL = legacy default stream). Host-side
 *     validation happens before anything is enqueued; a call that returns an
 *     error has enqueued nothing.
 *   - Index errors that only the device can see (a slot, page or length out of
 *     range inside a device array) never fault: the kernel skips the access and
 *     records the first such error in a device error word, read with
 *     kv4_get_device_error(). No call traps, aborts or throws across the ABI.
 *   - head_dim is 128 and page_size is 16; other values return KV4_ERR_UNSUPPORTED.
 *   - A call that takes a cache runs on the device the cache was created on: it makes
 *     that device current for the call and restores the caller's device before it
 *     returns. The stream passed must belong to that device.
 */
#ifndef KV4_H
#define KV4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct kv4_cache kv4_cache;

typedef enum {
    KV4_OK = 0,
    KV4_ERR_INVALID_ARG = -1,   /* null pointer, negative size, inconsistent sizes */
    KV4_ERR_UNSUPPORTED = -2,   /* head_dim != 128, page_size != 16, s + w > 256, s or w not a
                                   multiple of 16, group size */
    KV4_ERR_OUT_OF_MEMORY = -3, /* a pool or workspace allocation failed at create */
    KV4_ERR_CUDA = -4,          /* a CUDA runtime call failed; the cache stays usable if it can */
    KV4_ERR_OUT_OF_RANGE = -5,  /* batch, q heads or tokens above the cache's configured limits */
    KV4_ERR_DEVICE_FAULT = -6   /* reported by kv4_get_device_error: see kv4_device_error */
} kv4_status;

/* Codes stored in the device error word (first error wins; 0 = none). */
typedef enum {
    KV4_DEVERR_NONE = 0,
    KV4_DEVERR_BAD_SLOT = 1,       /* slot id outside [0, max_slots) */
    KV4_DEVERR_BAD_PAGE = 2,       /* block-table entry outside [0, num_pages) */
    KV4_DEVERR_BAD_POSITION = 3,   /* position beyond block_table_stride pages, or negative */
    KV4_DEVERR_LEN_MISMATCH = 4,   /* decode context_len differs from the slot's appended length */
    KV4_DEVERR_WAIT_TIMEOUT = 5,   /* a shared-memory staging wait gave up (no data arrived) */
    KV4_DEVERR_BAD_TOKENS = 6      /* cu_tokens not non-decreasing or not ending at total_tokens */
} kv4_device_error;

/* Cache formats. KV4_FORMAT_INT4_HYBRID is the method: INT4 pages for every
 * position plus the bounded INT8 side buffer of sink and recent positions.
 * KV4_FORMAT_INT8 is the whole-cache 8-bit configuration the pages compare it
 * against (KV8, [zh] 核心发现 (2)): the same 8-bit group-affine codes as the side
 * buffer for every position, in pages, and no side buffer (sink = window = 0). */
typedef enum {
    KV4_FORMAT_INT4_HYBRID = 0,
    KV4_FORMAT_INT8 = 1,
    KV4_FORMAT_NVFP4 = 2,     /* NVFP4 for every position (E2M1 values, E4M3 scales per 16
                                 dims, an FP32 scale per token-head vector), no side buffer */
    KV4_FORMAT_MXFP4 = 3      /* MXFP4 for every position (E2M1 values, an E8M0 power-of-two
                                 scale per 32 dims), no side buffer */
} kv4_format;

typedef struct {
    int32_t num_kv_heads;    /* H_kv >= 1 */
    int32_t head_dim;        /* must be 128 (one quantization group per token-head, [zh] 分组仿射 KV 量化) */
    int32_t page_size;       /* must be 16 */
    int32_t sink;            /* s >= 0: INT8-protected sink positions (16 in [zh] 核心方法) */
    int32_t window;          /* w >= 0: INT8-protected recent positions (128 in [zh] 核心方法); s + w <= 256;
                                s and w multiples of 16 (the protected weights are formed per page,
                                and this keeps each page's protected rows in one side group) */
    int64_t num_pages;       /* physical pages in the INT4 pool (each holds 16 positions of every KV head) */
    int32_t max_slots;       /* sequences that own a side buffer (slot ids are 0 .. max_slots-1) */
    int32_t max_batch;       /* largest batch of one decode call */
    int32_t max_q_heads;     /* largest H_q of one decode call (H_q = G * H_kv, G in {1, 2, 4}) */
    int32_t max_work_items;  /* reserved: must be >= 0 and is otherwise ignored (the decode
                                workspace is sized from max_batch, max_q_heads and the SM count) */
    int32_t format;          /* kv4_format; KV4_FORMAT_INT8, KV4_FORMAT_NVFP4 and
                                KV4_FORMAT_MXFP4 require sink = window = 0 */
} kv4_cache_config;

/*
 * Memory layout (all blocks 16-byte aligned; pools zeroed at create).
 *
 * INT4 page pool: num_pages * H_kv blocks of KV4_PAGE_BLOCK_BYTES = 2176 bytes;
 * the block of (page p, KV head h) starts at (p * H_kv + h) * 2176. Inside it,
 * for the 16 token slots t of the page:
 *   [0,    1024)  K codes (rotated K): tokens t and t+8 (t < 8) share bytes, token t in
 *                 the low nibble. Code d of token t sits in the byte at
 *                 512*(i/4) + 16*(4*(t%8) + d/32) + 4*(i%4) + {0, 2, 1, 3}[d%4] with
 *                 i = (d%32)/4 (two planes of eight 16-byte slots per token pair)
 *   [1024, 2048)  V codes: one byte per (dim pair j, token t) = c_t[2j] | c_t[2j+1] << 4, at
 *                 offset 4*(8*(4*(j%8) + t%4) + j/8) + t/4 (32 groups of eight 32-bit
 *                 words; each word holds one dim pair of tokens u, u+4, u+8, u+12 with
 *                 u = t%4, one tensor-core fragment)
 *   [2048, 2176)  K and V metadata, {fp16 delta, fp16 min} (4 bytes) per token: 8 rows
 *                 of 16 bytes, row r = [K of token r | K of token r+8 | V of token r |
 *                 V of token r+8], so one 16-byte load brings both tokens a lane scores
 * Side pool: max_slots * H_kv blocks of side_block_bytes = ceil((s+w)/16) * 4352;
 * block (slot, h) at (slot * H_kv + h) * side_block_bytes. Side row i (i = p for a
 * sink position p < s, i = s + p mod w for a ring position) is row r = i%16 of group
 * i/16; group g starts at g * 4352 and holds two 2176-byte blocks. For dim d write
 * W = (d%32)/4; a code byte (u8, INT8 grid) sits at:
 *   K block [0, 2176):    1024*(W/4) + 64*r + 16*(d/32) + 4*(W%4) + d%4   (rotated K)
 *                         K metadata {fp16 delta, fp16 min} of row r at 2048 + 8*(r%8) + 4*(r/8)
 *   V block [2176, 4352): with n = 4*(d%8) + r%4, W' = 2*(d/16) + (d/8)%2 and
 *                         b' = (r/8)%2 + 2*((r/4)%2): 2176 + 16*(32*(W'/4) + n) + 4*(W'%4) + b'
 *                         V metadata of row r at 2176 + 2048 + 16*(r%4) + 4*b'
 * so each lane of a warp reads its tensor-core fragments with 16-byte loads.
 * KV4_FORMAT_INT8 pages: num_pages * H_kv blocks of KV4_PAGE_BLOCK_BYTES_INT8 = 4352
 * bytes, block (p, h) at (p * H_kv + h) * 4352, each laid out as one side group
 * above with row r = t, the page's token slot t; there is no side pool.
 * KV4_FORMAT_NVFP4 pages: num_pages * H_kv blocks of KV4_PAGE_BLOCK_BYTES_NVFP4 = 2432 bytes,
 * block (p, h) at (p * H_kv + h) * 2432: a K half at 0 and a V half at 1216, each with
 *   [0, 1024)    E2M1 codes (sign in bit 3), two per byte:
 *                K: one byte per (token, dim pair): dims 2j (low nibble) and 2j+1 (high)
 *                   of token t, j = 8b + jj (block b, jj < 8), at
 *                   16*(32*(b/4) + 4*(t%8) + jj%4) + 4*(b%4) + t/8 + 2*(jj/4)
 *                V: one byte per (dim, token pair): dim d = 16m + r (r < 16) of tokens
 *                   t (low nibble) and t+8 (high nibble), t%16 < 8, at
 *                   16*(32*(m/4) + 4*(r%8) + t%4) + 4*(m%4) + 2*((t/4)%2) + r/8
 *                   (an append writes a token's nibbles with atomic clear-and-set of
 *                   their 32-bit word, which holds four tokens' nibbles)
 *   [1024, 1152) E4M3 block scales (block b = dims 16b .. 16b+15) of token t:
 *                K: byte 16*(t%8) + 2*b + t/8      (tokens t, t+8 of a block paired)
 *                V: byte 32*(t%4) + 4*b + {0,2,1,3}[t/4]  (tokens t, t+8, t+4, t+12)
 *   [1152, 1216) FP32 vector scales, float of token t at byte 8*(t%8) + 4*(t/8)
 * KV4_FORMAT_MXFP4 pages: num_pages * H_kv blocks of KV4_PAGE_BLOCK_BYTES_MXFP4 = 2176 bytes,
 * block (p, h) at (p * H_kv + h) * 2176: a K half at 0 and a V half at 1088, each with
 *   [0, 1024)    E2M1 codes, bytes as in KV4_FORMAT_NVFP4
 *   [1024, 1088) E8M0 scales (biased exponents s + 127) of block b = dims 32b .. 32b+31
 *                of token t: K: byte 8*(t%8) + 2*b + t/8; V: byte 16*(t%4) + 4*b +
 *                {0,2,1,3}[t/4]
 * Lengths: int32 per slot, the slot's length after its last append.
 */
#define KV4_HEAD_DIM 128
#define KV4_PAGE_SIZE 16
#define KV4_PAGE_BLOCK_BYTES 2176
#define KV4_PAGE_BLOCK_BYTES_INT8 4352
#define KV4_PAGE_BLOCK_BYTES_NVFP4 2432
#define KV4_PAGE_BLOCK_BYTES_MXFP4 2176

typedef struct {
    void   *page_pool_dev;   size_t page_pool_bytes;
    void   *side_pool_dev;   size_t side_pool_bytes;   size_t side_block_bytes;   /* per (slot, head) */
    int32_t *seq_len_dev;    /* [max_slots] */
    int32_t num_sms;         /* SMs of the device the cache lives on */
    int32_t decode_grid;     /* persistent CTAs launched by decode */
    int32_t device;
} kv4_cache_info;

/* Allocate the pools and the decode workspace on the current device (cudaMalloc),
 * zero them, size the persistent decode grid. *out receives the handle.
 * Errors: KV4_ERR_INVALID_ARG, KV4_ERR_UNSUPPORTED, KV4_ERR_OUT_OF_MEMORY, KV4_ERR_CUDA. */
kv4_status kv4_cache_create(const kv4_cache_config *config, kv4_cache **out);

/* Free everything the cache owns (synchronises the device first). NULL is a no-op. */
kv4_status kv4_cache_free(kv4_cache *cache);

/* Pointers and sizes of the cache's pools (for inspection and tests). */
kv4_status kv4_cache_get_info(const kv4_cache *cache, kv4_cache_info *info);

/*
 * kv4_cache_set_rope — fuse RoPE into the cache's appends and decodes.
 * [zh] 核心方法 (keys take the Hadamard rotation after RoPE), 方法步骤详情 step 2
 * (the query takes the same rotations before attention).
 * With a table set, kv4_append takes PRE-RoPE keys and rotates each key by RoPE at
 * its position before the Hadamard transform, and kv4_decode_attention(_debug)
 * takes PRE-RoPE queries and rotates the query of sequence b at position L_b - 1.
 * Pairs are (i, i + 64) ("rotate half"): with a = x_i, b = x_{i+64},
 * x_i' = fmaf(a, cos, -(b*sin)) and x_{i+64}' = fmaf(b, cos, a*sin) in FP32.
 *   cos_sin_dev : [max_pos][128] fp32 device table, 16-byte aligned, owned by the caller
 *                 and valid while set: cos of pair i at position p at [p][i], its sin
 *                 at [p][64 + i]; NULL clears the setting (inputs are post-RoPE again)
 *   max_pos     : rows of the table (>= 1 when cos_sin_dev is set)
 * A position at or beyond max_pos is a device-side error (KV4_DEVERR_BAD_POSITION):
 * an append skips the sequence, a decode uses the unrotated query. Errors:
 * KV4_ERR_INVALID_ARG. kv4_decode_attention_noalloc never applies RoPE.
 */
kv4_status kv4_cache_set_rope(kv4_cache *cache, const float *cos_sin_dev, int max_pos);

/*
 * kv4_append — quantize and store new tokens of n_seqs sequences.
 * [zh] 方法步骤详情 steps 2-3, 前置知识 › 分组仿射 KV 量化; [ko] 전제와 한계.
 * For each token-head: rotate K (post-RoPE, supplied by the caller) with the
 * orthonormal 128-point Hadamard transform H/sqrt(128); quantize rotated K and
 * (unrotated) V to 4-bit affine codes with fp16 delta = up-rounded step and
 * fp16 min = down-rounded minimum; write them to page block_table[i][pos/16],
 * slot pos%16. A position p < s also gets an 8-bit copy in sink row p; a
 * position p >= L_new - w (L_new = start_pos[i] + its token count) gets an
 * 8-bit copy in ring row s + p mod w. The slot's length becomes L_new.
 * KV4_FORMAT_INT8 caches store the 8-bit codes (n = 255, same rounding) of
 * rotated K and V for every position in row pos%16 of the page's block instead;
 * KV4_FORMAT_NVFP4 caches store the NVFP4 codes and scales of rotated K and V:
 * g = amax / 2688, s_b = e4m3(amax_b / fl(6 g)), code = e2m1(x * fl(1 / fl(s_b g)))
 * (nearest, ties to even, saturating).
 *   k_bf16_dev, v_bf16_dev : [total_tokens][H_kv][128] bf16, finite, tokens of sequence
 *                            i at rows cu_tokens[i] .. cu_tokens[i+1]-1 (an infinite or
 *                            NaN value makes its token-head's codes and scales undefined)
 *   cu_tokens_dev          : [n_seqs+1] int32, non-decreasing, cu[0] = 0, cu[n] = total_tokens
 *   slot_ids_dev           : [n_seqs] int32 side-buffer slot of each sequence (distinct)
 *   start_pos_dev          : [n_seqs] int32 position of each sequence's first new token
 *   block_table_dev        : [n_seqs][block_table_stride] int32 physical page per 16 positions
 * Sequences must not repeat a slot within one call. Appends of one slot must be
 * issued in position order on one stream (a later call sees earlier writes).
 */
kv4_status kv4_append(kv4_cache *cache, const void *k_bf16_dev, const void *v_bf16_dev,
                      const int32_t *cu_tokens_dev, const int32_t *slot_ids_dev,
                      const int32_t *start_pos_dev, const int32_t *block_table_dev,
                      int block_table_stride, int n_seqs, int total_tokens, void *stream);

/*
 * kv4_decode_attention — one decode step of attention for a batch of sequences.
 * [ko] 전제와 한계; [zh] 核心方法, 方法步骤详情 step 4.
 * Per q head (q head hq uses KV head hq / G, G = num_q_heads / H_kv):
 *   q' = Hadamard(q); q8 = rint(q' * 127/max|q'|) with s_q = max|q'|/127.
 *   INT4 region [s, L-w): integer dot q8 . c, score scale/offset applied after
 *     the dot; per page, p' = 2^(sigma - page max) and w = p' * Delta_V, quantized to
 *     u8 with one power-of-two scale per page: e = floor(log2 max w),
 *     w^ = min(rint(w * 2^(7-e)), 255); integer PV sum w^ * c_V, page output
 *     2^(e-7) * sum + sum p' * m_V, pages rescaled in FP32.
 *   Protected region [0, min(s,L)) U [max(s, L-w), L): the same q8 against INT8
 *     side keys; per 16-position page of the protected positions, p = 2^(sigma -
 *     that page's max) rounded to bf16, side values dequantized to bf16, PV
 *     accumulated in FP32.
 *   The regions' outputs and log-normalizers are merged exactly (log-sum-exp),
 *   split-K partials over pages likewise.
 *   KV4_FORMAT_INT8 caches: every position takes the protected region's arithmetic
 *   (INT8 keys, bf16 weights and values, FP32 PV) from its page.
 *   KV4_FORMAT_NVFP4 caches: the same q8 against the E2M1 keys, block dots exact and
 *   scaled after the dot (fma chain over the blocks, then g, s_q); per page, the exact
 *   E2M1 values times fp16 weights that carry the value scales,
 *   fp16(fp16(p * g * 2^-k) * s_b) with 2^k the power of two just above the page's
 *   largest V vector scale, FP32 PV scaled by 2^k.
 *   q_bf16_dev       : [batch][num_q_heads][128] bf16 (post-RoPE, unrotated)
 *   slot_ids_dev     : [batch] int32
 *   context_lens_dev : [batch] int32 L_b, including the token appended this step;
 *                      must equal the slot's appended length
 *   block_table_dev  : [batch][block_table_stride] int32
 *   sm_scale         : softmax scale (1/sqrt(128) for standard attention)
 *   out_dev          : [batch][num_q_heads][128] fp32, normalized output
 *   lse_dev          : [batch][num_q_heads] fp32 natural-log normalizer, or NULL
 * L_b = 0 gives a zero output and lse = -inf. Uses the cache's workspace, so
 * decode calls on one cache must not overlap (issue them on one stream).
 */
kv4_status kv4_decode_attention(kv4_cache *cache, const void *q_bf16_dev, int num_q_heads,
                                const int32_t *slot_ids_dev, const int32_t *context_lens_dev,
                                const int32_t *block_table_dev, int block_table_stride, int batch,
                                float sm_scale, float *out_dev, float *lse_dev, void *stream);

/*
 * kv4_decode_attention_debug — the same kernels, also writing their integer
 * intermediates (any pointer may be NULL):
 *   q8_dev     : [batch][num_q_heads][128] int8 quantized rotated query
 *   q_scale_dev: [batch][num_q_heads] fp32 s_q
 *   qk_dev     : [batch][num_q_heads][debug_stride] int32 QK accumulator per position
 *                (INT4 codes in the INT4 region, INT8 side codes in the protected region,
 *                INT8 page codes in KV4_FORMAT_INT8); KV4_FORMAT_NVFP4 has no single
 *                integer dot, and the record holds the bits of the FP32 score sigma
 *                (log2 domain: the block-scaled dot times g, s_q and sm_scale * log2 e)
 *   w_hat_dev  : [batch][num_q_heads][debug_stride] u8 PV weight per INT4-region position
 *   p_bits_dev : [batch][num_q_heads][debug_stride] uint16 bits of the PV weight of each
 *                protected position as the product takes it: BF16 p (hybrid protected
 *                region, KV4_FORMAT_INT8), fp16 p·g·2^-k before the block scale (NVFP4),
 *                fp16 p before the block powers of two (MXFP4)
 * Positions >= debug_stride are not written. For tests; slower than the plain call.
 */
kv4_status kv4_decode_attention_debug(kv4_cache *cache, const void *q_bf16_dev, int num_q_heads,
                                      const int32_t *slot_ids_dev, const int32_t *context_lens_dev,
                                      const int32_t *block_table_dev, int block_table_stride,
                                      int batch, float sm_scale, float *out_dev, float *lse_dev,
                                      int8_t *q8_dev, float *q_scale_dev, int32_t *qk_dev,
                                      uint8_t *w_hat_dev, uint16_t *p_bits_dev, int debug_stride,
                                      void *stream);

/*
 * kv4_decode_attention_noalloc — the same decode attention for callers that
 * cannot allocate device memory: for example code that runs inside a host
 * framework whose allocator has already reserved the whole GPU for its own
 * arena, or a plugin that is handed device buffers but has no right to call
 * cudaMalloc itself. The paper has no counterpart of this entry point.
 * It reads the pools through plain pointers laid out as described above (the
 * caller may own them, or take them from kv4_cache_get_info), and it keeps its
 * split-K scratch in a 16 MiB array that libkv4 reserves statically on every
 * GPU that loads it, until the process exits. The call itself allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 * A page is read whole, including its slots past a sequence's length, whose
 * scores are masked: those slots must hold finite metadata and scales, as a
 * zeroed pool (what kv4_cache_create makes) or earlier appends leave them.
 *   config          : the cache geometry the pools were built with
 *   page_pool_dev, side_pool_dev, seq_len_dev : the pools (16-byte aligned) and slot lengths
 *                     (side_pool_dev may be NULL for a KV4_FORMAT_INT8, KV4_FORMAT_MXFP4 or
 *                     KV4_FORMAT_NVFP4 configuration)
 *   other arguments : as kv4_decode_attention
 * Limits: batch <= 4096, and the call's workspace must fit in the 16 MiB. The
 * workspace is six sections, each rounded up to a multiple of 256 bytes: a 16-byte
 * plan header; 4 * (batch + 1) bytes of cost starts; 4 * (batch * H_kv + 1) bytes of
 * unit offsets; 144 bytes per q head (batch * H_q); and 8 * G and 512 * G bytes for
 * each of 2 * batch * H_kv + W partials, W being the persistent warps of the decode
 * grid (16 per resident CTA, one CTA per SM on a GB300). On a 152-SM GB300 with
 * H_q = 32, H_kv = 8 that admits batch <= 308. The limit depends on the SM count and
 * the occupancy; KV4_ERR_OUT_OF_RANGE, returned before anything is enqueued, is the
 * authoritative check. The first call on each device looks up the device addresses of
 * the scratch array and of an error word with that device current; make that first
 * call before any stream capture. Every call on a device shares the one array and
 * leaves its contents behind (each call writes everything it reads there before
 * reading it), so calls whose kernels overlap on the GPU race: issue them on one
 * stream. Device-side errors (index errors, which are skipped, and staging waits that
 * gave up, which leave out and lse of that call incomplete) go to that error word,
 * first error wins: read it with kv4_get_device_error(NULL, ...) with the device
 * current.
 */
kv4_status kv4_decode_attention_noalloc(const kv4_cache_config *config,
                                        const void *page_pool_dev, const void *side_pool_dev,
                                        const int32_t *seq_len_dev, const void *q_bf16_dev,
                                        int num_q_heads, const int32_t *slot_ids_dev,
                                        const int32_t *context_lens_dev,
                                        const int32_t *block_table_dev, int block_table_stride,
                                        int batch, float sm_scale, float *out_dev, float *lse_dev,
                                        void *stream);

/*
 * kv4_linear_bf16 — Y = X · Wᵀ on the tcgen05 tensor cores (the QKV projection ahead
 * of the cache): BF16 inputs, FP32 accumulation in tensor memory, BF16 output
 * (round to nearest). Tiles of 128 × 256 outputs (128 × 128 when 256-wide tiles would
 * leave SMs idle), TMA loads with a 128-byte swizzle. With M <= 128 the k range of each
 * 128 × 128 tile is split over the CTAs of a thread-block cluster (up to 8, as many as
 * fit on the GPU at once), whose FP32 partial sums are added in a fixed order through
 * distributed shared memory: the result does not depend on scheduling. The same call
 * shape always takes the same split, and kv4_qkv_append takes the same one, so the two
 * produce the same sums.
 *   x_dev   : [M][K] bf16, K contiguous, 16-byte aligned
 *   w_dev   : [N][K] bf16, K contiguous (the nn.Linear weight layout), 16-byte aligned
 *   y_dev   : [M][N] bf16, 16-byte aligned
 *   M >= 1; N a multiple of 128; K a multiple of 64
 *   err_dev : device int32 error word (KV4_DEVERR_WAIT_TIMEOUT if a staging wait gave
 *             up, leaving the output incomplete), or NULL
 * Errors: KV4_ERR_INVALID_ARG (sizes, alignment), KV4_ERR_CUDA.
 */
kv4_status kv4_linear_bf16(const void *x_dev, const void *w_dev, void *y_dev, int M, int N, int K,
                           int32_t *err_dev, void *stream);

/*
 * kv4_qkv_append — the attention input projection with the append fused into its
 * epilogue ([zh] 核心方法: keys take RoPE, then the Hadamard rotation, then the cache
 * quantization): Y = X · W_qkvᵀ on the tcgen05 tensor cores (BF16 operands, FP32
 * accumulation), Y rounded to BF16; the Q columns are written to q_out and the K and V
 * columns of every token are appended to the cache exactly as kv4_append would append
 * those BF16 rows (RoPE when a table is set, either cache format).
 *   x_dev     : [total_tokens][d_model] bf16 hidden states, 16-byte aligned
 *   w_qkv_dev : [(num_q_heads + 2 H_kv) * 128][d_model] bf16, rows in the order Q heads,
 *               then K head 0, V head 0, K head 1, V head 1, ... (128 rows each)
 *   q_out_dev : [total_tokens][num_q_heads][128] bf16 projected queries (pre-RoPE)
 *   d_model   : a multiple of 64; num_q_heads * 128 a multiple of 256
 *   other arguments: as kv4_append (the token order of x is the order of cu_tokens)
 * Errors: as kv4_append, KV4_ERR_INVALID_ARG for the sizes above.
 */
kv4_status kv4_qkv_append(kv4_cache *cache, const void *x_dev, const void *w_qkv_dev, int num_q_heads,
                          int d_model, void *q_out_dev, const int32_t *cu_tokens_dev,
                          const int32_t *slot_ids_dev, const int32_t *start_pos_dev,
                          const int32_t *block_table_dev, int block_table_stride, int n_seqs,
                          int total_tokens, void *stream);

/* Per-kernel device time of decode calls, from CUDA events recorded around each
 * of the three decode launches on the caller's stream while profiling is on. */
typedef struct {
    int32_t calls;       /* decode calls recorded */
    float plan_ms;       /* summed device time of the plan kernel */
    float split_ms;      /* summed device time of the split-K attention kernel */
    float merge_ms;      /* summed device time of the merge kernel */
} kv4_profile;

/* Start recording events around the next max_calls decode calls of this cache
 * (creates 4 * max_calls CUDA events; no device memory). */
kv4_status kv4_profile_start(kv4_cache *cache, int max_calls);

/* Stop recording, wait for the recorded events and return the summed times. */
kv4_status kv4_profile_stop(kv4_cache *cache, kv4_profile *out);

/* Read (synchronously: waits for the device) and optionally clear the device
 * error word of a cache, or, with cache = NULL, the error word that
 * kv4_decode_attention_noalloc reports to on the current device. *code receives a
 * kv4_device_error value. Errors: KV4_ERR_INVALID_ARG (code NULL), KV4_ERR_CUDA. */
kv4_status kv4_get_device_error(kv4_cache *cache, int32_t *code, int clear);

/* Static description of a status code. */
const char *kv4_status_string(kv4_status status);

#ifdef __cplusplus
}
#endif
#endif /* KV4_H */
