// append_common.cuh — the per-token work of an append, shared by the append kernel and
// the fused projection epilogue: page and side-group byte layouts, the 8-bit row store,
// and the rotation + quantization + packing of one token-head.
//
// Pages cited (title, then section):
//   [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速" — 方法步骤详情 steps 2-3,
//        前置知识 › 分组仿射 KV 量化
//   [ko] "INT4 KV 캐시로 비동기 RLVR 롤아웃을 1.8배 가속한다" — 전제와 한계
#pragma once

#include "device_common.cuh"
#include "kv4_internal.h"

namespace kv4 {

// Byte of (dim pair j, token t) inside a page's V code block. The block is 32 lanes x
// 8 words: word (l, m) holds pair j = 8m + (l >> 2) for tokens u, u+4, u+8, u+12 with
// u = l & 3 (bytes 0..3), so one lane's eight words are one tensor-core fragment per
// 16-dim tile and sit in 32 contiguous bytes.
__device__ __forceinline__ int v_byte_offset(int j, int t)
{
    return ((((j & 7) << 2) + (t & 3)) * 8 + (j >> 3)) * 4 + (t >> 2);
}

// Side K code byte of (row r, dim d): the QK A fragments of the protected path take,
// per 32-dim chunk c = d / 32, eight words of four consecutive dims in two planes, so
// one byte permute widens two codes of one fragment register.
__device__ __forceinline__ int side_k_offset(int r, int d)
{
    const int word = (d & 31) >> 2;
    return 1024 * (word >> 2) + 64 * r + 16 * (d >> 5) + 4 * (word & 3) + (d & 3);
}

// Byte of side row r inside a V fragment word (rows t, t+8, t+4, t+12 with t = r % 4).
__device__ __forceinline__ int side_v_byte(int r) { return ((r >> 3) & 1) | (((r >> 2) & 1) << 1); }

// Side V code byte of (row r, dim d): lane n = 4 (d % 8) + r % 4 of the PV A fragments,
// word 2 (d / 16) + (d / 8) % 2 of its sixteen, stored as four 512-byte planes.
__device__ __forceinline__ int side_v_offset(int r, int d)
{
    const int n = 4 * (d & 7) + (r & 3);
    const int word = 2 * (d >> 4) + ((d >> 3) & 1);
    return 16 * (32 * (word >> 2) + n) + 4 * (word & 3) + side_v_byte(r);
}

// One row rr of a 16-row INT8 group (a side group, or a page of the 8-bit format):
// this lane's four K and V codes (dims 4 lane .. 4 lane + 3) and, from lane 0, the
// row's metadata.
// ... its K half (codes and metadata) and its V half, for callers that hold one of them
__device__ __forceinline__ void store_int8_k(uint8_t* g, int rr, const uint32_t (&k8)[4], __half k8d,
                                             __half k8m, int lane)
{
    // the K codes of four consecutive dims are one word in natural order
    *reinterpret_cast<uint32_t*>(g + kSideKCodeOff + side_k_offset(rr, 4 * lane)) =
        k8[0] | (k8[1] << 8) | (k8[2] << 16) | (k8[3] << 24);
    if (lane == 0)
        *reinterpret_cast<__half2*>(g + kSideKMetaOff + 8 * (rr & 7) + 4 * (rr >> 3)) = __halves2half2(k8d, k8m);
}
__device__ __forceinline__ void store_int8_v(uint8_t* g, int rr, const uint32_t (&v8)[4], __half v8d,
                                             __half v8m, int lane)
{
#pragma unroll
    for (int i = 0; i < 4; ++i) g[kSideVCodeOff + side_v_offset(rr, 4 * lane + i)] = (uint8_t)v8[i];
    if (lane == 0)
        *reinterpret_cast<__half2*>(g + kSideVMetaOff + 16 * (rr & 3) + 4 * side_v_byte(rr)) =
            __halves2half2(v8d, v8m);
}
__device__ __forceinline__ void store_int8_row(uint8_t* g, int rr, const uint32_t (&k8)[4],
                                               const uint32_t (&v8)[4], __half k8d, __half k8m,
                                               __half v8d, __half v8m, int lane)
{
    store_int8_k(g, rr, k8, k8d, k8m, lane);
    store_int8_v(g, rr, v8, v8d, v8m, lane);
}

// Page K codes: tokens t and t+8 share bytes (t in the low nibble). Lane l of a warp
// holding dims 4l..4l+3 owns one 32-bit word per token pair: dims 4i, 4i+2, 4i+1,
// 4i+3 of chunk c (i = l % 8, c = l / 8) in bytes 0..3, at plane i / 4 (512 bytes),
// slot 4t + c (16 bytes), word i % 4 -- the QK fragment of lane (t, c) of the MMAs.
__device__ __forceinline__ int k_word_offset(int t, int lane)
{
    const int i = lane & 7, c = lane >> 3;
    return (i >> 2) * 512 + (4 * t + c) * 16 + (i & 3) * 4;
}

// Quantize and store one token-head: V to 4-bit codes in the page block, the metadata,
// and the 8-bit side copies when the position is protected. Returns the lane's K codes
// as a nibble word (bytes: dims 4i, 4i+2, 4i+1, 4i+3, low nibbles); the caller stores K.
__device__ __forceinline__ uint32_t append_head(const AppendArgs& a, float (&kx)[4], float (&vx)[4],
                                                uint8_t* blk, int ts, uint8_t* sb, bool to_sink,
                                                bool to_ring, int pos, int lane)
{
    warp_fwht128(kx, lane);                 // keys are stored in the rotated basis; V is not rotated
    uint32_t kc[4], vc[4];
    __half kd, km, vd, vm;
    warp_quant<15>(kx, kc, kd, km);
    warp_quant<15>(vx, vc, vd, vm);
    const uint32_t kn = kc[0] | (kc[2] << 8) | (kc[1] << 16) | (kc[3] << 24);
    // V dim pairs 2l and 2l+1 of token ts, at their places in the tile-interleaved layout
    blk[kVCodeOff + v_byte_offset(2 * lane, ts)] = (uint8_t)(vc[0] | (vc[1] << 4));
    blk[kVCodeOff + v_byte_offset(2 * lane + 1, ts)] = (uint8_t)(vc[2] | (vc[3] << 4));
    if (lane == 0) {
        // metadata row ts % 8: [K ts, K ts+8, V ts, V ts+8] for ts < 8, the same row for ts >= 8
        uint8_t* mrow = blk + kMetaOff + 16 * (ts & 7) + 4 * (ts >> 3);
        *reinterpret_cast<__half2*>(mrow) = __halves2half2(kd, km);
        *reinterpret_cast<__half2*>(mrow + 8) = __halves2half2(vd, vm);
    }

    // INT8 side copies: sink row pos (pos < s), ring row s + pos mod w for the last
    // w positions of this append. Earlier positions of a long chunk would map to the
    // same ring rows and be overwritten anyway; skipping them avoids the race.
    if (to_sink || to_ring) {
        const int s = a.sink, w = a.window;
        uint32_t k8[4], v8[4];
        __half k8d, k8m, v8d, v8m;
        warp_quant<255>(kx, k8, k8d, k8m);
        warp_quant<255>(vx, v8, v8d, v8m);
        int idx[2];
        int n = 0;
        if (to_sink) idx[n++] = pos;
        if (to_ring) idx[n++] = s + pos % w;
        for (int k = 0; k < n; ++k)
            store_int8_row(sb + (idx[k] >> 4) * kSideGroupBytes, idx[k] & 15, k8, v8, k8d, k8m, v8d,
                           v8m, lane);
    }
    return kn;
}

// Tokens A = t and B = t + 8 (t < 8) of one page and KV head together, the bytes of
// append_head for each: K of both (k2[i] = (A, B), after RoPE when a table is set)
// rotated with packed fp32x2 arithmetic; the four
// 4-bit quantizers (K and V of A and B) reduce their min/max, and lanes 0..3 compute the
// parameters of groups KA, KB, VA, VB (one pass for all four; lane g also stores group
// g's metadata) before the codes come out pairwise. Writes the V
// codes, the metadata and the side rows; returns the lane's K word with A in the low and
// B in the high nibbles.
// Byte offsets of a lane's four V bytes of tokens tsA and tsA + 8 in a page block.
struct PairVOffsets {
    int a0, a1, b0, b1;
    __device__ __forceinline__ PairVOffsets(int tsA, int lane)
        : a0(kVCodeOff + v_byte_offset(2 * lane, tsA)), a1(kVCodeOff + v_byte_offset(2 * lane + 1, tsA)),
          b0(kVCodeOff + v_byte_offset(2 * lane, tsA + 8)), b1(kVCodeOff + v_byte_offset(2 * lane + 1, tsA + 8))
    {
    }
};

__device__ __forceinline__ uint32_t append_head_pair(const AppendArgs& a, float2 (&k2)[4], const float (&vA)[4],
                                                     const float (&vB)[4], uint8_t* blk, int tsA,
                                                     const PairVOffsets& vo, uint8_t* sb, bool sinkA,
                                                     bool ringA, bool sinkB, bool ringB, int posA, int lane)
{
    warp_fwht128x2(k2, lane);
    float kA[4], kB[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        kA[i] = k2[i].x;
        kB[i] = k2[i].y;
    }
    // group extremes, each reduced over the warp
    auto lmin = [](const float (&x)[4]) { return fminf(fminf(x[0], x[1]), fminf(x[2], x[3])); };
    auto lmax = [](const float (&x)[4]) { return fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])); };
    const float loKA = warp_min_f32(lmin(kA)), hiKA = warp_max_f32(lmax(kA));
    const float loKB = warp_min_f32(lmin(kB)), hiKB = warp_max_f32(lmax(kB));
    const float loVA = warp_min_f32(lmin(vA)), hiVA = warp_max_f32(lmax(vA));
    const float loVB = warp_min_f32(lmin(vB)), hiVB = warp_max_f32(lmax(vB));
    // lane g (mod 4) takes group g = KA, KB, VA, VB
    const int g = lane & 3;
    const float lo = g == 0 ? loKA : g == 1 ? loKB : g == 2 ? loVA : loVB;
    const float hi = g == 0 ? hiKA : g == 1 ? hiKB : g == 2 ? hiVA : hiVB;
    __half min_h, delta_h;
    float m, inv;
    quant_params<15>(lo, hi, min_h, delta_h, m, inv);
    // metadata [K ts | K ts+8 | V ts | V ts+8] of row tsA: group g at 4 g
    if (lane < 4)
        *reinterpret_cast<__half2*>(blk + kMetaOff + 16 * tsA + 4 * g) = __halves2half2(delta_h, min_h);
    const float2 mK = make_float2(__shfl_sync(kFull, m, 0), __shfl_sync(kFull, m, 1));
    const float2 iK = make_float2(__shfl_sync(kFull, inv, 0), __shfl_sync(kFull, inv, 1));
    const float2 mV = make_float2(__shfl_sync(kFull, m, 2), __shfl_sync(kFull, m, 3));
    const float2 iV = make_float2(__shfl_sync(kFull, inv, 2), __shfl_sync(kFull, inv, 3));
    uint32_t kb[4], vab[4], vbb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint2 ck = code_pair(k2[i], mK, iK);
        const uint2 cv = code_pair(make_float2(vA[i], vB[i]), mV, iV);
        kb[i] = ck.x | (ck.y << 4);                                                      // A | B << 4
        vab[i] = cv.x;
        vbb[i] = cv.y;
    }
    // V dim pairs 2l and 2l+1 of each token, at their places in the tile-interleaved layout
    blk[vo.a0] = (uint8_t)(vab[0] | (vab[1] << 4));
    blk[vo.a1] = (uint8_t)(vab[2] | (vab[3] << 4));
    blk[vo.b0] = (uint8_t)(vbb[0] | (vbb[1] << 4));
    blk[vo.b1] = (uint8_t)(vbb[2] | (vbb[3] << 4));

    // INT8 side copies of protected positions (sink rows, the ring rows of the last w)
    if (sinkA || ringA || sinkB || ringB) {
        const int s = a.sink, w = a.window;
#pragma unroll
        for (int tk = 0; tk < 2; ++tk) {
            const bool to_sink = tk ? sinkB : sinkA, to_ring = tk ? ringB : ringA;
            if (!(to_sink || to_ring)) continue;
            const int pos = posA + 8 * tk;
            uint32_t k8[4], v8[4];
            __half k8d, k8m, v8d, v8m;
            warp_quant<255>(tk ? kB : kA, k8, k8d, k8m);
            warp_quant<255>(tk ? vB : vA, v8, v8d, v8m);
            if (to_sink)
                store_int8_row(sb + (pos >> 4) * kSideGroupBytes, pos & 15, k8, v8, k8d, k8m, v8d, v8m, lane);
            if (to_ring) {
                const int i = s + pos % w;
                store_int8_row(sb + (i >> 4) * kSideGroupBytes, i & 15, k8, v8, k8d, k8m, v8d, v8m, lane);
            }
        }
    }
    // bytes: dims 4i, 4i+2, 4i+1, 4i+3
    return kb[0] | (kb[2] << 8) | (kb[1] << 16) | (kb[3] << 24);
}

// The K half and the V half of append_head, for callers that hold one of the two
// tensors: the same bytes (K codes returned as the nibble word, K metadata and K side
// rows; V codes, V metadata and V side rows).
__device__ __forceinline__ uint32_t append_k(const AppendArgs& a, float (&kx)[4], uint8_t* blk, int ts,
                                             uint8_t* sb, bool to_sink, bool to_ring, int pos, int lane)
{
    warp_fwht128(kx, lane);
    uint32_t kc[4];
    __half kd, km;
    warp_quant<15>(kx, kc, kd, km);
    if (lane == 0)
        *reinterpret_cast<__half2*>(blk + kMetaOff + 16 * (ts & 7) + 4 * (ts >> 3)) = __halves2half2(kd, km);
    if (to_sink || to_ring) {
        uint32_t k8[4];
        __half k8d, k8m;
        warp_quant<255>(kx, k8, k8d, k8m);
        if (to_sink) store_int8_k(sb + (pos >> 4) * kSideGroupBytes, pos & 15, k8, k8d, k8m, lane);
        if (to_ring) {
            const int i = a.sink + pos % a.window;
            store_int8_k(sb + (i >> 4) * kSideGroupBytes, i & 15, k8, k8d, k8m, lane);
        }
    }
    return kc[0] | (kc[2] << 8) | (kc[1] << 16) | (kc[3] << 24);
}
__device__ __forceinline__ void append_v(const AppendArgs& a, float (&vx)[4], uint8_t* blk, int ts,
                                         uint8_t* sb, bool to_sink, bool to_ring, int pos, int lane)
{
    uint32_t vc[4];
    __half vd, vm;
    warp_quant<15>(vx, vc, vd, vm);
    blk[kVCodeOff + v_byte_offset(2 * lane, ts)] = (uint8_t)(vc[0] | (vc[1] << 4));
    blk[kVCodeOff + v_byte_offset(2 * lane + 1, ts)] = (uint8_t)(vc[2] | (vc[3] << 4));
    if (lane == 0)
        *reinterpret_cast<__half2*>(blk + kMetaOff + 16 * (ts & 7) + 4 * (ts >> 3) + 8) = __halves2half2(vd, vm);
    if (to_sink || to_ring) {
        uint32_t v8[4];
        __half v8d, v8m;
        warp_quant<255>(vx, v8, v8d, v8m);
        if (to_sink) store_int8_v(sb + (pos >> 4) * kSideGroupBytes, pos & 15, v8, v8d, v8m, lane);
        if (to_ring) {
            const int i = a.sink + pos % a.window;
            store_int8_v(sb + (i >> 4) * kSideGroupBytes, i & 15, v8, v8d, v8m, lane);
        }
    }
}

// ---- NVFP4 (E2M1 values, an E4M3 scale per 16 dims, an FP32 scale per vector)
// E4M3 bits of t >= 0: nearest value, ties to the even mantissa, held at 448 (0x7E).
// Quantum 2^(e-3) for exponent e = floor(log2 t) >= -6, 2^-9 below (subnormals).
__device__ __forceinline__ uint32_t e4m3_rn(float t)
{
    if (!(t > 0.0f)) return 0u;
    if (t >= 448.0f) return 0x7Eu;
    const int e = max(-6, (int)((__float_as_uint(t) >> 23) & 0xffu) - 127);
    const float m = rintf(__fmul_rn(t, __uint_as_float((uint32_t)(127 + 3 - e) << 23)));   // t / 2^(e-3)
    const float v = __fmul_rn(m, __uint_as_float((uint32_t)(127 - 3 + e) << 23));
    if (v >= 448.0f) return 0x7Eu;
    if (v == 0.0f) return 0u;
    if (v < 0x1p-6f) return (uint32_t)__float2int_rn(__fmul_rn(v, 512.0f));             // E = 0
    const int ev = (int)((__float_as_uint(v) >> 23) & 0xffu) - 127;
    const int mant = __float2int_rn(__fmul_rn(v, __uint_as_float((uint32_t)(127 + 3 - ev) << 23))) - 8;
    return (uint32_t)(((ev + 7) << 3) | mant);
}
__device__ __forceinline__ float e4m3_value(uint32_t bits)
{
    const int E = (bits >> 3) & 15, m = bits & 7;
    return E == 0 ? __fmul_rn((float)m, 0x1p-9f)
                  : __fmul_rn((float)(8 + m), __uint_as_float((uint32_t)(127 - 10 + E) << 23));
}
// E2M1 code of v: magnitude code (0, 0.5, 1, 1.5, 2, 3, 4, 6) nearest with ties to the
// even code, held at 6, sign in bit 3; a zero magnitude is code 0.
__device__ __forceinline__ uint32_t e2m1_rn(float v)
{
    const float a = fabsf(v);
    uint32_t k;
    if (a <= 0.25f) k = 0;
    else if (a < 0.75f) k = 1;
    else if (a <= 1.25f) k = 2;
    else if (a < 1.75f) k = 3;
    else if (a <= 2.5f) k = 4;
    else if (a < 3.5f) k = 5;
    else if (a <= 5.0f) k = 6;
    else k = 7;
    return k == 0 ? 0u : (k | (v < 0.0f ? 8u : 0u));
}
// The warp's 128 values (4 per lane: dims 4l .. 4l+3) to NVFP4: the lane's codes, its
// block's E4M3 scale bits (lanes 4b .. 4b+3 hold block b) and the vector scale g.
__device__ __forceinline__ void warp_quant_nvfp4(const float (&x)[4], uint32_t (&c)[4], uint32_t& sb,
                                                 float& g)
{
    float la = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    const float amax = __uint_as_float(__reduce_max_sync(kFull, __float_as_uint(la)));
    g = __fdiv_rn(amax, 2688.0f);
    const float d = __fmul_rn(g, 6.0f);
    la = fmaxf(la, __shfl_xor_sync(kFull, la, 1));
    la = fmaxf(la, __shfl_xor_sync(kFull, la, 2));              // the block's max |x|
    sb = d > 0.0f ? e4m3_rn(__fdiv_rn(la, d)) : 0u;
    const float scale = __fmul_rn(e4m3_value(sb), g);
    const float inv = scale > 0.0f ? __frcp_rn(scale) : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = scale > 0.0f ? e2m1_rn(__fmul_rn(x[i], inv)) : 0u;
}
// E2M1 codes of one token-head in a K or V half (NVFP4 and MXFP4). K: a byte holds
// dims 2j, 2j + 1 of one token, in the QK fragment order.
__device__ __forceinline__ void store_e2m1_k(uint8_t* half, int ts, const uint32_t (&c)[4], int lane)
{
    const int b = lane >> 2;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
        const int jj = 2 * (lane & 3) + e;
        half[16 * (32 * (b >> 2) + 4 * (ts & 7) + (jj & 3)) + 4 * (b & 3) + (ts >> 3) + 2 * (jj >> 2)] =
            (uint8_t)(c[2 * e] | (c[2 * e + 1] << 4));
    }
}
// V codes: a byte holds one dim of tokens t (low nibble) and t + 8 (high nibble), the
// pairs of a PV A fragment, so a reader widens it with one conversion per register; the
// word of (dim group 16m + g, token t mod 4) holds dims g, g + 8 of tokens {t, t + 8} in
// bytes 0, 1 and of tokens {t + 4, t + 12} in bytes 2, 3. A token owns one nibble of each
// of two bytes of a word that three other tokens share: it clears and sets its nibbles
// with atomics, whatever order the tokens of a page are written in.
__device__ __forceinline__ void store_e2m1_v(uint8_t* half, int ts, const uint32_t (&c)[4], int lane)
{
    const int m = lane >> 2;
    uint32_t hi[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) hi[i] = __shfl_xor_sync(kFull, c[i], 2);
    const int sh = 16 * ((ts >> 2) & 1) + 4 * (ts >> 3);          // this token's nibble in byte 0 of its pair
    const uint32_t mask = (0xfu << sh) | (0xfu << (sh + 8));
    if ((lane & 2) == 0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int gq = 4 * (lane & 3) + i;
            uint32_t* w = reinterpret_cast<uint32_t*>(half + 16 * (32 * (m >> 2) + 4 * gq + (ts & 3)) + 4 * (m & 3));
            atomicAnd(w, ~mask);
            atomicOr(w, (c[i] << sh) | (hi[i] << (sh + 8)));
        }
    }
}
// One token-head in an NVFP4 page block: the K half (codes in the QK fragment order) or
// the V half (codes in the PV fragment order), its block scales and vector scale. The K
// scales of tokens t, t + 8 sit side by side per block, the V scales of tokens t, t + 8,
// t + 4, t + 12 per block, and the vector scales of t, t + 8 side by side, each in the
// order a decode lane reads them.
__device__ __forceinline__ void store_nvfp4_k(uint8_t* half, int ts, const uint32_t (&c)[4], uint32_t sb, float g,
                                              int lane)
{
    store_e2m1_k(half, ts, c, lane);
    const int b = lane >> 2;
    if ((lane & 3) == 0) half[kFp4ScaleOff + 16 * (ts & 7) + 2 * b + (ts >> 3)] = (uint8_t)sb;
    if (lane == 0) *reinterpret_cast<float*>(half + kFp4GlobalOff + 8 * (ts & 7) + 4 * (ts >> 3)) = g;
}
__device__ __forceinline__ void store_nvfp4_v(uint8_t* half, int ts, const uint32_t (&c)[4], uint32_t sb, float g,
                                              int lane)
{
    store_e2m1_v(half, ts, c, lane);
    const int m = lane >> 2;
    const int q4 = ts >> 2, kb = ((q4 & 1) << 1) | (q4 >> 1);     // tokens t, t+8, t+4, t+12 -> bytes 0..3
    if ((lane & 3) == 0) half[kFp4ScaleOff + 32 * (ts & 3) + 4 * m + kb] = (uint8_t)sb;
    if (lane == 0) *reinterpret_cast<float*>(half + kFp4GlobalOff + 8 * (ts & 7) + 4 * (ts >> 3)) = g;
}

// ---- MXFP4 (E2M1 values, one E8M0 power-of-two scale per 32 values)
// The warp's 128 values (4 per lane: dims 4l .. 4l+3) to MXFP4: the lane's codes and its
// block's biased exponent e = s + 127 (lanes 8b .. 8b+7 hold block b), where
// s = floor(log2 amax_b) - 2 held in [-127, 127]; an all-zero block takes s = -127.
__device__ __forceinline__ void warp_quant_mxfp4(const float (&x)[4], uint32_t (&c)[4], uint32_t& e)
{
    float la = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    la = fmaxf(la, __shfl_xor_sync(kFull, la, 1));
    la = fmaxf(la, __shfl_xor_sync(kFull, la, 2));
    la = fmaxf(la, __shfl_xor_sync(kFull, la, 4));              // the block's max |x|
    // floor(log2 amax) is the biased exponent field minus 127 for a normal amax; a
    // subnormal or zero amax lands below -127 and is held there
    const int ef = (int)((__float_as_uint(la) >> 23) & 0xffu);
    const int sx = min(127, max(-127, ef - 127 - 2));
    e = (uint32_t)(sx + 127);
    // 2^-s as a normal float (s <= 125 for finite inputs); the products are exact unless
    // they fall below the normal range, where they round to nearest like any product
    const float inv = __uint_as_float((uint32_t)(127 - sx) << 23);
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = la > 0.0f ? e2m1_rn(__fmul_rn(x[i], inv)) : 0u;
}
// One token-head in an MXFP4 page block: codes as NVFP4, E8M0 scales of tokens t, t + 8
// side by side per block (K) or of tokens t, t + 8, t + 4, t + 12 per block (V).
__device__ __forceinline__ void store_mxfp4_k(uint8_t* half, int ts, const uint32_t (&c)[4], uint32_t e, int lane)
{
    store_e2m1_k(half, ts, c, lane);
    const int b = lane >> 3;
    if ((lane & 7) == 0) half[kMxScaleOff + 8 * (ts & 7) + 2 * b + (ts >> 3)] = (uint8_t)e;
}
__device__ __forceinline__ void store_mxfp4_v(uint8_t* half, int ts, const uint32_t (&c)[4], uint32_t e, int lane)
{
    store_e2m1_v(half, ts, c, lane);
    const int b = lane >> 3, q4 = ts >> 2, kb = ((q4 & 1) << 1) | (q4 >> 1);
    if ((lane & 7) == 0) half[kMxScaleOff + 16 * (ts & 3) + 4 * b + kb] = (uint8_t)e;
}

// Where token tok of an append goes: its sequence entry i (cu_tokens[i] <= tok <
// cu_tokens[i+1]), slot, position, the sequence's length after the append and the
// page of the position. False, with the error reported, when an input is invalid.
struct TokenLoc {
    int i, c0, c1, slot, start, pos, new_len, page;
};

__device__ __forceinline__ bool locate_token(const AppendArgs& a, int tok, int lane, TokenLoc& L)
{
    int i = (int)(((int64_t)tok * a.n_seqs) / a.total_tokens);     // proportional guess
    int c0 = __ldg(&a.cu_tokens[i]);
    int c1 = __ldg(&a.cu_tokens[i + 1]);
    if (!(c0 <= tok && tok < c1)) {
        int lo = 0, hi = a.n_seqs;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(&a.cu_tokens[mid]) <= tok) lo = mid; else hi = mid;
        }
        i = lo;
        c0 = __ldg(&a.cu_tokens[i]);
        c1 = __ldg(&a.cu_tokens[i + 1]);
    }
    if (tok < c0 || tok >= c1) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_TOKENS);
        return false;
    }
    L.i = i;
    L.c0 = c0;
    L.c1 = c1;
    L.slot = __ldg(&a.slot_ids[i]);
    L.start = __ldg(&a.start_pos[i]);
    L.pos = L.start + (tok - c0);
    L.new_len = L.start + (c1 - c0);
    if (L.slot < 0 || L.slot >= a.max_slots) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_SLOT);
        return false;
    }
    if (L.start < 0 || L.pos / kPage >= a.stride || (a.rope && L.new_len > a.rope_max_pos)) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_POSITION);
        return false;
    }
    L.page = __ldg(&a.block_table[(int64_t)i * a.stride + L.pos / kPage]);
    if (L.page < 0 || (int64_t)L.page >= a.num_pages) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_PAGE);
        return false;
    }
    return true;
}

}  // namespace kv4
