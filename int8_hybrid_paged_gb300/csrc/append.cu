// append.cu — kv4_append: Hadamard-rotate K, quantize K and V to 4-bit affine
// codes, pack them into the page of each position, and write the 8-bit side
// copies of sink and recent positions.
//
// Pages cited (title, then section):
//   [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速" — 方法步骤详情 steps 2-3,
//        前置知识 › 分组仿射 KV 量化
//   [ko] "INT4 KV 캐시로 비동기 RLVR 롤아웃을 1.8배 가속한다" — 전제와 한계
//
// One warp per token, looping over its KV heads: lane l holds dims 4l..4l+3 of K
// and V of a head (one 8-byte load each, 256 contiguous bytes per warp), the
// rotation and both min/max reductions run in registers and shuffles, and the warp
// writes the token's 64-byte K code row in one coalesced store.
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
__device__ __forceinline__ void store_int8_row(uint8_t* g, int rr, const uint32_t (&k8)[4],
                                               const uint32_t (&v8)[4], __half k8d, __half k8m,
                                               __half v8d, __half v8m, int lane)
{
    // the K codes of four consecutive dims are one word in natural order
    *reinterpret_cast<uint32_t*>(g + kSideKCodeOff + side_k_offset(rr, 4 * lane)) =
        k8[0] | (k8[1] << 8) | (k8[2] << 16) | (k8[3] << 24);
#pragma unroll
    for (int i = 0; i < 4; ++i) g[kSideVCodeOff + side_v_offset(rr, 4 * lane + i)] = (uint8_t)v8[i];
    if (lane == 0) {
        *reinterpret_cast<__half2*>(g + kSideKMetaOff + 8 * (rr & 7) + 4 * (rr >> 3)) =
            __halves2half2(k8d, k8m);
        *reinterpret_cast<__half2*>(g + kSideVMetaOff + 16 * (rr & 3) + 4 * side_v_byte(rr)) =
            __halves2half2(v8d, v8m);
    }
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

// One warp per (token, group of hpw KV heads): the sequence lookup, validation and
// page lookup happen once per warp, then the warp quantizes its heads one by one (for
// a token pair t, t + 8 both tokens' loads and arithmetic are in flight together).
template <bool ROPE>
__global__ void __launch_bounds__(256) kv4_append_kernel(AppendArgs a, int hpw)
{
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int groups = (a.num_heads + hpw - 1) / hpw;   // head groups per token
    const int tok = gw / groups;
    if (tok >= a.total_tokens) return;      // whole warp leaves together
    const int h_lo = (gw - tok * groups) * hpw, h_hi = min(a.num_heads, h_lo + hpw);

    // this token's K/V rows do not depend on the lookup below: start them towards L2
    if (lane < 2 * (h_hi - h_lo)) {
        const uint16_t* src = (lane & 1 ? a.v : a.k) + ((int64_t)tok * a.num_heads + h_lo + (lane >> 1)) * kHeadDim;
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(src + 64));
    }

    // sequence i of this token: the largest i with cu[i] <= tok (cu[n] = total > tok).
    // First guess in proportion (exact when the sequences append equal counts, e.g.
    // one token each; its slot and start are loaded alongside), then a binary search
    // if the guess misses.
    int i = (int)(((int64_t)tok * a.n_seqs) / a.total_tokens);
    int c0 = __ldg(&a.cu_tokens[i]);
    int c1 = __ldg(&a.cu_tokens[i + 1]);
    int slot = __ldg(&a.slot_ids[i]);
    int start = __ldg(&a.start_pos[i]);
    if (!(c0 <= tok && tok < c1)) {
        int lo = 0, hi = a.n_seqs;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(&a.cu_tokens[mid]) <= tok) lo = mid; else hi = mid;
        }
        i = lo;
        c0 = __ldg(&a.cu_tokens[i]);
        c1 = __ldg(&a.cu_tokens[i + 1]);
        slot = __ldg(&a.slot_ids[i]);
        start = __ldg(&a.start_pos[i]);
    }
    if (tok < c0 || tok >= c1) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_TOKENS);
        return;
    }
    const int pos = start + (tok - c0);
    const int new_len = start + (c1 - c0);
    if (slot < 0 || slot >= a.max_slots) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_SLOT);
        return;
    }
    if (start < 0 || pos / kPage >= a.stride) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_POSITION);
        return;
    }
    if (ROPE && new_len > a.rope_max_pos) {           // positions beyond the RoPE table
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_POSITION);
        return;
    }
    const int page = __ldg(&a.block_table[(int64_t)i * a.stride + pos / kPage]);
    if (page < 0 || (int64_t)page >= a.num_pages) {
        if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_PAGE);
        return;
    }

    const int H = a.num_heads, ts = pos % kPage;
    if (a.kv8) {
        // whole-cache 8-bit format: row ts of the page's group, every head of the warp
        uint8_t* blk8 = a.pages + (int64_t)page * H * kPageBlock8;
        const uint16_t* krow = a.k + (int64_t)tok * H * kHeadDim + 4 * lane;
        const uint16_t* vrow = a.v + (int64_t)tok * H * kHeadDim + 4 * lane;
        RopeRow rr{};
        if (ROPE) rr = rope_row(a.rope + (int64_t)pos * kHeadDim, lane);   // one row for all heads
        for (int h = h_lo; h < h_hi; ++h) {
            float kx[4], vx[4];
            load_bf16x4(krow + h * kHeadDim, kx);
            load_bf16x4(vrow + h * kHeadDim, vx);
            if (ROPE) warp_rope128(kx, rr, lane);
            warp_fwht128(kx, lane);
            uint32_t k8[4], v8[4];
            __half k8d, k8m, v8d, v8m;
            warp_quant<255>(kx, k8, k8d, k8m);
            warp_quant<255>(vx, v8, v8d, v8m);
            store_int8_row(blk8 + h * kPageBlock8, ts, k8, v8, k8d, k8m, v8d, v8m, lane);
        }
        if (lane == 0 && h_lo == 0 && tok == c1 - 1) a.seq_len[slot] = new_len;
        return;
    }
    // tokens t and t+8 of a page share their K bytes. When both are in this append,
    // their 2 x groups warps split the heads of both tokens and each writes whole
    // words; a token without its partner merges its nibbles into the word (the partner
    // was written by an earlier append or is not written yet)
    const bool lower = ts < 8;
    const bool pair = lower ? (pos + 8 < new_len) : (pos - 8 >= start);
    const int posA = pair && !lower ? pos - 8 : pos;       // first token of the work
    const int tokA = tok - (pos - posA);
    const int posB = posA + 8;
    int hb = h_lo, he = h_hi;
    if (pair) {
        const int k = (lower ? 0 : groups) + h_lo / hpw;     // warp of the pair, 0 .. 2 groups
        hb = k * H / (2 * groups);
        he = (k + 1) * H / (2 * groups);
    }
    const bool sinkA = posA < a.sink, ringA = (a.window > 0) && (posA >= new_len - a.window);
    const bool sinkB = posB < a.sink, ringB = (a.window > 0) && (posB >= new_len - a.window);
    const uint16_t* krow = a.k + (int64_t)tokA * H * kHeadDim + 4 * lane;
    const uint16_t* vrow = a.v + (int64_t)tokA * H * kHeadDim + 4 * lane;
    const int64_t rowB = (int64_t)8 * H * kHeadDim;        // token tokA + 8
    uint8_t* blk0 = a.pages + (int64_t)page * H * kPageBlock;
    uint8_t* sb0 = a.side + (int64_t)slot * H * a.side_block_bytes;
    const int tsA = posA % kPage;
    const int kw = kKCodeOff + k_word_offset(tsA & 7, lane);
    RopeRow rA{}, rB{};                     // the tokens' RoPE rows, shared by all heads
    if (ROPE) {
        rA = rope_row(a.rope + (int64_t)posA * kHeadDim, lane);
        if (pair) rB = rope_row(a.rope + (int64_t)posB * kHeadDim, lane);
    }
    if (pair) {
        for (int h = hb; h < he; ++h) {
            uint8_t* blk = blk0 + h * kPageBlock;
            uint8_t* sb = sb0 + h * a.side_block_bytes;
            float kxA[4], vxA[4], kxB[4], vxB[4];
            load_bf16x4(krow + h * kHeadDim, kxA);
            load_bf16x4(vrow + h * kHeadDim, vxA);
            load_bf16x4(krow + rowB + h * kHeadDim, kxB);
            load_bf16x4(vrow + rowB + h * kHeadDim, vxB);
            if (ROPE) {
                warp_rope128(kxA, rA, lane);
                warp_rope128(kxB, rB, lane);
            }
            const uint32_t knA = append_head(a, kxA, vxA, blk, tsA, sb, sinkA, ringA, posA, lane);
            const uint32_t knB = append_head(a, kxB, vxB, blk, tsA + 8, sb, sinkB, ringB, posB, lane);
            *reinterpret_cast<uint32_t*>(blk + kw) = knA | (knB << 4);
        }
    } else {
        for (int h = hb; h < he; ++h) {
            uint8_t* blk = blk0 + h * kPageBlock;
            uint32_t* kp = reinterpret_cast<uint32_t*>(blk + kw);
            const uint32_t old = *kp;                       // issued before the arithmetic
            float kx[4], vx[4];
            load_bf16x4(krow + h * kHeadDim, kx);
            load_bf16x4(vrow + h * kHeadDim, vx);
            if (ROPE) warp_rope128(kx, rA, lane);
            const uint32_t kn = append_head(a, kx, vx, blk, tsA, sb0 + h * a.side_block_bytes,
                                            sinkA, ringA, posA, lane);
            *kp = lower ? ((old & 0xf0f0f0f0u) | kn) : ((old & 0x0f0f0f0fu) | (kn << 4));
        }
    }
    if (lane == 0 && hb == 0 && he > 0 && (pair ? tokA + 8 : tok) == c1 - 1) a.seq_len[slot] = new_len;
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream)
{
    if (a.total_tokens == 0) return cudaSuccess;
    // all heads of a token in one warp when there are enough tokens to fill the GPU
    // (the per-token lookup is paid once); one head per warp for small appends
    const int hpw = (int64_t)a.total_tokens >= 16384 ? a.num_heads : 1;
    const int64_t warps = (int64_t)a.total_tokens * ((a.num_heads + hpw - 1) / hpw);
    const int64_t blocks = (warps + 7) / 8;
    if (a.rope) kv4_append_kernel<true><<<(unsigned)blocks, 256, 0, stream>>>(a, hpw);
    else kv4_append_kernel<false><<<(unsigned)blocks, 256, 0, stream>>>(a, hpw);
    return cudaGetLastError();
}

}  // namespace kv4
