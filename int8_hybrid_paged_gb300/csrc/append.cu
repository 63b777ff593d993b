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
#include "append_common.cuh"
#include "device_common.cuh"
#include "kv4_internal.h"

namespace kv4 {

// One warp per (token, group of hpw KV heads): the sequence lookup, validation and
// page lookup happen once per warp, then the warp quantizes its heads one by one (for
// a token pair t, t + 8 both tokens' loads and arithmetic are in flight together).
template <bool ROPE>
__global__ void __launch_bounds__(256, 4) kv4_append_kernel(AppendArgs a, int hpw)
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
    if (a.fp4) {
        // NVFP4 format: the K and V halves of the page's block, every head of the warp
        uint8_t* blk4 = a.pages + (int64_t)page * H * kPageBlock4f;
        const uint16_t* krow = a.k + (int64_t)tok * H * kHeadDim + 4 * lane;
        const uint16_t* vrow = a.v + (int64_t)tok * H * kHeadDim + 4 * lane;
        RopeRow rr{};
        if (ROPE) rr = rope_row(a.rope + (int64_t)pos * kHeadDim, lane);
        for (int h = h_lo; h < h_hi; ++h) {
            float kx[4], vx[4];
            load_bf16x4(krow + h * kHeadDim, kx);
            load_bf16x4(vrow + h * kHeadDim, vx);
            if (ROPE) warp_rope128(kx, rr, lane);
            warp_fwht128(kx, lane);
            uint32_t kc[4], vc[4], ksb, vsb;
            float kg, vg;
            warp_quant_nvfp4(kx, kc, ksb, kg);
            warp_quant_nvfp4(vx, vc, vsb, vg);
            uint8_t* b = blk4 + h * kPageBlock4f;
            store_nvfp4_k(b, ts, kc, ksb, kg, lane);
            store_nvfp4_v(b + kFp4Half, ts, vc, vsb, vg, lane);
        }
        if (lane == 0 && h_lo == 0 && tok == c1 - 1) a.seq_len[slot] = new_len;
        return;
    }
    if (a.mx) {
        // MXFP4 format: the K and V halves of the page's block, every head of the warp
        uint8_t* blkm = a.pages + (int64_t)page * H * kPageBlockMx;
        const uint16_t* krow = a.k + (int64_t)tok * H * kHeadDim + 4 * lane;
        const uint16_t* vrow = a.v + (int64_t)tok * H * kHeadDim + 4 * lane;
        RopeRow rr{};
        if (ROPE) rr = rope_row(a.rope + (int64_t)pos * kHeadDim, lane);
        for (int h = h_lo; h < h_hi; ++h) {
            float kx[4], vx[4];
            load_bf16x4(krow + h * kHeadDim, kx);
            load_bf16x4(vrow + h * kHeadDim, vx);
            if (ROPE) warp_rope128(kx, rr, lane);
            warp_fwht128(kx, lane);
            uint32_t kc[4], vc[4], ke, ve;
            warp_quant_mxfp4(kx, kc, ke);
            warp_quant_mxfp4(vx, vc, ve);
            uint8_t* b = blkm + h * kPageBlockMx;
            store_mxfp4_k(b, ts, kc, ke, lane);
            store_mxfp4_v(b + kMxHalf, ts, vc, ve, lane);
        }
        if (lane == 0 && h_lo == 0 && tok == c1 - 1) a.seq_len[slot] = new_len;
        return;
    }
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
    RopeRow rA{};                           // a lone token's RoPE row, shared by all heads
    if (ROPE && !pair) rA = rope_row(a.rope + (int64_t)posA * kHeadDim, lane);
    if (pair) {
        // per-head pointers advance by one head; the offsets inside a block are fixed
        const PairVOffsets vo(tsA, lane);
        const int64_t sbb = a.side_block_bytes;
        uint8_t* blk = blk0 + hb * kPageBlock;
        uint8_t* sb = sb0 + hb * sbb;
        const uint16_t* kr = krow + hb * kHeadDim;
        const uint16_t* vr = vrow + hb * kHeadDim;
#pragma unroll 1
        for (int h = hb; h < he; ++h, blk += kPageBlock, sb += sbb, kr += kHeadDim, vr += kHeadDim) {
            float kxA[4], vxA[4], kxB[4], vxB[4];
            load_bf16x4(kr, kxA);
            load_bf16x4(vr, vxA);
            load_bf16x4(kr + rowB, kxB);
            load_bf16x4(vr + rowB, vxB);
            float2 k2[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) k2[i] = make_float2(kxA[i], kxB[i]);
            // the tokens' RoPE rows are read again for every head (from L1): holding them
            // across the loop costs more registers than the loads cost
            if (ROPE)
                warp_rope128x2(k2, rope_row(a.rope + (int64_t)posA * kHeadDim, lane),
                               rope_row(a.rope + (int64_t)posB * kHeadDim, lane), lane);
            *reinterpret_cast<uint32_t*>(blk + kw) =
                append_head_pair(a, k2, vxA, vxB, blk, tsA, vo, sb, sinkA, ringA, sinkB, ringB, posA, lane);
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
