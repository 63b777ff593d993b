// qkv.cu — the projection ahead of the cache on the 5th-generation tensor cores:
// Y = X · Wᵀ with X [M][K] and W [N][K] in BF16 (both K-contiguous, the nn.Linear
// layout), FP32 accumulation in tensor memory.
//
// One CTA computes a 128 × BN tile of Y (BN = 256, or 128 when that leaves SMs idle):
// one thread streams 128 × 64 tiles of X and BN × 64 tiles of W into a ring of
// shared-memory stages with TMA (128-byte swizzle); one thread issues tcgen05.mma
// (M = 128, N = BN, K = 16 per instruction) into a TMEM accumulator and
// frees each stage with tcgen05.commit; then the four warps read their 32 TMEM lanes
// (rows) back with tcgen05.ld and write the tile. Every wait is bounded: a wait that
// gives up records an error and the CTA still releases its tensor memory.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "append_common.cuh"
#include "device_common.cuh"
#include "kv4_internal.h"

namespace kv4 {

namespace {

constexpr int kBM = 128, kBK = 64;                 // kBK * 2 bytes = one 128-byte swizzle row
// TMA ring depth: 4 stages of 48 KB for 256-wide tiles, 6 of 32 KB for 128-wide ones
// (a deeper ring keeps more bytes in flight per SM when few tiles share the GPU)
template <int BN>
constexpr int gemm_stages() { return BN == 256 ? 4 : 6; }
constexpr int kTileBytes = kBM * kBK * 2;           // 16 KB: the X tile
constexpr int kGemmThreads = 128;

// BN = 128 or 256 output columns per tile (the W tile and the TMEM accumulator width)
template <int BN>
struct __align__(1024) GemmSmem {
    static constexpr int kStages = gemm_stages<BN>();
    uint8_t a[kStages][kTileBytes];                 // 1024-byte aligned: swizzle atoms
    uint8_t b[kStages][BN * kBK * 2];
    uint64_t full[kStages], empty[kStages], accum;
    uint32_t tmem_base;
    int32_t abort;
};

// ---- TMA, tcgen05 (inline PTX)
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void arrive_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile in the 128-byte swizzle
// layout: start address, leading offset (unused for this layout, 16 bytes), stride
// between 8-row groups 1024 bytes, descriptor version 1, swizzle mode 2 (128 bytes).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr)
{
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)(16u >> 4) << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: FP32 accumulator, BF16 A and B, both K-major,
// N = BN, M = kBM.
template <int BN>
constexpr uint32_t idesc_bf16()
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc,
                                          uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
        ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 ::"r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tmem_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tmem_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive FP32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Bounded wait on an mbarrier phase (about 2 s), false when it gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity)
{
    if (mbar_try_wait_at(bar, parity)) return true;
    return mbar_wait_slow(bar, parity);
}

// The tile's main loop over k blocks [kb0, kb1): barrier and TMEM set-up, thread 0
// streams the X and W tiles of every k block, thread 32 issues the MMAs, threads 64 and
// up run pre(tid - 64) (work that does not need the tile: no warp-collective
// operations), and every thread then waits for the accumulator. True when the
// accumulator holds the finished tile.
template <int BN, class PreWait>
__device__ __forceinline__ bool gemm_tile(GemmSmem<BN>& sm, const CUtensorMap& map_x,
                                          const CUtensorMap& map_w, int m0, int n0, int kb0, int kb1,
                                          int32_t* err, PreWait&& pre)
{
    constexpr int kWBytes = BN * kBK * 2;
    constexpr int kS = GemmSmem<BN>::kStages;
    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < kS; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], 1);
        }
        mbar_init(&sm.accum, 1);
        sm.abort = 0;
        fence_mbar_init();
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_x)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_w)) : "memory");
    }
    if (warp == 0) {
        // the accumulator: BN columns x 128 lanes of tensor memory
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                     ::"r"(smem_u32(&sm.tmem_base)), "r"((uint32_t)BN)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem = sm.tmem_base;

    if (tid == 0) {
        // ---- producer: TMA of the X and W tiles of every k block
        for (int kb = kb0; kb < kb1; ++kb) {
            const int i = kb - kb0, s = i % kS, r = i / kS;
            if (r > 0 && !wait_phase(smem_u32(&sm.empty[s]), (r - 1) & 1)) {
                report_error(err, KV4_DEVERR_WAIT_TIMEOUT);
                atomicExch(&sm.abort, 1);
                break;
            }
            const uint32_t fb = smem_u32(&sm.full[s]);
            arrive_expect_tx(fb, kTileBytes + kWBytes);
            tma_load_2d(smem_u32(sm.a[s]), &map_x, kb * kBK, m0, fb);
#pragma unroll
            for (int h = 0; h < BN / 128; ++h)              // boxes of 128 W rows
                tma_load_2d(smem_u32(sm.b[s]) + h * kTileBytes, &map_w, kb * kBK, n0 + 128 * h, fb);
        }
    } else if (tid == 32) {
        // ---- MMA issuer: four K = 16 steps per stage, accumulate after the first
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
            const int i = kb - kb0, s = i % kS, r = i / kS;
            if (!wait_phase(smem_u32(&sm.full[s]), r & 1)) {
                report_error(err, KV4_DEVERR_WAIT_TIMEOUT);
                atomicExch(&sm.abort, 1);
                ok = false;
                break;
            }
            tmem_fence_after();
            const uint64_t ad = smem_desc_sw128(smem_u32(sm.a[s]));
            const uint64_t bd = smem_desc_sw128(smem_u32(sm.b[s]));
#pragma unroll
            for (int k = 0; k < kBK / 16; ++k)              // +32 bytes along K = +2 in the address field
                umma_bf16(tmem, ad + 2 * k, bd + 2 * k, idesc_bf16<BN>(), (i | k) != 0);
            umma_commit(smem_u32(&sm.empty[s]));          // stage free once these MMAs have read it
        }
        if (ok) umma_commit(smem_u32(&sm.accum));
        else asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&sm.accum)) : "memory");
    } else if (tid >= 64) {
        pre(tid - 64);
    }
    const bool got = wait_phase(smem_u32(&sm.accum), 0);
    tmem_fence_after();
    if (!got && (tid & 31) == 0) report_error(err, KV4_DEVERR_WAIT_TIMEOUT);
    // one answer for the whole CTA: the warp-collective TMEM loads that follow must be
    // executed by every lane of every warp or by none
    return __syncthreads_and(got && !sm.abort) != 0;
}

// Release the tile's tensor memory (after every warp's last tcgen05.ld).
template <int BN>
__device__ __forceinline__ void gemm_release(GemmSmem<BN>& sm)
{
    tmem_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(sm.tmem_base),
                     "r"((uint32_t)BN)
                     : "memory");
    }
}

// Columns [0, 32 * nc) of this thread's accumulator row as BF16 (round to nearest)
// into dst (16-byte aligned, 64 bytes per 32 columns) when write is set. The TMEM
// loads are warp-collective (.sync.aligned): every lane of the warp must call this,
// with write false for rows that are not stored.
__device__ __forceinline__ void store_row_bf16(uint32_t taddr, int nc, uint16_t* dst, bool write)
{
#pragma unroll 1
    for (int c = 0; c < nc; ++c) {
        float v[32];
        tmem_ld32(taddr + (uint32_t)(32 * c), v);
        if (!write) continue;
        uint4* d4 = reinterpret_cast<uint4*>(dst + 32 * c);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const __nv_bfloat162 h = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
                w[e] = *reinterpret_cast<const uint32_t*>(&h);
            }
            d4[q] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int BN>
__global__ void __launch_bounds__(kGemmThreads, 1)
kv4_linear_bf16_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                       uint16_t* __restrict__ y, int M, int N, int K, int32_t* err)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GemmSmem<BN>& sm = *reinterpret_cast<GemmSmem<BN>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * BN;
    const bool ok = gemm_tile<BN>(sm, map_x, map_w, m0, n0, 0, K / kBK, err, [](int) {});
    const int row = m0 + 32 * warp + lane;
    if (ok)                                  // CTA-uniform: every lane loads, rows < M store
        store_row_bf16(sm.tmem_base + ((uint32_t)(32 * warp) << 16), BN / 32, y + (int64_t)row * N + n0,
                       row < M);
    gemm_release<BN>(sm);
}

// Fused projection + append. Output columns: [Q heads | K0 V0 | K1 V1 | ...], 128 each;
// a 256-wide tile is two Q heads or the K and V heads of one KV head.
struct QkvArgs {
    AppendArgs ap;                // the cache append (ap.k, ap.v unused)
    uint16_t* q_out;              // [T][Hq * 128] bf16
    int32_t q_cols;               // Hq * 128
};

// 16 warps: warps w, w + 4, w + 8, w + 12 read the same TMEM lane quarter (rows
// 32 (w % 4) ..), each a quarter of the 256 columns; all 16 share the append loop.
constexpr int kQkvThreads = 512;

// Where each token of a K/V tile goes, found by the idle threads while the tile's MMAs
// run (the lookups are dependent global loads: done in the append loop they would come
// one token after another); kept in shared memory past the GEMM's stages.
struct TokenLocS {
    TokenLoc L;
    int32_t ok;
};
__device__ __forceinline__ void locate_tile_tokens(const AppendArgs& a, TokenLocS* loc, int m0, int t,
                                                   int r0 = 0, int r1 = kBM)
{
    for (int rr = r0 + t; rr < r1; rr += kQkvThreads - 64) {
        const int tok = m0 + rr;
        TokenLocS e{};
        e.ok = tok < a.total_tokens && locate_token(a, tok, 0, e.L);
        loc[rr] = e;
    }
}

// The append of the K and V heads of KV head h for rows [r0, r1) of a row tile that starts
// at token m0: warp w takes rows r0 + w, r0 + w + 16, ...; load_row(rr, kx, vx) gives this
// lane's four K and four V values (dims 4 lane .. 4 lane + 3) of row rr, already rounded
// to BF16 as the projection's output is.
template <int FMT, class LoadRow>
__device__ __forceinline__ void append_kv_rows(const AppendArgs& a, const TokenLocS* loc, int m0, int r0, int r1,
                                               int h, int warp, int lane, LoadRow&& load_row)
{
    const int H = a.num_heads, T = a.total_tokens;
#pragma unroll 1
    for (int rr = r0 + warp; rr < r1; rr += kQkvThreads / 32) {
        const int tok = m0 + rr;
        if (tok >= T) break;
        if (!loc[rr].ok) continue;
        const TokenLoc L = loc[rr].L;
        const int ts = L.pos % kPage;
        float kxA[4], vxA[4];
        load_row(rr, kxA, vxA);
        if (a.rope) warp_rope128(kxA, rope_row(a.rope + (int64_t)L.pos * kHeadDim, lane), lane);
        if (FMT == 3) {
            warp_fwht128(kxA, lane);
            uint32_t kc[4], vc[4], ke, ve;
            warp_quant_mxfp4(kxA, kc, ke);
            warp_quant_mxfp4(vxA, vc, ve);
            uint8_t* b = a.pages + ((int64_t)L.page * H + h) * kPageBlockMx;
            store_mxfp4_k(b, ts, kc, ke, lane);
            store_mxfp4_v(b + kMxHalf, ts, vc, ve, lane);
            if (lane == 0 && h == 0 && tok == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
            continue;
        }
        if (FMT == 2) {
            warp_fwht128(kxA, lane);
            uint32_t kc[4], vc[4], ksb, vsb;
            float kg, vg;
            warp_quant_nvfp4(kxA, kc, ksb, kg);
            warp_quant_nvfp4(vxA, vc, vsb, vg);
            uint8_t* b = a.pages + ((int64_t)L.page * H + h) * kPageBlock4f;
            store_nvfp4_k(b, ts, kc, ksb, kg, lane);
            store_nvfp4_v(b + kFp4Half, ts, vc, vsb, vg, lane);
            if (lane == 0 && h == 0 && tok == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
            continue;
        }
        if (FMT == 1) {
            warp_fwht128(kxA, lane);
            uint32_t k8[4], v8[4];
            __half k8d, k8m, v8d, v8m;
            warp_quant<255>(kxA, k8, k8d, k8m);
            warp_quant<255>(vxA, v8, v8d, v8m);
            store_int8_row(a.pages + ((int64_t)L.page * H + h) * kPageBlock8, ts, k8, v8, k8d, k8m, v8d, v8m,
                           lane);
            if (lane == 0 && h == 0 && tok == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
            continue;
        }
        // tokens t and t + 8 of a page share K bytes: a pair inside rows [r0, r1) is
        // written whole by the lower token's warp; a token whose partner is elsewhere
        // (other rows of this call, or an earlier append) merges its nibbles atomically
        const bool lower = ts < 8;
        const bool pair = lower ? (L.pos + 8 < L.new_len && rr + 8 < r1 && tok + 8 < T)
                                : (L.pos - 8 >= L.start && rr - 8 >= r0);
        if (pair && !lower) continue;                      // written with its lower partner
        uint8_t* blk = a.pages + ((int64_t)L.page * H + h) * kPageBlock;
        uint8_t* sb = a.side + ((int64_t)L.slot * H + h) * a.side_block_bytes;
        const int kwo = kKCodeOff + k_word_offset(ts & 7, lane);
        const bool sinkA = L.pos < a.sink, ringA = (a.window > 0) && (L.pos >= L.new_len - a.window);
        const uint32_t knA = append_head(a, kxA, vxA, blk, ts, sb, sinkA, ringA, L.pos, lane);
        uint32_t* kp = reinterpret_cast<uint32_t*>(blk + kwo);
        if (pair) {
            const int posB = L.pos + 8;
            float kxB[4], vxB[4];
            load_row(rr + 8, kxB, vxB);
            if (a.rope) warp_rope128(kxB, rope_row(a.rope + (int64_t)posB * kHeadDim, lane), lane);
            const bool sinkB = posB < a.sink, ringB = (a.window > 0) && (posB >= L.new_len - a.window);
            const uint32_t knB = append_head(a, kxB, vxB, blk, ts + 8, sb, sinkB, ringB, posB, lane);
            *kp = knA | (knB << 4);
        } else if (lower) {
            atomicAnd(kp, 0xf0f0f0f0u);
            atomicOr(kp, knA);
        } else {
            atomicAnd(kp, 0x0f0f0f0fu);
            atomicOr(kp, knA << 4);
        }
        if (lane == 0 && h == 0 && (pair ? tok + 8 : tok) == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
    }
}

// FMT: 0 the method's format (INT4 pages + side buffer), 1 the 8-bit format, 2 NVFP4,
// 3 MXFP4
template <int FMT>
__global__ void __launch_bounds__(kQkvThreads, 1)
kv4_qkv_append_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                      const QkvArgs qa, int K)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GemmSmem<256>& sm = *reinterpret_cast<GemmSmem<256>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const AppendArgs& a = qa.ap;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * 256;
    const int T = a.total_tokens;
    TokenLocS* loc = reinterpret_cast<TokenLocS*>(reinterpret_cast<uint8_t*>(&sm) + sizeof(GemmSmem<256>));
    const bool kv_tile = n0 >= qa.q_cols;
    const bool ok = gemm_tile<256>(sm, map_x, map_w, m0, n0, 0, K / kBK, a.err, [&](int t) {
        if (kv_tile) locate_tile_tokens(a, loc, m0, t);
    });
    const int quarter = warp & 3, colq = warp >> 2;                 // TMEM lane quarter, column quarter
    const uint32_t trow = sm.tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(64 * colq);
    const int r = 32 * quarter + lane, row = m0 + r;
    if (n0 < qa.q_cols) {
        // ---- two Q heads: the projection itself
        if (ok) store_row_bf16(trow, 2, qa.q_out + (int64_t)row * qa.q_cols + n0 + 64 * colq, row < T);
        gemm_release<256>(sm);
        return;
    }
    // ---- K and V of KV head h for tokens m0 .. m0+127: rounded to BF16 as the projection
    // would be, staged in the (now idle) W stages, then appended token by token
    const int h = (n0 - qa.q_cols) / 256;
    uint16_t* kt = reinterpret_cast<uint16_t*>(sm.b[0]);              // [128][128] bf16
    uint16_t* vt = kt + 128 * 128;
    fence_proxy_async();                    // the MMAs' reads of the stages precede these writes
    if (ok)                                  // CTA-uniform; rows past T are staged but never read
        store_row_bf16(trow, 2, (colq >= 2 ? vt : kt) + 128 * r + 64 * (colq & 1), true);
    gemm_release<256>(sm);                                            // ends with a CTA barrier
    if (!ok) return;
    append_kv_rows<FMT>(a, loc, m0, 0, kBM, h, warp, lane,
                        [&](int rr, float (&kx)[4], float (&vx)[4]) {
                            const uint2 kw2 = *reinterpret_cast<const uint2*>(kt + 128 * rr + 4 * lane);
                            const uint2 vw2 = *reinterpret_cast<const uint2*>(vt + 128 * rr + 4 * lane);
                            kx[0] = bf16_lo(kw2.x); kx[1] = bf16_hi(kw2.x); kx[2] = bf16_lo(kw2.y); kx[3] = bf16_hi(kw2.y);
                            vx[0] = bf16_lo(vw2.x); vx[1] = bf16_hi(vw2.x); vx[2] = bf16_lo(vw2.y); vx[3] = bf16_hi(vw2.y);
                        });
}

// The append of one 128-column K or V tile (KV head h) for rows [r0, r1) of a row tile
// that starts at token m0: warp w takes rows r0 + w, r0 + w + 16, ...; load_row(rr, x)
// gives this lane's four values (dims 4 lane .. 4 lane + 3) of row rr, already rounded to
// BF16 as the projection's output is. The K or V half of the per-token routine writes
// the same bytes as the combined one.
template <int FMT, class LoadRow>
__device__ __forceinline__ void append_half_rows(const AppendArgs& a, const TokenLocS* loc, int m0, int r0,
                                                 int r1, int h, bool is_v, int warp, int lane,
                                                 LoadRow&& load_row)
{
    const int H = a.num_heads, T = a.total_tokens;
#pragma unroll 1
    for (int rr = r0 + warp; rr < r1; rr += kQkvThreads / 32) {
        const int tok = m0 + rr;
        if (tok >= T) break;
        if (!loc[rr].ok) continue;
        const TokenLoc L = loc[rr].L;
        const int ts = L.pos % kPage;
        float xA[4];
        load_row(rr, xA);
        if (!is_v && a.rope) warp_rope128(xA, rope_row(a.rope + (int64_t)L.pos * kHeadDim, lane), lane);
        if (FMT == 3) {
            uint8_t* b = a.pages + ((int64_t)L.page * H + h) * kPageBlockMx;
            uint32_t c4[4], e4;
            if (!is_v) {
                warp_fwht128(xA, lane);
                warp_quant_mxfp4(xA, c4, e4);
                store_mxfp4_k(b, ts, c4, e4, lane);
                if (lane == 0 && h == 0 && tok == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
            } else {
                warp_quant_mxfp4(xA, c4, e4);
                store_mxfp4_v(b + kMxHalf, ts, c4, e4, lane);
            }
            continue;
        }
        if (FMT == 2) {
            uint8_t* b = a.pages + ((int64_t)L.page * H + h) * kPageBlock4f;
            uint32_t c4[4], sb4;
            float g4;
            if (!is_v) {
                warp_fwht128(xA, lane);
                warp_quant_nvfp4(xA, c4, sb4, g4);
                store_nvfp4_k(b, ts, c4, sb4, g4, lane);
                if (lane == 0 && h == 0 && tok == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
            } else {
                warp_quant_nvfp4(xA, c4, sb4, g4);
                store_nvfp4_v(b + kFp4Half, ts, c4, sb4, g4, lane);
            }
            continue;
        }
        if (FMT == 1) {
            uint8_t* g = a.pages + ((int64_t)L.page * H + h) * kPageBlock8;
            uint32_t c8[4];
            __half d8, m8;
            if (!is_v) {
                warp_fwht128(xA, lane);
                warp_quant<255>(xA, c8, d8, m8);
                store_int8_k(g, ts, c8, d8, m8, lane);
                if (lane == 0 && h == 0 && tok == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
            } else {
                warp_quant<255>(xA, c8, d8, m8);
                store_int8_v(g, ts, c8, d8, m8, lane);
            }
            continue;
        }
        uint8_t* blk = a.pages + ((int64_t)L.page * H + h) * kPageBlock;
        uint8_t* sb = a.side + ((int64_t)L.slot * H + h) * a.side_block_bytes;
        const bool sinkA = L.pos < a.sink, ringA = (a.window > 0) && (L.pos >= L.new_len - a.window);
        if (is_v) {
            append_v(a, xA, blk, ts, sb, sinkA, ringA, L.pos, lane);
            continue;
        }
        // K: tokens t and t + 8 of a page inside rows [r0, r1) are written together,
        // others merge their nibbles
        const bool lower = ts < 8;
        const bool pair = lower ? (L.pos + 8 < L.new_len && rr + 8 < r1 && tok + 8 < T)
                                : (L.pos - 8 >= L.start && rr - 8 >= r0);
        if (pair && !lower) continue;
        const uint32_t knA = append_k(a, xA, blk, ts, sb, sinkA, ringA, L.pos, lane);
        uint32_t* kp = reinterpret_cast<uint32_t*>(blk + kKCodeOff + k_word_offset(ts & 7, lane));
        if (pair) {
            const int posB = L.pos + 8;
            float xB[4];
            load_row(rr + 8, xB);
            if (a.rope) warp_rope128(xB, rope_row(a.rope + (int64_t)posB * kHeadDim, lane), lane);
            const bool sinkB = posB < a.sink, ringB = (a.window > 0) && (posB >= L.new_len - a.window);
            const uint32_t knB = append_k(a, xB, blk, ts + 8, sb, sinkB, ringB, posB, lane);
            *kp = knA | (knB << 4);
        } else if (lower) {
            atomicAnd(kp, 0xf0f0f0f0u);
            atomicOr(kp, knA);
        } else {
            atomicAnd(kp, 0x0f0f0f0fu);
            atomicOr(kp, knA << 4);
        }
        if (lane == 0 && h == 0 && (pair ? tok + 8 : tok) == L.c1 - 1) a.seq_len[L.slot] = L.new_len;
    }
}

// The same with 128-wide tiles, for calls with few tokens (twice the CTAs): a tile is one
// Q head, or the K or the V head of one KV head, appended with the K or V half of the
// per-token routine (the same bytes as the combined one).
template <int FMT>
__global__ void __launch_bounds__(kQkvThreads, 1)
kv4_qkv_append_narrow_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                             const QkvArgs qa, int K)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    GemmSmem<128>& sm = *reinterpret_cast<GemmSmem<128>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const AppendArgs& a = qa.ap;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int m0 = blockIdx.y * kBM, n0 = blockIdx.x * 128;
    const int T = a.total_tokens;
    TokenLocS* loc = reinterpret_cast<TokenLocS*>(reinterpret_cast<uint8_t*>(&sm) + sizeof(GemmSmem<128>));
    const bool kv_tile = n0 >= qa.q_cols;
    const bool ok = gemm_tile<128>(sm, map_x, map_w, m0, n0, 0, K / kBK, a.err, [&](int t) {
        if (kv_tile) locate_tile_tokens(a, loc, m0, t);
    });
    const int quarter = warp & 3, colq = warp >> 2;                 // TMEM lane quarter, column quarter
    const uint32_t trow = sm.tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)(32 * colq);
    const int r = 32 * quarter + lane, row = m0 + r;
    if (n0 < qa.q_cols) {
        if (ok) store_row_bf16(trow, 1, qa.q_out + (int64_t)row * qa.q_cols + n0 + 32 * colq, row < T);
        gemm_release<128>(sm);
        return;
    }
    const int kvj = (n0 - qa.q_cols) / 128, h = kvj >> 1;
    const bool is_v = (kvj & 1) != 0;
    uint16_t* xt = reinterpret_cast<uint16_t*>(sm.b[0]);              // [128][128] bf16: K or V
    fence_proxy_async();
    if (ok) store_row_bf16(trow, 1, xt + 128 * r + 32 * colq, true);
    gemm_release<128>(sm);
    if (!ok) return;
    append_half_rows<FMT>(a, loc, m0, 0, kBM, h, is_v, warp, lane, [&](int rr, float (&x)[4]) {
        const uint2 w2 = *reinterpret_cast<const uint2*>(xt + 128 * rr + 4 * lane);
        x[0] = bf16_lo(w2.x); x[1] = bf16_hi(w2.x); x[2] = bf16_lo(w2.y); x[3] = bf16_hi(w2.y);
    });
}

// ---- split-K for few tokens (a small decode step): the S CTAs of a thread-block cluster
// share one 128 x 128 tile, CTA c taking k blocks [c nk / S, (c + 1) nk / S). Each CTA parks its partial sums in its own
// shared memory; after a cluster barrier, CTA c adds the S partials (in rank order, the
// same for every caller) of its share of the rows through distributed shared memory and
// runs the tile's epilogue on them: BF16 rows for the plain projection and for Q, the
// append for K and V. A second cluster barrier keeps every CTA's partials in place until
// the others have read them.
struct SplitKArgs {
    QkvArgs qa;                   // the fused call (FMT >= 0)
    uint16_t* y;                  // the plain projection (FMT < 0): [M][N] bf16
    int32_t M, N, nk;             // rows, output columns, k blocks of 64
    int32_t* err;                 // the plain projection's error word
};

struct SplitKSmem {
    GemmSmem<128> g;              // its stages hold the parked partials after the main loop
    TokenLocS loc[kBM];
    int32_t ok;
};

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
// every thread of every CTA of the cluster: writes before it are visible to reads after it
__device__ __forceinline__ void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ int32_t ld_cluster_s32(uint32_t addr)
{
    int32_t v;
    asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void round_bf16x4(float (&x)[4])
{
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __bfloat162float(__float2bfloat16_rn(x[i]));
}

// Grid: column tiles x S CTAs, clusters of S. FMT: -1 the plain projection; 0..3 the
// fused call in the cache's format (as above), whose tiles are one Q head, or the K or
// the V head of one KV head.
template <int FMT>
__global__ void __launch_bounds__(kQkvThreads, 1)
kv4_gemm_splitk_kernel(const __grid_constant__ CUtensorMap map_x, const __grid_constant__ CUtensorMap map_w,
                       const SplitKArgs ka)
{
    // parked rows: 132 floats, so that the 16-byte chunks written by 8 consecutive rows
    // fall in distinct bank groups
    constexpr int BN = 128, kPS = BN + 4;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    SplitKSmem& sm = *reinterpret_cast<SplitKSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    static_assert(kBM * kPS * 4 <= sizeof(sm.g.a) + sizeof(sm.g.b), "partials exceed the stages");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = (int)cluster_size(), c = (int)cluster_rank();
    const int n0 = (int)(blockIdx.x / S) * BN, m0 = 0;
    const int kb0 = c * ka.nk / S, kb1 = (c + 1) * ka.nk / S;
    constexpr int R = kBM;
    const int share = ((R + S - 1) / S + 15) & ~15;                  // rows per CTA, whole 16-row groups
    const int r0 = min(R, c * share), r1 = min(R, r0 + share);
    const AppendArgs& a = ka.qa.ap;
    const bool kv_tile = FMT >= 0 && n0 >= ka.qa.q_cols;
    const int M = FMT >= 0 ? a.total_tokens : ka.M;
    const bool ok = gemm_tile<BN>(sm.g, map_x, map_w, m0, n0, kb0, kb1, FMT >= 0 ? a.err : ka.err,
                                      [&](int t) {
                                          if (kv_tile) locate_tile_tokens(a, sm.loc, m0, t, r0, r1);
                                      });
    // park this CTA's partial sums: TMEM -> shared memory rows; warp w reads TMEM lane
    // quarter w % 4, column quarter w / 4
    float* P = reinterpret_cast<float*>(&sm.g.a[0][0]);
    fence_proxy_async();                    // the stages were last written by TMA, read by the MMAs
    if (ok) {                               // CTA-uniform
        const int quarter = warp & 3, col = 32 * (warp >> 2);
        float v[32];
        tmem_ld32(sm.g.tmem_base + ((uint32_t)(32 * quarter) << 16) + (uint32_t)col, v);
        float4* d = reinterpret_cast<float4*>(P + (32 * quarter + lane) * kPS + col);
#pragma unroll
        for (int q = 0; q < 8; ++q) d[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    }
    gemm_release<BN>(sm.g);                 // CTA barrier, TMEM freed
    if (threadIdx.x == 0) sm.ok = ok ? 1 : 0;
    cluster_sync_all();
    const uint32_t p_loc = smem_u32(P);
    bool all_ok = true;
    for (int j = 0; j < S; ++j) all_ok = all_ok && ld_cluster_s32(cluster_map(smem_u32(&sm.ok), (uint32_t)j)) != 0;
    // this lane's four columns 128 c + 4 lane .. (c < NC) of rows rows[i] (i < NR): the S
    // partials added in rank order; the loads go out four ranks at a time for all NR rows
    // together (one round trip for S <= 4)
    auto sum_cols = [&](const auto& rows, auto& x) {
        constexpr int NR = sizeof(rows) / sizeof(rows[0]);
        constexpr int NC = sizeof(x[0]) / sizeof(x[0][0]);
        float4 acc[NR][NC];
#pragma unroll 1
        for (int j0 = 0; j0 < S; j0 += 4) {
            float4 v[NR][NC][4];
#pragma unroll
            for (int i = 0; i < NR; ++i)
#pragma unroll
                for (int cc = 0; cc < NC; ++cc)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        if (j0 + j < S)
                            v[i][cc][j] = ld_cluster_f4(cluster_map(
                                p_loc + (uint32_t)((rows[i] * kPS + 128 * cc + 4 * lane) * 4), (uint32_t)(j0 + j)));
#pragma unroll
            for (int i = 0; i < NR; ++i)
#pragma unroll
                for (int cc = 0; cc < NC; ++cc)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (j0 + j >= S) continue;
                        if (j0 + j == 0) {
                            acc[i][cc] = v[i][cc][0];
                        } else {
                            acc[i][cc].x += v[i][cc][j].x;
                            acc[i][cc].y += v[i][cc][j].y;
                            acc[i][cc].z += v[i][cc][j].z;
                            acc[i][cc].w += v[i][cc][j].w;
                        }
                    }
        }
#pragma unroll
        for (int i = 0; i < NR; ++i)
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                x[i][cc][0] = acc[i][cc].x; x[i][cc][1] = acc[i][cc].y;
                x[i][cc][2] = acc[i][cc].z; x[i][cc][3] = acc[i][cc].w;
            }
    };
    if (all_ok) {
        if (!kv_tile) {
            // BF16 rows: the plain projection's Y, or the fused call's Q heads; two rows per pass
            uint16_t* dst = FMT >= 0 ? ka.qa.q_out : ka.y;
            const int ld = FMT >= 0 ? ka.qa.q_cols : ka.N;
            const int rend = min(r1, M - m0);
#pragma unroll 1
            for (int rr = r0 + warp; rr < rend; rr += 2 * (kQkvThreads / 32)) {
                const int rb = rr + kQkvThreads / 32;
                const bool two = rb < rend;
                const int rows[2] = {rr, two ? rb : rr};
                float x[2][BN / 128][4];
                sum_cols(rows, x);
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    if (i == 1 && !two) break;
#pragma unroll
                    for (int j = 0; j < BN / 128; ++j) {
                        const __nv_bfloat162 lo = __floats2bfloat162_rn(x[i][j][0], x[i][j][1]),
                                             hi = __floats2bfloat162_rn(x[i][j][2], x[i][j][3]);
                        *reinterpret_cast<uint2*>(dst + (int64_t)(m0 + rows[i]) * ld + n0 + 128 * j + 4 * lane) =
                            make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
                    }
                }
            }
        } else if constexpr (FMT >= 0) {
            const int kvj = (n0 - ka.qa.q_cols) / 128;
            append_half_rows<FMT>(a, sm.loc, m0, r0, r1, kvj >> 1, (kvj & 1) != 0, warp, lane,
                                  [&](int rr, float (&xo)[4]) {
                                      const int rows[1] = {rr};
                                      float x[1][1][4];
                                      sum_cols(rows, x);
#pragma unroll
                                      for (int q = 0; q < 4; ++q) xo[q] = x[0][0][q];
                                      round_bf16x4(xo);
                                  });
        }
    }
    cluster_sync_all();                     // the partials stay until every CTA has read them
}

// ---- host: tensor maps through the driver entry point
PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, []() {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// rows x K BF16, K contiguous; boxes of kBK x 128 rows, 128-byte swizzle; rows past
// the end read as zero
bool make_map(CUtensorMap* map, const void* base, int rows, int K)
{
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {(cuuint32_t)kBK, 128u};
    const cuuint32_t estr[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

template <int FMT>
static cudaError_t splitk_attr()
{
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, []() {
        attr = cudaFuncSetAttribute(kv4_gemm_splitk_kernel<FMT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)(sizeof(SplitKSmem) + 1024));
    });
    return attr;
}

// Clusters of S one-SM CTAs that the GPU can hold at once (queried once per device and S;
// 0 when none or the query fails). Thread-block clusters are placed within a GPC, so for
// S > 2 this is below the SM count / S.
static int max_clusters(int S)
{
    static std::mutex mu;
    static int cache[64][9] = {};           // 0 = not asked yet, else count + 1
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev >= 64 || S < 1 || S > 8) return 0;
    std::lock_guard<std::mutex> g(mu);
    if (cache[dev][S] == 0) {
        int n = 0;
        if (splitk_attr<-1>() == cudaSuccess) {
            cudaLaunchConfig_t cfg{};
            cfg.gridDim = dim3((unsigned)S);
            cfg.blockDim = dim3(kQkvThreads);
            cfg.dynamicSmemBytes = sizeof(SplitKSmem) + 1024;
            cudaLaunchAttribute at[1];
            at[0].id = cudaLaunchAttributeClusterDimension;
            at[0].val.clusterDim.x = (unsigned)S;
            at[0].val.clusterDim.y = 1;
            at[0].val.clusterDim.z = 1;
            cfg.attrs = at;
            cfg.numAttrs = 1;
            if (cudaOccupancyMaxActiveClusters(&n, kv4_gemm_splitk_kernel<-1>, &cfg) != cudaSuccess) {
                cudaGetLastError();
                n = 0;
            }
        }
        cache[dev][S] = n + 1;
    }
    return cache[dev][S] - 1;
}

// Split-K plan for an M x N x K projection of one row tile (M <= 128): 128-wide tiles and
// the largest S <= 8 (S <= the k blocks) whose clusters all fit on the GPU at once. (Wider
// tiles run fewer MMAs but park and exchange twice the partial bytes per CTA, and the
// exchange through distributed shared memory costs more than the MMAs save.) With two row
// tiles the tile kernel already fills as many SMs and skips the exchange, so there is no
// split. S = 1: no split. The plain and the fused projection take the same plan, so their
// sums agree bit for bit.
struct SplitKPlan {
    int groups, S;                // 128-wide column tiles (one cluster each), CTAs per cluster
};
static SplitKPlan splitk_plan(int M, int N, int K, int sms)
{
    SplitKPlan p{N / 128, 1};
    if (M > kBM) return p;
    const int nk = K / kBK;
    for (int S = std::min(8, nk); S >= 2; --S)
        if ((int64_t)p.groups * S <= sms && p.groups <= max_clusters(S)) {
            p.S = S;
            return p;
        }
    return p;
}

template <int FMT>
static cudaError_t launch_splitk(const CUtensorMap& mx, const CUtensorMap& mw, const SplitKArgs& ka,
                                 const SplitKPlan& pl, cudaStream_t stream)
{
    const cudaError_t attr = splitk_attr<FMT>();
    if (attr != cudaSuccess) return attr;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3((unsigned)(pl.groups * pl.S));
    cfg.blockDim = dim3(kQkvThreads);
    cfg.dynamicSmemBytes = sizeof(SplitKSmem) + 1024;
    cfg.stream = stream;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = (unsigned)pl.S;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kv4_gemm_splitk_kernel<FMT>, mx, mw, ka);
}

template <int BN>
static cudaError_t launch_bn(const CUtensorMap& mx, const CUtensorMap& mw, void* y, int M, int N, int K,
                             int32_t* err, cudaStream_t stream)
{
    const size_t smem = sizeof(GemmSmem<BN>) + 1024;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [smem]() {
        attr = cudaFuncSetAttribute(kv4_linear_bf16_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)smem);
    });
    if (attr != cudaSuccess) return attr;
    const dim3 grid((unsigned)(N / BN), (unsigned)((M + kBM - 1) / kBM));
    kv4_linear_bf16_kernel<BN><<<grid, kGemmThreads, smem, stream>>>(mx, mw, static_cast<uint16_t*>(y), M, N,
                                                                      K, err);
    return cudaGetLastError();
}

cudaError_t launch_qkv_append(const AppendArgs& ap, const void* x, const void* w, void* q_out, int num_q_heads,
                              int d_model, cudaStream_t stream)
{
    const int T = ap.total_tokens;
    const int N = (num_q_heads + 2 * ap.num_heads) * kHeadDim;
    CUtensorMap mx, mw;
    if (!make_map(&mx, x, T, d_model) || !make_map(&mw, w, N, d_model)) return cudaErrorInvalidValue;
    QkvArgs qa{};
    qa.ap = ap;
    qa.q_out = static_cast<uint16_t*>(q_out);
    qa.q_cols = num_q_heads * kHeadDim;
    const size_t smem_w = sizeof(GemmSmem<256>) + sizeof(TokenLocS) * kBM + 1024,
                 smem_n = sizeof(GemmSmem<128>) + sizeof(TokenLocS) * kBM + 1024;
    static std::once_flag once;
    static cudaError_t attr = cudaSuccess;
    std::call_once(once, [smem_w, smem_n]() {
        const int sw = (int)smem_w, sn = (int)smem_n;
        for (auto k : {kv4_qkv_append_kernel<0>, kv4_qkv_append_kernel<1>, kv4_qkv_append_kernel<2>,
                       kv4_qkv_append_kernel<3>})
            if (attr == cudaSuccess) attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, sw);
        for (auto k : {kv4_qkv_append_narrow_kernel<0>, kv4_qkv_append_narrow_kernel<1>,
                       kv4_qkv_append_narrow_kernel<2>, kv4_qkv_append_narrow_kernel<3>})
            if (attr == cudaSuccess) attr = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, sn);
    });
    if (attr != cudaSuccess) return attr;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const SplitKPlan pl = splitk_plan(T, N, d_model, sms);
    if (pl.S > 1) {
        SplitKArgs ka{};
        ka.qa = qa;
        ka.M = T;
        ka.N = N;
        ka.nk = d_model / kBK;
        if (ap.mx) return launch_splitk<3>(mx, mw, ka, pl, stream);
        if (ap.fp4) return launch_splitk<2>(mx, mw, ka, pl, stream);
        if (ap.kv8) return launch_splitk<1>(mx, mw, ka, pl, stream);
        return launch_splitk<0>(mx, mw, ka, pl, stream);
    }
    const int mt = (T + kBM - 1) / kBM;
    if ((int64_t)mt * (N / 256) >= sms) {
        const dim3 grid((unsigned)(N / 256), (unsigned)mt);
        if (ap.mx) kv4_qkv_append_kernel<3><<<grid, kQkvThreads, smem_w, stream>>>(mx, mw, qa, d_model);
        else if (ap.fp4) kv4_qkv_append_kernel<2><<<grid, kQkvThreads, smem_w, stream>>>(mx, mw, qa, d_model);
        else if (ap.kv8) kv4_qkv_append_kernel<1><<<grid, kQkvThreads, smem_w, stream>>>(mx, mw, qa, d_model);
        else kv4_qkv_append_kernel<0><<<grid, kQkvThreads, smem_w, stream>>>(mx, mw, qa, d_model);
    } else {
        // few tokens: 128-wide tiles double the CTAs
        const dim3 grid((unsigned)(N / 128), (unsigned)mt);
        if (ap.mx) kv4_qkv_append_narrow_kernel<3><<<grid, kQkvThreads, smem_n, stream>>>(mx, mw, qa, d_model);
        else if (ap.fp4) kv4_qkv_append_narrow_kernel<2><<<grid, kQkvThreads, smem_n, stream>>>(mx, mw, qa, d_model);
        else if (ap.kv8) kv4_qkv_append_narrow_kernel<1><<<grid, kQkvThreads, smem_n, stream>>>(mx, mw, qa, d_model);
        else kv4_qkv_append_narrow_kernel<0><<<grid, kQkvThreads, smem_n, stream>>>(mx, mw, qa, d_model);
    }
    return cudaGetLastError();
}

cudaError_t launch_linear_bf16(const void* x, const void* w, void* y, int M, int N, int K, int32_t* err,
                               cudaStream_t stream)
{
    CUtensorMap mx, mw;
    if (!make_map(&mx, x, M, K) || !make_map(&mw, w, N, K)) return cudaErrorInvalidValue;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const SplitKPlan pl = splitk_plan(M, N, K, sms);
    if (pl.S > 1) {
        SplitKArgs ka{};
        ka.y = static_cast<uint16_t*>(y);
        ka.M = M;
        ka.N = N;
        ka.nk = K / kBK;
        ka.err = err;
        return launch_splitk<-1>(mx, mw, ka, pl, stream);
    }
    // 256-wide tiles halve the operand bytes per multiply-add; when they would leave SMs
    // idle (few row tiles), 128-wide tiles double the CTAs
    const int mt = (M + kBM - 1) / kBM;
    if (N % 256 == 0 && (int64_t)mt * (N / 256) >= sms)
        return launch_bn<256>(mx, mw, y, M, N, K, err, stream);
    return launch_bn<128>(mx, mw, y, M, N, K, err, stream);
}

}  // namespace kv4
