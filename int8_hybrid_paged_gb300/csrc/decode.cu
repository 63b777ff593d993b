// decode.cu — kv4_decode_attention: plan, split-K-over-pages attention, exact merge.
//
// Pages cited (title, then section):
//   [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速" — 核心方法 (regions read in
//        parallel, exact softmax merge), 方法步骤详情 step 4, 前置知识 › 分组仿射 KV 量化
//        (scale and offset applied after the dot product)
//   [ko] "INT4 KV 캐시로 비동기 RLVR 롤아웃을 1.8배 가속한다" — 전제와 한계 (INT8 query,
//        integer QK·PV on INT4 codes; INT8 side keys with BF16 values and FP32
//        accumulation; disjoint regions merged by their log-normalizers)
//
// Three launches on the caller's stream:
//   plan   (1 CTA)   per sequence: INT4 pages, chunk size, work-item prefix sums.
//   split  (persistent, SMs × resident CTAs) each CTA takes work items from an
//          atomic ticket: an item is (sequence b, KV head h, chunk of INT4 pages)
//          or (b, h, protected region). Pages are staged into shared memory with
//          1-D bulk copies on per-warp mbarrier rings; each warp streams its own
//          pages, so no CTA-wide barrier sits inside the page loop.
//   merge  (warp per q head) exact log-sum-exp merge of the item partials.
#include <float.h>

#include <mutex>

#include "device_common.cuh"
#include "kv4_internal.h"

namespace kv4 {

constexpr int kWarps = kDecodeThreads / 32;
constexpr int kMaxG = 4;
constexpr int kMinChunkPages = 16;

struct __align__(128) SplitSmem {
    uint8_t stage[kWarps][kStages][kPageBlock];   // page staging, per warp
    int8_t q8[kMaxG][kHeadDim];                   // INT8 rotated query of the item's heads
    float qscale[kMaxG];
    int32_t qsum[kMaxG];
    uint8_t wbuf[kWarps][kMaxG][16];              // u8 PV weights of the page in flight
    float pbuf[kWarps][kMaxG][16];                // protected-path weights of a position group
    float wM[kWarps][kMaxG];                      // per-warp running max (log2)
    float wL[kWarps][kMaxG];                      // per-warp normalizer
    uint64_t bar[kWarps][kStages];
    int32_t item;
    int32_t abort;
};

__device__ __forceinline__ int int4_pages(int L, int s, int w)
{
    // pages touched by the INT4 region [s, L - w)
    return (L - w > s) ? ((L - w - 1) / kPage - s / kPage + 1) : 0;
}

// ---------------------------------------------------------------- plan
// Chunk size C (pages per item) aims at about `target_items` items in total and is
// raised if the workspace could not hold the items otherwise:
// items ≤ H·(T/C + 2B) ≤ max_items  ⇐  C ≥ H·T / (max_items − 2·H·B).
__global__ void __launch_bounds__(1024) kv4_decode_plan_kernel(DecodeArgs a)
{
    __shared__ long long s_red[32];
    __shared__ int s_scan[32];
    __shared__ int s_chunk;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int B = a.batch, H = a.num_heads;
    const int per = (B + 1023) / 1024;
    const int b0 = min(B, tid * per), b1 = min(B, b0 + per);

    long long T = 0;
    for (int b = b0; b < b1; ++b) T += int4_pages(max(0, a.context_lens[b]), a.sink, a.window);
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) T += __shfl_xor_sync(kFull, T, m);
    if (lane == 0) s_red[warp] = T;
    __syncthreads();
    if (tid == 0) {
        long long tot = 0;
        for (int k = 0; k < 32; ++k) tot += s_red[k];
        long long need = tot * H;
        long long C = (need + a.target_items - 1) / max(1, a.target_items);
        if (C < kMinChunkPages) C = kMinChunkPages;
        const long long room = (long long)a.max_items - 2LL * H * B;
        if (room > 0) {
            long long Cmin = (need + room - 1) / room;
            if (C < Cmin) C = Cmin;
        }
        if (C > (1 << 30)) C = 1 << 30;
        s_chunk = (int)C;
    }
    __syncthreads();
    const int C = s_chunk;

    int local = 0;
    for (int b = b0; b < b1; ++b) {
        const int n = int4_pages(max(0, a.context_lens[b]), a.sink, a.window);
        local += H * ((n + C - 1) / C + 1);
    }
    // block-wide exclusive scan of the per-thread counts
    int incl = local;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int v = __shfl_up_sync(kFull, incl, m);
        if (lane >= m) incl += v;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = s_scan[lane];
        int x = v;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int u = __shfl_up_sync(kFull, x, m);
            if (lane >= m) x += u;
        }
        s_scan[lane] = x - v;   // exclusive offset of each warp
    }
    __syncthreads();
    int off = s_scan[warp] + incl - local;
    for (int b = b0; b < b1; ++b) {
        a.item_start[b] = off;
        const int n = int4_pages(max(0, a.context_lens[b]), a.sink, a.window);
        off += H * ((n + C - 1) / C + 1);
    }
    if (tid == 1023) {
        a.item_start[B] = off;        // thread 1023 owns the last range (possibly empty)
        a.plan->chunk_pages = C;
        a.plan->total_items = off;
        a.plan->counter = 0;
    }
}

// ---------------------------------------------------------------- split: helpers

// Per-warp running state of one item: o is relative to 2^M, l likewise.
template <int G>
struct WarpState {
    float o[G][4];      // dims 4·lane .. 4·lane+3 of each head
    float M[G];         // running max (log2 domain), uniform over the warp
    float l[G];         // this lane's share of the normalizer
    float bias[G];      // this lane's share of Σ p'·m^V (INT4 path)
};

template <int G>
__device__ __forceinline__ void state_init(WarpState<G>& st)
{
#pragma unroll
    for (int g = 0; g < G; ++g) {
        st.M[g] = -INFINITY;
        st.l[g] = 0.f;
        st.bias[g] = 0.f;
#pragma unroll
        for (int d = 0; d < 4; ++d) st.o[g][d] = 0.f;
    }
}

// Heads scored by a lane: with G ≥ 2 the two lanes of a token pair split the
// heads (half 0 takes the first G/2); with G = 1 both score head 0.
template <int G>
struct HeadSplit {
    static constexpr int GL = (G >= 2) ? G / 2 : 1;
    __device__ static int head(int half, int j) { return (G >= 2) ? half * GL + j : 0; }
    // does the lane own head gg's normalizer contribution?
    __device__ static bool owns(int half, int gg) { return (G >= 2) ? (gg / GL == half) : (half == 0); }
};

// Exchange per-lane values of the lane's own heads so every lane knows all G.
template <int G>
__device__ __forceinline__ void share_heads(const float (&mine)[HeadSplit<G>::GL], int half,
                                            float (&all)[G])
{
    constexpr int GL = HeadSplit<G>::GL;
    float other[GL];
#pragma unroll
    for (int j = 0; j < GL; ++j) other[j] = __shfl_xor_sync(kFull, mine[j], 1);
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
        if (G >= 2) {
            const int jj = gg % GL, hh = gg / GL;
            all[gg] = (hh == half) ? mine[jj] : other[jj];
        } else {
            all[gg] = mine[0];
        }
    }
}

// max over the 16 token lanes of the same half (lane bits 1..4)
__device__ __forceinline__ float token_max(float v)
{
#pragma unroll
    for (int m = 2; m < 32; m <<= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}

template <int G>
__device__ __forceinline__ int pick(const int (&v)[G], int g)
{
    int r = v[0];
#pragma unroll
    for (int gg = 1; gg < G; ++gg)
        if (gg == g) r = v[gg];
    return r;
}

// ---------------------------------------------------------------- split: INT4 page
// One staged page (16 positions) against the item's G query heads.
// QK: lane pair (t, half) covers token t; each lane dots 64 dims (8 words of 8
// codes) against the matching query bytes with dp4a, the pair sums by shuffle.
// PV: lane l owns dims 4l..4l+3; the u8 weights of all 16 tokens are broadcast
// from shared memory and dotted with 4-token code words.
template <int G, bool DEBUG>
__device__ __forceinline__ void int4_page(const DecodeArgs& a, SplitSmem& sm, WarpState<G>& st,
                                          const uint8_t* pg, int lp, int r4_lo, int r4_hi,
                                          const uint32_t (&qlo)[G][8], const uint32_t (&qhi)[G][8],
                                          const float (&qs)[G], const float (&qsumf)[G],
                                          int b, int h, int warp, int lane)
{
    using HS = HeadSplit<G>;
    constexpr int GL = HS::GL;
    const int t = lane >> 1, half = lane & 1;

    // ---- integer QK
    const uint4 ka = *reinterpret_cast<const uint4*>(pg + kKCodeOff + t * 64 + half * 32);
    const uint4 kb = *reinterpret_cast<const uint4*>(pg + kKCodeOff + t * 64 + half * 32 + 16);
    const uint32_t kw[8] = {ka.x, ka.y, ka.z, ka.w, kb.x, kb.y, kb.z, kb.w};
    int dot[G];
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t lo = kw[i] & 0x0F0F0F0Fu;
        const uint32_t hi = (kw[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            dot[g] = dp4a_su(qlo[g][i], lo, dot[g]);
            dot[g] = dp4a_su(qhi[g][i], hi, dot[g]);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] += __shfl_xor_sync(kFull, dot[g], 1);

    const int pos = lp * kPage + t;
    const bool valid = pos >= r4_lo && pos < r4_hi;
    const __half2 kmeta = *reinterpret_cast<const __half2*>(pg + kKMetaOff + t * 4);
    const __half2 vmeta = *reinterpret_cast<const __half2*>(pg + kVMetaOff + t * 4);
    const float kd = __low2float(kmeta), kmin = __high2float(kmeta);
    const float vd = __low2float(vmeta), vmin = __high2float(vmeta);

    // ---- scores, page max, page-local weights, u8 quantization (lane's own heads)
    float pmax[GL], wmx[GL], pp[GL];
#pragma unroll
    for (int j = 0; j < GL; ++j) {
        const int g = HS::head(half, j);
        const int d = pick<G>(dot, g);
        float sqg = qs[0], qsg = qsumf[0];
#pragma unroll
        for (int gg = 1; gg < G; ++gg)
            if (gg == g) { sqg = qs[gg]; qsg = qsumf[gg]; }
        const float u = __fmaf_rn(kd, (float)d, __fmul_rn(kmin, qsg));
        const float sig = valid ? __fmul_rn(__fmul_rn(u, sqg), a.log2_scale) : -INFINITY;
        const float Mp = token_max(sig);
        const float p = valid ? exp2_poly(__fsub_rn(sig, Mp)) : 0.f;
        const float wv = valid ? __fmul_rn(p, vd) : 0.f;
        const float wmax = token_max(wv);
        const bool qz = wmax > 0x1p-64f;
        const float iw = qz ? __fdiv_rn(255.f, wmax) : 0.f;
        int wh = 0;
        if (valid && qz) wh = min(__float2int_rn(__fmul_rn(wv, iw)), 255);
        if (G >= 2 || half == 0) sm.wbuf[warp][g][t] = (uint8_t)wh;
        if (DEBUG && valid && pos < a.dbg_stride && (G >= 2 || half == 0)) {
            const int64_t o = ((int64_t)b * a.num_q_heads + h * G + g) * a.dbg_stride + pos;
            if (a.dbg_qk) a.dbg_qk[o] = d;
            if (a.dbg_w) a.dbg_w[o] = (uint8_t)wh;
        }
        pmax[j] = Mp;
        wmx[j] = qz ? __fmul_rn(wmax, 1.0f / 255.0f) : 0.f;
        pp[j] = p;
    }
    float Mall[G], swall[G];
    share_heads<G>(pmax, half, Mall);
    share_heads<G>(wmx, half, swall);

    // ---- rescale factors; normalizer and offset-term shares of this lane
    float alpha[G], scale[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float Mn = fmaxf(st.M[g], Mall[g]);
        const bool none = (Mn == -INFINITY);            // no valid position yet
        alpha[g] = none ? 1.f : exp2_fast(st.M[g] - Mn);
        const float beta = none ? 0.f : exp2_fast(Mall[g] - Mn);
        scale[g] = beta * swall[g];
        st.M[g] = Mn;
        float contrib = 0.f;
        if (HS::owns(half, g)) contrib = pp[(G >= 2) ? g % GL : 0];
        st.l[g] = st.l[g] * alpha[g] + beta * contrib;
        st.bias[g] = st.bias[g] * alpha[g] + beta * (valid ? contrib * vmin : 0.f);
    }
    __syncwarp();

    // ---- integer PV
    uint32_t W[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const uint4 wq = *reinterpret_cast<const uint4*>(&sm.wbuf[warp][g][0]);
        W[g][0] = wq.x; W[g][1] = wq.y; W[g][2] = wq.z; W[g][3] = wq.w;
    }
    const uint4 va = *reinterpret_cast<const uint4*>(pg + kVCodeOff + lane * 32);
    const uint4 vb = *reinterpret_cast<const uint4*>(pg + kVCodeOff + lane * 32 + 16);
    const uint32_t v0[4] = {va.x, va.y, va.z, va.w};   // dim pair 2l, token quads 0..3
    const uint32_t v1[4] = {vb.x, vb.y, vb.z, vb.w};   // dim pair 2l+1
    int acc[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int d = 0; d < 4; ++d) acc[g][d] = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t lo0 = v0[k] & 0x0F0F0F0Fu, hi0 = (v0[k] >> 4) & 0x0F0F0F0Fu;
        const uint32_t lo1 = v1[k] & 0x0F0F0F0Fu, hi1 = (v1[k] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            acc[g][0] = dp4a_uu(lo0, W[g][k], acc[g][0]);
            acc[g][1] = dp4a_uu(hi0, W[g][k], acc[g][1]);
            acc[g][2] = dp4a_uu(lo1, W[g][k], acc[g][2]);
            acc[g][3] = dp4a_uu(hi1, W[g][k], acc[g][3]);
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int d = 0; d < 4; ++d) st.o[g][d] = fmaf(scale[g], (float)acc[g][d], st.o[g][d] * alpha[g]);
    __syncwarp();
}

template <int G>
__device__ __forceinline__ float pickf(const float (&v)[G], int g)
{
    float r = v[0];
#pragma unroll
    for (int gg = 1; gg < G; ++gg)
        if (gg == g) r = v[gg];
    return r;
}

// ---------------------------------------------------------------- split: protected group
// 16 protected positions (group `grp`) against the item's G heads. The same INT8
// query meets the 8-bit side keys (natural dim order, query bytes broadcast from
// shared memory); side values are dequantized to bf16 and accumulated in FP32.
template <int G, bool DEBUG>
__device__ __forceinline__ void protected_group(const DecodeArgs& a, SplitSmem& sm,
                                                WarpState<G>& st, const uint8_t* sb, int S,
                                                int grp, int npos, int n_sink, int ring_lo,
                                                const float (&qs)[G], const float (&qsumf)[G],
                                                int b, int h, int warp, int lane)
{
    using HS = HeadSplit<G>;
    constexpr int GL = HS::GL;
    const int t = lane >> 1, half = lane & 1;
    const int s = a.sink, w = a.window;
    const int k = grp * 16 + t;
    const bool valid = k < npos;
    int tpos = 0, sidx = 0;
    if (valid) {
        tpos = (k < n_sink) ? k : ring_lo + (k - n_sink);
        sidx = (tpos < s) ? tpos : s + tpos % w;
    }
    int dot[G];
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] = 0;
    if (valid) {
        const uint4* kr = reinterpret_cast<const uint4*>(sb + sidx * 128 + half * 64);
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
            const uint4 c4 = __ldg(kr + q4);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const uint4 qv = *reinterpret_cast<const uint4*>(&sm.q8[g][half * 64 + q4 * 16]);
                dot[g] = dp4a_su(qv.x, c4.x, dot[g]);
                dot[g] = dp4a_su(qv.y, c4.y, dot[g]);
                dot[g] = dp4a_su(qv.z, c4.z, dot[g]);
                dot[g] = dp4a_su(qv.w, c4.w, dot[g]);
            }
        }
    }
#pragma unroll
    for (int g = 0; g < G; ++g) dot[g] += __shfl_xor_sync(kFull, dot[g], 1);

    float kd = 0.f, kmin = 0.f;
    if (valid) {
        const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(sb + S * 256 + sidx * 4));
        const __half2 km = *reinterpret_cast<const __half2*>(&mw);
        kd = __low2float(km);
        kmin = __high2float(km);
    }
    float sig[GL], gmax[GL];
#pragma unroll
    for (int j = 0; j < GL; ++j) {
        const int g = HS::head(half, j);
        const int d = pick<G>(dot, g);
        const float sqg = pickf<G>(qs, g), qsg = pickf<G>(qsumf, g);
        const float u = __fmaf_rn(kd, (float)d, __fmul_rn(kmin, qsg));
        sig[j] = valid ? __fmul_rn(__fmul_rn(u, sqg), a.log2_scale) : -INFINITY;
        gmax[j] = token_max(sig[j]);
        if (DEBUG && valid && a.dbg_qk && tpos < a.dbg_stride && (G >= 2 || half == 0))
            a.dbg_qk[((int64_t)b * a.num_q_heads + h * G + g) * a.dbg_stride + tpos] = d;
    }
    float Mall[G];
    share_heads<G>(gmax, half, Mall);
    float alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float Mn = fmaxf(st.M[g], Mall[g]);
        alpha[g] = (Mn == -INFINITY) ? 1.f : exp2_fast(st.M[g] - Mn);
        st.M[g] = Mn;
    }
    float p[GL];
#pragma unroll
    for (int j = 0; j < GL; ++j) {
        const int g = HS::head(half, j);
        p[j] = valid ? exp2_poly(__fsub_rn(sig[j], pickf<G>(st.M, g))) : 0.f;
        if (G >= 2 || half == 0) sm.pbuf[warp][g][t] = p[j];
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float contrib = HS::owns(half, g) ? p[(G >= 2) ? g % GL : 0] : 0.f;
        st.l[g] = st.l[g] * alpha[g] + contrib;
#pragma unroll
        for (int d = 0; d < 4; ++d) st.o[g][d] *= alpha[g];
    }
    __syncwarp();
    const int n_here = min(16, npos - grp * 16);
    for (int tt = 0; tt < n_here; ++tt) {
        const int kk = grp * 16 + tt;
        const int tp = (kk < n_sink) ? kk : ring_lo + (kk - n_sink);
        const int si = (tp < s) ? tp : s + tp % w;
        const uint32_t vcw = __ldg(reinterpret_cast<const uint32_t*>(sb + S * 128 + si * 128 + 4 * lane));
        const uint32_t mw = __ldg(reinterpret_cast<const uint32_t*>(sb + S * 260 + si * 4));
        const __half2 vm = *reinterpret_cast<const __half2*>(&mw);
        const float vd = __low2float(vm), vmin = __high2float(vm);
        float v[4];
#pragma unroll
        for (int m = 0; m < 4; ++m)
            v[m] = __bfloat162float(
                __float2bfloat16_rn(__fmaf_rn(vd, (float)((vcw >> (8 * m)) & 255u), vmin)));
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float pw = sm.pbuf[warp][g][tt];
#pragma unroll
            for (int m = 0; m < 4; ++m) st.o[g][m] = fmaf(pw, v[m], st.o[g][m]);
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- split kernel
template <int G, bool DEBUG>
__global__ void __launch_bounds__(kDecodeThreads) kv4_decode_split_kernel(DecodeArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SplitSmem& sm = *reinterpret_cast<SplitSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int H = a.num_heads, s = a.sink, w = a.window;

    if (tid == 0) {
        for (int ww = 0; ww < kWarps; ++ww)
            for (int k = 0; k < kStages; ++k) mbar_init(&sm.bar[ww][k], 1);
        fence_mbar_init();
        sm.abort = 0;
    }
    __syncthreads();
    uint32_t phase = 0;                    // bit k: parity awaited next on this warp's stage k
    const int total = a.plan->total_items;
    const int C = a.plan->chunk_pages;

    for (;;) {
        if (tid == 0) sm.item = atomicAdd(&a.plan->counter, 1);
        __syncthreads();
        const int item = sm.item;
        if (item >= total || sm.abort) break;

        // ---- which sequence, head and chunk
        int lo = 0, hi = a.batch;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(&a.item_start[mid]) <= item) lo = mid; else hi = mid;
        }
        const int b = lo;
        const int i0 = __ldg(&a.item_start[b]), i1 = __ldg(&a.item_start[b + 1]);
        const int per_head = (i1 - i0) / H;
        const int r = item - i0;
        const int h = r / per_head, c = r - h * per_head;
        const bool prot = (c == per_head - 1);
        const int L = max(0, __ldg(&a.context_lens[b]));
        const int slot = __ldg(&a.slot_ids[b]);
        const bool slot_ok = slot >= 0 && slot < a.max_slots;

        // ---- rotate and quantize the item's G query heads (one warp per head)
        if (warp < G) {
            const int hq = h * G + warp;
            float x[4];
            load_bf16x4(a.q + ((int64_t)b * a.num_q_heads + hq) * kHeadDim + 4 * lane, x);
            warp_fwht128(x, lane);
            const float amax =
                warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
            int q[4] = {0, 0, 0, 0};
            float sq = 0.f;
            if (amax > 0.f) {
                const float inv = __fdiv_rn(127.0f, amax);
#pragma unroll
                for (int i = 0; i < 4; ++i) q[i] = __float2int_rn(__fmul_rn(x[i], inv));
                sq = __fdiv_rn(amax, 127.0f);
            }
            const int qsum = warp_sum_int(q[0] + q[1] + q[2] + q[3]);
            const uint32_t packed = (uint32_t)(q[0] & 255) | ((uint32_t)(q[1] & 255) << 8) |
                                    ((uint32_t)(q[2] & 255) << 16) | ((uint32_t)(q[3] & 255) << 24);
            *reinterpret_cast<uint32_t*>(&sm.q8[warp][4 * lane]) = packed;
            if (lane == 0) {
                sm.qscale[warp] = sq;
                sm.qsum[warp] = qsum;
            }
            if (DEBUG && prot) {
                const int64_t o = ((int64_t)b * a.num_q_heads + hq);
                if (a.dbg_q8) *reinterpret_cast<uint32_t*>(a.dbg_q8 + o * kHeadDim + 4 * lane) = packed;
                if (a.dbg_qscale && lane == 0) a.dbg_qscale[o] = sq;
            }
        }
        __syncthreads();

        WarpState<G> st;
        state_init<G>(st);
        float qs[G], qsumf[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            qs[g] = sm.qscale[g];
            qsumf[g] = (float)sm.qsum[g];
        }

        if (!prot) {
            // ---- INT4 region [s, L - w): pages cp0 .. cp1-1, warp w takes every 4th
            const int r4_lo = s, r4_hi = L - w;
            const int cp0 = s / kPage + c * C;
            const int cp1 = min(cp0 + C, (r4_hi - 1) / kPage + 1);
            const int np = max(0, cp1 - cp0);
            const int nl = (np > warp) ? (np - warp + kWarps - 1) / kWarps : 0;
            uint32_t qlo[G][8], qhi[G][8];
            {
                const int half = lane & 1;
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int base = 64 * half + 8 * i;
                        const uint32_t A = *reinterpret_cast<const uint32_t*>(&sm.q8[g][base]);
                        const uint32_t B = *reinterpret_cast<const uint32_t*>(&sm.q8[g][base + 4]);
                        qlo[g][i] = prmt(A, B, 0x6420);   // dims base+0, +2, +4, +6 (low nibbles)
                        qhi[g][i] = prmt(A, B, 0x7531);   // dims base+1, +3, +5, +7 (high nibbles)
                    }
            }
            const int64_t bt_row = (int64_t)b * a.stride;
            const uint8_t* head_base = a.pages + (int64_t)h * kPageBlock;
            const int64_t page_stride = (int64_t)H * kPageBlock;
            auto issue = [&](int stg, int j) {
                const int lp = cp0 + warp + kWarps * j;
                int page = 0;
                if (lp < a.stride) page = __ldg(&a.block_table[bt_row + lp]);
                else report_error(a.err, KV4_DEVERR_BAD_POSITION);
                if (page < 0 || (int64_t)page >= a.num_pages) {
                    report_error(a.err, KV4_DEVERR_BAD_PAGE);
                    page = 0;
                }
                fence_proxy_async();
                mbar_expect_tx(&sm.bar[warp][stg], kPageBlock);
                bulk_g2s(sm.stage[warp][stg], head_base + (int64_t)page * page_stride, kPageBlock,
                         &sm.bar[warp][stg]);
            };
            if (lane == 0)
                for (int k = 0; k < kStages && k < nl; ++k) issue(k, k);
            __syncwarp();
            for (int j = 0; j < nl; ++j) {
                const int stg = j % kStages;
                const bool ok = mbar_wait_bounded(&sm.bar[warp][stg], (phase >> stg) & 1u);
                phase ^= 1u << stg;
                if (!ok && lane == 0) {
                    report_error(a.err, KV4_DEVERR_WAIT_TIMEOUT);
                    sm.abort = 1;
                }
                int4_page<G, DEBUG>(a, sm, st, sm.stage[warp][stg], cp0 + warp + kWarps * j, r4_lo,
                                    r4_hi, qlo, qhi, qs, qsumf, b, h, warp, lane);
                if (lane == 0 && j + kStages < nl) issue(stg, j + kStages);
                __syncwarp();
            }
        } else {
            // ---- protected region [0, min(s, L)) ∪ [max(s, L - w), L) from the side buffer
            if (tid == 0) {
                if (!slot_ok) report_error(a.err, KV4_DEVERR_BAD_SLOT);
                else if (L != __ldg(&a.seq_len[slot])) report_error(a.err, KV4_DEVERR_LEN_MISMATCH);
            }
            const int n_sink = slot_ok ? min(s, L) : 0;
            const int ring_lo = max(s, L - w);
            const int n_ring = slot_ok ? max(0, L - ring_lo) : 0;
            const int npos = n_sink + n_ring;
            const int S = s + w;
            const uint8_t* sb = a.side + ((int64_t)(slot_ok ? slot : 0) * H + h) * a.side_block_bytes;
            for (int grp = warp; grp * 16 < npos; grp += kWarps)
                protected_group<G, DEBUG>(a, sm, st, sb, S, grp, npos, n_sink, ring_lo, qs, qsumf, b,
                                          h, warp, lane);
        }

        // ---- warp totals -> shared memory (own stage 0 is idle now)
        float ltot[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float l = st.l[g], bb = st.bias[g];
#pragma unroll
            for (int m = 16; m > 0; m >>= 1) {
                l += __shfl_xor_sync(kFull, l, m);
                bb += __shfl_xor_sync(kFull, bb, m);
            }
            ltot[g] = l;
#pragma unroll
            for (int d = 0; d < 4; ++d) st.o[g][d] += bb;
        }
        float* red = reinterpret_cast<float*>(sm.stage[warp][0]);
#pragma unroll
        for (int g = 0; g < G; ++g)
            *reinterpret_cast<float4*>(&red[g * kHeadDim + 4 * lane]) =
                make_float4(st.o[g][0], st.o[g][1], st.o[g][2], st.o[g][3]);
        if (lane < G) {
            sm.wM[warp][lane] = pickf<G>(st.M, lane);
            sm.wL[warp][lane] = pickf<G>(ltot, lane);
        }
        __syncthreads();

        // ---- combine the warps (thread = dim) and write the item's partial
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float Mx = -INFINITY;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) Mx = fmaxf(Mx, sm.wM[ww][g]);
            float acc = 0.f, lsum = 0.f;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) {
                const float Mw = sm.wM[ww][g];
                if (Mw == -INFINITY) continue;
                const float f = exp2_fast(Mw - Mx);
                acc = fmaf(f, reinterpret_cast<const float*>(sm.stage[ww][0])[g * kHeadDim + tid], acc);
                lsum = fmaf(f, sm.wL[ww][g], lsum);
            }
            a.part_o[((int64_t)item * G + g) * kHeadDim + tid] = acc;
            if (tid == 0) a.part_ml[(int64_t)item * G + g] = make_float2(Mx, lsum);
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- merge
// Exact log-sum-exp merge of a q head's partials: M* = max M_i,
// O = Σ 2^(M_i − M*) o_i / Σ 2^(M_i − M*) l_i, lse = (M* + log2 den) · ln 2.
template <int G>
__global__ void __launch_bounds__(128) kv4_decode_merge_kernel(DecodeArgs a)
{
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (gw >= a.batch * a.num_q_heads) return;
    const int b = gw / a.num_q_heads, hq = gw - b * a.num_q_heads;
    const int h = hq / G, g = hq - h * G;
    const int i0 = a.item_start[b], i1 = a.item_start[b + 1];
    const int per_head = (i1 - i0) / a.num_heads;
    const int first = i0 + h * per_head;
    float Mx = -INFINITY;
    for (int k = lane; k < per_head; k += 32) Mx = fmaxf(Mx, a.part_ml[(int64_t)(first + k) * G + g].x);
    Mx = warp_max(Mx);
    float den = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Mx != -INFINITY) {
        for (int k = 0; k < per_head; ++k) {
            const float2 ml = a.part_ml[(int64_t)(first + k) * G + g];
            if (ml.x == -INFINITY) continue;
            const float f = exp2f(ml.x - Mx);
            den = fmaf(f, ml.y, den);
            const float4 v = *reinterpret_cast<const float4*>(
                &a.part_o[((int64_t)(first + k) * G + g) * kHeadDim + 4 * lane]);
            o.x = fmaf(f, v.x, o.x);
            o.y = fmaf(f, v.y, o.y);
            o.z = fmaf(f, v.z, o.z);
            o.w = fmaf(f, v.w, o.w);
        }
    }
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (den > 0.f) res = make_float4(o.x / den, o.y / den, o.z / den, o.w / den);
    *reinterpret_cast<float4*>(&a.out[((int64_t)b * a.num_q_heads + hq) * kHeadDim + 4 * lane]) = res;
    if (a.lse && lane == 0)
        a.lse[(int64_t)b * a.num_q_heads + hq] =
            (den > 0.f) ? (Mx + log2f(den)) * 0.69314718055994531f : -INFINITY;
}

// ---------------------------------------------------------------- launchers
template <int G, bool DEBUG>
static cudaError_t launch_g(const DecodeArgs& a, int grid, cudaStream_t stream, cudaEvent_t* ev)
{
    if (ev) cudaEventRecord(ev[0], stream);
    kv4_decode_plan_kernel<<<1, 1024, 0, stream>>>(a);
    if (ev) cudaEventRecord(ev[1], stream);
    kv4_decode_split_kernel<G, DEBUG><<<grid, kDecodeThreads, sizeof(SplitSmem), stream>>>(a);
    if (ev) cudaEventRecord(ev[2], stream);
    const int warps = a.batch * a.num_q_heads;
    kv4_decode_merge_kernel<G><<<(warps + 3) / 4, 128, 0, stream>>>(a);
    if (ev) cudaEventRecord(ev[3], stream);
    return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t stream, cudaEvent_t* ev)
{
    const bool dbg = a.dbg_q8 || a.dbg_qscale || a.dbg_qk || a.dbg_w;
    switch (a.group) {
    case 1: return dbg ? launch_g<1, true>(a, grid, stream, ev) : launch_g<1, false>(a, grid, stream, ev);
    case 2: return dbg ? launch_g<2, true>(a, grid, stream, ev) : launch_g<2, false>(a, grid, stream, ev);
    case 4: return dbg ? launch_g<4, true>(a, grid, stream, ev) : launch_g<4, false>(a, grid, stream, ev);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t decode_ctas_per_sm(int group, int* ctas)
{
    const size_t smem = sizeof(SplitSmem);
    switch (group) {
    case 1: return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kv4_decode_split_kernel<1, false>, kDecodeThreads, smem);
    case 2: return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kv4_decode_split_kernel<2, false>, kDecodeThreads, smem);
    case 4: return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kv4_decode_split_kernel<4, false>, kDecodeThreads, smem);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace kv4

// ---------------------------------------------------------------- decode without allocation
// A variant of kv4_decode_attention for callers that cannot make device
// allocations: its split-K scratch (plan header, item offsets, partial outputs)
// lives in the file-scope array below instead of a cache-owned workspace, and it
// reads caller-provided pools, so nothing is allocated by anyone for the call.
// The array is reserved on every GPU that loads this library, until the process
// exits. In host code its name is only a host-side stand-in; the kernels get its
// device address, looked up once per device with that device current.
namespace kv4 {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kNoAllocMaxBatch = 4096;
constexpr size_t kNoAllocHeaderBytes = 256;
constexpr size_t kNoAllocStartBytes = ((size_t)(kNoAllocMaxBatch + 1) * 4 + 255) / 256 * 256;

static __device__ __align__(256) unsigned char g_kv4_noalloc_scratch[kNoAllocScratchBytes];

}  // namespace kv4

namespace {

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
    std::once_flag once;
    unsigned char* scratch = nullptr;   // device address of g_kv4_noalloc_scratch
    cudaError_t status = cudaSuccess;
    int grid[5] = {0, 0, 0, 0, 0};
};

NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Set-up on the current device, once: resolve the scratch array's device address
// and size the persistent grid. Allocates nothing.
NoAllocDevice* noalloc_device(int dev)
{
    if (dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
    NoAllocDevice* d = &g_noalloc_dev[dev];
    std::call_once(d->once, [d, dev]() {
        void* p = nullptr;
        d->status = cudaGetSymbolAddress(&p, kv4::g_kv4_noalloc_scratch);
        if (d->status != cudaSuccess) return;
        d->scratch = static_cast<unsigned char*>(p);
        int sms = 0;
        d->status = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (d->status != cudaSuccess) return;
        for (int g = 1; g <= 4; g <<= 1) {
            int per_sm = 0;
            if (kv4::decode_ctas_per_sm(g, &per_sm) != cudaSuccess || per_sm < 1) per_sm = 1;
            d->grid[g] = sms * per_sm;
        }
    });
    return d;
}

}  // namespace

extern "C" kv4_status kv4_decode_attention_noalloc(
    const kv4_cache_config* cfg, const void* page_pool_dev, const void* side_pool_dev,
    const int32_t* seq_len_dev, const void* q_bf16_dev, int num_q_heads,
    const int32_t* slot_ids_dev, const int32_t* context_lens_dev, const int32_t* block_table_dev,
    int block_table_stride, int batch, float sm_scale, float* out_dev, float* lse_dev, void* stream)
{
    using namespace kv4;
    if (!cfg || batch < 0 || num_q_heads < 1 || block_table_stride < 0) return KV4_ERR_INVALID_ARG;
    if (cfg->head_dim != KV4_HEAD_DIM || cfg->page_size != KV4_PAGE_SIZE) return KV4_ERR_UNSUPPORTED;
    if (cfg->num_kv_heads < 1 || cfg->sink < 0 || cfg->window < 0 || cfg->num_pages < 1 ||
        cfg->max_slots < 1)
        return KV4_ERR_INVALID_ARG;
    if (cfg->sink + cfg->window > kMaxProtected || cfg->num_pages > INT32_MAX) return KV4_ERR_UNSUPPORTED;
    if (batch == 0) return KV4_OK;
    if (!page_pool_dev || !side_pool_dev || !seq_len_dev || !q_bf16_dev || !slot_ids_dev ||
        !context_lens_dev || !block_table_dev || !out_dev || block_table_stride < 1)
        return KV4_ERR_INVALID_ARG;
    if (!(sm_scale == sm_scale) || sm_scale == INFINITY || sm_scale == -INFINITY) return KV4_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(q_bf16_dev) & 7) || (reinterpret_cast<uintptr_t>(out_dev) & 15) ||
        (reinterpret_cast<uintptr_t>(page_pool_dev) & 15) || (reinterpret_cast<uintptr_t>(side_pool_dev) & 15))
        return KV4_ERR_INVALID_ARG;
    const int H = cfg->num_kv_heads;
    if (num_q_heads % H != 0) return KV4_ERR_INVALID_ARG;
    const int G = num_q_heads / H;
    if (G != 1 && G != 2 && G != 4) return KV4_ERR_UNSUPPORTED;
    // sizes beyond the scratch array are refused: at most 4096 sequences, and room for
    // at least 3 * batch * H_kv partials of G heads
    if (batch > kNoAllocMaxBatch) return KV4_ERR_OUT_OF_RANGE;
    const size_t per_item = (size_t)G * (kHeadDim * sizeof(float) + sizeof(float2));
    const size_t avail = kNoAllocScratchBytes - kNoAllocHeaderBytes - kNoAllocStartBytes - 256;
    const size_t items_cap = avail / per_item;
    if ((size_t)3 * batch * H > items_cap) return KV4_ERR_OUT_OF_RANGE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KV4_ERR_CUDA;
    NoAllocDevice* d = noalloc_device(dev);
    if (!d) return KV4_ERR_UNSUPPORTED;
    if (d->status != cudaSuccess || !d->scratch) return KV4_ERR_CUDA;

    unsigned char* base = d->scratch;
    const size_t ml_off = kNoAllocHeaderBytes + kNoAllocStartBytes;
    const size_t o_off = ml_off + (items_cap * G * sizeof(float2) + 255) / 256 * 256;

    DecodeArgs a{};
    a.q = static_cast<const uint16_t*>(q_bf16_dev);
    a.slot_ids = slot_ids_dev;
    a.context_lens = context_lens_dev;
    a.block_table = block_table_dev;
    a.stride = block_table_stride;
    a.batch = batch;
    a.num_q_heads = num_q_heads;
    a.num_heads = H;
    a.group = G;
    a.sink = cfg->sink;
    a.window = cfg->window;
    a.max_slots = cfg->max_slots;
    a.num_pages = cfg->num_pages;
    a.log2_scale = (float)((double)sm_scale * 1.4426950408889634074);
    a.pages = static_cast<const uint8_t*>(page_pool_dev);
    a.side = static_cast<const uint8_t*>(side_pool_dev);
    a.side_block_bytes = (int64_t)(((size_t)(cfg->sink + cfg->window) * 264 + 15) / 16 * 16);
    a.seq_len = seq_len_dev;
    a.err = nullptr;                      // no error word: device index errors are skipped silently
    a.plan = reinterpret_cast<PlanHeader*>(base);
    a.item_start = reinterpret_cast<int32_t*>(base + kNoAllocHeaderBytes);
    a.part_ml = reinterpret_cast<float2*>(base + ml_off);
    a.part_o = reinterpret_cast<float*>(base + o_off);
    a.max_items = (int32_t)items_cap;
    a.target_items = 16 * d->grid[G];
    a.out = out_dev;
    a.lse = lse_dev;
    const cudaError_t e = launch_decode(a, d->grid[G], static_cast<cudaStream_t>(stream), nullptr);
    return e == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
}
