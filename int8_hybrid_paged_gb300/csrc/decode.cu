// decode.cu — kv4_decode_attention: prep, stream-K split attention, exact merge.
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
//   prep   block 0 plans the call: every (sequence b, KV head h) is a unit of
//          "stage items" — its INT4 pages (one 2176-byte block each) and its
//          protected run (the side-buffer groups, two page-sized blocks per 16 rows),
//          with positions for the setup of each run — and the units are laid end to
//          end in one cost line, cut into equal spans, one per warp of the split grid;
//          block 0 records where each unit's partials go. The other blocks rotate and
//          quantize every q head once (INT8 query, its scale, sum and widening offsets).
//   split  persistent, a programmatic dependent of prep; each CTA repeats the plan's
//          arithmetic for its own warps (one block-wide scan over the batch) and
//          issues its first copies before it waits for prep. Each warp walks its span
//          alone: a producer (lane 0 issues, all lanes track) keeps a 5-deep ring of
//          1-D bulk copies (global -> shared, mbarrier-completed) running across run
//          boundaries, and the consumer turns INT4 pages into integer QK / integer PV
//          on the tensor cores and protected groups into INT8 QK / BF16 PV with FP32
//          accumulation. Each run piece ends in one partial (output relative to its
//          max, max, normalizer).
//   merge  a programmatic dependent of split; warp per q head: exact log-sum-exp
//          merge of that head's partials.
// No ticket or search sits on the data path, and the spans are balanced to one run
// piece, whatever the length mix.
#include <float.h>

#include <mutex>
#include <type_traits>

#include "device_common.cuh"
#include "kv4_internal.h"

namespace kv4 {

constexpr int kWarps = kDecodeThreads / 32;
constexpr int kMaxG = 4;

// Per-warp query state of the current (b, h): INT8 rotated query of its G heads,
// s_q, Σq8 and the QK widening offsets of each dim half.
struct __align__(16) WarpQ {
    int8_t q8[kMaxG][kHeadDim];
    float scale[kMaxG];
    float qsum[kMaxG];
    float corr[kMaxG][2];     // QK widening offsets per dim half
};

// Span walker state (one per producer and consumer of a warp): the current (b, h) of
// the span and the item reached in it.
struct Walk {
    int lo, hi;
    int b, h;
    int L, n, cp, cbh, csb, slot;   // of the current b (cp: protected stage items per unit)
    int k;                      // current item of (b, h): k < n INT4 page, else protected item
    int a1;                     // end of the span's INT4 pages of (b, h)
    int g0, g1;                 // the span's protected groups of (b, h): first items in [lo, hi)
    int done;
};

// PV operands of an INT4 page pair: the u8 weights (as fp16) in the B-fragment order of
// each page's MMA (columns 4p..4p+3 of page p; the rest stay zero) and the page scales.
struct PairSmem {
    uint32_t wfrag[2][8][8];
    float ksc[2][kMaxG];
};

struct __align__(128) SplitSmem {
    uint8_t stage[kWarps][kStages][kPageBlock];   // staging ring of each warp
    WarpQ wq[kWarps];
    uint4 qfrag[kWarps][4][32];                   // QK B fragments: [k step pair][lane]
    union {
        PairSmem pair;                            // PV B operands of a page pair / side group
    } xb[kWarps];
    Walk walk[kWarps][2];                         // producer, consumer
    uint64_t bar[kWarps][kStages];
};

__device__ __forceinline__ int int4_pages(int L, int s, int w)
{
    // pages touched by the INT4 region [s, L - w)
    return (L - w > s) ? ((L - w - 1) / kPage - s / kPage + 1) : 0;
}

// Stage items of a protected unit: two page-sized blocks per 16-row side group,
// or one empty item when there is no side buffer (so every (b, h) has a unit).
__device__ __forceinline__ int prot_items(int S) { return S > 0 ? 2 * ((S + 15) >> 4) : 1; }

// Cost-line length of a (b, h) unit: its n INT4 pages, its cp protected items and the
// positions that stand for the setup of its two runs and its flush.
__device__ __forceinline__ int unit_cost(int n, int cp)
{
    return kRunSetup + kPageCost * n + kProtSetup + kProtCost * cp + kUnitFlush;
}
// Cost positions of a unit starting at base: its first INT4 page, its first protected item.
__device__ __forceinline__ int int4_start(int base) { return base + kRunSetup; }
__device__ __forceinline__ int prot_start(int base, int n) { return base + kRunSetup + kPageCost * n + kProtSetup; }

// Protected groups of a unit: ceil(S/16) groups of two stage items (a side K block and
// a side V block), or one empty item when there is no side buffer.
__device__ __forceinline__ int group_items(int cp) { return cp > 1 ? 2 : 1; }
__device__ __forceinline__ int prot_groups(int cp) { return cp > 1 ? cp >> 1 : 1; }
// Cost-line extent from the first to the last group's first item (inclusive).
__device__ __forceinline__ int prot_span_len(int cp)
{
    return kProtCost * group_items(cp) * (prot_groups(cp) - 1) + 1;
}
// Groups of a unit whose first item lies before cost position pstart + x.
__device__ __forceinline__ int groups_before(int x, int cp)
{
    const int gc = kProtCost * group_items(cp);
    return x <= 0 ? 0 : min(prot_groups(cp), (x + gc - 1) / gc);
}
// INT4 pages of a unit (of n) whose cost position lies before int4_start(base) + x.
__device__ __forceinline__ int pages_before(int x, int n)
{
    return x <= 0 ? 0 : min(n, (x + kPageCost - 1) / kPageCost);
}
// Cost-line extent from the first to the last INT4 page (inclusive), 0 for none.
__device__ __forceinline__ int int4_span_len(int n) { return n > 0 ? kPageCost * (n - 1) + 1 : 0; }

// Number of warp-span pieces of n INT4 pages whose first sits at cost position first.
__device__ __forceinline__ int n_pieces(int first, int n, int span)
{
    return n > 0 ? (first + kPageCost * (n - 1)) / span - first / span + 1 : 0;
}

// Division of non-negative 32-bit values by one divisor d >= 2 with a multiply-high:
// m = floor(2^32 (2^s - d) / d) + 1 with s = ceil(log2 d), q = (t + ((x - t) >> 1)) >> (s - 1)
// where t = mulhi(x, m) (exact for every x < 2^32).
struct SpanDiv {
    uint32_t m, s;
    __device__ explicit SpanDiv(uint32_t d)
    {
        s = 32u - (uint32_t)__clz(d - 1u);
        m = (uint32_t)((((1ull << 32) * ((1ull << s) - d)) / d) + 1ull);
    }
    __device__ __forceinline__ int operator()(int x) const
    {
        const uint32_t t = __umulhi((uint32_t)x, m);
        return (int)((t + (((uint32_t)x - t) >> 1)) >> (s - 1u));
    }
    // pieces of [base, base + n) as n_pieces
    __device__ __forceinline__ int pieces(int base, int n) const
    {
        return n > 0 ? (*this)(base + n - 1) - (*this)(base) + 1 : 0;
    }
};

// Span of each warp on a cost line of length total: a span holds at least one item
// position of any unit it lies inside (pages are kPageCost apart, protected groups
// 2 kProtCost), so every piece index is written. The plan kernel and the split kernel
// both compute it, from the same inputs.
__device__ __forceinline__ int plan_span(int total, int num_warps)
{
    return max(2 * kProtCost, (total + num_warps - 1) / num_warps);
}

// First partial of unit (b, h), laid out by the plan: per unit its INT4 pieces, then
// its protected pieces (spans holding the first item of one of its groups).
__device__ __forceinline__ int unit_first_partial(const DecodeArgs& a, int b, int h)
{
    return __ldg(&a.unit_seg[b * a.num_heads + h]);
}
// Block-wide exclusive scan (up to 1024 threads); returns the thread's offset and the total.
__device__ __forceinline__ int block_scan(int v, int* s_scan, int& total)
{
    const int nwarps = blockDim.x >> 5;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const int u = __shfl_up_sync(kFull, incl, m);
        if (lane >= m) incl += u;
    }
    if (lane == 31) s_scan[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const int x0 = lane < nwarps ? s_scan[lane] : 0;
        int x = x0;
#pragma unroll
        for (int m = 1; m < 32; m <<= 1) {
            const int u = __shfl_up_sync(kFull, x, m);
            if (lane >= m) x += u;
        }
        s_scan[lane] = x - x0;
        if (lane == 31) s_scan[32] = x;
    }
    __syncthreads();
    const int off = s_scan[warp] + incl - v;
    total = s_scan[32];
    __syncthreads();
    return off;
}

// ---------------------------------------------------------------- prep
constexpr int kPrepThreads = 256;

__global__ void __launch_bounds__(kPrepThreads) kv4_decode_prep_kernel(DecodeArgs a)
{
    // the split kernel may be scheduled now; it waits for this grid's writes itself
    grid_launch_dependents();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (blockIdx.x == 0) {
        // ---- plan: cost line, spans, piece counts
        __shared__ int s_scan[33];
        const int B = a.batch, H = a.num_heads, s = a.sink, w = a.window;
        const bool kv8 = a.kv8 != 0;
        // INT4 pages and protected stage items of sequence b's units (KV8: all of its
        // positions are protected rows of its pages)
        auto n_of = [&](int L) { return kv8 ? 0 : int4_pages(L, s, w); };
        auto cp_of = [&](int L) { return prot_items(kv8 ? L : s + w); };
        const int per = (B + kPrepThreads - 1) / kPrepThreads;
        const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
        int cost = 0;
        for (int b = b0; b < b1; ++b) {
            const int L = max(0, a.context_lens[b]);
            cost += H * unit_cost(n_of(L), cp_of(L));
        }
        int total = 0;
        int off = block_scan(cost, s_scan, total);
        const int span = plan_span(total, a.num_warps);
        const SpanDiv sd((uint32_t)span);
        int segs = 0;
        for (int b = b0; b < b1; ++b) {
            a.cost_start[b] = off;
            const int L = max(0, a.context_lens[b]);
            const int n = n_of(L), cp = cp_of(L), plen = prot_span_len(cp);
            for (int h = 0; h < H; ++h) {
                const int base = off + h * unit_cost(n, cp);
                segs += sd.pieces(int4_start(base), int4_span_len(n)) + sd.pieces(prot_start(base, n), plen);
            }
            off += H * unit_cost(n, cp);
        }
        int nseg = 0;
        int soff = block_scan(segs, s_scan, nseg);
        for (int b = b0; b < b1; ++b) {
            const int L = max(0, a.context_lens[b]);
            const int n = n_of(L), cp = cp_of(L), plen = prot_span_len(cp);
            const int cs = a.cost_start[b];
            for (int h = 0; h < H; ++h) {
                a.unit_seg[b * H + h] = soff;
                const int base = cs + h * unit_cost(n, cp);
                soff += sd.pieces(int4_start(base), int4_span_len(n)) + sd.pieces(prot_start(base, n), plen);
            }
        }
        if (tid == kPrepThreads - 1) {
            a.cost_start[B] = total;
            a.unit_seg[B * H] = nseg;
            a.plan->total_cost = total;
            a.plan->span = span;
            a.plan->total_items = nseg;
        }
        return;
    }
    // ---- query: rotate and quantize one q head per warp
    const int gw = (blockIdx.x - 1) * (kPrepThreads / 32) + warp;
    if (gw >= a.batch * a.num_q_heads) return;
    float x[4];
    load_bf16x4(a.q + (int64_t)gw * kHeadDim + 4 * lane, x);
    if (a.rope) {
        // the query of this step sits at position L - 1 of its sequence
        const int L = __ldg(&a.context_lens[gw / a.num_q_heads]);
        if (L > a.rope_max_pos) {
            if (lane == 0) report_error(a.err, KV4_DEVERR_BAD_POSITION);
        } else if (L > 0) {
            warp_rope128(x, rope_row(a.rope + (int64_t)(L - 1) * kHeadDim, lane), lane);
        }
    }
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
    // QK widening offsets: every code slot carries 1024 q, so each dim half is offset by
    // 1024 times its query sum
    int hsum = q[0] + q[1] + q[2] + q[3];
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) hsum += __shfl_xor_sync(kFull, hsum, m);
    const int qsum = hsum + __shfl_xor_sync(kFull, hsum, 16);
    const float corr = 1024.f * (float)hsum;
    const float corr_hi = __shfl_sync(kFull, corr, 16);
    const uint32_t packed = (uint32_t)(q[0] & 255) | ((uint32_t)(q[1] & 255) << 8) |
                            ((uint32_t)(q[2] & 255) << 16) | ((uint32_t)(q[3] & 255) << 24);
    uint8_t* rec = a.qinfo + (int64_t)gw * kQInfoBytes;
    *reinterpret_cast<uint32_t*>(rec + 4 * lane) = packed;
    if (lane == 0)
        *reinterpret_cast<float4*>(rec + kHeadDim) = make_float4(sq, (float)qsum, corr, corr_hi);
    if (a.dbg_q8) *reinterpret_cast<uint32_t*>(a.dbg_q8 + (int64_t)gw * kHeadDim + 4 * lane) = packed;
    if (a.dbg_qscale && lane == 0) a.dbg_qscale[gw] = sq;
}

// ---------------------------------------------------------------- tensor-core integer dots
// Integer codes enter the fp16 MMA as exact fp16 values 1024 + x, where x is a whole
// byte (a code pair or an INT8 code) or 16 times a high nibble, cut from the 32-bit
// word by one LOP3 or byte permute; the INT8 query enters as fp16 q. Every product is
// exact, every partial sum an integer below 2^24, and the accumulator is seeded with
// minus the widening offset (1024·Σq per dim half for QK, 1024·Σŵ for PV), so the
// fp32 result is the exact integer dot; row or slot differences then separate the
// two nibbles of a byte.
// QK: m16n8k16, rows = the 16 tokens of a page, 8 columns = 4 heads x 2 halves of
// the 128 dims. PV: rows = 16 dims, k = the 16 tokens of one page, 8 columns =
// 2 pages x 4 heads (pages are taken in pairs). No column is padding.

__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1, float c0, float c1,
                                        float c2, float c3)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2),
          "f"(c3));
}

// (a & b) | c in one LOP3 (lookup table 0xEA), all three operands in registers.
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// bytes 0 and 2 whole (two nibbles) as fp16 1024 + byte
__device__ __forceinline__ uint32_t wide_byte(uint32_t w) { return and_or(w, 0x00ff00ffu, 0x64006400u); }
// nibbles 1 and 5 of w as fp16 (1024 + 16 n1, 1024 + 16 n5)
__device__ __forceinline__ uint32_t wide_hi(uint32_t w)
{
    return and_or(w, 0x00F000F0u, 0x64006400u);
}

__device__ __forceinline__ uint32_t half2_bits(__half lo, __half hi)
{
    __half2 v = __halves2half2(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t half2_u32(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 u32_half2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

__device__ __forceinline__ uint32_t lds32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }

// ---------------------------------------------------------------- span walker
// Walks the stage items of one warp's span [lo, hi) of the cost line: for each
// (b, h) touched, the INT4 pages of the span's overlap, then the protected unit
// if its first item lies in the span (its owner takes all of it).

// KV8: no INT4 pages; every position is a protected row of its page, so the
// protected items of a unit follow its length.
// csb: the cost position of b's first unit (the previous sequence's plus its H units)
template <bool KV8>
__device__ __forceinline__ void walk_load_b(Walk& W, const DecodeArgs& a, int b, int cp, int csb)
{
    W.b = b;
    W.L = max(0, __ldg(&a.context_lens[b]));
    W.n = KV8 ? 0 : int4_pages(W.L, a.sink, a.window);
    W.cp = KV8 ? prot_items(W.L) : cp;
    W.cbh = unit_cost(W.n, W.cp);
    W.csb = csb;
    W.slot = __ldg(&a.slot_ids[b]);
}

// Position the walker at the first item of (b, h) inside the span; false if none.
__device__ __forceinline__ bool walk_enter(Walk& W)
{
    const int cp = W.cp;
    const int base = W.csb + W.h * W.cbh;
    const int a0 = pages_before(W.lo - int4_start(base), W.n);
    W.a1 = pages_before(W.hi - int4_start(base), W.n);
    const int pstart = prot_start(base, W.n);
    W.g0 = groups_before(W.lo - pstart, cp);
    W.g1 = groups_before(W.hi - pstart, cp);
    if (a0 < W.a1) { W.k = a0; return true; }
    if (W.g0 < W.g1) { W.k = W.n + group_items(cp) * W.g0; return true; }
    return false;
}

template <bool KV8>
__device__ __forceinline__ void walk_next_bh(Walk& W, const DecodeArgs& a, int cp)
{
    for (;;) {
        if (++W.h == a.num_heads) {
            if (W.b + 1 >= a.batch) { W.done = true; return; }
            walk_load_b<KV8>(W, a, W.b + 1, cp, W.csb + a.num_heads * W.cbh);
            W.h = 0;
        }
        if (W.csb + W.h * W.cbh >= W.hi) { W.done = true; return; }
        if (walk_enter(W)) return;
    }
}

// b, csb: the sequence whose units hold cost position lo, and its first unit's position
template <bool KV8>
__device__ __forceinline__ void walk_init(Walk& W, const DecodeArgs& a, int lo, int hi, int cp, int b, int csb)
{
    W.lo = lo;
    W.hi = hi;
    W.done = lo >= hi;
    if (W.done) return;
    walk_load_b<KV8>(W, a, b, cp, csb);
    W.h = min(a.num_heads - 1, (lo - W.csb) / W.cbh);
    if (!walk_enter(W)) walk_next_bh<KV8>(W, a, cp);
}


// ---------------------------------------------------------------- INT4 page pair
// Lane (g', t') = (lane >> 2, lane & 3) scores tokens g' and g' + 8 of each page for
// head hs = 2(t' & 1) + (t' >> 1), and accumulates output dims 16m + 2g' + {0, 1}
// (m = 0..7) of heads 2(t' & 1), 2(t' & 1) + 1 from page t' >> 1 of each pair.
//
// QK columns: column n of the B operand is head n (n < 4) or n ^ 5 (n >= 4) over the
// dim half n & 1, so lane t' < 2 holds (head hs, half 0 | head hs + 1, half 1) and its
// partner t' + 2 holds (head hs + 1, half 0 | head hs, half 1): each lane keeps its
// first column and adds its partner's second, with no select on either side.
//
// PV columns: n = 4 page + head. The u8 weights go to shared memory as packed half2
// words (token g', token g' + 8) in the B-fragment order of each page's MMA; the
// columns of the other page stay zero, so each MMA takes its operand with one load.
// Component c of a float2 (c a compile-time constant in the unrolled loops).
__device__ __forceinline__ float& fc(float2& v, int c) { return c ? v.y : v.x; }

struct Int4State {
    float2 o[8][2];      // [m][r] = (column 0, column 1) of rows r of tile m: packed FFMA2 operands
    float M, l, bias;    // running max, normalizer and offset-term share of the scored head
    float wacc;          // Σ over pages of (page scale) x Σ u8 weights, for the widening offset
};

__device__ __forceinline__ uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 lds128(const void* p) { return *reinterpret_cast<const uint4*>(p); }

// position of word w (tokens w, w + 8) inside a column's 8 B-fragment words:
// a lane reads words t' and t' + 4 with one 8-byte load
__device__ __forceinline__ int wfrag_pos(int w) { return 2 * (w & 3) + (w >> 2); }

template <int G, bool DEBUG>
__device__ __forceinline__ void int4_pair(const DecodeArgs& a, SplitSmem& sm, Int4State& st,
                                          const uint4* __restrict__ qf, float cq0, float cq1,
                                          float sqh, float qsh, const uint8_t* pg0,
                                          const uint8_t* pg1, bool two, int lp0, int r4_hi, int b,
                                          int h, int warp, int lane)
{
    const int gq = lane >> 2, tq = lane & 3;
    const int half = tq >> 1;
    const int hs = 2 * (tq & 1) + half;            // head scored by this lane
    const uint8_t* pgs[2] = {pg0, pg1};
    PairSmem& ps = sm.xb[warp].pair;

    // ---- integer QK of both pages (two independent MMA chains). A page word holds one
    // dim of tokens gq (low nibble) and gq + 8 (high nibble): rows gq take the whole byte
    // (1024 + c + 16 c'), rows gq + 8 take 1024 + 16 c'; row differences recover both dots
    uint4 kp0[2], kp1[2], mt[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        kp0[p] = lds128(pgs[p] + kKCodeOff + 16 * lane);
        kp1[p] = lds128(pgs[p] + kKCodeOff + 512 + 16 * lane);
        mt[p] = lds128(pgs[p] + kMetaOff + 16 * gq);
    }
    float d[2][4];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        d[p][0] = cq0;
        d[p][1] = cq1;
        d[p][2] = cq0;
        d[p][3] = cq1;
    }
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
        const uint4 qv = qf[32 * ii];                // B fragments of MMAs 2ii, 2ii + 1
#pragma unroll
        for (int p = 0; p < 2; ++p) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int i = 2 * ii + e;                // MMA (word) index
                const uint4& kq = i < 4 ? kp0[p] : kp1[p];
                const uint32_t wd = (i & 3) == 0 ? kq.x : (i & 3) == 1 ? kq.y : (i & 3) == 2 ? kq.z : kq.w;
                const uint32_t x = prmt(wd, 0x64646464u, 0x4341u);
                mma_f16(d[p], wide_byte(wd), wide_hi(wd), x, x & 0xfff0fff0u, e ? qv.z : qv.x,
                        e ? qv.w : qv.y, d[p][0], d[p][1], d[p][2], d[p][3]);
            }
        }
    }

    // ---- scores of head hs, tokens gq and gq + 8 of each page
    const int hi_eff = two ? r4_hi : min(r4_hi, (lp0 + 1) * kPage);
    float2 sig[2], vdl[2], vmn[2];
    bool v0[2], v1[2];
    float Mp[2];
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        // column sums: rows gq hold dot(gq) + 16 dot(gq+8), rows gq + 8 hold 16 dot(gq+8)
        const float2 own = __fadd2_rn(make_float2(d[p][0], d[p][1]), make_float2(-d[p][2], -d[p][3]));
        const float r0 = __shfl_xor_sync(kFull, own.y, 2);
        const float r1 = __shfl_xor_sync(kFull, d[p][3], 2);
        const float2 dot = __fmul2_rn(__fadd2_rn(make_float2(own.x, d[p][2]), make_float2(r0, r1)),
                                      make_float2(1.f, 0.0625f));
        const __half2 km0 = u32_half2(mt[p].x), km1 = u32_half2(mt[p].y);
        const __half2 vm0 = u32_half2(mt[p].z), vm1 = u32_half2(mt[p].w);
        vdl[p] = make_float2(__low2float(vm0), __low2float(vm1));
        vmn[p] = make_float2(__high2float(vm0), __high2float(vm1));
        const float2 kd = make_float2(__low2float(km0), __low2float(km1));
        const float2 kmin = make_float2(__high2float(km0), __high2float(km1));
        const float2 u = __ffma2_rn(kd, dot, __fmul2_rn(kmin, make_float2(qsh, qsh)));
        const float2 sg =
            __fmul2_rn(__fmul2_rn(u, make_float2(sqh, sqh)), make_float2(a.log2_scale, a.log2_scale));
        // INT4 pages start at s (a multiple of 16): a position is masked only past the
        // region's end or, for a lone page, past that page
        const int pos0 = (lp0 + p) * kPage + gq;
        v0[p] = pos0 < hi_eff;
        v1[p] = pos0 + 8 < hi_eff;
        sig[p] = make_float2(v0[p] ? sg.x : -INFINITY, v1[p] ? sg.y : -INFINITY);
        if (DEBUG && a.dbg_qk && hs < G) {
            const int64_t row = ((int64_t)b * a.num_q_heads + h * G + hs) * a.dbg_stride;
            if (v0[p] && pos0 < a.dbg_stride) a.dbg_qk[row + pos0] = (int)dot.x;
            if (v1[p] && pos0 + 8 < a.dbg_stride) a.dbg_qk[row + pos0 + 8] = (int)dot.y;
        }
        float m = fmaxf(sig[p].x, sig[p].y);
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, msk));
        Mp[p] = m;
    }

    // ---- running max of head hs and rescale factors. The first page's first position
    // lies inside the region, so Mn is finite; st.M or a masked page's -inf gives 0
    const float Mn = fmaxf(st.M, fmaxf(Mp[0], Mp[1]));
    const float alpha = exp2_fast(st.M - Mn);
    const float beta[2] = {exp2_fast(Mp[0] - Mn), exp2_fast(Mp[1] - Mn)};
    st.M = Mn;

    // ---- page-local weights, u8 with one power-of-two scale per (page, head)
    float ksc[2];
    float2 lb = make_float2(0.f, 0.f);             // (Σ β p, Σ β p · V min)
    float wsum = 0.f;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        // masked tokens give -inf - Mp (or NaN for an empty page): exp2_poly2 returns 0
        const float2 pp = exp2_poly2(__fadd2_rn(sig[p], make_float2(-Mp[p], -Mp[p])));
        const float2 wv = __fmul2_rn(pp, vdl[p]);
        float wmax = fmaxf(wv.x, wv.y);
#pragma unroll
        for (int msk = 4; msk < 32; msk <<= 1) wmax = fmaxf(wmax, __shfl_xor_sync(kFull, wmax, msk));
        const bool qz = wmax > 0x1p-64f;
        const uint32_t eb = __float_as_uint(wmax) & 0x7f800000u;       // 2^floor(log2 wmax)
        const float up = __uint_as_float(0x82800000u - eb);              // 2^(7-e)
        // rint by the 1.5·2^23 shift (round half to even), then the u8 ceiling
        const float2 sc = __fmul2_rn(wv, make_float2(up, up));
        const float2 rr = __fadd2_rn(__fadd2_rn(sc, make_float2(12582912.f, 12582912.f)),
                                     make_float2(-12582912.f, -12582912.f));
        const float wh0 = fminf(rr.x, 255.f), wh1 = fminf(rr.y, 255.f);
        const uint32_t wpk = qz ? half2_u32(__floats2half2_rn(wh0, wh1)) : 0u;
        ps.wfrag[p][4 * p + hs][wfrag_pos(gq)] = wpk;
        ksc[p] = qz ? beta[p] * __uint_as_float(eb - 0x03800000u) : 0.f;   // β·2^(e-7)
        wsum = fmaf(ksc[p], wh0 + wh1, wsum);
        if (DEBUG && a.dbg_w && hs < G) {
            const int64_t row = ((int64_t)b * a.num_q_heads + h * G + hs) * a.dbg_stride;
            const int pos0 = (lp0 + p) * kPage + gq;
            if (v0[p] && pos0 < a.dbg_stride) a.dbg_w[row + pos0] = qz ? (uint8_t)wh0 : 0;
            if (v1[p] && pos0 + 8 < a.dbg_stride) a.dbg_w[row + pos0 + 8] = qz ? (uint8_t)wh1 : 0;
        }
        const float2 bb = make_float2(beta[p], beta[p]);
        lb = __ffma2_rn(bb, make_float2(pp.x + pp.y, fmaf(pp.x, vmn[p].x, pp.y * vmn[p].y)), lb);
    }
    st.l = fmaf(st.l, alpha, lb.x);
    st.bias = fmaf(st.bias, alpha, lb.y);
    st.wacc = fmaf(st.wacc, alpha, wsum);
    if (gq == 0) {
        ps.ksc[0][hs] = ksc[0];
        ps.ksc[1][hs] = ksc[1];
    }
    // rescale of the output accumulators when a head's max moved
    if (__any_sync(kFull, alpha != 1.f)) {
        const int srcA = (lane & ~3) | (tq & 1);
        const float aA = __shfl_sync(kFull, alpha, srcA), aB = __shfl_sync(kFull, alpha, srcA | 2);
#pragma unroll
        for (int m = 0; m < 8; ++m)
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                st.o[m][r] = __fmul2_rn(st.o[m][r], make_float2(aA, aB));
            }
    }
    __syncwarp();

    // ---- integer PV of both pages; the widening offsets are removed at the flush
    const float2 kk = *reinterpret_cast<const float2*>(&ps.ksc[half][2 * (tq & 1)]);
    const uint2 bw0 = lds64(&ps.wfrag[0][gq][2 * tq]);
    const uint2 bw1 = lds64(&ps.wfrag[1][gq][2 * tq]);
    const uint4 va0 = lds128(pg0 + kVCodeOff + lane * 32);
    const uint4 va1 = lds128(pg0 + kVCodeOff + lane * 32 + 16);
    const uint4 vb0 = lds128(pg1 + kVCodeOff + lane * 32);
    const uint4 vb1 = lds128(pg1 + kVCodeOff + lane * 32 + 16);
    const uint32_t vA[8] = {va0.x, va0.y, va0.z, va0.w, va1.x, va1.y, va1.z, va1.w};
    const uint32_t vB[8] = {vb0.x, vb0.y, vb0.z, vb0.w, vb1.x, vb1.y, vb1.z, vb1.w};
    const float kA = kk.x, kB = kk.y;
    const float kAh = kA * 0.0625f, kBh = kB * 0.0625f;
#pragma unroll
    for (int m = 0; m < 8; ++m) {
        float c[4];
        // rows g' (dim 2j) take the whole byte, 1024 + lo + 16 hi; rows g' + 8 (dim 2j+1)
        // take 1024 + 16 hi; the flush removes 16 x the second from the first
        const uint32_t xa = prmt(vA[m], 0x64646464u, 0x4341u);
        const uint32_t xb = prmt(vB[m], 0x64646464u, 0x4341u);
        mma_f16(c, wide_byte(vA[m]), wide_hi(vA[m]), xa, xa & 0xfff0fff0u, bw0.x, bw0.y, 0.f, 0.f,
                0.f, 0.f);
        mma_f16(c, wide_byte(vB[m]), wide_hi(vB[m]), xb, xb & 0xfff0fff0u, bw1.x, bw1.y, c[0], c[1],
                c[2], c[3]);
        st.o[m][0] = __ffma2_rn(make_float2(kA, kB), make_float2(c[0], c[1]), st.o[m][0]);
        st.o[m][1] = __ffma2_rn(make_float2(kAh, kBh), make_float2(c[2], c[3]), st.o[m][1]);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- protected group
// One 16-row side group on the tensor cores, lane roles as on an INT4 page.
// QK: an INT8 code widens to 1024 + c, one byte permute per two codes, so the query
// B fragments and accumulator seeds of the INT4 path serve unchanged.
// PV: values dequantized to BF16 (A; rows = dims), weights p against the group's max
// rounded to BF16 (B; columns = heads, k order t, t+8, t+4, t+12 so a scoring lane's
// pair of rows is one B word), FP32 accumulation, folded into the running output.
struct ProtState {
    float2 o[8][2];    // [m][0]: dim 16m + g', [m][1]: dim 16m + g' + 8, of the lane's two columns
    float M, l;        // running max and normalizer share of head hs
};

__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1, float c0, float c1,
                                         float c2, float c3)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%10,%11,%12,%13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c0), "f"(c1), "f"(c2), "f"(c3));
}

// INT8 codes of bytes 0, 1 (resp. 2, 3) as fp16 1024 + c
__device__ __forceinline__ uint32_t w8_lo(uint32_t w) { return prmt(w, 0x64646464u, 0x4140u); }
__device__ __forceinline__ uint32_t w8_hi(uint32_t w) { return prmt(w, 0x64646464u, 0x4342u); }

__device__ __forceinline__ uint32_t bf16x2_u32(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Four side V codes of one dim (rows t, t+8, t+4, t+12) to two BF16 pairs
// bf16(fmaf(Δ, c, m)) with each row's metadata.
__device__ __forceinline__ void dequant_word(uint32_t w, float2 dA, float2 mA, float2 dB, float2 mB,
                                             uint32_t& lo, uint32_t& hi)
{
    const float k = 8388608.0f;                      // 2^23: float bits 0x4b0000cc = 2^23 + c
    const float x0 = __uint_as_float(prmt(w, 0x4b000000u, 0x7440u));
    const float x1 = __uint_as_float(prmt(w, 0x4b000000u, 0x7441u));
    const float x2 = __uint_as_float(prmt(w, 0x4b000000u, 0x7442u));
    const float x3 = __uint_as_float(prmt(w, 0x4b000000u, 0x7443u));
    const float2 c01 = __fadd2_rn(make_float2(x0, x1), make_float2(-k, -k));
    const float2 c23 = __fadd2_rn(make_float2(x2, x3), make_float2(-k, -k));
    const float2 v01 = __ffma2_rn(dA, c01, mA);
    const float2 v23 = __ffma2_rn(dB, c23, mB);
    lo = bf16x2_u32(v01.x, v01.y);
    hi = bf16x2_u32(v23.x, v23.y);
}

// Position held by side row rr at context length L, or -1 if the row is not in
// the protected set [0, min(s, L)) ∪ [max(s, L - w), L).
__device__ __forceinline__ int side_row_position(int rr, int s, int w, int L)
{
    if (rr < s) return rr < L ? rr : -1;
    if (rr >= s + w || L <= 0) return -1;
    const int k = rr - s;
    const int d = ((L - 1 - k) % w + w) % w;        // the latest position p < L with p mod w = k
    const int p = L - 1 - d;
    return p >= s ? p : -1;
}

// Running-max step of a 16-row group: lane (g', t') holds the scores of rows g', g' + 8
// for head hs. The weights p = 2^(score - group max) go, rounded to BF16, to the PV B tile
// (column hs, k order t, t+8, t+4, t+12); the running output and normalizer are rescaled
// to the new running max. Returns the group's fold factors 2^(group max - running max)
// of the two heads whose output this lane accumulates.
// F16W (NVFP4): the weights carry their row's value scale, p·wsc·inv with inv = 2^-k
// for the power of two 2^k just above the group's largest value scale, and go in fp16;
// the fold factors carry up = 2^k. No weight exceeds 1; the normalizer still sums the
// plain p.
template <bool F16W>
__device__ __forceinline__ float2 group_weights(ProtState& st, PairSmem& ps, float2 sig, int lane,
                                                float2 wsc, float inv, float up, uint32_t& wbits)
{
    const int gq = lane >> 2, tq = lane & 3;
    const int hs = 2 * (tq & 1) + (tq >> 1);
    float m = fmaxf(sig.x, sig.y);
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, msk));
    // weights against the group's own max (so their BF16 rounding does not depend on
    // which groups share a piece), folded in by 2^(group max - running max)
    const float Mn = fmaxf(st.M, m);
    const bool none = (Mn == -INFINITY);
    const float alpha = none ? 1.f : exp2_fast(st.M - Mn);
    const float beta = none ? 0.f : exp2_fast(m - Mn);
    st.M = Mn;
    // masked rows give -inf - m (NaN for an empty group): exp2_poly2 returns 0
    const float2 pp = exp2_poly2(__fadd2_rn(sig, make_float2(-m, -m)));
    st.l = fmaf(st.l, alpha, beta * (pp.x + pp.y));
    float fold = beta;
    if (F16W) {
        const float2 wn = __fmul2_rn(__fmul2_rn(pp, wsc), make_float2(inv, inv));
        wbits = half2_u32(__floats2half2_rn(wn.x, wn.y));
        fold = beta * up;
    } else {
        wbits = bf16x2_u32(pp.x, pp.y);
    }
    ps.wfrag[0][hs][wfrag_pos(gq)] = wbits;
    const int srcA = (lane & ~3) | (tq & 1);
    const float bA = __shfl_sync(kFull, fold, srcA), bB = __shfl_sync(kFull, fold, srcA | 2);
    if (__any_sync(kFull, alpha != 1.f)) {
        const float aA = __shfl_sync(kFull, alpha, srcA), aB = __shfl_sync(kFull, alpha, srcA | 2);
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
            st.o[mm][0] = __fmul2_rn(st.o[mm][0], make_float2(aA, aB));
            st.o[mm][1] = __fmul2_rn(st.o[mm][1], make_float2(aA, aB));
        }
    }
    __syncwarp();
    return make_float2(bA, bB);
}

// Running-max step of a side group of the hybrid cache. A ring group whose residues the
// window start cuts holds positions of two pages, the window's oldest and its newest;
// each page's weights are formed against that page's own max. inA/inB say which of the
// two column sets each of the lane's rows gq, gq + 8 belongs to (neither: a masked row);
// each set holds the rows of one page. Set A's weights go to columns hs of the PV B
// tile, set B's to columns 4 + hs (zero when the group holds one page). Lanes t' < 2
// then accumulate set A's product and lanes t' >= 2 set B's, each with its page's fold
// factors 2^(page max - running max), returned here; the two halves are added at the
// end of the piece. wA, wB: the BF16 weight pairs written.
__device__ __forceinline__ float2 group_weights_pages(ProtState& st, PairSmem& ps, float2 sig, bool inA0,
                                                      bool inA1, bool inB0, bool inB1, int lane,
                                                      uint32_t& wA, uint32_t& wB)
{
    const int gq = lane >> 2, tq = lane & 3;
    const int hs = 2 * (tq & 1) + (tq >> 1);
    // both pages' maxima in one reduction chain
    float mA = fmaxf(inA0 ? sig.x : -INFINITY, inA1 ? sig.y : -INFINITY);
    float mB = fmaxf(inB0 ? sig.x : -INFINITY, inB1 ? sig.y : -INFINITY);
#pragma unroll
    for (int msk = 4; msk < 32; msk <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(kFull, mA, msk));
        mB = fmaxf(mB, __shfl_xor_sync(kFull, mB, msk));
    }
    const float Mn = fmaxf(st.M, fmaxf(mA, mB));
    const bool none = (Mn == -INFINITY);
    const float alpha = none ? 1.f : exp2_fast(st.M - Mn);
    const float betaA = none ? 0.f : exp2_fast(mA - Mn);     // exp2(-inf) = 0 for a missing page
    const float betaB = none ? 0.f : exp2_fast(mB - Mn);
    st.M = Mn;
    // each row against its own page's max; rows of neither page (masked, -inf) give 0
    const float2 pp = exp2_poly2(__fadd2_rn(sig, make_float2(inA0 ? -mA : -mB, inA1 ? -mA : -mB)));
    st.l = fmaf(st.l, alpha, fmaf(inA0 ? betaA : betaB, pp.x, (inA1 ? betaA : betaB) * pp.y));
    wA = bf16x2_u32(inA0 ? pp.x : 0.f, inA1 ? pp.y : 0.f);
    wB = bf16x2_u32(inB0 ? pp.x : 0.f, inB1 ? pp.y : 0.f);
    ps.wfrag[0][hs][wfrag_pos(gq)] = wA;
    ps.wfrag[0][4 + hs][wfrag_pos(gq)] = wB;
    // fold factors: every lane of a scoring column holds its head's betaA and betaB after
    // the reduction, so even rows publish betaA and odd rows betaB; lanes t' < 2 (set A)
    // read an even row, lanes t' >= 2 (set B) an odd one
    const float pub = (gq & 1) ? betaB : betaA;
    const int src = ((lane & ~7) | ((tq >> 1) << 2)) | (tq & 1);
    const float f0 = __shfl_sync(kFull, pub, src), f1 = __shfl_sync(kFull, pub, src | 2);
    if (__any_sync(kFull, alpha != 1.f)) {
        const int srcA = (lane & ~3) | (tq & 1);
        const float aA = __shfl_sync(kFull, alpha, srcA), aB = __shfl_sync(kFull, alpha, srcA | 2);
#pragma unroll
        for (int mm = 0; mm < 8; ++mm) {
            st.o[mm][0] = __fmul2_rn(st.o[mm][0], make_float2(aA, aB));
            st.o[mm][1] = __fmul2_rn(st.o[mm][1], make_float2(aA, aB));
        }
    }
    __syncwarp();
    return make_float2(f0, f1);
}

// BF16 PV of one side group (values dequantized with each row's metadata, weights
// from the B tile in shared memory), FP32 accumulation into the running output with
// this lane's fold factors.
__device__ __forceinline__ void prot_pv(ProtState& st, const PairSmem& ps, const uint8_t* pv, float2 fold,
                                        int lane)
{
    const int gq = lane >> 2, tq = lane & 3;
    const float bA = fold.x, bB = fold.y;
    const uint2 bw = lds64(&ps.wfrag[0][gq][2 * tq]);
    const uint4 vmw = lds128(pv + (kSideVMetaOff - kPageBlock) + 16 * tq);
    const __half2 vt0 = u32_half2(vmw.x), vt8 = u32_half2(vmw.y);
    const __half2 vt4 = u32_half2(vmw.z), vt12 = u32_half2(vmw.w);
    const float2 dA = make_float2(__low2float(vt0), __low2float(vt8));
    const float2 mA = make_float2(__high2float(vt0), __high2float(vt8));
    const float2 dB = make_float2(__low2float(vt4), __low2float(vt12));
    const float2 mB = make_float2(__high2float(vt4), __high2float(vt12));
    uint4 vq[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) vq[i] = lds128(pv + (kSideVCodeOff - kPageBlock) + 16 * (32 * i + lane));
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) {
        const uint4 q4 = vq[mm >> 1];
        const uint32_t w0 = (mm & 1) ? q4.z : q4.x;      // dim 16 mm + gq
        const uint32_t w1 = (mm & 1) ? q4.w : q4.y;      // dim 16 mm + gq + 8
        uint32_t a0, a1, a2, a3;
        dequant_word(w0, dA, mA, dB, mB, a0, a2);
        dequant_word(w1, dA, mA, dB, mB, a1, a3);
        float c[4];
        mma_bf16(c, a0, a1, a2, a3, bw.x, bw.y, 0.f, 0.f, 0.f, 0.f);
        st.o[mm][0] = __ffma2_rn(make_float2(bA, bB), make_float2(c[0], c[1]), st.o[mm][0]);
        st.o[mm][1] = __ffma2_rn(make_float2(bA, bB), make_float2(c[2], c[3]), st.o[mm][1]);
    }
    __syncwarp();
}

// Debug record of a lane's two rows: the bits of each row's weight (one half of wbits).
__device__ __forceinline__ void record_weights(const DecodeArgs& a, int b, int hq, int pos0, int pos1,
                                               uint32_t w0bits, uint32_t w1bits)
{
    const int64_t row = ((int64_t)b * a.num_q_heads + hq) * a.dbg_stride;
    if (pos0 >= 0 && pos0 < a.dbg_stride) a.dbg_p[row + pos0] = (uint16_t)(w0bits & 0xffffu);
    if (pos1 >= 0 && pos1 < a.dbg_stride) a.dbg_p[row + pos1] = (uint16_t)(w1bits >> 16);
}

template <int G, bool DEBUG, bool KV8>
__device__ __forceinline__ void prot_group(const DecodeArgs& a, SplitSmem& sm, ProtState& st,
                                           const uint4* __restrict__ qf, float cq0, float cq1,
                                           float sqh, float qsh, const uint8_t* pk,
                                           const uint8_t* pv, int grp, int L, int b, int h,
                                           int warp, int lane)
{
    const int gq = lane >> 2, tq = lane & 3, half = tq >> 1;
    const int hs = 2 * (tq & 1) + half;
    PairSmem& ps = sm.xb[warp].pair;

    // ---- INT8 QK of rows gq, gq + 8 (two planes of four words per row and lane)
    const uint4 k00 = lds128(pk + kSideKCodeOff + 64 * gq + 16 * tq);
    const uint4 k01 = lds128(pk + kSideKCodeOff + 1024 + 64 * gq + 16 * tq);
    const uint4 k10 = lds128(pk + kSideKCodeOff + 64 * (gq + 8) + 16 * tq);
    const uint4 k11 = lds128(pk + kSideKCodeOff + 1024 + 64 * (gq + 8) + 16 * tq);
    const uint32_t wa[8] = {k00.x, k00.y, k00.z, k00.w, k01.x, k01.y, k01.z, k01.w};
    const uint32_t wb[8] = {k10.x, k10.y, k10.z, k10.w, k11.x, k11.y, k11.z, k11.w};
    float d[4] = {cq0, cq1, cq0, cq1};
#pragma unroll
    for (int ii = 0; ii < 4; ++ii) {
        const uint4 qv = qf[32 * ii];
        mma_f16(d, w8_lo(wa[2 * ii]), w8_lo(wb[2 * ii]), w8_hi(wa[2 * ii]), w8_hi(wb[2 * ii]), qv.x,
                qv.y, d[0], d[1], d[2], d[3]);
        mma_f16(d, w8_lo(wa[2 * ii + 1]), w8_lo(wb[2 * ii + 1]), w8_hi(wa[2 * ii + 1]),
                w8_hi(wb[2 * ii + 1]), qv.z, qv.w, d[0], d[1], d[2], d[3]);
    }
    const float r0 = __shfl_xor_sync(kFull, d[1], 2);
    const float r1 = __shfl_xor_sync(kFull, d[3], 2);
    const float2 dot = __fadd2_rn(make_float2(d[0], d[2]), make_float2(r0, r1));
    const uint2 kmw = lds64(pk + kSideKMetaOff + 8 * gq);
    const __half2 km0 = u32_half2(kmw.x), km1 = u32_half2(kmw.y);
    const float2 kd = make_float2(__low2float(km0), __low2float(km1));
    const float2 kmin = make_float2(__high2float(km0), __high2float(km1));
    const float2 u = __ffma2_rn(kd, dot, __fmul2_rn(kmin, make_float2(qsh, qsh)));
    const float2 sg =
        __fmul2_rn(__fmul2_rn(u, make_float2(sqh, sqh)), make_float2(a.log2_scale, a.log2_scale));
    // rows of a side group hold the positions of the ring/sink rule; rows of a KV8
    // page hold its 16 consecutive positions
    const int pos0 = KV8 ? (16 * grp + gq < L ? 16 * grp + gq : -1)
                         : side_row_position(16 * grp + gq, a.sink, a.window, L);
    const int pos1 = KV8 ? (16 * grp + gq + 8 < L ? 16 * grp + gq + 8 : -1)
                         : side_row_position(16 * grp + gq + 8, a.sink, a.window, L);
    const float2 sig = make_float2(pos0 >= 0 ? sg.x : -INFINITY, pos1 >= 0 ? sg.y : -INFINITY);
    if (DEBUG && a.dbg_qk && hs < G) {
        const int64_t row = ((int64_t)b * a.num_q_heads + h * G + hs) * a.dbg_stride;
        if (pos0 >= 0 && pos0 < a.dbg_stride) a.dbg_qk[row + pos0] = (int)dot.x;
        if (pos1 >= 0 && pos1 < a.dbg_stride) a.dbg_qk[row + pos1] = (int)dot.y;
    }

    if (KV8) {
        // ---- a KV8 group is one page: weights against its max, BF16 PV
        uint32_t wbits;
        const float2 fold = group_weights<false>(st, ps, sig, lane, make_float2(0.f, 0.f), 0.f, 0.f, wbits);
        if (DEBUG && a.dbg_p && hs < G) record_weights(a, b, h * G + hs, pos0, pos1, wbits, wbits);
        prot_pv(st, ps, pv, fold, lane);
        return;
    }
    // ---- hybrid side group: weights per page of the positions its rows hold, against
    // each page's own max. With s and w multiples of the page size (the host enforces it)
    // all protected positions of a page sit in one side group, and a group holds at most
    // two pages: a sink page, a whole window page, or the window's oldest and newest
    // partial pages when the window start cuts a page (ring rows share residues mod w).
    // Rows of the newest page (positions from ns = 16 floor((L - 1) / 16)) go to the
    // second column set, every other row to the first, which separates the two pages of
    // any group. (Taking the two-set step for every group measured faster than branching
    // to the one-page step for groups that hold one page.)
    const int ns = (L - 1) & ~(kPage - 1);
    uint32_t wA, wB;
    const float2 fold = group_weights_pages(st, ps, sig, pos0 >= 0 && pos0 < ns, pos1 >= 0 && pos1 < ns,
                                            pos0 >= ns, pos1 >= ns, lane, wA, wB);
    if (DEBUG && a.dbg_p && hs < G)
        record_weights(a, b, h * G + hs, pos0, pos1, pos0 < ns ? wA : wB, pos1 < ns ? wA : wB);
    prot_pv(st, ps, pv, fold, lane);
}

// ---------------------------------------------------------------- NVFP4 page
// One page of the NVFP4 format (16 positions of one KV head), lane roles as in a
// protected group; the K and V halves arrive in two stage slots.
// QK: per 16-dim block one fp16 MMA of the E2M1 codes (A: rows = positions) with the
// INT8 query (B: even columns 2t' hold head [0, 2, 1, 3][t'], odd columns are zero), so
// lane t' finds its head's block dots of rows g', g' + 8 in c0, c2. The dots are exact
// (halves times integers, sums below 2^14); they enter an FP32 fma chain over the
// blocks with the E4M3 block scales, then the vector scale g, s_q and C. The block
// scales are widened to FP32 once per page into scratch space past the K half in its
// stage slot (the bulk copy never writes there).
// PV: fp16 MMA of the E2M1 values (A: rows = dims, exact) with weights that carry the
// value scales, p·g / 2^k (from group_weights; 2^k just above the page's largest g)
// times the E4M3 scale of the block: the B tile of block m is one packed multiply per
// register. The FP32 results fold into the running output with 2^k.
__device__ __forceinline__ void e2m1x4_f16x2(uint32_t w, uint32_t (&o)[4])
{
    // byte k of w holds two E2M1 codes; its low nibble becomes the low half of o[k]
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\tmov.b32 {c0, c1, c2, c3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, c0;\n\tcvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, c2;\n\tcvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
        : "=r"(o[0]), "=r"(o[1]), "=r"(o[2]), "=r"(o[3])
        : "r"(w));
}
// four E4M3 bytes to two fp16 pairs (bytes 0, 1 -> lo; 2, 3 -> hi); every E4M3 value is
// exact in fp16
__device__ __forceinline__ void e4m3x4_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi)
{
    asm("{\n\t.reg .b16 p0, p1;\n\tmov.b32 {p0, p1}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, p0;\n\tcvt.rn.f16x2.e4m3x2 %1, p1;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b)
{
    return half2_u32(__hmul2(u32_half2(a), u32_half2(b)));
}

template <int G, bool DEBUG>
__device__ __forceinline__ void fp4_group(const DecodeArgs& a, SplitSmem& sm, ProtState& st,
                                          const uint4* __restrict__ qf, float sqh, uint8_t* pk,
                                          const uint8_t* pv, int grp, int L, int b, int h, int warp,
                                          int lane)
{
    const int gq = lane >> 2, tq = lane & 3;
    const int hs = 2 * (tq & 1) + (tq >> 1);
    PairSmem& ps = sm.xb[warp].pair;
    uint8_t* ksc = pk + kFp4Half;
    const int pos0 = 16 * grp + gq < L ? 16 * grp + gq : -1;
    const int pos1 = 16 * grp + gq + 8 < L ? 16 * grp + gq + 8 : -1;

    // ---- the PV weights' power of two 2^k, just above the largest V vector scale of the
    // page's positions: g >= 0 orders as its bits; the biased exponent e gives
    // g in [2^(e-127), 2^(e-126)), so k = e - 126 (e <= 243: g <= FLT_MAX / 2688)
    const float2 vg = *reinterpret_cast<const float2*>(pv + kFp4GlobalOff + 8 * gq);
    const uint32_t gb = __reduce_max_sync(
        kFull, max(pos0 >= 0 ? __float_as_uint(vg.x) : 0u, pos1 >= 0 ? __float_as_uint(vg.y) : 0u));
    const uint32_t ge = (gb >> 23) & 255u;
    const float pinv = __uint_as_float((253u - ge) << 23), pup = __uint_as_float((ge + 1u) << 23);

    // ---- K block scales to FP32: lane l widens blocks 2c, 2c + 1 (c = l >> 3) of positions
    // t, t + 8 (t = l & 7), stored as (s of t, of t + 8) pairs in 16-byte chunk c ^ ((t >> 1) & 3)
    // of row t, so that every load and store below is conflict-free
    {
        const int t = lane & 7, c = lane >> 3;
        uint32_t lo, hi;
        e4m3x4_f16x2(lds32(pk + kFp4ScaleOff + 16 * t + 4 * c), lo, hi);
        const float2 f0 = __half22float2(u32_half2(lo)), f1 = __half22float2(u32_half2(hi));
        *reinterpret_cast<float4*>(ksc + 64 * t + 16 * (c ^ ((t >> 1) & 3))) = make_float4(f0.x, f0.y, f1.x, f1.y);
    }
    __syncwarp();

    // ---- QK: block dots of rows gq, gq + 8 and the fma chain over the blocks
    const uint4 kc0 = lds128(pk + 16 * lane);            // blocks 0..3
    const uint4 kc1 = lds128(pk + 512 + 16 * lane);      // blocks 4..7
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // (s_b of rows gq, gq + 8) for blocks 2i, 2i + 1
        const float4 sp = *reinterpret_cast<const float4*>(ksc + 64 * gq + 16 * (i ^ ((gq >> 1) & 3)));
        const uint4 qv = qf[32 * i];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int bb = 2 * i + e;
            const uint4 kc = bb < 4 ? kc0 : kc1;
            const uint32_t wd = (bb & 3) == 0 ? kc.x : (bb & 3) == 1 ? kc.y : (bb & 3) == 2 ? kc.z : kc.w;
            uint32_t A[4];
            e2m1x4_f16x2(wd, A);
            float d[4];
            mma_f16(d, A[0], A[1], A[2], A[3], e ? qv.z : qv.x, e ? qv.w : qv.y, 0.f, 0.f, 0.f, 0.f);
            acc = __ffma2_rn(e ? make_float2(sp.z, sp.w) : make_float2(sp.x, sp.y), make_float2(d[0], d[2]), acc);
        }
    }
    const float2 kg = *reinterpret_cast<const float2*>(pk + kFp4GlobalOff + 8 * gq);
    const float2 sg = __fmul2_rn(__fmul2_rn(__fmul2_rn(acc, kg), make_float2(sqh, sqh)),
                                 make_float2(a.log2_scale, a.log2_scale));
    const float2 sig = make_float2(pos0 >= 0 ? sg.x : -INFINITY, pos1 >= 0 ? sg.y : -INFINITY);
    if (DEBUG && a.dbg_qk && hs < G) {
        // no single integer dot here: the record holds the score's FP32 bits
        const int64_t row = ((int64_t)b * a.num_q_heads + h * G + hs) * a.dbg_stride;
        if (pos0 >= 0 && pos0 < a.dbg_stride) a.dbg_qk[row + pos0] = __float_as_int(sg.x);
        if (pos1 >= 0 && pos1 < a.dbg_stride) a.dbg_qk[row + pos1] = __float_as_int(sg.y);
    }

    uint32_t wbits;
    const float2 bAB = group_weights<true>(st, ps, sig, lane, vg, pinv, pup, wbits);
    if (DEBUG && a.dbg_p && hs < G) record_weights(a, b, h * G + hs, pos0, pos1, wbits, wbits);
    const float bA = bAB.x, bB = bAB.y;

    // ---- fp16 PV, FP32 accumulation into the running output
    const uint2 pw = lds64(&ps.wfrag[0][gq][2 * tq]);    // weights of tokens (tq, tq+8), (tq+4, tq+12)
    const uint4 vc0 = lds128(pv + 16 * lane);            // blocks 0..3
    const uint4 vc1 = lds128(pv + 512 + 16 * lane);      // blocks 4..7
    const uint4 vs0 = lds128(pv + kFp4ScaleOff + 32 * tq);        // E4M3 scales, blocks 0..3
    const uint4 vs1 = lds128(pv + kFp4ScaleOff + 32 * tq + 16);   // blocks 4..7
#pragma unroll
    for (int mm = 0; mm < 8; ++mm) {
        const uint4 vc = mm < 4 ? vc0 : vc1;
        const uint4 vs = mm < 4 ? vs0 : vs1;
        const uint32_t wd = (mm & 3) == 0 ? vc.x : (mm & 3) == 1 ? vc.y : (mm & 3) == 2 ? vc.z : vc.w;
        const uint32_t sw = (mm & 3) == 0 ? vs.x : (mm & 3) == 1 ? vs.y : (mm & 3) == 2 ? vs.z : vs.w;
        uint32_t hv[4];                                  // the A fragment: (dim d | d + 8) x tokens
        e2m1x4_f16x2(wd, hv);                            // (t, t+8), (t+4, t+12)
        uint32_t s01, s23;                               // block scales of tokens (t, t+8), (t+4, t+12)
        e4m3x4_f16x2(sw, s01, s23);
        float c[4];
        mma_f16(c, hv[0], hv[1], hv[2], hv[3], hmul2_u32(pw.x, s01), hmul2_u32(pw.y, s23), 0.f, 0.f, 0.f, 0.f);
        // scalar fmas here: the packed form measured slower in this routine
        fc(st.o[mm][0], 0) = fmaf(bA, c[0], fc(st.o[mm][0], 0));
        fc(st.o[mm][0], 1) = fmaf(bB, c[1], fc(st.o[mm][0], 1));
        fc(st.o[mm][1], 0) = fmaf(bA, c[2], fc(st.o[mm][1], 0));
        fc(st.o[mm][1], 1) = fmaf(bB, c[3], fc(st.o[mm][1], 1));
    }
    __syncwarp();
}

// ---------------------------------------------------------------- MXFP4 page
// One page of the MXFP4 format, lane roles and fragment orders as in an NVFP4 page. QK:
// the two fp16 MMAs of a 32-value block chain their accumulators (the block dot stays
// exact, below 2^24) and the fma chain runs over the four blocks with their powers of two.
// PV: the weights are fp16(p) from group_weights, times 2^(s_b - k) per block and token
// (one packed fp16 multiply per register), 2^k the page's largest block scale; the fold
// factor carries 2^k.
__device__ __forceinline__ float e8m0_f32(uint32_t e)
{
    return e ? __uint_as_float(e << 23) : __uint_as_float(0x00400000u);     // 2^(e - 127)
}
// 2^(e - emax) for a biased exponent e <= emax, as a float that rounds to fp16 (0 below
// 2^-24 after rounding: 2^-25 is a tie to the even 0). A masked position's stale scale may
// exceed emax; it gets 0, like its weight.
__device__ __forceinline__ float pow2_rel(uint32_t e, uint32_t emax)
{
    const int j = (int)e - (int)emax;
    return (j <= 0 && j >= -126) ? __uint_as_float((uint32_t)(j + 127) << 23) : 0.f;
}
__device__ __forceinline__ uint32_t pow2_pair_f16(uint32_t e0, uint32_t e1, uint32_t emax)
{
    return half2_u32(__floats2half2_rn(pow2_rel(e0, emax), pow2_rel(e1, emax)));
}

template <int G, bool DEBUG>
__device__ __forceinline__ void mx_group(const DecodeArgs& a, SplitSmem& sm, ProtState& st,
                                         const uint4* __restrict__ qf, float sqh, const uint8_t* pk,
                                         const uint8_t* pv, int grp, int L, int b, int h, int warp,
                                         int lane)
{
    const int gq = lane >> 2, tq = lane & 3;
    const int hs = 2 * (tq & 1) + (tq >> 1);
    PairSmem& ps = sm.xb[warp].pair;
    const int pos0 = 16 * grp + gq < L ? 16 * grp + gq : -1;
    const int pos1 = 16 * grp + gq + 8 < L ? 16 * grp + gq + 8 : -1;

    // ---- V block scales of tokens tq, tq+8, tq+4, tq+12 (bytes 0..3 of word b) and the
    // page's largest one over its valid positions
    const uint4 vs = lds128(pv + kMxScaleOff + 16 * tq);
    const int p0 = 16 * grp + tq;
    const uint32_t vmask = (p0 < L ? 0xffu : 0u) | (p0 + 8 < L ? 0xff00u : 0u) |
                           (p0 + 4 < L ? 0xff0000u : 0u) | (p0 + 12 < L ? 0xff000000u : 0u);
    uint32_t m4 = __vmaxu4(__vmaxu4(vs.x & vmask, vs.y & vmask), __vmaxu4(vs.z & vmask, vs.w & vmask));
    m4 = max(max(m4 & 0xffu, (m4 >> 8) & 0xffu), max((m4 >> 16) & 0xffu, m4 >> 24));
    const uint32_t emax = __reduce_max_sync(kFull, m4);

    // ---- QK: the four 32-value block dots of rows gq, gq + 8 and the fma chain
    const uint2 ks = lds64(pk + kMxScaleOff + 8 * gq);   // (t, t+8) of blocks 0, 1 | 2, 3
    const uint4 kc0 = lds128(pk + 16 * lane);            // 16-value blocks 0..3
    const uint4 kc1 = lds128(pk + 512 + 16 * lane);      // 16-value blocks 4..7
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < 4; ++i) {                        // 32-value block i = 16-value blocks 2i, 2i+1
        const uint4 qv = qf[32 * i];
        const uint4 kc = i < 2 ? kc0 : kc1;
        const uint32_t w0 = (i & 1) ? kc.z : kc.x, w1 = (i & 1) ? kc.w : kc.y;
        uint32_t A0[4], A1[4];
        e2m1x4_f16x2(w0, A0);
        e2m1x4_f16x2(w1, A1);
        float d[4];
        mma_f16(d, A0[0], A0[1], A0[2], A0[3], qv.x, qv.y, 0.f, 0.f, 0.f, 0.f);
        mma_f16(d, A1[0], A1[1], A1[2], A1[3], qv.z, qv.w, d[0], d[1], d[2], d[3]);
        const uint32_t sw = (i < 2) ? ks.x : ks.y;
        const uint32_t e0 = (sw >> (16 * (i & 1))) & 0xffu, e1 = (sw >> (16 * (i & 1) + 8)) & 0xffu;
        acc = __ffma2_rn(make_float2(e8m0_f32(e0), e8m0_f32(e1)), make_float2(d[0], d[2]), acc);
    }
    const float2 sg = __fmul2_rn(__fmul2_rn(acc, make_float2(sqh, sqh)), make_float2(a.log2_scale, a.log2_scale));
    const float2 sig = make_float2(pos0 >= 0 ? sg.x : -INFINITY, pos1 >= 0 ? sg.y : -INFINITY);
    if (DEBUG && a.dbg_qk && hs < G) {
        // no single integer dot here: the record holds the score's FP32 bits
        const int64_t row = ((int64_t)b * a.num_q_heads + h * G + hs) * a.dbg_stride;
        if (pos0 >= 0 && pos0 < a.dbg_stride) a.dbg_qk[row + pos0] = __float_as_int(sg.x);
        if (pos1 >= 0 && pos1 < a.dbg_stride) a.dbg_qk[row + pos1] = __float_as_int(sg.y);
    }

    uint32_t wbits;
    const float2 bAB = group_weights<true>(st, ps, sig, lane, make_float2(1.f, 1.f), 1.f, e8m0_f32(emax), wbits);
    if (DEBUG && a.dbg_p && hs < G) record_weights(a, b, h * G + hs, pos0, pos1, wbits, wbits);
    const float bA = bAB.x, bB = bAB.y;

    // ---- fp16 PV, FP32 accumulation into the running output
    const uint2 pw = lds64(&ps.wfrag[0][gq][2 * tq]);    // fp16(p) of tokens (tq, tq+8), (tq+4, tq+12)
    const uint4 vc0 = lds128(pv + 16 * lane);
    const uint4 vc1 = lds128(pv + 512 + 16 * lane);
#pragma unroll
    for (int bb = 0; bb < 4; ++bb) {
        const uint32_t sw = bb == 0 ? vs.x : bb == 1 ? vs.y : bb == 2 ? vs.z : vs.w;
        const uint32_t b0 = hmul2_u32(pw.x, pow2_pair_f16(sw & 0xffu, (sw >> 8) & 0xffu, emax));
        const uint32_t b1 = hmul2_u32(pw.y, pow2_pair_f16((sw >> 16) & 0xffu, sw >> 24, emax));
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int mm = 2 * bb + e;
            const uint4 vc = mm < 4 ? vc0 : vc1;
            const uint32_t wd = (mm & 3) == 0 ? vc.x : (mm & 3) == 1 ? vc.y : (mm & 3) == 2 ? vc.z : vc.w;
            uint32_t hv[4];
            e2m1x4_f16x2(wd, hv);                        // the A fragment, as in an NVFP4 page
            float c[4];
            mma_f16(c, hv[0], hv[1], hv[2], hv[3], b0, b1, 0.f, 0.f, 0.f, 0.f);
            // scalar fmas here: the packed form measured slower in this routine
            fc(st.o[mm][0], 0) = fmaf(bA, c[0], fc(st.o[mm][0], 0));
            fc(st.o[mm][0], 1) = fmaf(bB, c[1], fc(st.o[mm][0], 1));
            fc(st.o[mm][1], 0) = fmaf(bA, c[2], fc(st.o[mm][1], 0));
            fc(st.o[mm][1], 1) = fmaf(bB, c[3], fc(st.o[mm][1], 1));
        }
    }
    __syncwarp();
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------- split kernel
// The two walkers of a warp (producer, consumer) live in shared memory and are
// read and written only where a run begins or ends, so the page loop keeps
// nothing of them in registers.
__device__ __forceinline__ Walk walk_load(const volatile Walk& s)
{
    Walk w;
    w.lo = s.lo; w.hi = s.hi; w.b = s.b; w.h = s.h; w.L = s.L; w.n = s.n; w.cp = s.cp; w.cbh = s.cbh;
    w.csb = s.csb; w.slot = s.slot; w.k = s.k; w.a1 = s.a1; w.g0 = s.g0; w.g1 = s.g1; w.done = s.done;
    return w;
}

__device__ __forceinline__ void walk_store(volatile Walk& d, const Walk& w)
{
    d.lo = w.lo; d.hi = w.hi; d.b = w.b; d.h = w.h; d.L = w.L; d.n = w.n; d.cp = w.cp; d.cbh = w.cbh;
    d.csb = w.csb; d.slot = w.slot; d.k = w.k; d.a1 = w.a1; d.g0 = w.g0; d.g1 = w.g1; d.done = w.done;
}

// FMT: 0 the method's format (INT4 pages + side groups), 1 the 8-bit format, 2 NVFP4,
// 3 MXFP4; the last three walk every page as one group.
template <int G, bool DEBUG, int FMT>
__global__ void __launch_bounds__(kDecodeThreads, 1) kv4_decode_split_kernel(DecodeArgs a)
{
    constexpr bool KV8 = FMT != 0, FP4 = FMT == 2, MX = FMT == 3;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    SplitSmem& sm = *reinterpret_cast<SplitSmem*>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int ww = 0; ww < kWarps; ++ww)
            for (int k = 0; k < kStages; ++k) mbar_init(&sm.bar[ww][k], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int H = a.num_heads, s = a.sink, w = a.window, S = s + w;
    const int cp = prot_items(S);
    // whole-cache formats: a page block and each of its two stage items (K half, V half)
    constexpr int kBlock8 = FP4 ? kPageBlock4f : MX ? kPageBlockMx : kPageBlock8;
    constexpr int kItem8 = FP4 ? kFp4Half : MX ? kMxHalf : kPageBlock;
    const int wg = blockIdx.x * kWarps + warp;
    volatile Walk& Psm = sm.walk[warp][0];
    volatile Walk& Csm = sm.walk[warp][1];
    // ---- this CTA's share of the plan, from the call's inputs alone, so that it and the
    // first bulk copies run before the dependency wait, alongside the plan kernel: the
    // cost line's length (one block-wide scan over the batch, the plan kernel's
    // arithmetic) and, for each of the CTA's warps, the sequence whose units hold the
    // start of its span (left in the warp's consumer walker slot)
    int span, total;
    {
        int* s_scan = reinterpret_cast<int*>(&sm.wq[0]);    // free until the first query load
        const int B = a.batch;
        const int per = (B + kDecodeThreads - 1) / kDecodeThreads;
        const int b0 = min(B, tid * per), b1 = min(B, b0 + per);
        auto unit_of = [&](int L) {
            return KV8 ? unit_cost(0, prot_items(L)) : unit_cost(int4_pages(L, s, w), cp);
        };
        int cost = 0;
        for (int b = b0; b < b1; ++b) cost += H * unit_of(max(0, __ldg(&a.context_lens[b])));
        int off = block_scan(cost, s_scan, total);
        span = plan_span(total, a.num_warps);
        const int wg0 = blockIdx.x * kWarps;
        for (int b = b0; b < b1; ++b) {
            const int end = off + H * unit_of(max(0, __ldg(&a.context_lens[b])));
            const int first = max(wg0, (off + span - 1) / span), last = min(wg0 + kWarps, (end + span - 1) / span);
            for (int wgi = first; wgi < last; ++wgi) {
                sm.walk[wgi - wg0][1].b = b;
                sm.walk[wgi - wg0][1].csb = off;
            }
            off = end;
        }
        __syncthreads();
        const int lo = min(total, wg * span), hi = min(total, lo + span);
        const int b_lo = Csm.b, csb_lo = Csm.csb;
        __syncwarp();
        Walk W;
        walk_init<KV8>(W, a, lo, hi, cp, b_lo, csb_lo);
        if (lane == 0) {
            walk_store(Psm, W);
            walk_store(Csm, W);
        }
        __syncwarp();
    }
    const int p_first = s / kPage;
    int prod = 0, cons = 0;                 // items issued / consumed
    int pst = 0, cst = 0;                   // stage of the next item to issue / consume
    uint32_t cph = 0;                       // parity awaited on stage cst (flips as cst wraps)
    bool aborted = false;
    const uint32_t stage0 = smem_u32(&sm.stage[warp][0][0]);
    const uint32_t bar0 = smem_u32(&sm.bar[warp][0]);
    const uint32_t is_l0 = lane == 0;

    // Producer: walks the span run by run; within a run the items are consecutive
    // pages (block-table window of 32 entries, one load per lane) or consecutive
    // side blocks. All lanes track it; lane 0 issues (predicated, no branch).
    int r_kind = -1;                        // 0 INT4 pages, 1 side blocks, 2 empty item; -1 none
    int r_i = 0, r_end = 0, win_lo = 0, win = 0, r_b = 0;
    const uint8_t* r_src = nullptr;
    auto next_run = [&]() -> bool {
        Walk P = walk_load(Psm);
        if (r_kind >= 0) {                  // leave the run that just ended
            if (r_kind == 0 && P.g0 < P.g1) P.k = P.n + group_items(P.cp) * P.g0;
            else walk_next_bh<KV8>(P, a, cp);
        }
        bool more = !P.done;
        if (more) {
            if (P.k < P.n) {
                r_kind = 0;
                r_i = P.k;
                r_end = P.a1;
                r_b = P.b;
                r_src = a.pages + (int64_t)P.h * kPageBlock;
                win_lo = -64;               // force a window load
            } else if (KV8) {
                // the unit's pages, two stage items (K block, V block) each
                r_kind = P.L > 0 ? 3 : 2;
                r_i = P.k;
                r_end = group_items(P.cp) * P.g1;
                r_b = P.b;
                r_src = a.pages + (int64_t)P.h * kBlock8;
                win_lo = -64;               // force a window load
            } else {
                r_kind = S > 0 ? 1 : 2;
                r_i = P.k - P.n;
                r_end = group_items(P.cp) * P.g1;
                const int slot = (P.slot >= 0 && P.slot < a.max_slots) ? P.slot : 0;
                r_src = a.side + ((int64_t)slot * H + P.h) * a.side_block_bytes;
            }
        } else {
            r_kind = -1;
        }
        __syncwarp();
        if (lane == 0) walk_store(Psm, P);
        __syncwarp();
        return more;
    };
    const int64_t page_stride = (int64_t)H * kPageBlock;
    const int64_t page_stride8 = (int64_t)H * kBlock8;
    auto produce = [&]() {
        // common case: two more pages of the current INT4 run, both inside the
        // block-table window, and two free stages
        if (r_kind == 0 && prod + 2 <= cons + kStages && r_i + 2 <= r_end) {
            const int o0 = p_first + r_i - win_lo;
            if ((unsigned)o0 < 31u) {
                const int pg0 = __shfl_sync(kFull, win, o0);
                const int pg1 = __shfl_sync(kFull, win, o0 + 1);
                const int p1 = (pst + 1 == kStages) ? 0 : pst + 1;
                issue_bulk(stage0 + (uint32_t)(kPageBlock * pst), r_src + (int64_t)pg0 * page_stride,
                           kPageBlock, bar0 + 8u * pst, is_l0);
                issue_bulk(stage0 + (uint32_t)(kPageBlock * p1), r_src + (int64_t)pg1 * page_stride,
                           kPageBlock, bar0 + 8u * p1, is_l0);
                r_i += 2;
                prod += 2;
                pst = (p1 + 1 == kStages) ? 0 : p1 + 1;
                return;
            }
        }
        // whole-cache formats: the next two items of the run (page halves), their pages'
        // entries inside the block-table window, two free stages
        if (KV8 && r_kind == 3 && prod + 2 <= cons + kStages && r_i + 2 <= r_end) {
            const int o0 = (r_i >> 1) - win_lo, o1 = ((r_i + 1) >> 1) - win_lo;
            if ((unsigned)o0 < 32u && (unsigned)o1 < 32u) {
                const int h0 = (r_i & 1) * kItem8, h1 = kItem8 - h0;
                const uint8_t* src0 = r_src + (int64_t)__shfl_sync(kFull, win, o0) * page_stride8 + h0;
                const uint8_t* src1 = r_src + (int64_t)__shfl_sync(kFull, win, o1) * page_stride8 + h1;
                const int p1 = (pst + 1 == kStages) ? 0 : pst + 1;
                issue_bulk(stage0 + (uint32_t)(kPageBlock * pst), src0, kItem8, bar0 + 8u * pst, is_l0);
                issue_bulk(stage0 + (uint32_t)(kPageBlock * p1), src1, kItem8, bar0 + 8u * p1, is_l0);
                r_i += 2;
                prod += 2;
                pst = (p1 + 1 == kStages) ? 0 : p1 + 1;
                return;
            }
        }
#pragma unroll 1
        while (prod < cons + kStages) {
            if (r_i >= r_end) {
                if (!next_run()) break;
            }
            const uint32_t bar = bar0 + 8u * pst;
            const uint32_t dst = stage0 + (uint32_t)(kPageBlock * pst);
            if (r_kind == 0) {
                const int lp = p_first + r_i;
                if ((unsigned)(lp - win_lo) >= 32u) {
                    win_lo = lp;
                    const int e = lp + lane;
                    int pg = -1;
                    if (e < a.stride) pg = __ldg(&a.block_table[(int64_t)r_b * a.stride + e]);
                    // entries past the sequence's pages are never issued; report the rest
                    if (e < p_first + r_end && (e >= a.stride || pg < 0 || (int64_t)pg >= a.num_pages)) {
                        report_error(a.err, e >= a.stride ? KV4_DEVERR_BAD_POSITION : KV4_DEVERR_BAD_PAGE);
                        pg = 0;
                    }
                    win = pg;
                }
                const int page = __shfl_sync(kFull, win, lp - win_lo);
                issue_bulk(dst, r_src + (int64_t)page * page_stride, kPageBlock, bar, is_l0);
            } else if (r_kind == 1) {
                issue_bulk(dst, r_src + (int64_t)r_i * kPageBlock, kPageBlock, bar, is_l0);
            } else if (KV8 && r_kind == 3) {
                const int lp = r_i >> 1;
                if ((unsigned)(lp - win_lo) >= 32u) {
                    win_lo = lp;
                    const int e = lp + lane;
                    int pg = -1;
                    if (e < a.stride) pg = __ldg(&a.block_table[(int64_t)r_b * a.stride + e]);
                    // entries past the unit's pages are never issued; report the rest
                    if (e < (r_end >> 1) && (e >= a.stride || pg < 0 || (int64_t)pg >= a.num_pages)) {
                        report_error(a.err, e >= a.stride ? KV4_DEVERR_BAD_POSITION : KV4_DEVERR_BAD_PAGE);
                        pg = 0;
                    }
                    win = pg;
                }
                const int page = __shfl_sync(kFull, win, lp - win_lo);
                issue_bulk(dst, r_src + (int64_t)page * page_stride8 + (r_i & 1) * kItem8, kItem8, bar,
                           is_l0);
            } else {
                arrive_pred(bar, is_l0);    // empty protected item: no side buffer
            }
            ++r_i;
            ++prod;
            pst = (pst + 1 == kStages) ? 0 : pst + 1;
        }
    };
    // consume the next item: wait for its stage, advance the consumer position
    auto wait_next = [&]() -> int {
        const int stg = cst;
        if (!aborted) {
            const uint32_t bar = bar0 + 8u * stg;
            if (!mbar_try_wait_at(bar, cph) && !mbar_wait_slow(bar, cph)) {
                if (lane == 0) report_error(a.err, KV4_DEVERR_WAIT_TIMEOUT);
                aborted = true;
            }
        }
        if (++cst == kStages) {
            cst = 0;
            cph ^= 1u;
        }
        ++cons;
        return stg;
    };

    produce();
    // launched as a programmatic dependent of the prep kernel: everything above ran
    // alongside its tail; the query records and the partials' layout are read only
    // past this wait
    grid_dependency_wait();
    grid_launch_dependents();
    int q_b = -1, q_h = -1;
    const int gq = lane >> 2, tq = lane & 3, half = tq >> 1;
    while (!aborted) {
        int b, h, k, n, a1, L, slot, g0, g1;
        {
            const Walk C = walk_load(Csm);
            if (C.done) break;
            b = C.b; h = C.h; k = C.k; n = C.n; a1 = C.a1; L = C.L; slot = C.slot; g0 = C.g0; g1 = C.g1;
        }
        // ---- query state of (b, h) into this warp's shared memory
        if (b != q_b || h != q_h) {
            __syncwarp();
            const uint8_t* rec = a.qinfo + ((int64_t)b * a.num_q_heads + h * G) * kQInfoBytes;
            if (lane < G * 8) {
                const int g = lane >> 3, part = lane & 7;
                *reinterpret_cast<uint4*>(&sm.wq[warp].q8[g][part * 16]) =
                    __ldg(reinterpret_cast<const uint4*>(rec + g * kQInfoBytes + part * 16));
            }
            if (lane < G) {
                const float4 f = __ldg(reinterpret_cast<const float4*>(rec + lane * kQInfoBytes + kHeadDim));
                sm.wq[warp].scale[lane] = f.x;
                sm.wq[warp].qsum[lane] = f.y;
                sm.wq[warp].corr[lane][0] = f.z;
                sm.wq[warp].corr[lane][1] = f.w;
            }
            __syncwarp();
            if (FP4 || MX) {
                // NVFP4 / MXFP4 QK B fragments: even column g' is head [0, 2, 1, 3][g' / 2], odd
                // columns are zero; block bb takes k rows 2t', 2t'+1, 2t'+8, 2t'+9 as dims
                // 16bb + 2t' + {0, 1, 8, 9}. Slot ii holds blocks 2ii, 2ii + 1.
                const int bh = 2 * ((gq >> 1) & 1) + (gq >> 2);
                const bool bok = !(gq & 1) && bh < G;
                const int8_t* qq = sm.wq[warp].q8[bok ? bh : 0];
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    uint32_t f[4];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int base = 16 * (2 * ii + e) + 2 * tq;
                        f[2 * e] = bok ? half2_bits(__int2half_rn(qq[base]), __int2half_rn(qq[base + 1])) : 0u;
                        f[2 * e + 1] = bok ? half2_bits(__int2half_rn(qq[base + 8]), __int2half_rn(qq[base + 9])) : 0u;
                    }
                    sm.qfrag[warp][ii][lane] = make_uint4(f[0], f[1], f[2], f[3]);
                }
            } else {
                // QK B fragments. Column g' = head(g') over dim half g' & 1 with
                // head(n) = n < 4 ? n : n ^ 5; k rows 2t', 2t'+1, 2t'+8, 2t'+9 come from code
                // lane t', whose dims lie in half t' >> 1. Lane (g', t') keeps its column's
                // fragments.
                const int bh = gq < 4 ? gq : (gq ^ 5);
                const bool bok = (half == (gq & 1)) && (bh < G);
                const int8_t* qq = sm.wq[warp].q8[bok ? bh : 0];
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    uint32_t f[4];
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        // MMA i = 2ii + e: k rows 2t', 2t'+1 are dims 4i, 4i+1 of chunk t',
                        // k rows 2t'+8, 2t'+9 are dims 4i+2, 4i+3
                        const int base = 32 * tq + 4 * (2 * ii + e);
                        f[2 * e] = bok ? half2_bits(__int2half_rn(qq[base]), __int2half_rn(qq[base + 1])) : 0u;
                        f[2 * e + 1] = bok ? half2_bits(__int2half_rn(qq[base + 2]), __int2half_rn(qq[base + 3])) : 0u;
                    }
                    sm.qfrag[warp][ii][lane] = make_uint4(f[0], f[1], f[2], f[3]);
                }
            }
            __syncwarp();
            q_b = b;
            q_h = h;
        }
        const WarpQ& wq = sm.wq[warp];
        const int hs = 2 * (tq & 1) + half;
        const float sqh = hs < G ? wq.scale[hs] : 0.f;
        const float qsh = hs < G ? wq.qsum[hs] : 0.f;
        const uint4* qf = &sm.qfrag[warp][0][lane];
        // the weight tiles' unused columns must read zero; the other run kind shares them
        reinterpret_cast<uint4*>(&sm.xb[warp].pair.wfrag[0][0][0])[lane] = make_uint4(0u, 0u, 0u, 0u);
        __syncwarp();

        if (!KV8 && k < n) {
            // ---- INT4 run: pages k .. a1-1 of (b, h)
            // accumulator seeds: minus the widening offsets of (head hs, half 0) and
            // (head hs ^ 1, half 1), the two columns this lane's C fragment covers
            const float cq0 = hs < G ? -wq.corr[hs][0] : 0.f;
            const float cq1 = (hs ^ 1) < G ? -wq.corr[hs ^ 1][1] : 0.f;
            Int4State st;
#pragma unroll
            for (int m = 0; m < 8; ++m)
#pragma unroll
                for (int r = 0; r < 2; ++r) st.o[m][r] = make_float2(0.f, 0.f);
            st.M = -INFINITY;
            st.l = 0.f;
            st.bias = 0.f;
            st.wacc = 0.f;
            const int r4_hi = L - w;
#pragma unroll 1
            for (int j = k; j < a1; j += 2) {
                const bool two = j + 1 < a1;
                const int s0 = wait_next();
                const int s1 = two ? wait_next() : s0;
                const int lp0 = p_first + j;
                const uint8_t* pg0 = sm.stage[warp][s0];
                const uint8_t* pg1 = sm.stage[warp][s1];
                int4_pair<G, DEBUG>(a, sm, st, qf, cq0, cq1, sqh, qsh, pg0, pg1, two, lp0, r4_hi, b, h,
                                    warp, lane);
                produce();
            }
            // ---- partial of this piece: normalizer, offset terms and weight sums over the
            // 8 lanes that scored a head, handed to the PV lanes; output halves (pages of a
            // pair) over lanes t' and t' ^ 2
#pragma unroll
            for (int msk = 4; msk < 32; msk <<= 1) {
                st.l += __shfl_xor_sync(kFull, st.l, msk);
                st.bias += __shfl_xor_sync(kFull, st.bias, msk);
                st.wacc += __shfl_xor_sync(kFull, st.wacc, msk);
            }
            const int srcA = (lane & ~3) | (tq & 1);
            const float biasA = __shfl_sync(kFull, st.bias, srcA);
            const float biasB = __shfl_sync(kFull, st.bias, srcA | 2);
            const float waccA = __shfl_sync(kFull, st.wacc, srcA);
            const float waccB = __shfl_sync(kFull, st.wacc, srcA | 2);
            // rows r = 1 (dim 2j+1) carry (1024 + 16 code)/16: remove 64 x the scaled weight
            // sums; rows r = 0 (dim 2j) carry 1024 + code(2j) + 16 code(2j+1): remove 16 x
            // the raw r = 1 value, which takes the offset and the other nibble with it
            const float offA1 = biasA - 64.f * waccA, offB1 = biasB - 64.f * waccB;
#pragma unroll
            for (int m = 0; m < 8; ++m) {
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const float lo = fc(st.o[m][0], c) + __shfl_xor_sync(kFull, fc(st.o[m][0], c), 2);
                    const float hi = fc(st.o[m][1], c) + __shfl_xor_sync(kFull, fc(st.o[m][1], c), 2);
                    fc(st.o[m][0], c) = fmaf(-16.f, hi, lo) + (c ? biasB : biasA);
                    fc(st.o[m][1], c) = hi + (c ? offB1 : offA1);
                }
            }
            Walk C = walk_load(Csm);
            const int base = C.csb + h * C.cbh;
            const int idx = unit_first_partial(a, b, h) + (wg - int4_start(base) / span);
            if (tq < 2) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hd = 2 * (tq & 1) + j;
                    if (hd >= G) continue;
                    float* po = a.part_o + ((int64_t)idx * G + hd) * kHeadDim;
#pragma unroll
                    for (int m = 0; m < 8; ++m)
                        *reinterpret_cast<float2*>(po + 16 * m + 2 * gq) =
                            make_float2(fc(st.o[m][0], j), fc(st.o[m][1], j));
                }
            }
            if (gq == 0 && hs < G) a.part_ml[(int64_t)idx * G + hs] = make_float2(st.M, st.l);
            if (C.g0 < C.g1) C.k = C.n + group_items(C.cp) * C.g0;
            else walk_next_bh<KV8>(C, a, cp);
            __syncwarp();
            if (lane == 0) walk_store(Csm, C);
            __syncwarp();
        } else {
            // ---- protected unit of (b, h), owned by this span
            ProtState st;
#pragma unroll
            for (int mm = 0; mm < 8; ++mm)
#pragma unroll
                for (int r = 0; r < 2; ++r) st.o[mm][r] = make_float2(0.f, 0.f);
            st.M = -INFINITY;
            st.l = 0.f;
            const float cq0 = hs < G ? -wq.corr[hs][0] : 0.f;
            const float cq1 = (hs ^ 1) < G ? -wq.corr[hs ^ 1][1] : 0.f;
            const bool slot_ok = slot >= 0 && slot < a.max_slots;
            const int Lp = slot_ok ? L : 0;
            if (lane == 0) {
                if (!slot_ok) report_error(a.err, KV4_DEVERR_BAD_SLOT);
                else if (L != __ldg(&a.seq_len[slot])) report_error(a.err, KV4_DEVERR_LEN_MISMATCH);
            }
            if (KV8 ? L > 0 : S > 0) {
#pragma unroll 1
                for (int grp = g0; grp < g1; ++grp) {
                    const int s0 = wait_next();
                    const int s1 = wait_next();
                    if (FP4)
                        fp4_group<G, DEBUG>(a, sm, st, qf, sqh, sm.stage[warp][s0], sm.stage[warp][s1],
                                            grp, Lp, b, h, warp, lane);
                    else if (MX)
                        mx_group<G, DEBUG>(a, sm, st, qf, sqh, sm.stage[warp][s0], sm.stage[warp][s1],
                                           grp, Lp, b, h, warp, lane);
                    else
                        prot_group<G, DEBUG, KV8>(a, sm, st, qf, cq0, cq1, sqh, qsh, sm.stage[warp][s0],
                                                  sm.stage[warp][s1], grp, Lp, b, h, warp, lane);
                    produce();
                }
            } else {
                wait_next();
                produce();
            }
#pragma unroll
            for (int msk = 4; msk < 32; msk <<= 1) st.l += __shfl_xor_sync(kFull, st.l, msk);
            if (!KV8) {
                // lanes t' >= 2 hold the products of the second column set: add them in
#pragma unroll
                for (int mm = 0; mm < 8; ++mm)
#pragma unroll
                    for (int r = 0; r < 2; ++r) {
                        st.o[mm][r].x += __shfl_xor_sync(kFull, st.o[mm][r].x, 2);
                        st.o[mm][r].y += __shfl_xor_sync(kFull, st.o[mm][r].y, 2);
                    }
            }
            int pidx;
            {
                const Walk C = walk_load(Csm);
                const int base = C.csb + h * C.cbh;
                pidx = unit_first_partial(a, b, h) +
                       n_pieces(int4_start(base), C.n, span) + (wg - prot_start(base, C.n) / span);
            }
            float* po = a.part_o + ((int64_t)pidx * G) * kHeadDim;
            if (tq < 2) {
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int hd = 2 * tq + j;
                    if (hd >= G) continue;
#pragma unroll
                    for (int mm = 0; mm < 8; ++mm) {
                        po[hd * kHeadDim + 16 * mm + gq] = fc(st.o[mm][0], j);
                        po[hd * kHeadDim + 16 * mm + gq + 8] = fc(st.o[mm][1], j);
                    }
                }
            }
            if (gq == 0 && hs < G) a.part_ml[(int64_t)pidx * G + hs] = make_float2(st.M, st.l);
            Walk C = walk_load(Csm);
            walk_next_bh<KV8>(C, a, cp);
            __syncwarp();
            if (lane == 0) walk_store(Csm, C);
            __syncwarp();
        }
    }
}

// ---------------------------------------------------------------- merge
// Exact log-sum-exp merge, one warp per q head, over the partials (INT4 pieces and
// protected pieces) of its (b, h). Lane k loads the (max, normalizer) of item k;
// every lane then loads its four dims of four items at once, so the merge costs a
// few load round trips whatever the number of pieces.
template <int G>
__global__ void __launch_bounds__(128) kv4_decode_merge_kernel(DecodeArgs a)
{
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * 4 + (threadIdx.x >> 5);
    const bool live = gw < a.batch * a.num_q_heads;
    const int b = gw / a.num_q_heads, hq = gw - b * a.num_q_heads;
    const int h = hq / G, g = hq - h * G;
    // a unit's partials are consecutive: its count is the next unit's first minus its own.
    // The plan kernel wrote these before the split kernel began, so they are read before
    // the wait for the split kernel's partials.
    const int u = b * a.num_heads + h;
    const int first = live ? __ldg(&a.unit_seg[u]) : 0;
    const int nit = live ? __ldg(&a.unit_seg[u + 1]) - first : 0;
    grid_dependency_wait();                 // the split kernel's partials are complete past here
    if (!live) return;
    auto item = [&](int k) { return first + k; };
    auto pout = [&](int it) {
        return __ldg(reinterpret_cast<const float4*>(&a.part_o[((int64_t)it * G + g) * kHeadDim + 4 * lane]));
    };
    if (nit <= 32) {
        // one round for the (max, normalizer) of every item and the first four outputs
        float2 ml = make_float2(-INFINITY, 0.f);
        if (lane < nit) ml = __ldg(&a.part_ml[(int64_t)item(lane) * G + g]);
        float4 v[4];
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) v[kk] = pout(item(min(kk, nit - 1)));   // weight 0 past the last
        const float Mx = warp_max(ml.x);
        float den = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Mx != -INFINITY) {
            const float f = (ml.x != -INFINITY) ? exp2f(ml.x - Mx) : 0.f;
            den = warp_sum(f * ml.y);
            for (int c0 = 0; c0 < nit; c0 += 4) {
                if (c0 > 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) v[kk] = pout(item(min(c0 + kk, nit - 1)));
                }
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const float fk = __shfl_sync(kFull, f, (c0 + kk) & 31);
                    o.x = fmaf(fk, v[kk].x, o.x);
                    o.y = fmaf(fk, v[kk].y, o.y);
                    o.z = fmaf(fk, v[kk].z, o.z);
                    o.w = fmaf(fk, v[kk].w, o.w);
                }
            }
        }
        float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
        if (den > 0.f) {
            const float r = 1.f / den;
            res = make_float4(o.x * r, o.y * r, o.z * r, o.w * r);
        }
        *reinterpret_cast<float4*>(&a.out[((int64_t)b * a.num_q_heads + hq) * kHeadDim + 4 * lane]) = res;
        if (a.lse && lane == 0)
            a.lse[(int64_t)b * a.num_q_heads + hq] =
                (den > 0.f) ? (Mx + log2f(den)) * 0.69314718055994531f : -INFINITY;
        return;
    }
    float Mx = -INFINITY;
    for (int c0 = 0; c0 < nit; c0 += 32)
        if (c0 + lane < nit) Mx = fmaxf(Mx, __ldg(&a.part_ml[(int64_t)item(c0 + lane) * G + g].x));
    Mx = warp_max(Mx);
    float den = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (Mx != -INFINITY) {
        for (int c0 = 0; c0 < nit; c0 += 4) {
            float f = 0.f;
            if (lane < 4 && c0 + lane < nit) {
                const float2 ml = __ldg(&a.part_ml[(int64_t)item(c0 + lane) * G + g]);
                if (ml.x != -INFINITY) {
                    f = exp2f(ml.x - Mx);
                    den = fmaf(f, ml.y, den);
                }
            }
            float4 v[4];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const int it = item(min(c0 + kk, nit - 1));      // weight 0 past the last item
                v[kk] = __ldg(reinterpret_cast<const float4*>(
                    &a.part_o[((int64_t)it * G + g) * kHeadDim + 4 * lane]));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float fk = __shfl_sync(kFull, f, kk);
                o.x = fmaf(fk, v[kk].x, o.x);
                o.y = fmaf(fk, v[kk].y, o.y);
                o.z = fmaf(fk, v[kk].z, o.z);
                o.w = fmaf(fk, v[kk].w, o.w);
            }
        }
        den = warp_sum(den);
    }
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (den > 0.f) {
        const float r = 1.f / den;
        res = make_float4(o.x * r, o.y * r, o.z * r, o.w * r);
    }
    *reinterpret_cast<float4*>(&a.out[((int64_t)b * a.num_q_heads + hq) * kHeadDim + 4 * lane]) = res;
    if (a.lse && lane == 0)
        a.lse[(int64_t)b * a.num_q_heads + hq] =
            (den > 0.f) ? (Mx + log2f(den)) * 0.69314718055994531f : -INFINITY;
}

// ---------------------------------------------------------------- launchers
// Launch k(a) on the stream; dependent = programmatic dependent launch (the kernel
// may start while the previous one drains and waits for its writes on the device).
static cudaError_t launch_k(void (*k)(DecodeArgs), int grid, int block, size_t smem,
                            cudaStream_t stream, const DecodeArgs& a, bool dependent)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = dependent ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, a);
}

template <int G, bool DEBUG, int FMT>
static cudaError_t launch_g(const DecodeArgs& a, int grid, cudaStream_t stream, cudaEvent_t* ev)
{
    // with profiling events between the kernels each one runs alone, so the events
    // time it; otherwise split and merge are programmatic dependents of their predecessor
    const bool dep = ev == nullptr;
    if (ev) cudaEventRecord(ev[0], stream);
    const int prep_blocks = 1 + (a.batch * a.num_q_heads + kPrepThreads / 32 - 1) / (kPrepThreads / 32);
    cudaError_t e = launch_k(kv4_decode_prep_kernel, prep_blocks, kPrepThreads, 0, stream, a, false);
    if (ev) cudaEventRecord(ev[1], stream);
    if (e == cudaSuccess)
        e = launch_k(kv4_decode_split_kernel<G, DEBUG, FMT>, grid, kDecodeThreads, sizeof(SplitSmem),
                     stream, a, dep);
    if (ev) cudaEventRecord(ev[2], stream);
    const int warps = a.batch * a.num_q_heads;
    if (e == cudaSuccess)
        e = launch_k(kv4_decode_merge_kernel<G>, (warps + 3) / 4, 128, 0, stream, a, dep);
    if (ev) cudaEventRecord(ev[3], stream);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_decode(const DecodeArgs& a, int grid, cudaStream_t stream, cudaEvent_t* ev)
{
    const bool dbg = a.dbg_q8 || a.dbg_qscale || a.dbg_qk || a.dbg_w || a.dbg_p;
    const int fmt = a.mx ? 3 : a.fp4 ? 2 : a.kv8 ? 1 : 0;
    const int sel = 2 * fmt + (dbg ? 1 : 0);
    auto go = [&](auto g) -> cudaError_t {
        constexpr int Gc = decltype(g)::value;
        switch (sel) {
        case 0: return launch_g<Gc, false, 0>(a, grid, stream, ev);
        case 1: return launch_g<Gc, true, 0>(a, grid, stream, ev);
        case 2: return launch_g<Gc, false, 1>(a, grid, stream, ev);
        case 3: return launch_g<Gc, true, 1>(a, grid, stream, ev);
        case 4: return launch_g<Gc, false, 2>(a, grid, stream, ev);
        case 5: return launch_g<Gc, true, 2>(a, grid, stream, ev);
        case 6: return launch_g<Gc, false, 3>(a, grid, stream, ev);
        default: return launch_g<Gc, true, 3>(a, grid, stream, ev);
        }
    };
    switch (a.group) {
    case 1: return go(std::integral_constant<int, 1>{});
    case 2: return go(std::integral_constant<int, 2>{});
    case 4: return go(std::integral_constant<int, 4>{});
    default: return cudaErrorInvalidValue;
    }
}

// Opt every split-kernel instantiation in to its dynamic shared memory (above the
// 48 KB default) on the current device, then report resident CTAs per SM.
template <int G>
static cudaError_t split_setup(int* ctas)
{
    const int smem = (int)sizeof(SplitSmem);
    cudaError_t e = cudaSuccess;
    for (auto k : {kv4_decode_split_kernel<G, false, 0>, kv4_decode_split_kernel<G, true, 0>,
                   kv4_decode_split_kernel<G, false, 1>, kv4_decode_split_kernel<G, true, 1>,
                   kv4_decode_split_kernel<G, false, 2>, kv4_decode_split_kernel<G, true, 2>,
                   kv4_decode_split_kernel<G, false, 3>, kv4_decode_split_kernel<G, true, 3>})
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas, kv4_decode_split_kernel<G, false, 0>,
                                                         kDecodeThreads, smem);
}

cudaError_t decode_ctas_per_sm(int group, int* ctas)
{
    switch (group) {
    case 1: return split_setup<1>(ctas);
    case 2: return split_setup<2>(ctas);
    case 4: return split_setup<4>(ctas);
    default: return cudaErrorInvalidValue;
    }
}

size_t decode_workspace_bytes(int batch, int num_q_heads, int num_kv_heads, int group, int grid,
                              DecodeWorkspace* ws, unsigned char* base)
{
    // plan header | cost_start[B+1] | unit_seg[B*H+1] | query records | partial (M, l) |
    // partial o
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t items = (size_t)2 * batch * num_kv_heads + (size_t)grid * kWarps;
    size_t off = 0;
    const size_t o_plan = off;  off = up(off + sizeof(PlanHeader));
    const size_t o_cost = off;  off = up(off + sizeof(int32_t) * (batch + 1));
    const size_t o_seg = off;   off = up(off + sizeof(int32_t) * ((size_t)batch * num_kv_heads + 1));
    const size_t o_q = off;     off = up(off + (size_t)kQInfoBytes * batch * num_q_heads);
    const size_t o_ml = off;    off = up(off + sizeof(float2) * items * group);
    const size_t o_o = off;     off = up(off + sizeof(float) * items * group * kHeadDim);
    if (ws && base) {
        ws->plan = reinterpret_cast<PlanHeader*>(base + o_plan);
        ws->cost_start = reinterpret_cast<int32_t*>(base + o_cost);
        ws->unit_seg = reinterpret_cast<int32_t*>(base + o_seg);
        ws->qinfo = base + o_q;
        ws->part_ml = reinterpret_cast<float2*>(base + o_ml);
        ws->part_o = reinterpret_cast<float*>(base + o_o);
    }
    return off;
}

}  // namespace kv4

// ---------------------------------------------------------------- decode without allocation
// A variant of kv4_decode_attention for callers that cannot make device
// allocations: its workspace (plan, query records, partial outputs) lives in the
// file-scope array below instead of a cache-owned buffer, and it reads
// caller-provided pools, so nothing is allocated by anyone for the call. The
// array is reserved on every GPU that loads this library, until the process
// exits. In host code its name is only a host-side stand-in; the kernels get its
// device address, looked up once per device with that device current.
namespace kv4 {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kNoAllocMaxBatch = 4096;

static __device__ __align__(256) unsigned char g_kv4_noalloc_scratch[kNoAllocScratchBytes];
// Device error word of the allocation-free decode (first error wins, 0 = none), the
// counterpart of a cache's error word: index errors and staging-wait timeouts of its
// kernels land here.
static __device__ int32_t g_kv4_noalloc_err;

}  // namespace kv4

namespace {

constexpr int kNoAllocMaxDevices = 64;

struct NoAllocDevice {
    std::once_flag once;
    unsigned char* scratch = nullptr;   // device address of g_kv4_noalloc_scratch
    int32_t* err = nullptr;             // device address of g_kv4_noalloc_err
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
        d->status = cudaGetSymbolAddress(&p, kv4::g_kv4_noalloc_err);
        if (d->status != cudaSuccess) return;
        d->err = static_cast<int32_t*>(p);
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
    if (cfg->format < KV4_FORMAT_INT4_HYBRID || cfg->format > KV4_FORMAT_MXFP4)
        return KV4_ERR_INVALID_ARG;
    const bool kv8 = cfg->format != KV4_FORMAT_INT4_HYBRID;
    if (kv8 && (cfg->sink != 0 || cfg->window != 0)) return KV4_ERR_INVALID_ARG;
    if (cfg->sink % KV4_PAGE_SIZE != 0 || cfg->window % KV4_PAGE_SIZE != 0) return KV4_ERR_UNSUPPORTED;
    if (batch == 0) return KV4_OK;
    if (!page_pool_dev || (!side_pool_dev && !kv8) || !seq_len_dev || !q_bf16_dev || !slot_ids_dev ||
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
    if (batch > kNoAllocMaxBatch) return KV4_ERR_OUT_OF_RANGE;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return KV4_ERR_CUDA;
    NoAllocDevice* d = noalloc_device(dev);
    if (!d) return KV4_ERR_UNSUPPORTED;
    if (d->status != cudaSuccess || !d->scratch || !d->err) return KV4_ERR_CUDA;
    // a call whose workspace would not fit in the array is refused before anything runs
    if (decode_workspace_bytes(batch, num_q_heads, H, G, d->grid[G], nullptr, nullptr) >
        kNoAllocScratchBytes)
        return KV4_ERR_OUT_OF_RANGE;

    DecodeWorkspace ws{};
    decode_workspace_bytes(batch, num_q_heads, H, G, d->grid[G], &ws, d->scratch);
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
    a.side_block_bytes = (int64_t)((cfg->sink + cfg->window + 15) / 16) * kSideGroupBytes;
    a.seq_len = seq_len_dev;
    a.err = d->err;
    a.plan = ws.plan;
    a.cost_start = ws.cost_start;
    a.unit_seg = ws.unit_seg;
    a.qinfo = ws.qinfo;
    a.part_o = ws.part_o;
    a.part_ml = ws.part_ml;
    a.num_warps = d->grid[G] * (kDecodeThreads / 32);
    a.out = out_dev;
    a.lse = lse_dev;
    a.kv8 = kv8;
    a.fp4 = cfg->format == KV4_FORMAT_NVFP4;
    a.mx = cfg->format == KV4_FORMAT_MXFP4;
    const cudaError_t e = launch_decode(a, d->grid[G], static_cast<cudaStream_t>(stream), nullptr);
    return e == cudaSuccess ? KV4_OK : KV4_ERR_CUDA;
}

namespace kv4 {

// Read (and optionally clear) the allocation-free decode's error word on the current
// device. Synchronous; allocates nothing.
cudaError_t noalloc_device_error(int32_t* code, bool clear)
{
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpyFromSymbol(code, g_kv4_noalloc_err, sizeof(int32_t));
    if (e == cudaSuccess && clear) {
        const int32_t zero = 0;
        e = cudaMemcpyToSymbol(g_kv4_noalloc_err, &zero, sizeof(int32_t));
    }
    return e;
}

}  // namespace kv4
