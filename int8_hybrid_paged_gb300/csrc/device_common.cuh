// device_common.cuh — device helpers shared by the append and decode kernels.
//
// Pages cited (title, then section):
//   [zh] "KV4-RL:用 INT4 KV 缓存量化为 RLVR 异步 Rollout 提速"
//   [ko] "INT4 KV 캐시로 비동기 RLVR 롤아웃을 1.8배 가속한다"
//
// Every float operation that feeds an integer decision (a code, an INT8 query
// value, a u8 PV weight) is spelled with an explicit-rounding intrinsic, so the
// compiler cannot contract or reorder it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace kv4 {

constexpr unsigned kFull = 0xffffffffu;

// ---------------------------------------------------------------- errors
__device__ __forceinline__ void report_error(int32_t* err, int32_t code)
{
    if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---------------------------------------------------------------- bf16 loads
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// 4 consecutive bf16 values (8 bytes, 8-byte aligned) -> float.
__device__ __forceinline__ void load_bf16x4(const uint16_t* p, float (&x)[4])
{
    uint2 r = __ldg(reinterpret_cast<const uint2*>(p));
    x[0] = bf16_lo(r.x);
    x[1] = bf16_hi(r.x);
    x[2] = bf16_lo(r.y);
    x[3] = bf16_hi(r.y);
}

// ---------------------------------------------------------------- warp reductions
__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}
__device__ __forceinline__ float warp_min(float v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, m));
    return v;
}
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}
__device__ __forceinline__ int warp_sum_int(int v)
{
#pragma unroll
    for (int m = 16; m > 0; m >>= 1) v += __shfl_xor_sync(kFull, v, m);
    return v;
}

// ---------------------------------------------------------------- Hadamard rotation
// Orthonormal 128-point Walsh–Hadamard transform (H/√128) over one warp; lane l
// holds dims 4l..4l+3. Stages h = 1, 2 run inside the lane, h = 4 … 64 pair lane
// l with lane l ^ (h/4). Within a stage each pair (i, i+h) becomes
// (x_i + x_{i+h}, x_i − x_{i+h}); the stage order is fixed, so the rounded result
// does not depend on how the pairs are spread over lanes.
// [zh] 前置知识 › 分组仿射 KV 量化 (QH(HK)^T = QK^T); 方法步骤详情 step 2.
__device__ __forceinline__ void warp_fwht128(float (&x)[4], int lane)
{
    float a0 = __fadd_rn(x[0], x[1]), a1 = __fsub_rn(x[0], x[1]);
    float a2 = __fadd_rn(x[2], x[3]), a3 = __fsub_rn(x[2], x[3]);
    x[0] = __fadd_rn(a0, a2);
    x[2] = __fsub_rn(a0, a2);
    x[1] = __fadd_rn(a1, a3);
    x[3] = __fsub_rn(a1, a3);
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        // lower lane: x + y; upper lane: y - x (its partner's value minus its own),
        // one fma with an exact ±1 product, so each rounds once as an add/sub would
        const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float y = __shfl_xor_sync(kFull, x[i], m);
            x[i] = __fmaf_rn(x[i], sg, y);
        }
    }
    const float inv_sqrt128 = 0x1.6a09e6p-4f;   // nearest float to 1/√128
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __fmul_rn(x[i], inv_sqrt128);
}

// The same transform of two vectors at once (x[i] = (value of one, of the other)), with
// packed fp32x2 arithmetic: every element rounds exactly as in warp_fwht128.
__device__ __forceinline__ void warp_fwht128x2(float2 (&x)[4], int lane)
{
    const float2 a0 = __fadd2_rn(x[0], x[1]);
    const float2 a1 = __fadd2_rn(x[0], make_float2(-x[1].x, -x[1].y));
    const float2 a2 = __fadd2_rn(x[2], x[3]);
    const float2 a3 = __fadd2_rn(x[2], make_float2(-x[3].x, -x[3].y));
    x[0] = __fadd2_rn(a0, a2);
    x[2] = __fadd2_rn(a0, make_float2(-a2.x, -a2.y));
    x[1] = __fadd2_rn(a1, a3);
    x[3] = __fadd2_rn(a1, make_float2(-a3.x, -a3.y));
#pragma unroll
    for (int m = 1; m < 32; m <<= 1) {
        const float sg = (lane & m) ? -1.0f : 1.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float2 y = make_float2(__shfl_xor_sync(kFull, x[i].x, m), __shfl_xor_sync(kFull, x[i].y, m));
            x[i] = __ffma2_rn(x[i], make_float2(sg, sg), y);
        }
    }
    const float inv_sqrt128 = 0x1.6a09e6p-4f;
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __fmul2_rn(x[i], make_float2(inv_sqrt128, inv_sqrt128));
}

// ---------------------------------------------------------------- affine quantizer
// One group = the warp's 128 values. x^ = Δc + m with fp16 Δ, m:
// m = fp16 rounded down from min x (a zero minimum is taken as +0),
// Δ = fp16 rounded up from (max x − m)/LEVELS, itself rounded up in float,
// c = clamp(rint((x − m) · fl(1/Δ)), 0, LEVELS); Δ = 0 gives c = 0.
// [zh] 前置知识 › 分组仿射 KV 量化; 方法步骤详情 step 2 (fp16 Δ, m computed online).
// The smallest fp16 value >= r / n for r >= 0, i.e. the quotient rounded up to fp16
// (rounding up to fp32 first and then to fp16 gives the same value). An fp32 estimate
// r * fl(1/n), within a few fp32 ulps, is rounded up to fp16 and then moved by at most
// one fp16 step, decided by exact comparisons: c * n is exact for an 11-bit c and an
// integer n below 2^13.
__device__ __forceinline__ __half half_div_up(float r, float n, float inv_n)
{
    const __half c = __float2half_ru(__fmul_rn(r, inv_n));
    const unsigned short cb = __half_as_ushort(c);
    const unsigned short pb = (unsigned short)(cb - 1);
    const bool below = __fmul_rn(__half2float(c), n) < r;                     // estimate below the quotient
    const bool above = cb != 0 && __fmul_rn(__half2float(__ushort_as_half(pb)), n) >= r;   // one step too high
    // selects, not branches: lanes that hold different groups take different cases
    return __ushort_as_half(below ? (unsigned short)(cb + 1) : (above ? pb : cb));
}

// The quantizer's parameters of one group from its min lo and max hi: fp16 m rounded
// down, fp16 Δ rounded up, their float values and inv = fl(1/Δ) (0 when Δ = 0, which
// makes every code 0).
template <int LEVELS>
__device__ __forceinline__ void quant_params(float lo, float hi, __half& min_h, __half& delta_h, float& m,
                                             float& inv)
{
    lo = __fadd_rn(lo, 0.0f);
    min_h = __float2half_rd(lo);
    m = __half2float(min_h);
    const float r = __fadd_ru(hi, -m);
    delta_h = half_div_up(r, (float)LEVELS, 1.0f / (float)LEVELS);
    const float delta = __half2float(delta_h);
    inv = delta == 0.0f ? 0.0f : __frcp_rn(delta);
}

// The codes of a pair of values, rint(fl(fl(x − m)·inv)) with ties to even. The clamp
// to [0, LEVELS] of the definition never acts: m ≤ min x makes x − m ≥ 0, and
// m + LEVELS·Δ ≥ max x with fl(1/Δ) and the two roundings keeps the product below
// LEVELS + 1/2.
__device__ __forceinline__ uint2 code_pair(float2 x, float2 m, float2 inv)
{
    const float2 v = __fmul2_rn(__fadd2_rn(x, make_float2(-m.x, -m.y)), inv);
    return make_uint2((uint32_t)__float2int_rn(v.x), (uint32_t)__float2int_rn(v.y));
}

// Warp-wide min and max of a float (sm_100 redux on floats; -0 orders below +0).
__device__ __forceinline__ float warp_min_f32(float v)
{
    float r;
    asm volatile("redux.sync.min.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float warp_max_f32(float v)
{
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

template <int LEVELS>
__device__ __forceinline__ void warp_quant(const float (&x)[4], uint32_t (&c)[4],
                                           __half& delta_h, __half& min_h)
{
    const float lo = warp_min_f32(fminf(fminf(x[0], x[1]), fminf(x[2], x[3])));
    const float hi = warp_max_f32(fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));
    float m, inv;
    quant_params<LEVELS>(lo, hi, min_h, delta_h, m, inv);
    const uint2 c01 = code_pair(make_float2(x[0], x[1]), make_float2(m, m), make_float2(inv, inv));
    const uint2 c23 = code_pair(make_float2(x[2], x[3]), make_float2(m, m), make_float2(inv, inv));
    c[0] = c01.x;
    c[1] = c01.y;
    c[2] = c23.x;
    c[3] = c23.y;
}

// ---------------------------------------------------------------- exp2
// exp2 for the page-local PV weights, identical on every device and on the host
// oracle: 2^x = 2^n · 2^f, n = rint(x), f = x − n ∈ [−½, ½], 2^f by the Taylor
// series Σ (f ln2)^k / k! up to k = 7 in Horner form with fused multiply-adds.
// Coefficients: (ln 2)^k / k! rounded to float. Used for x ≤ 0; x < −125 gives 0,
// so every nonzero result is a normal float and the 2^n scaling is exact.
__device__ __forceinline__ float exp2_poly(float x)
{
    if (!(x >= -125.0f)) return 0.0f;
    const int n = __float2int_rn(x);
    const float f = __fsub_rn(x, (float)n);
    float p = 0x1.ffcbfcp-17f;
    p = __fmaf_rn(p, f, 0x1.430912p-13f);
    p = __fmaf_rn(p, f, 0x1.5d87fep-10f);
    p = __fmaf_rn(p, f, 0x1.3b2ab6p-7f);
    p = __fmaf_rn(p, f, 0x1.c6b08ep-5f);
    p = __fmaf_rn(p, f, 0x1.ebfbe0p-3f);
    p = __fmaf_rn(p, f, 0x1.62e430p-1f);
    p = __fmaf_rn(p, f, 1.0f);
    return __int_as_float(__float_as_int(p) + (n << 23));
}

// The same exp2 on two values with packed fp32 arithmetic; bit-identical to
// exp2_poly (rint(x) is taken as (x + 1.5·2^23) − 1.5·2^23, exact for |x| < 2^22).
__device__ __forceinline__ float2 exp2_poly2(float2 x)
{
    const float kMagic = 12582912.0f;
    const float2 xm = __fadd2_rn(x, make_float2(kMagic, kMagic));
    const float2 n = __fadd2_rn(xm, make_float2(-kMagic, -kMagic));
    const float2 f = __ffma2_rn(n, make_float2(-1.0f, -1.0f), x);
    float2 p = make_float2(0x1.ffcbfcp-17f, 0x1.ffcbfcp-17f);
    p = __ffma2_rn(p, f, make_float2(0x1.430912p-13f, 0x1.430912p-13f));
    p = __ffma2_rn(p, f, make_float2(0x1.5d87fep-10f, 0x1.5d87fep-10f));
    p = __ffma2_rn(p, f, make_float2(0x1.3b2ab6p-7f, 0x1.3b2ab6p-7f));
    p = __ffma2_rn(p, f, make_float2(0x1.c6b08ep-5f, 0x1.c6b08ep-5f));
    p = __ffma2_rn(p, f, make_float2(0x1.ebfbe0p-3f, 0x1.ebfbe0p-3f));
    p = __ffma2_rn(p, f, make_float2(0x1.62e430p-1f, 0x1.62e430p-1f));
    p = __ffma2_rn(p, f, make_float2(1.0f, 1.0f));
    const int n0 = __float_as_int(xm.x) - __float_as_int(kMagic);
    const int n1 = __float_as_int(xm.y) - __float_as_int(kMagic);
    return make_float2(x.x >= -125.0f ? __int_as_float(__float_as_int(p.x) + (n0 << 23)) : 0.0f,
                       x.y >= -125.0f ? __int_as_float(__float_as_int(p.y) + (n1 << 23)) : 0.0f);
}

// Fast exp2 (hardware approximation) for rescaling factors that decide no integer.
__device__ __forceinline__ float exp2_fast(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---------------------------------------------------------------- integer dots
// Σ_k a_k·b_k over four byte lanes: a signed (INT8 query), b unsigned (codes).
__device__ __forceinline__ int dp4a_su(uint32_t a, uint32_t b, int c)
{
    int d;
    asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}
// both unsigned (u8 PV weights against codes)
__device__ __forceinline__ int dp4a_uu(uint32_t a, uint32_t b, int c)
{
    uint32_t d;
    asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return (int)d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// ---------------------------------------------------------------- bulk copies + mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// RoPE of one 128-dim vector held 4 dims per lane (lane l: dims 4l .. 4l+3) with one
// row of the caller's table (cos of pair i at row[i], sin at row[64 + i]): dims i and
// i + 64 (lanes l and l ^ 16) rotate together, x_i' = fma(x_i, cos, -(x_{i+64} sin)),
// x_{i+64}' = fma(x_{i+64}, cos, x_i sin), each product and fma rounded once.
struct RopeRow {
    float4 c, s;                 // this lane's cos and sin (pairs 4 (l mod 16) .. +3)
};
__device__ __forceinline__ RopeRow rope_row(const float* __restrict__ row, int lane)
{
    const int i0 = 4 * (lane & 15);
    return {__ldg(reinterpret_cast<const float4*>(row + i0)),
            __ldg(reinterpret_cast<const float4*>(row + 64 + i0))};
}
__device__ __forceinline__ void warp_rope128(float (&x)[4], const RopeRow& r, int lane)
{
    const float cc[4] = {r.c.x, r.c.y, r.c.z, r.c.w}, ss[4] = {r.s.x, r.s.y, r.s.z, r.s.w};
    const bool lo = lane < 16;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float y = __shfl_xor_sync(0xffffffffu, x[j], 16);       // the paired dim
        x[j] = lo ? __fmaf_rn(x[j], cc[j], -__fmul_rn(y, ss[j]))
                  : __fmaf_rn(x[j], cc[j], __fmul_rn(y, ss[j]));
    }
}

// The same rotation of two vectors at once (x[j] = (value of one, of the other)), each
// with its own table row; every element rounds exactly as in warp_rope128.
__device__ __forceinline__ void warp_rope128x2(float2 (&x)[4], const RopeRow& ra, const RopeRow& rb, int lane)
{
    const float ca[4] = {ra.c.x, ra.c.y, ra.c.z, ra.c.w}, sa[4] = {ra.s.x, ra.s.y, ra.s.z, ra.s.w};
    const float cb[4] = {rb.c.x, rb.c.y, rb.c.z, rb.c.w}, sb[4] = {rb.s.x, rb.s.y, rb.s.z, rb.s.w};
    const float sg = lane < 16 ? -1.0f : 1.0f;        // lower half: x cos - y sin; upper: x cos + y sin
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float2 y = make_float2(__shfl_xor_sync(0xffffffffu, x[j].x, 16),
                                     __shfl_xor_sync(0xffffffffu, x[j].y, 16));
        const float2 t = __fmul2_rn(y, make_float2(sg * sa[j], sg * sb[j]));   // exact sign flip
        x[j] = __ffma2_rn(x[j], make_float2(ca[j], cb[j]), t);
    }
}

// Programmatic dependent launch: wait until the grid this one depends on has completed
// and its memory is visible (returns at once for an ordinary launch), and allow the
// next grid on the stream to be scheduled.
__device__ __forceinline__ void grid_dependency_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> shared (16-byte aligned addresses, size multiple of 16),
// completion counted on `bar`. Plain (non-multicast) form.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Test phase `parity` of `bar`; a waiting thread may be suspended for up to
// ~20 us (the hint, in ns) or until the phase completes, instead of spinning.
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Lane-predicated (pred != 0) arm of `bar` for `bytes` and 1-D bulk copy global ->
// shared completing on it: one asm block, no branch around it.
__device__ __forceinline__ void issue_bulk(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                           uint32_t pred)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%3], %2;\n\t"
        "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "r"(pred)
        : "memory");
}

// Lane-predicated plain arrive on `bar` (an item with nothing to copy).
__device__ __forceinline__ void arrive_pred(uint32_t bar, uint32_t pred)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %1, 0;\n\t"
        "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(bar), "r"(pred)
        : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_at(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(20000u)
        : "memory");
    return ok != 0;
}

// Slow path of a wait whose first try failed: retry, giving up after ~2 s.
static __device__ __noinline__ bool mbar_wait_slow(uint32_t bar, uint32_t parity)
{
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait_at(bar, parity)) return true;
        if (globaltimer_ns() - t0 > 2000000000ull) return false;
    }
}

// Wait for phase `parity` of `bar`, giving up after ~2 s. Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > 2000000000ull) return false;
    }
}

}  // namespace kv4
