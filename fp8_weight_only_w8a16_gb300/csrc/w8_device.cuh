// w8_device.cuh -- device helpers shared by the GEMV kernels of libw8:
// streaming weight loads, the exact E4M3 -> bf16 and MXFP4 -> bf16
// widenings, the weight operand fragments of the packed layout (w8_layout.h),
// rounding, asynchronous copies and programmatic-dependent-launch controls.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "w8_layout.h"

namespace w8 {
namespace {

// Streaming 16-byte weight load: read-only path, no L1 allocation, 256-byte
// L2 fetch granule (a warp's 512-byte run is two granules).
__device__ __forceinline__ uint4 ld_stream(const uint8_t *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(p));
    return v;
}

// Two E4M3fn codes -> two bf16, exactly.  `sel` picks bytes (0,2) or (1,3) of
// the word and puts each code in the low byte of a 16-bit lane with its sign
// replicated across the high byte (prmt's sign-replicate mode).  Shifting left
// by 4 and masking leaves the sign at bit 15 and the 7 exponent+mantissa bits
// at bits 10..4: a bf16 whose exponent field is the E4M3 exponent field
// (bias 127 instead of 7) and whose top 3 mantissa bits are the E4M3 mantissa
// (a bf16 subnormal when the exponent field is 0, just as E4M3 subnormals).
// Multiplying by 2^120 moves the bias from 127 to 7; the product is exact for
// every finite code, including subnormals and zeros.  (The two NaN codes come
// out as +-480; their rows carry a NaN scale instead, set at bind.)
template <uint32_t kSel>
__device__ __forceinline__ uint32_t widen_e4m3x2(uint32_t w)
{
    uint32_t d, r;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(w), "n"(kSel));
    d = (d << 4) & 0x87F087F0u;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(d), "r"(0x7B807B80u)); // 2^120, 2^120
    return r;
}
constexpr uint32_t kSelRowG = 0xA280u;  // bytes 0 and 2 (row g)
constexpr uint32_t kSelRowG8 = 0xB391u; // bytes 1 and 3 (row g+8)

// fp32 -> bf16, round to nearest even (NaN stays NaN, overflow gives inf).
__device__ __forceinline__ uint16_t to_bf16(float f)
{
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}

// The output column of packed row p: p itself on a plain plane; on a gate_up
// plane (packed tile t = gate rows 8t..8t+7, then up rows 8t..8t+7, of a
// [2*half, K] merged projection) the source row, which is also the column of
// SiLU-and-multiply's output for a gate row.
__device__ __forceinline__ int out_col(int p, bool gated, int half)
{
    if (!gated)
        return p;
    const int t = p >> 4, i = p & 15;
    return i < 8 ? 8 * t + i : half + 8 * t + (i - 8);
}

// SiLU-and-multiply of one gate/up pair, from the scaled fp32 row sums: g
// and u are rounded to bf16 first (the projection's outputs), then
// h = bf16(silu(g) * u) with silu(g) = g / (1 + exp(-g)) in fp32 (CUDA's
// expf and a correctly rounded division: the library is compiled without
// fast-math).
__device__ __forceinline__ uint16_t silu_mul_bf16(float g_sum, float u_sum)
{
    const float g = __uint_as_float(uint32_t(to_bf16(g_sum)) << 16);
    const float u = __uint_as_float(uint32_t(to_bf16(u_sum)) << 16);
    const float s = g / (1.0f + expf(-g));
    return to_bf16(s * u);
}

// 4-byte asynchronous copy global -> shared (the CTA's row scales).
__device__ __forceinline__ void cp_async4(float *smem, const float *gmem)
{
    const uint32_t s = uint32_t(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit()
{
    asm volatile("cp.async.commit_group;" ::: "memory");
}
// Wait until at most N of this thread's committed copy groups are pending.
template <int N> __device__ __forceinline__ void cp_async_wait_group()
{
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all()
{
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_all;" ::: "memory");
}

// Programmatic dependent launch: let the next kernel of the stream begin
// launching, and wait until the previous one has finished and its writes are
// visible.  Both are no-ops when the launch carries no programmatic edge.
__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Hint: fetch `bytes` at p into L2 (a bulk prefetch; nothing waits on it).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ float ld_cg_f32(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// Weight operand of one (row tile, K block) for one lane: 16 bytes of E4M3
// codes, 32 bytes of bf16, or 8 bytes of MXFP4 codes plus the word of its
// rows' block scales (bf16 of row g, bf16 of row g+8).
template <int kDt> struct WFrag;
template <> struct WFrag<kDtFp8> { uint4 v; };
template <> struct WFrag<kDtBf16> { uint4 v[2]; };
template <> struct WFrag<kDtFp4> { uint2 v; uint32_t s; };
template <> struct WFrag<kDtFp4Wide> { uint2 v; uint32_t s; };

// Predicated streaming loads: fill the destination only when ok (it keeps
// its value otherwise).
__device__ __forceinline__ void ld_stream_pred(uint4 &v, const uint8_t *p, uint32_t ok)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t"
                 "@q ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
                 : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
                 : "l"(p), "r"(ok));
}
__device__ __forceinline__ void ld_stream8_pred(uint2 &v, const uint8_t *p, uint32_t ok)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %3, 0;\n\t"
                 "@q ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];\n\t}"
                 : "+r"(v.x), "+r"(v.y)
                 : "l"(p), "r"(ok));
}
__device__ __forceinline__ void ld_stream4_pred(uint32_t &v, const uint8_t *p, uint32_t ok)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %2, 0;\n\t"
                 "@q ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];\n\t}"
                 : "+r"(v)
                 : "l"(p), "r"(ok));
}

// Load the lane's fragment of the run at p (p already includes the lane's
// offset into the run; soff is the offset from p to the lane's scale word,
// MXFP4 only), predicated on ok.
template <int kDt>
__device__ __forceinline__ void load_w_pred(WFrag<kDt> &f, const uint8_t *p, int soff, uint32_t ok)
{
    if constexpr (kDt == kDtFp8) {
        ld_stream_pred(f.v, p, ok);
    } else if constexpr (kDt == kDtBf16) {
        ld_stream_pred(f.v[0], p, ok);
        ld_stream_pred(f.v[1], p + 512, ok);
    } else {
        ld_stream8_pred(f.v, p, ok);
        ld_stream4_pred(f.s, p + soff, ok);
    }
}
template <int kDt>
__device__ __forceinline__ void load_w(WFrag<kDt> &f, const uint8_t *p, int soff)
{
    load_w_pred<kDt>(f, p, soff, 1u);
}
// The same load with no predicate at all (the steady part of a stream).
template <int kDt>
__device__ __forceinline__ void load_w_now(WFrag<kDt> &f, const uint8_t *p, int soff)
{
    if constexpr (kDt == kDtFp8) {
        f.v = ld_stream(p);
    } else if constexpr (kDt == kDtBf16) {
        f.v[0] = ld_stream(p);
        f.v[1] = ld_stream(p + 512);
    } else {
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v2.u32 {%0,%1}, [%2];"
                     : "=r"(f.v.x), "=r"(f.v.y)
                     : "l"(p));
        asm volatile("ld.global.nc.L1::no_allocate.L2::256B.u32 %0, [%1];" : "=r"(f.s) : "l"(p + soff));
    }
}

template <int kDt>
__device__ __forceinline__ void zero_w(WFrag<kDt> &f)
{
    if constexpr (kDt == kDtFp8) {
        f.v = make_uint4(0, 0, 0, 0);
    } else if constexpr (kDt == kDtBf16) {
        f.v[0] = make_uint4(0, 0, 0, 0);
        f.v[1] = make_uint4(0, 0, 0, 0);
    } else {
        f.v = make_uint2(0, 0);
        f.s = 0;
    }
}

// MXFP4 A registers from a packed code word (the bit places of w8_layout.h):
// the bf16x2 bit patterns of two E2M1 values times 2^-126, exactly -- sign to
// bit 15, exponent bits to 8..7, mantissa bit to 6, so a normal code e >= 1
// reads as (1 + m/2) 2^(e - 127) and the subnormal one (e = 0) as m/2 2^-126.
constexpr uint32_t kFp4Mask = 0x81C081C0u; // magnitudes at 6..8, 22..24, signs at 15, 31
template <int kReg>
__device__ __forceinline__ uint32_t e2m1x2_bits(uint32_t w)
{
    if constexpr (kReg == 0)
        return (w << 6) & kFp4Mask;
    else if constexpr (kReg == 1)
        return (w << 3) & kFp4Mask;
    else if constexpr (kReg == 2)
        return w & kFp4Mask;
    else // bits 10, 11 -> 6, 7; 13 -> 8; 14 -> 15 (and the same 16 higher)
        return ((w >> 4) & 0x00C000C0u) | ((w >> 5) & 0x01000100u) | ((w << 1) & 0x80008000u);
}
__device__ __forceinline__ uint32_t mul_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// The eight A registers of one lane for one block (two m16n8k16 steps).
template <int kDt>
__device__ __forceinline__ void a_operands(uint32_t (&a)[8], const WFrag<kDt> &f)
{
    if constexpr (kDt == kDtFp8) {
        a[0] = widen_e4m3x2<kSelRowG>(f.v.x);
        a[1] = widen_e4m3x2<kSelRowG8>(f.v.x);
        a[2] = widen_e4m3x2<kSelRowG>(f.v.y);
        a[3] = widen_e4m3x2<kSelRowG8>(f.v.y);
        a[4] = widen_e4m3x2<kSelRowG>(f.v.z);
        a[5] = widen_e4m3x2<kSelRowG8>(f.v.z);
        a[6] = widen_e4m3x2<kSelRowG>(f.v.w);
        a[7] = widen_e4m3x2<kSelRowG8>(f.v.w);
    } else if constexpr (kDt == kDtBf16) {
        a[0] = f.v[0].x; a[1] = f.v[0].y; a[2] = f.v[0].z; a[3] = f.v[0].w;
        a[4] = f.v[1].x; a[5] = f.v[1].y; a[6] = f.v[1].z; a[7] = f.v[1].w;
    } else {
        // E2M1 x 2^-126 (exact) x the stored factor: 2^126 x the block scale
        // 2^(e-127) = 2^(e-1) for kDtFp4 (exact: bf16 holds 2^(e-1) for e <=
        // 128, and the product keeps 2 significant bits within bf16's range),
        // or 2^126 and then the scale for kDtFp4Wide (scales past 2^1).  A NaN
        // scale gives NaN, a product past bf16's range gives inf.
        uint32_t sg, sg8;
        asm("prmt.b32 %0, %1, 0, 0x1010;" : "=r"(sg) : "r"(f.s));  // (row g, row g)
        asm("prmt.b32 %0, %1, 0, 0x3232;" : "=r"(sg8) : "r"(f.s)); // (row g+8, row g+8)
        constexpr uint32_t k2p126 = 0x7E807E80u;                  // 2^126, 2^126
#pragma unroll
        for (int q = 0; q < 2; ++q) {
            const uint32_t w = q ? f.v.y : f.v.x;
            if constexpr (kDt == kDtFp4Wide) {
                a[4 * q + 0] = mul_bf16x2(mul_bf16x2(e2m1x2_bits<0>(w), k2p126), sg);
                a[4 * q + 1] = mul_bf16x2(mul_bf16x2(e2m1x2_bits<1>(w), k2p126), sg8);
                a[4 * q + 2] = mul_bf16x2(mul_bf16x2(e2m1x2_bits<2>(w), k2p126), sg);
                a[4 * q + 3] = mul_bf16x2(mul_bf16x2(e2m1x2_bits<3>(w), k2p126), sg8);
            } else {
                a[4 * q + 0] = mul_bf16x2(e2m1x2_bits<0>(w), sg);
                a[4 * q + 1] = mul_bf16x2(e2m1x2_bits<1>(w), sg8);
                a[4 * q + 2] = mul_bf16x2(e2m1x2_bits<2>(w), sg);
                a[4 * q + 3] = mul_bf16x2(e2m1x2_bits<3>(w), sg8);
            }
        }
    }
}

} // namespace
} // namespace w8
