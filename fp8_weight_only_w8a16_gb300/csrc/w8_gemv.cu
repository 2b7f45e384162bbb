// w8_gemv.cu -- the w8a16 / bf16 decode GEMV for sm_103a.
//
// Computes, per output row n and decode token m (ATOM PR #2980, Summary and
// Changes),
//     y[m,n] = bf16_rne( scale[n] * sum_k widen(W[n,k]) * x[m,k] )
// with fp32 accumulation.  The E4M3 codes widen exactly to bf16 in registers,
// feed bf16 tensor-core steps (mma.sync m16n8k16, fp32 accumulators) with the
// decode tokens as the instruction's N = 8 dimension, and the fp32 row scale
// multiplies the reduced row right before the single bf16 rounding.
//
// Why tensor cores for a GEMV: at M = 8 every weight byte costs 8 multiply-adds;
// at the HBM rate that is ~5e13 FMA/s, more than the fp32 pipes sustain once
// the widening is added, so the multiply-adds go to the tensor pipe and the
// integer/fp pipes only widen.  The weights are still read exactly once, with
// fully coalesced 16-byte loads that stream past L1.
//
// Data flow of one CTA (8 warps, see w8_layout.h for the packed layout):
//   1. issue the first D weight loads of every warp (they do not depend on x);
//   2. stage x[0..8*NT)[k range] into shared memory (zero past M and past K);
//   3. per K block: one 16-byte weight load per lane per row tile (D blocks
//      ahead), one 16-byte shared-memory load of activations per 8 tokens,
//      widen, two tensor-core steps per (row tile, 8 tokens);
//   4. splits == 1: scale, round, store.  splits > 1: store fp32 partials,
//      count arrivals; the last CTA of the row group sums the partials in
//      split order, scales, rounds and stores.  No CTA waits on another.
#include <cuda_runtime.h>
#include <stdint.h>

#include "w8_internal.h"

namespace w8 {
namespace {

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------

// Streaming 16-byte weight load: read-only path, no L1 allocation, 256-byte
// L2 fetch granule (a warp's 512-byte run is two granules).
__device__ __forceinline__ uint4 ld_stream(const uint8_t *p)
{
    uint4 v;
    asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
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

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// fp32 -> bf16, round to nearest even (NaN stays NaN, overflow gives inf).
__device__ __forceinline__ uint16_t to_bf16(float f)
{
    uint16_t h;
    asm("cvt.rn.bf16.f32 %0, %1;" : "=h"(h) : "f"(f));
    return h;
}

__device__ __forceinline__ float ld_cg_f32(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

// Weight operand of one (row tile, K block) for one lane.
template <bool kFp8> struct WFrag;
template <> struct WFrag<true> { uint4 v; };
template <> struct WFrag<false> { uint4 v[2]; };

template <bool kFp8>
__device__ __forceinline__ void load_w(WFrag<kFp8> &f, const uint8_t *p)
{
    if constexpr (kFp8) {
        f.v = ld_stream(p);
    } else {
        f.v[0] = ld_stream(p);
        f.v[1] = ld_stream(p + 512);
    }
}

template <bool kFp8>
__device__ __forceinline__ void zero_w(WFrag<kFp8> &f)
{
    if constexpr (kFp8) {
        f.v = make_uint4(0, 0, 0, 0);
    } else {
        f.v[0] = make_uint4(0, 0, 0, 0);
        f.v[1] = make_uint4(0, 0, 0, 0);
    }
}

// The two tensor-core steps of one K block for one (row tile, 8 tokens).
template <bool kFp8>
__device__ __forceinline__ void block_mma(float (&c)[4], const uint32_t (&a)[8], uint4 xb)
{
    mma_bf16(c, a[0], a[1], a[2], a[3], xb.x, xb.y);
    mma_bf16(c, a[4], a[5], a[6], a[7], xb.z, xb.w);
}

template <bool kFp8>
__device__ __forceinline__ void a_operands(uint32_t (&a)[8], const WFrag<kFp8> &f)
{
    if constexpr (kFp8) {
        a[0] = widen_e4m3x2<kSelRowG>(f.v.x);
        a[1] = widen_e4m3x2<kSelRowG8>(f.v.x);
        a[2] = widen_e4m3x2<kSelRowG>(f.v.y);
        a[3] = widen_e4m3x2<kSelRowG8>(f.v.y);
        a[4] = widen_e4m3x2<kSelRowG>(f.v.z);
        a[5] = widen_e4m3x2<kSelRowG8>(f.v.z);
        a[6] = widen_e4m3x2<kSelRowG>(f.v.w);
        a[7] = widen_e4m3x2<kSelRowG8>(f.v.w);
    } else {
        a[0] = f.v[0].x; a[1] = f.v[0].y; a[2] = f.v[0].z; a[3] = f.v[0].w;
        a[4] = f.v[1].x; a[5] = f.v[1].y; a[6] = f.v[1].z; a[7] = f.v[1].w;
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <bool kFp8, int NT, int R, int D, int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gemv_kernel(const GemvArgs a)
{
    extern __shared__ __align__(16) uint8_t xs[];
    constexpr int kRun = kFp8 ? kRunFp8 : kRunBf16;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t = lane & 3;

    const int rg = blockIdx.x / a.splits;
    const int sp = blockIdx.x - rg * a.splits;
    const int kb0 = int((int64_t(sp) * a.kb) / a.splits);
    const int kb1 = int((int64_t(sp + 1) * a.kb) / a.splits);
    const int nkb = kb1 - kb0;

    // ---- 1. the warp's row tiles and its first D weight loads ------------
    int rt[R];
    bool valid[R];
    const uint8_t *wptr[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
        rt[r] = rg * (kWarps * R) + r * kWarps + warp;
        valid[r] = rt[r] < a.rt;
        const int64_t tile = valid[r] ? rt[r] : 0; // idle warps re-read tile 0
        wptr[r] = a.wp + (tile * a.kb + kb0) * kRun + lane * 16;
    }
    WFrag<kFp8> ring[D][R];
#pragma unroll
    for (int i = 0; i < D; ++i)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (i < nkb)
                load_w<kFp8>(ring[i][r], wptr[r] + int64_t(i) * kRun);
            else
                zero_w<kFp8>(ring[i][r]);
        }

    // ---- 2. stage x[tokens][k range] ----------------------------------------
    {
        const int cols8 = nkb * 4;            // 8-column chunks in the range
        const int64_t kbase = int64_t(kb0) * kTileK;
        const int items = NT * 8 * cols8;
        for (int idx = threadIdx.x; idx < items; idx += kThreads) {
            const int tok = idx / cols8;
            const int c8 = idx - tok * cols8;
            const int64_t col = kbase + c8 * 8;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (tok < a.m) {
                const uint16_t *src = a.x + int64_t(tok) * a.ldx + col;
                if (a.x_vec && col + 8 <= a.k) {
                    v = __ldg(reinterpret_cast<const uint4 *>(src));
                } else {
                    uint16_t h[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        h[e] = (col + e < a.k) ? src[e] : uint16_t(0);
                    v.x = h[0] | (uint32_t(h[1]) << 16);
                    v.y = h[2] | (uint32_t(h[3]) << 16);
                    v.z = h[4] | (uint32_t(h[5]) << 16);
                    v.w = h[6] | (uint32_t(h[7]) << 16);
                }
            }
            *reinterpret_cast<uint4 *>(xs + tok * a.x_stride + c8 * 16) = v;
        }
    }
    __syncthreads();

    // ---- 3. stream the K range ---------------------------------------------
    float acc[R][NT][4];
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                acc[r][j][e] = 0.0f;

    const uint8_t *xrow = xs + g * a.x_stride + t * 16;
    for (int base = 0; base < nkb; base += D) {
#pragma unroll
        for (int i = 0; i < D; ++i) {
            const int b = base + i;
            if (b < nkb) {
                WFrag<kFp8> cur[R];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    cur[r] = ring[i][r];
                if (b + D < nkb) {
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        load_w<kFp8>(ring[i][r], wptr[r] + int64_t(b + D) * kRun);
                }
                uint32_t aop[R][8];
#pragma unroll
                for (int r = 0; r < R; ++r)
                    a_operands<kFp8>(aop[r], cur[r]);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint4 xb =
                        *reinterpret_cast<const uint4 *>(xrow + j * 8 * a.x_stride + b * 64);
#pragma unroll
                    for (int r = 0; r < R; ++r)
                        block_mma<kFp8>(acc[r][j], aop[r], xb);
                }
            }
        }
    }

    // ---- 4. epilogue ----------------------------------------------------------
    // Accumulator e of (r, j): row rt*16 + g + 8*(e >> 1), token 8j + 2t + (e & 1).
    if (a.splits == 1) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            if (!valid[r])
                continue;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int row = rt[r] * kTileN + g + 8 * h;
                if (row >= a.n)
                    continue;
                const float sc = kFp8 ? a.scale[row] : 1.0f;
#pragma unroll
                for (int j = 0; j < NT; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int tok = 8 * j + 2 * t + e;
                        if (tok < a.m) {
                            const float v = acc[r][j][2 * h + e];
                            a.y[int64_t(tok) * a.ldy + row] = to_bf16(kFp8 ? sc * v : v);
                        }
                    }
            }
        }
        return;
    }

    // splits > 1: partials [split][row][token]
    const int64_t rows_pad = int64_t(a.rt) * kTileN;
#pragma unroll
    for (int r = 0; r < R; ++r) {
        if (!valid[r])
            continue;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = rt[r] * kTileN + g + 8 * h;
            float *dst = a.partial + (int64_t(sp) * rows_pad + row) * a.m;
#pragma unroll
            for (int j = 0; j < NT; ++j)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = 8 * j + 2 * t + e;
                    if (tok < a.m)
                        dst[tok] = acc[r][j][2 * h + e];
                }
        }
    }
    __threadfence();
    __syncthreads();
    __shared__ int s_last;
    if (threadIdx.x == 0) {
        const int prev = atomicAdd(a.counters + rg, 1);
        s_last = (prev == a.splits - 1);
    }
    __syncthreads();
    if (!s_last)
        return;
    __threadfence();

    // The last CTA of the row group: sum the partials in split order.
    const int row0 = rg * kWarps * R * kTileN;
    int row_end = row0 + kWarps * R * kTileN;
    if (row_end > a.n)
        row_end = a.n;
    const int nrows = row_end - row0;
    const int items = nrows * a.m;
    for (int idx = threadIdx.x; idx < items; idx += kThreads) {
        const int tok = idx / nrows;
        const int row = row0 + (idx - tok * nrows);
        float v = 0.0f;
        for (int s = 0; s < a.splits; ++s)
            v += ld_cg_f32(a.partial + (int64_t(s) * rows_pad + row) * a.m + tok);
        a.y[int64_t(tok) * a.ldy + row] = to_bf16(kFp8 ? a.scale[row] * v : v);
    }
    if (threadIdx.x == 0)
        a.counters[rg] = 0; // ready for the next call on this workspace
}

// ---------------------------------------------------------------------------
// instance table
// ---------------------------------------------------------------------------
template <bool kFp8, int NT>
struct Inst {
    static constexpr int R = NT <= 2 ? 1 : 2;
    static constexpr int D = NT <= 2 ? 8 : 4;
    static constexpr int B = NT <= 2 ? 2 : 1;
    static void *fn() { return reinterpret_cast<void *>(&gemv_kernel<kFp8, NT, R, D, B>); }
};

template <bool kFp8>
void *pick(int nt)
{
    switch (nt) {
    case 1: return Inst<kFp8, 1>::fn();
    case 2: return Inst<kFp8, 2>::fn();
    case 4: return Inst<kFp8, 4>::fn();
    default: return Inst<kFp8, 8>::fn();
    }
}

} // namespace

cudaError_t prepare_gemv_kernels()
{
    const int nts[4] = {1, 2, 4, 8};
    for (int i = 0; i < 4; ++i) {
        for (int f = 0; f < 2; ++f) {
            void *fn = f ? pick<true>(nts[i]) : pick<false>(nts[i]);
            const int budget = (nts[i] <= 2 ? 100 : 200) * 1024;
            cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 budget);
            if (e != cudaSuccess)
                return e;
        }
    }
    return cudaSuccess;
}

cudaError_t launch_gemv(bool fp8, const Plan &plan, const GemvArgs &a, cudaStream_t s)
{
    void *fn = fp8 ? pick<true>(plan.nt) : pick<false>(plan.nt);
    void *args[] = {const_cast<GemvArgs *>(&a)};
    return cudaLaunchKernel(fn, dim3(plan.grid), dim3(kThreads), args, size_t(plan.smem), s);
}

} // namespace w8
