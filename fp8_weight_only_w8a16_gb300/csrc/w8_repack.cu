// w8_repack.cu -- bind-time repack of a row-major plane into W8_LAYOUT_MMA_16x32.
//
// The PR page (Changes) keeps each FP8 plane where it lies, in the (16, 16)
// preshuffle that AITER uses; here bind instead copies each plane once into the caller's
// packed buffer, in the order the GEMV's tensor-core A operand wants (see
// w8_layout.h).  One CTA per 16-row tile.  Each thread produces one lane's
// 16-byte vector of one K block: it reads 8 consecutive columns of rows g and
// g+8 of the tile (8- or 16-byte loads; the source rows are 16-byte aligned),
// zero-fills columns >= K and rows >= N, interleaves them and writes 16 bytes.
// A gate_up plane (a merged [2I, K] MLP projection) is read with its gate and
// up rows interleaved eight at a time, so that a tile's rows g and g+8 are a
// gate row and its up row.
// MXFP4 planes pack their codes into 288-byte runs (each code's four bits at
// the places the kernel's widening reads) whose last 32 bytes carry the rows'
// block scales as bf16 pairs.
// FP8 also writes the build's copy of the row scales; a row that holds a NaN
// code (0x7F or 0xFF) gets a NaN scale, so its outputs are NaN as the
// definition gives, while the GEMV's widening stays a fixed exact map.
// Block-scaled FP8 planes repack their codes the same way, take row scales
// of 1 (NaN for a row holding a NaN code) and copy their 128 x 128 block
// factors into the build, one dense row of ceil(K / 128) per 128 rows.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "w8_internal.h"

namespace w8 {
namespace {

// 8 consecutive bytes of one source row starting at column col (zero past K).
__device__ __forceinline__ uint2 load8_fp8(const uint8_t *row, int64_t col, int64_t k)
{
    if (col + 8 <= k)
        return *reinterpret_cast<const uint2 *>(row + col);
    uint8_t b[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        b[e] = (col + e < k) ? row[col + e] : uint8_t(0);
    uint2 v;
    v.x = b[0] | (uint32_t(b[1]) << 8) | (uint32_t(b[2]) << 16) | (uint32_t(b[3]) << 24);
    v.y = b[4] | (uint32_t(b[5]) << 8) | (uint32_t(b[6]) << 16) | (uint32_t(b[7]) << 24);
    return v;
}

// 8 consecutive bf16 of one source row starting at column col (zero past K).
__device__ __forceinline__ uint4 load8_bf16(const uint16_t *row, int64_t col, int64_t k)
{
    if (col + 8 <= k)
        return *reinterpret_cast<const uint4 *>(row + col);
    uint16_t h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        h[e] = (col + e < k) ? row[col + e] : uint16_t(0);
    return make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                      h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
}

__device__ __forceinline__ uint32_t byte_of(uint2 v, int j)
{
    return ((j < 4 ? v.x : v.y) >> (8 * (j & 3))) & 0xFFu;
}

__device__ __forceinline__ bool has_nan_code(uint2 v)
{
    // a byte whose low 7 bits are all ones is 0x7F or 0xFF
    uint32_t nan = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        nan |= ((byte_of(v, j) & 0x7Fu) == 0x7Fu);
    return nan != 0;
}

// The source row of packed row p (a gate_up plane interleaves gate and up
// rows eight at a time; a plain plane keeps its order).
__device__ __forceinline__ int64_t src_row(const RepackArgs &a, int64_t p)
{
    if (a.half == 0)
        return p;
    const int64_t t = p >> 4, i = p & 15;
    return i < 8 ? 8 * t + i : a.half + 8 * t + (i - 8);
}

__global__ void __launch_bounds__(256) repack_fp8_kernel(const RepackArgs a)
{
    __shared__ int nan_row[16];
    if (threadIdx.x < 16)
        nan_row[threadIdx.x] = 0;
    __syncthreads();

    const int64_t rt = blockIdx.x;
    const int64_t items = a.kb * 32;
    for (int64_t it = threadIdx.x; it < items; it += blockDim.x) {
        const int64_t kb = it >> 5;
        const int lane = int(it & 31);
        const int g = lane >> 2, t = lane & 3;
        const int64_t col = kb * kTileK + 8 * t;
        uint2 lo = make_uint2(0, 0), hi = make_uint2(0, 0);
        const int64_t n0 = rt * kTileN + g, n1 = n0 + 8;
        if (n0 < a.n)
            lo = load8_fp8(a.src + src_row(a, n0) * a.ld_bytes, col, a.k);
        if (n1 < a.n)
            hi = load8_fp8(a.src + src_row(a, n1) * a.ld_bytes, col, a.k);
        if (has_nan_code(lo))
            atomicOr(&nan_row[g], 1);
        if (has_nan_code(hi))
            atomicOr(&nan_row[g + 8], 1);
        // word w = 2q + h covers columns 4q + 2h (even) and 4q + 2h + 1 (odd):
        // bytes (row g even, row g+8 even, row g odd, row g+8 odd)
        uint32_t out[4];
#pragma unroll
        for (int w = 0; w < 4; ++w) {
            const int je = 2 * w, jo = 2 * w + 1; // columns 4q+2h, 4q+2h+1 == 2w, 2w+1
            out[w] = byte_of(lo, je) | (byte_of(hi, je) << 8) | (byte_of(lo, jo) << 16) |
                     (byte_of(hi, jo) << 24);
        }
        *reinterpret_cast<uint4 *>(a.dst + ((rt * a.kb + kb) * 32 + lane) * 16) =
            make_uint4(out[0], out[1], out[2], out[3]);
    }
    __syncthreads();
    if (threadIdx.x < 16) {
        const int64_t n = rt * kTileN + threadIdx.x;
        float s = 0.0f;
        if (n < a.n)
            s = nan_row[threadIdx.x] ? __int_as_float(0x7FC00000)
                : a.scale_src          ? a.scale_src[src_row(a, n)]
                                       : 1.0f; // block-scaled: the factors are the blocks'
        a.scale_dst[n] = s;
    }
}

__global__ void __launch_bounds__(256) repack_bf16_kernel(const RepackArgs a)
{
    const int64_t rt = blockIdx.x;
    const int64_t items = a.kb * 32;
    for (int64_t it = threadIdx.x; it < items; it += blockDim.x) {
        const int64_t kb = it >> 5;
        const int lane = int(it & 31);
        const int g = lane >> 2, t = lane & 3;
        const int64_t col = kb * kTileK + 8 * t;
        uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
        const int64_t n0 = rt * kTileN + g, n1 = n0 + 8;
        if (n0 < a.n)
            lo = load8_bf16(reinterpret_cast<const uint16_t *>(a.src + src_row(a, n0) * a.ld_bytes),
                            col, a.k);
        if (n1 < a.n)
            hi = load8_bf16(reinterpret_cast<const uint16_t *>(a.src + src_row(a, n1) * a.ld_bytes),
                            col, a.k);
        // half q: a01 = row g cols 4q+0,1; a23 = row g+8 cols 4q+0,1;
        //         a45 = row g cols 4q+2,3;  a67 = row g+8 cols 4q+2,3
        const uint4 h0 = make_uint4(lo.x, hi.x, lo.y, hi.y);
        const uint4 h1 = make_uint4(lo.z, hi.z, lo.w, hi.w);
        uint8_t *d = a.dst + (rt * a.kb + kb) * 2 * 512 + lane * 16;
        *reinterpret_cast<uint4 *>(d) = h0;
        *reinterpret_cast<uint4 *>(d + 512) = h1;
    }
}

// 8 codes (columns col .. col+7) of one MXFP4 source row as a 32-bit word,
// nibble j = column col + j (zero past K).  col is a multiple of 8, so the
// 4 bytes are 4-byte aligned (source rows are 16-byte aligned).
__device__ __forceinline__ uint32_t load8_fp4(const uint8_t *row, int64_t col, int64_t k)
{
    if (col + 8 <= k)
        return *reinterpret_cast<const uint32_t *>(row + col / 2);
    uint32_t v = 0;
    for (int j = 0; j < 8; ++j)
        if (col + j < k)
            v |= uint32_t((row[(col + j) / 2] >> (4 * ((col + j) & 1))) & 15u) << (4 * j);
    return v;
}

// E8M0 scale -> the bf16 factor stored beside the codes.  Folded (kDtFp4):
// 2^126 x 2^(e - 127) = 2^(e - 1), exponent field e + 126, for e <= 128.
// Otherwise (kDtFp4Wide) 2^(e - 127): the exponent field, except e = 0
// (2^-127, a bf16 subnormal).  e = 255 is NaN either way.
__device__ __forceinline__ uint32_t e8m0_to_bf16(uint32_t e, bool fold)
{
    if (e == 255)
        return 0x7FC0u;
    if (fold)
        return (e + 126u) << 7;
    return e == 0 ? 0x0040u : (e << 7);
}

// Whether any block scale of an MXFP4 plane lies in 129..254, where the
// folded factor 2^(e - 1) is past bf16's range: one CTA per source row.
__global__ void __launch_bounds__(256) fp4_scale_scan_kernel(const RepackArgs a, unsigned *wide)
{
    const int64_t row = blockIdx.x;
    for (int64_t kb = threadIdx.x; kb < a.kb; kb += blockDim.x) {
        const uint32_t e = a.bscale_src[row * a.ldb + kb];
        if (e > 128u && e < 255u) {
            atomicOr(wide, 1u);
            return;
        }
    }
}

__global__ void __launch_bounds__(256) repack_fp4_kernel(const RepackArgs a)
{
    const int64_t rt = blockIdx.x;
    const int64_t items = a.kb * 32;
    for (int64_t it = threadIdx.x; it < items; it += blockDim.x) {
        const int64_t kb = it >> 5;
        const int lane = int(it & 31);
        const int g = lane >> 2, t = lane & 3;
        const int64_t col = kb * kTileK + 8 * t;
        uint32_t lo = 0, hi = 0, slo = 0, shi = 0;
        const int64_t n0 = rt * kTileN + g, n1 = n0 + 8;
        if (n0 < a.n) {
            lo = load8_fp4(a.src + src_row(a, n0) * a.ld_bytes, col, a.k);
            slo = e8m0_to_bf16(a.bscale_src[src_row(a, n0) * a.ldb + kb], a.fp4_fold);
        }
        if (n1 < a.n) {
            hi = load8_fp4(a.src + src_row(a, n1) * a.ld_bytes, col, a.k);
            shi = e8m0_to_bf16(a.bscale_src[src_row(a, n1) * a.ldb + kb], a.fp4_fold);
        }
        // word q holds A registers reg = 0..3 of step q: (row g, cols 4q, +1),
        // (row g+8, same), (row g, cols 4q+2, +3), (row g+8, same) of the lane's
        // 8 columns, each element's mantissa, exponent-low, exponent-high and
        // sign bits at the places of mxfp4_code_bits (w8_layout.h)
        uint32_t out[2] = {0u, 0u};
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int reg = 0; reg < 4; ++reg)
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int c = 4 * q + 2 * (reg >> 1) + half;
                    const uint32_t code = (((reg & 1) ? hi : lo) >> (4 * c)) & 15u;
                    const int o = reg < 3 ? 3 * reg + 16 * half : 16 * half;
                    const int om = reg < 3 ? o : o + 10, oe0 = reg < 3 ? o + 1 : o + 11;
                    const int oe1 = reg < 3 ? o + 2 : o + 13, os = reg < 3 ? o + 9 : o + 14;
                    out[q] |= ((code & 1u) << om) | (((code >> 1) & 1u) << oe0) |
                              (((code >> 2) & 1u) << oe1) | (((code >> 3) & 1u) << os);
                }
        uint8_t *run = a.dst + (rt * a.kb + kb) * kRunFp4;
        *reinterpret_cast<uint2 *>(run + lane * 8) = make_uint2(out[0], out[1]);
        if (t == 0)
            *reinterpret_cast<uint32_t *>(run + kRunFp4Codes + 4 * g) = slo | (shi << 16);
    }
}

// Block-scaled FP8: the factors of one row block (CTA) into the build's copy.
__global__ void __launch_bounds__(256) copy_factors_kernel(const RepackArgs a)
{
    const int64_t rb = blockIdx.x;
    const int64_t cols = (a.k + kBlockB - 1) / kBlockB;
    for (int64_t c = threadIdx.x; c < cols; c += blockDim.x)
        a.bfac_dst[rb * cols + c] = a.bfac_src[rb * a.ldb + c];
}

} // namespace

cudaError_t fp4_scales_wide(const RepackArgs &a, unsigned *scratch, bool *wide, cudaStream_t s)
{
    *wide = false;
    if (a.n <= 0 || a.kb <= 0)
        return cudaSuccess;
    unsigned h = 0;
    cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(unsigned), s);
    if (e != cudaSuccess)
        return e;
    fp4_scale_scan_kernel<<<dim3(unsigned(a.n)), 256, 0, s>>>(a, scratch);
    if ((e = cudaGetLastError()) != cudaSuccess ||
        (e = cudaMemcpyAsync(&h, scratch, sizeof(unsigned), cudaMemcpyDeviceToHost, s)) !=
            cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return e;
    *wide = h != 0;
    return cudaSuccess;
}

cudaError_t launch_repack(int dt, const RepackArgs &a, cudaStream_t s)
{
    if (a.rt <= 0)
        return cudaSuccess;
    if (dt == kDtFp8B) {
        repack_fp8_kernel<<<dim3(unsigned(a.rt)), 256, 0, s>>>(a);
        copy_factors_kernel<<<dim3(unsigned((a.n + kBlockB - 1) / kBlockB)), 256, 0, s>>>(a);
    } else if (dt == kDtFp8)
        repack_fp8_kernel<<<dim3(unsigned(a.rt)), 256, 0, s>>>(a);
    else if (is_fp4(dt))
        repack_fp4_kernel<<<dim3(unsigned(a.rt)), 256, 0, s>>>(a);
    else
        repack_bf16_kernel<<<dim3(unsigned(a.rt)), 256, 0, s>>>(a);
    return cudaGetLastError();
}

} // namespace w8
