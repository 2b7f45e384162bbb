// w8_gemv.cu -- the w8a16 / bf16 / w4a16 decode GEMV for sm_103a.
//
// Computes, per output row n and decode token m (ATOM PR #2980, Summary and
// Changes),
//     y[m,n] = bf16_rne( scale[n] * sum_k widen(W[n,k]) * x[m,k] )
// with fp32 accumulation.  The E4M3 codes widen exactly to bf16 in registers,
// feed bf16 tensor-core steps (mma.sync m16n8k16, fp32 accumulators) with the
// decode tokens as the instruction's N = 8 dimension, and the fp32 row scale
// multiplies the reduced row right before the single bf16 rounding.  bf16
// planes skip the widening and the scale; MXFP4 planes (the ATOM Model
// Support Guide's FP4 GEMMs with 16-bit activations) widen each code times
// its E8M0 block scale exactly to bf16 instead, with no row scale.
// Block-scaled FP8 planes (one fp32 factor per 128 x 128 block, the
// blockscale GEMM's weights) widen like FP8 and sum each 128-column block
// apart: at the block's end its factor multiplies the block's sum into the
// row's accumulator (one fma), and the row scale is 1 (NaN for a row holding
// a NaN code).
//
// Why tensor cores for a GEMV: at M = 8 every weight byte costs 8 multiply-adds;
// at the HBM rate that is ~5e13 FMA/s, more than the fp32 pipes sustain once
// the widening is added, so the multiply-adds go to the tensor pipe and the
// integer/fp pipes only widen.  The weights are still read exactly once, with
// fully coalesced 16-byte loads that stream past L1.
//
// Work of one CTA (8 warps; see w8_layout.h for the layout and the plan):
//   1. each warp walks its K part of its R row tiles, one K block per step,
//      keeping D blocks of weights (HBM) and activations (L2/L1) in flight in
//      a register ring; per block: widen, two tensor-core steps per
//      (row tile, 8 tokens);
//   2. the warps' accumulators meet in shared memory; the wk K parts of each
//      row are added in K-part order;
//   3. splits == 1: scale, round, store.  splits > 1: store the fp32 partial,
//      count arrivals; the last CTA of the row group sums the partials in split
//      order, scales, rounds and stores.  No CTA ever waits on another.
// On a gate_up plane the store maps each packed row to its source row; for
// SiLU-and-multiply, accumulator e of a lane (tile row g, a gate row) meets
// accumulator e + 2 (row g + 8, its up row) and one bf16 h is stored.
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "w8_device.cuh"
#include "w8_internal.h"

namespace w8 {
namespace {

// ---------------------------------------------------------------------------
// device helpers of this kernel (the shared ones are in w8_device.cuh)
// ---------------------------------------------------------------------------

// D += A * B, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8 activations x[tok][col .. col+7] of one lane, loaded only when `ok`;
// otherwise v keeps its value (the ring slots of tokens >= m stay zero).
__device__ __forceinline__ void ld_act_pred(uint4 &v, const uint16_t *p, uint32_t ok)
{
    asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %5, 0;\n\t"
                 "@q ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];\n\t}"
                 : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w)
                 : "l"(p), "r"(ok));
}

// The same load with no predicate (the steady part of the stream).
__device__ __forceinline__ void ld_act(uint4 &v, const uint16_t *p)
{
    asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
}

// The activations of the K-tail block, element by element (zero past K).
__device__ __forceinline__ uint4 load_x_tail(const uint16_t *p, bool ok, int64_t col, int64_t k)
{
    uint16_t h[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        h[e] = (ok && col + e < k) ? p[e] : uint16_t(0);
    return make_uint4(h[0] | (uint32_t(h[1]) << 16), h[2] | (uint32_t(h[3]) << 16),
                      h[4] | (uint32_t(h[5]) << 16), h[6] | (uint32_t(h[7]) << 16));
}

// Block-scaled planes: lane l of the warp holds in fac[r] the factor of
// column block fbase + l of tile r's row block.  Before a stretch of K blocks
// whose column blocks end at hi, move the window to start at lo if hi lies
// past it (warp-uniform; at most once per 32 column blocks).
template <int R>
__device__ __forceinline__ void factor_window(float (&fac)[R], const float *const (&fac_row)[R],
                                              int &fbase, int lo, int hi, int lane, int nbf)
{
    if (hi - fbase >= 32) {
        fbase = lo;
#pragma unroll
        for (int r = 0; r < R; ++r)
            fac[r] = fbase + lane < nbf ? __ldg(fac_row[r] + fbase + lane) : 0.0f;
    }
}

// Block-scaled planes: close column block cb (inside the window) --
// acc += f * part, part = 0.  Warp-uniform: every lane calls it for the same cb.
template <int NT, int R>
__device__ __forceinline__ void close_block(float (&acc)[R][NT][4], float (&part)[R][NT][4],
                                            const float (&fac)[R], int fbase, int cb)
{
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const float f = __shfl_sync(0xffffffffu, fac[r], cb - fbase);
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[r][j][e] = fmaf(f, part[r][j][e], acc[r][j][e]);
                part[r][j][e] = 0.0f;
            }
    }
}

// One K block: widen the R weight fragments and run the two tensor-core steps
// of every (row tile, 8 tokens) into its accumulator.
template <int kDt, int NT, int R>
__device__ __forceinline__ void block_step(float (&acc)[R][NT][4], const WFrag<kDt> (&w)[R],
                                           const uint4 (&x)[NT])
{
#pragma unroll
    for (int r = 0; r < R; ++r) {
        uint32_t aop[8];
        a_operands<kDt>(aop, w[r]);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            mma_bf16(acc[r][j], aop[0], aop[1], aop[2], aop[3], x[j].x, x[j].y);
            mma_bf16(acc[r][j], aop[4], aop[5], aop[6], aop[7], x[j].z, x[j].w);
        }
    }
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
template <int kDt, int NT, int R, int DW, int DX, int kMinBlocks, bool kLong>
__global__ void __launch_bounds__(kThreads, kMinBlocks) gemv_kernel(const GemvArgs a)
{
    static_assert(DW % DX == 0, "the activation ring depth divides the weight ring depth");
    static_assert(kBlockB == 4 * kTileK, "a block factor covers four K blocks");
    static_assert(kDt != kDtFp8B || DW % 4 == 0, "block-scaled rings hold whole column blocks");
    extern __shared__ __align__(16) float red[]; // [warp][R][NT][4][32]
    constexpr bool kB128 = kDt == kDtFp8B;    // block factors inside the K loop
    constexpr int kW = kB128 ? kDtFp8 : kDt;   // the format of the weight codes
    constexpr bool kFp8 = kW == kDtFp8;        // row scales in the epilogue
    constexpr int kRun = kW == kDtFp8 ? kRunFp8 : is_fp4(kW) ? kRunFp4 : kRunBf16;
    constexpr int kLaneBytes = is_fp4(kDt) ? 8 : 16; // a lane's part of a run (bf16: twice)

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int t = lane & 3;
    const int wk = a.wk;
    const int wt = kWarps / wk;
    const int tg = warp / wk;       // tile group of this warp
    const int kp = warp - tg * wk;  // K part of this warp

    const int rg = blockIdx.x / a.splits;
    const int sp = blockIdx.x - rg * a.splits;
    // The CTA's and the warp's K blocks, split in units of kU blocks: single
    // blocks, or whole column blocks on block-scaled planes, so that every
    // warp's part starts on a column block and, with a ring of whole column
    // blocks, each column block ends at a fixed ring slot.
    constexpr int kU = kB128 ? kBlockB / kTileK : 1;
    const int nu = (a.kb + kU - 1) / kU;
    const int cu0 = int((int64_t(sp) * nu) / a.splits);
    const int cnu = int((int64_t(sp + 1) * nu) / a.splits) - cu0;
    const int u0 = cu0 + (kp * cnu) / wk;
    const int u1 = cu0 + ((kp + 1) * cnu) / wk;
    const int kb0 = u0 * kU;
    const int kb1 = u1 * kU < a.kb ? u1 * kU : a.kb;
    const int nkb = kb1 > kb0 ? kb1 - kb0 : 0;

    // ---- the warp's row tiles and activation rows ----------------------------
    // Blocks [0, nmain) of the warp's K part lie wholly inside K; when K is not
    // a multiple of 32 the plane's last block is partial and is handled after
    // the pipeline (it can only be the last block of the last K part).
    const int full_blocks = a.k / kTileK;
    int nmain = full_blocks - kb0;
    nmain = nmain < 0 ? 0 : (nmain > nkb ? nkb : nmain);
    const bool has_tail = nkb > nmain;

    const uint8_t *wptr[R]; // this lane's part of the warp's first run of each tile
#pragma unroll
    for (int r = 0; r < R; ++r) {
        const int tile = rg * (wt * R) + r * wt + tg;
        const int64_t t64 = tile < a.rt ? tile : 0; // idle slots re-read tile 0
        wptr[r] = a.wp + (t64 * a.kb + kb0) * kRun + lane * kLaneBytes;
    }
    // MXFP4: from the lane's codes to its rows' scale word (g) after the codes
    const int soff = is_fp4(kDt) ? kRunFp4Codes - kLaneBytes * lane + 4 * g : 0;
    const uint16_t *xptr[NT];
    uint32_t tok_ok[NT];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
        const int tok = 8 * j + g;
        tok_ok[j] = tok < a.m;
        xptr[j] = a.x + int64_t(tok < a.m ? tok : 0) * a.ldx + int64_t(kb0) * kTileK + 8 * t;
    }

    // Weights first: the packed plane is written only by w8_bind, which
    // finishes before any GEMV can be launched, so these loads may overlap the
    // tail of the previous kernel on the stream.  The ring holds blocks
    // [0, DW); for FP8 and MXFP4 planes, blocks up to kPf go to L2 now, and
    // every ring group sends the kPf-distant group after it (bulk
    // prefetches: no registers, no waits).  bf16 planes skip it: twice the
    // bytes ahead crowded L2 on the largest planes (lm_head, o_proj bf16) and
    // cost time.  Lane 0 issues them, so its wptr is the start of the warp's
    // runs.
    constexpr int kPf = kDt != kDtBf16 ? (DW > 16 ? DW : 16) : DW;
    if (kPf > DW && lane == 0 && nmain > DW) {
        const int hi = nmain < kPf ? nmain : kPf;
        if (hi > DW)
#pragma unroll
            for (int r = 0; r < R; ++r)
                prefetch_l2(wptr[r] + DW * kRun, uint32_t(hi - DW) * kRun);
    }
    WFrag<kW> wring[DW][R];
    uint4 xring[DX][NT];
#pragma unroll
    for (int i = 0; i < DW; ++i)
#pragma unroll
        for (int r = 0; r < R; ++r) {
            zero_w<kW>(wring[i][r]);
            if (i < nmain)
                load_w<kW>(wring[i][r], wptr[r] + i * kRun, soff);
        }
    // block-scaled planes: the first 32 factors of the warp's column blocks
    // (bind-time data too), one per lane, for each of its row tiles
    float fac[R];
    const float *fac_row[R];
    int fbase = kb0 >> 2;
    if constexpr (kB128) {
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const int tile = rg * (wt * R) + r * wt + tg;
            fac_row[r] = a.bfac + int64_t(tile < a.rt ? tile >> 3 : 0) * a.nbf;
            fac[r] = fbase + lane < a.nbf ? __ldg(fac_row[r] + fbase + lane) : 0.0f;
        }
    }
    // the CTA's row scales (bind-time data too) into shared memory
    __shared__ float s_scale[kWarps * 2 * kTileN];
    const int row0 = rg * wt * R * kTileN;
    if constexpr (kFp8) {
        if (threadIdx.x < wt * R * kTileN && row0 + int(threadIdx.x) < a.n)
            cp_async4(s_scale + threadIdx.x, a.scale + row0 + threadIdx.x);
    }
    pdl_launch_dependents();
    // Activations may be the previous kernel's output: wait for it.
    pdl_wait();
#pragma unroll
    for (int i = 0; i < DX; ++i)
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            xring[i][j] = make_uint4(0, 0, 0, 0);
            if (i < nmain)
                ld_act_pred(xring[i][j], xptr[j] + i * kTileK, tok_ok[j]);
        }

    // ---- stream the K part ------------------------------------------------------
    float acc[R][NT][4];
    float part[R][NT][4]; // block-scaled planes: the open column block's sum
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                acc[r][j][e] = 0.0f;
                part[r][j][e] = 0.0f;
            }

    // Blocks in ascending order.  Block b sits in weight slot b % DW and
    // activation slot b % DX; each slot is computed, then refilled (a
    // predicated load) with the block DW (weights) or DX (activations)
    // further on.
    int b = 0;
    if constexpr (kLong) {
        // The kLong copies of the 1..16-token FP8 (row- or block-scaled) and
        // one-group, one-tile MXFP4 instances, which the planner picks for K parts of at least four
        // ring groups: while every refill of a group lies inside the K part
        // (b + 2 DW <= nmain) the loads carry no predicate -- and activations
        // of tokens past m, whose sums are never stored, read token 0's row
        // instead of being masked; the last full group refills under
        // predicates.  Measured: o_proj 18.4 -> 17.8 us, MXFP4 o_proj 19.8 ->
        // 18.8 us at one token; compiled into the kernels of short K parts,
        // the second body made those 3-4 % slower, hence the separate copies.
        for (; b + 2 * DW <= nmain; b += DW) {
            if constexpr (kB128)
                factor_window<R>(fac, fac_row, fbase, (kb0 + b) >> 2, (kb0 + b + DW - 1) >> 2,
                                 lane, a.nbf);
            if (kPf > DW && lane == 0 && b + kPf < nmain) {
                const int hi = b + kPf + DW < nmain ? b + kPf + DW : nmain;
#pragma unroll
                for (int r = 0; r < R; ++r)
                    prefetch_l2(wptr[r] + (b + kPf) * kRun, uint32_t(hi - b - kPf) * kRun);
            }
#pragma unroll
            for (int i = 0; i < DW; ++i) {
                if constexpr (kB128) {
                    block_step<kW, NT, R>(part, wring[i], xring[i % DX]);
                    if ((i & 3) == 3) // kb0 and b are whole column blocks
                        close_block<NT, R>(acc, part, fac, fbase, (kb0 + b + i) >> 2);
                } else {
                    block_step<kW, NT, R>(acc, wring[i], xring[i % DX]);
                }
#pragma unroll
                for (int r = 0; r < R; ++r)
                    load_w_now<kW>(wring[i][r], wptr[r] + (b + DW + i) * kRun, soff);
#pragma unroll
                for (int j = 0; j < NT; ++j)
                    ld_act(xring[i % DX][j], xptr[j] + (b + DX + i) * kTileK);
            }
        }
    }
    for (; b + DW <= nmain; b += DW) {
        if constexpr (kB128)
            factor_window<R>(fac, fac_row, fbase, (kb0 + b) >> 2, (kb0 + b + DW - 1) >> 2, lane,
                             a.nbf);
        if (kPf > DW && lane == 0 && b + kPf < nmain) {
            const int hi = b + kPf + DW < nmain ? b + kPf + DW : nmain;
#pragma unroll
            for (int r = 0; r < R; ++r)
                prefetch_l2(wptr[r] + (b + kPf) * kRun, uint32_t(hi - b - kPf) * kRun);
        }
#pragma unroll
        for (int i = 0; i < DW; ++i) {
            if constexpr (kB128) {
                block_step<kW, NT, R>(part, wring[i], xring[i % DX]);
                if ((i & 3) == 3) // kb0 and b are whole column blocks
                    close_block<NT, R>(acc, part, fac, fbase, (kb0 + b + i) >> 2);
            } else {
                block_step<kW, NT, R>(acc, wring[i], xring[i % DX]);
            }
            const uint32_t more_w = (b + DW + i) < nmain;
#pragma unroll
            for (int r = 0; r < R; ++r)
                load_w_pred<kW>(wring[i][r], wptr[r] + (b + DW + i) * kRun, soff, more_w);
            const uint32_t more_x = (b + DX + i) < nmain;
#pragma unroll
            for (int j = 0; j < NT; ++j)
                ld_act_pred(xring[i % DX][j], xptr[j] + (b + DX + i) * kTileK,
                            tok_ok[j] & more_x);
        }
    }
    // the last partial group (fewer than DW blocks, all weights in flight)
    if constexpr (kB128)
        factor_window<R>(fac, fac_row, fbase, (kb0 + b) >> 2, (kb0 + b + DW - 1) >> 2, lane, a.nbf);
#pragma unroll
    for (int i = 0; i < DW - 1; ++i) {
        if (b + i < nmain) {
            if constexpr (kB128) {
                block_step<kW, NT, R>(part, wring[i], xring[i % DX]);
                if ((i & 3) == 3) // kb0 and b are whole column blocks
                    close_block<NT, R>(acc, part, fac, fbase, (kb0 + b + i) >> 2);
            } else {
                block_step<kW, NT, R>(acc, wring[i], xring[i % DX]);
            }
            const uint32_t more_x = (b + DX + i) < nmain;
#pragma unroll
            for (int j = 0; j < NT; ++j)
                ld_act_pred(xring[i % DX][j], xptr[j] + (b + DX + i) * kTileK,
                            tok_ok[j] & more_x);
        }
    }
    if (has_tail) {
        // the partial last block: zero activations past K (its weights past K
        // are zero-filled by the repack)
        WFrag<kW> tw[R];
        uint4 tx[NT];
#pragma unroll
        for (int r = 0; r < R; ++r)
            load_w<kW>(tw[r], wptr[r] + nmain * kRun, soff);
        const int64_t col = int64_t(kb0 + nmain) * kTileK + 8 * t;
#pragma unroll
        for (int j = 0; j < NT; ++j)
            tx[j] = load_x_tail(xptr[j] + nmain * kTileK, tok_ok[j] != 0, col, a.k);
        if constexpr (kB128)
            block_step<kW, NT, R>(part, tw, tx);
        else
            block_step<kW, NT, R>(acc, tw, tx);
    }
    // block-scaled planes: close the last column block unless the loop did
    if constexpr (kB128) {
        if (nkb > 0 && (has_tail || ((kb0 + nkb - 1) & 3) != 3)) {
            const int cb = (kb0 + nkb - 1) >> 2;
            factor_window<R>(fac, fac_row, fbase, cb, cb, lane, a.nbf);
            close_block<NT, R>(acc, part, fac, fbase, cb);
        }
    }

    // ---- K parts meet in shared memory ---------------------------------------
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                red[(((warp * R + r) * NT + j) * 4 + e) * 32 + lane] = acc[r][j][e];
    if constexpr (kFp8)
        cp_async_wait_all();
    __syncthreads();

    // One item per (tile group, r, j, e, lane): 8 * R * NT * 128 / wk items.
    // Accumulator e of lane (g, t): row g + 8*(e >> 1), token 8j + 2t + (e & 1).
    const int items = wt * R * NT * 128;
    const int64_t rows_pad = int64_t(a.rt) * kTileN;
    for (int it = threadIdx.x; it < items; it += kThreads) {
        const int ln = it & 31;
        const int e = (it >> 5) & 3;
        const int j = (it >> 7) % NT;
        const int r = ((it >> 7) / NT) % R;
        const int grp = ((it >> 7) / NT) / R;
        const int tile = rg * (wt * R) + r * wt + grp;
        const int row = tile * kTileN + (ln >> 2) + 8 * (e >> 1);
        const int tok = 8 * j + 2 * (ln & 3) + (e & 1);
        if (tile >= a.rt || tok >= a.m)
            continue;
        const float *src = red + ((((grp * wk) * R + r) * NT + j) * 4 + e) * 32 + ln;
        float v = src[0];
        for (int q = 1; q < wk; ++q)
            v += src[q * R * NT * 128];
        if (a.splits == 1) {
            if (row >= a.n)
                continue;
            const int64_t at = int64_t(tok) * a.ldy + out_col(row, a.act != kActPlain, a.half);
            if (a.act != kActSiluMul) {
                a.y[at] = to_bf16(kFp8 ? s_scale[row - row0] * v : v);
            } else if (e < 2) {
                // a gate row: its up row (row + 8) is accumulator e + 2 of this lane
                const float *su = src + 2 * 32;
                float vu = su[0];
                for (int q = 1; q < wk; ++q)
                    vu += su[q * R * NT * 128];
                a.y[at] = silu_mul_bf16(kFp8 ? s_scale[row - row0] * v : v,
                                        kFp8 ? s_scale[row + 8 - row0] * vu : vu);
            }
        } else {
            a.partial[(int64_t(sp) * rows_pad + row) * a.m + tok] = v;
        }
    }
    if (a.splits == 1)
        return;

    // ---- splits > 1: the last CTA of the row group adds the partials ---------
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

    int row_end = row0 + wt * R * kTileN;
    if (row_end > a.n)
        row_end = a.n;
    const int cnt = (row_end - row0) * a.m; // (row, token) pairs, token fastest
    const float *base = a.partial + int64_t(row0) * a.m;
    const int64_t split_stride = rows_pad * a.m;
    // the splits of one (row, token) partial, added in split order
    auto split_sum = [&](int off) {
        float v = 0.0f;
        int s = 0;
        for (; s + 8 <= a.splits; s += 8) {
            float p[8];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                p[q] = ld_cg_f32(base + (s + q) * split_stride + off);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                v += p[q];
        }
        for (; s < a.splits; ++s)
            v += ld_cg_f32(base + s * split_stride + off);
        return v;
    };
    for (int idx = threadIdx.x; idx < cnt; idx += kThreads) {
        const int row = row0 + idx / a.m;
        const int tok = idx - (idx / a.m) * a.m;
        if (a.act == kActSiluMul && (row & 8))
            continue; // an up row: added with its gate row (row - 8)
        const float v = split_sum(idx);
        const int64_t at = int64_t(tok) * a.ldy + out_col(row, a.act != kActPlain, a.half);
        if (a.act != kActSiluMul) {
            a.y[at] = to_bf16(kFp8 ? s_scale[row - row0] * v : v);
        } else {
            const float vu = split_sum(idx + 8 * a.m);
            a.y[at] = silu_mul_bf16(kFp8 ? s_scale[row - row0] * v : v,
                                    kFp8 ? s_scale[row + 8 - row0] * vu : vu);
        }
    }
    if (threadIdx.x == 0)
        a.counters[rg] = 0; // ready for the next call on this workspace
}

// ---------------------------------------------------------------------------
// instance table: one kernel per (dtype, NT, R, occupancy) with the depths of
// w8_layout.h
// ---------------------------------------------------------------------------
// Whether (dtype, token groups, row tiles per warp) has a kLong copy with
// the steady body (the copies whose registers hold it without spills).
constexpr bool has_long(int dt, int nt, int r)
{
    return nt <= 2 && (dt == kDtFp8 || dt == kDtFp8B || (is_fp4(dt) && nt == 1 && r == 1));
}

template <int kDt, int NT, int R, int OCC, bool kLong>
void *inst()
{
    constexpr int dw = depth_w_dt(NT, R, kDt, OCC), dx = depth_x_dt(NT, R, kDt, OCC);
    if constexpr (dw == 0) // a block-scaled instance that does not exist
        return nullptr;
    else if constexpr (kLong && !has_long(kDt, NT, R))
        return nullptr;
    else
        return reinterpret_cast<void *>(&gemv_kernel<kDt, NT, R, dw, dx, OCC, kLong>);
}

template <int kDt, int I, bool kLong>
void *inst_at()
{
    return inst<kDt, kInst[I].nt, kInst[I].r, kInst[I].occ, kLong>();
}

template <int kDt, bool kLong, int... Is>
void *pick_from(int idx, std::integer_sequence<int, Is...>)
{
    void *fn = nullptr;
    ((fn = (idx == Is ? inst_at<kDt, Is, kLong>() : fn)), ...);
    return fn;
}

template <int kDt>
void *pick(int nt, int r, int occ, bool lng)
{
    const int idx = inst_index(nt, r, occ);
    if (idx < 0)
        return nullptr;
    if (lng && has_long(kDt, nt, r))
        return pick_from<kDt, true>(idx, std::make_integer_sequence<int, kNumInst>{});
    return pick_from<kDt, false>(idx, std::make_integer_sequence<int, kNumInst>{});
}

void *pick_dt(int dt, int nt, int r, int occ, bool lng)
{
    return dt == kDtFp8    ? pick<kDtFp8>(nt, r, occ, lng)
           : dt == kDtFp4  ? pick<kDtFp4>(nt, r, occ, lng)
           : dt == kDtFp4Wide ? pick<kDtFp4Wide>(nt, r, occ, lng)
           : dt == kDtFp8B ? pick<kDtFp8B>(nt, r, occ, lng)
                           : pick<kDtBf16>(nt, r, occ, lng);
}

} // namespace

cudaError_t prepare_gemv_kernels()
{
    // the K-part reduction buffer: 8 warps x R x NT x 128 floats, at most 64 KB
    for (int i = 0; i < kNumInst; ++i) {
        for (int dt : {kDtBf16, kDtFp8, kDtFp4, kDtFp4Wide, kDtFp8B}) {
            for (bool lng : {false, true}) {
                void *fn = pick_dt(dt, kInst[i].nt, kInst[i].r, kInst[i].occ, lng);
                if (!fn)
                    continue;
                cudaError_t e = cudaFuncSetAttribute(
                    fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024);
                if (e != cudaSuccess)
                    return e;
            }
        }
    }
    return prepare_tc_kernels();
}

cudaError_t launch_gemv(int dt, const Plan &plan, const GemvArgs &a, cudaStream_t s)
{
    if (plan.tc)
        return is_fp4(dt) || dt == kDtFp8B ? cudaErrorInvalidValue
                                             : launch_tc(dt == kDtFp8, plan, a, s);
    void *fn = pick_dt(dt, plan.nt, plan.r, plan.occ, plan.long_k);
    if (!fn)
        return cudaErrorInvalidValue;
    void *args[] = {const_cast<GemvArgs *>(&a)};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(plan.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = size_t(plan.smem);
    cfg.stream = s;
    // programmatic dependent launch: this kernel may start while the previous
    // kernel of the stream drains; it reads no activation and writes nothing
    // before griddepcontrol.wait
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

} // namespace w8
