// w8_layout.h -- the packed weight layout and the launch planner of libw8.
//
// Packed layout W8_LAYOUT_MMA_16x32 (see include/w8.h).  The weight plane is
// cut into row tiles of 16 rows and K blocks of 32 columns.  Tile rt, block kb
// is one contiguous run, tiles outer, blocks inner:
//
//   FP8 : run = 512 bytes  = 32 lanes x 16 bytes
//   bf16: run = 1024 bytes = 2 halves x 32 lanes x 16 bytes
//
// so a warp streams a row tile with one fully coalesced 16-byte load per lane
// per block (two for bf16).  Inside a run, lane L = 4*g + t holds rows g and
// g+8 of the tile and columns 8t..8t+7 of the block.  Those 8 columns feed two
// m16n8k16 tensor-core steps: columns 8t+0..3 the first, 8t+4..7 the second.
// In each step the lane's four k slots (2t, 2t+1, 2t+8, 2t+9 in the
// instruction's own numbering) carry columns +0, +1, +2, +3, so the lane's B
// operand (8 consecutive activations x[token][8t..8t+7]) is one 16-byte load.
//
// A operand registers of one step: a01 = (row g, cols +0,+1), a23 = (row g+8,
// cols +0,+1), a45 = (row g, cols +2,+3), a67 = (row g+8, cols +2,+3).
//   bf16: the lane's 16 bytes of half q are exactly a01 a23 a45 a67 of step q.
//   FP8 : the lane's 16 bytes are 4 words; word 2q+h serves step q, columns
//         +2h,+2h+1; its bytes are (row g, even col), (row g+8, even col),
//         (row g, odd col), (row g+8, odd col), so bytes 0 and 2 widen to the
//         row-g register and bytes 1 and 3 to the row-(g+8) register.
#pragma once

#include <stddef.h>
#include <stdint.h>

#ifdef __CUDACC__
#define W8_HD __host__ __device__ __forceinline__
#else
#define W8_HD inline
#endif

namespace w8 {

constexpr int kTileN = 16;        // rows per tile (tensor-core M)
constexpr int kTileK = 32;        // columns per block (two k16 steps)
constexpr int kRunFp8 = 512;      // bytes of one (tile, block) run, FP8
constexpr int kRunBf16 = 1024;    // bytes of one (tile, block) run, bf16
constexpr int kWarps = 8;         // warps per CTA of the GEMV kernel
constexpr int kThreads = kWarps * 32;
constexpr int kMaxM = 64;         // decode tokens per call

W8_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
W8_HD size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

// Byte offset of element (row, col) inside one plane's packed weights.
W8_HD int64_t packed_offset_fp8(int64_t k_blocks, int64_t row, int64_t col)
{
    const int64_t rt = row >> 4, kb = col >> 5;
    const int r = int(row & 15), c = int(col & 31);
    const int g = r & 7, hi = r >> 3, t = c >> 3, j = c & 7;
    const int lane = g * 4 + t;
    const int q = j >> 2, jj = j & 3;
    const int word = q * 2 + (jj >> 1);
    const int byte = word * 4 + hi + ((jj & 1) << 1);
    return ((rt * k_blocks + kb) * 32 + lane) * 16 + byte;
}

W8_HD int64_t packed_offset_bf16(int64_t k_blocks, int64_t row, int64_t col)
{
    const int64_t rt = row >> 4, kb = col >> 5;
    const int r = int(row & 15), c = int(col & 31);
    const int g = r & 7, hi = r >> 3, t = c >> 3, j = c & 7;
    const int lane = g * 4 + t;
    const int q = j >> 2, jj = j & 3;
    const int reg = (jj >> 1) * 2 + hi;
    const int elem = reg * 2 + (jj & 1);
    return ((rt * k_blocks + kb) * 2 + q) * 512 + lane * 16 + elem * 2;
}

// ---------------------------------------------------------------------------
// Launch plan.  A function of (N, K, m, SM count) only -- never of the weight
// dtype -- so FP8 and bf16 planes of one shape sum in the same order.
//
// The grid is row_groups x splits CTAs.  A CTA owns kWarps*R row tiles (warp w
// takes tiles w, w+8, ...) and one contiguous range of K blocks; it stages
// that range of x in shared memory once and streams its weight runs straight
// into registers.  With splits > 1 each CTA writes fp32 partial sums to the
// workspace and the last CTA of a row group to arrive (an atomic counter; no
// CTA ever waits on another) adds them in split order, scales and rounds.
// ---------------------------------------------------------------------------
struct Plan {
    int nt;          // 8-token groups (tensor-core N = 8): 1, 2, 4 or 8
    int r;           // row tiles per warp
    int d;           // prefetch depth in blocks
    int ctas_per_sm; // occupancy the kernel is built for
    int64_t rt;      // row tiles of the plane
    int64_t kb;      // K blocks of the plane
    int row_groups;
    int splits;
    int kbs_max;     // most K blocks in one split
    int grid;
    int smem;        // dynamic shared memory bytes
    int x_stride;    // bytes between token rows of the staged x
    size_t ws_counters; // bytes of the counter head of the workspace
    size_t ws_bytes;    // total workspace bytes (0 when splits == 1)
};

W8_HD int nt_for_m(int m) { return m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8; }
W8_HD int r_for_nt(int nt) { return nt <= 2 ? 1 : 2; }
W8_HD int d_for_nt(int nt) { return nt <= 2 ? 8 : 4; }
W8_HD int ctas_per_sm_for_nt(int nt) { return nt <= 2 ? 2 : 1; }

// Token rows of the staged x are kbs*64 bytes long; the stride is padded so
// that it is 64 modulo 128 and the lanes' 16-byte reads hit distinct banks.
W8_HD int x_stride_bytes(int kbs) { return kbs * 64 + ((kbs & 1) ? 0 : 64); }

inline Plan make_plan(int64_t n, int64_t k, int m, int sm_count)
{
    Plan p{};
    p.nt = nt_for_m(m);
    p.r = r_for_nt(p.nt);
    p.d = d_for_nt(p.nt);
    p.ctas_per_sm = ctas_per_sm_for_nt(p.nt);
    p.rt = ceil_div(n, kTileN);
    p.kb = ceil_div(k, kTileK);
    const int64_t tiles_per_cta = int64_t(kWarps) * p.r;
    p.row_groups = int(ceil_div(p.rt, tiles_per_cta));

    const int smem_budget = (p.ctas_per_sm == 2 ? 100 : 200) * 1024;
    // largest split whose staged x fits the budget
    int kbs_cap = 1;
    while (kbs_cap < p.kb && p.nt * 8 * x_stride_bytes(kbs_cap + 1) <= smem_budget)
        ++kbs_cap;
    const int64_t s_min = ceil_div(p.kb, kbs_cap);

    const int64_t target = int64_t(sm_count > 0 ? sm_count : 1) * p.ctas_per_sm;
    int64_t s = (target + p.row_groups / 2) / p.row_groups; // round(target / row_groups)
    const int64_t s_cap = p.kb / 4 > 1 ? p.kb / 4 : 1;     // keep >= 4 blocks per split
    if (s > s_cap) s = s_cap;
    if (s < 1) s = 1;
    if (s < s_min) s = s_min;
    if (s > p.kb) s = p.kb;
    p.splits = int(s);
    p.kbs_max = int(ceil_div(p.kb, s));
    p.grid = p.row_groups * p.splits;
    p.x_stride = x_stride_bytes(p.kbs_max);
    p.smem = p.nt * 8 * p.x_stride;
    if (p.splits > 1) {
        p.ws_counters = align256(size_t(p.row_groups) * sizeof(int));
        p.ws_bytes = p.ws_counters + align256(size_t(p.splits) * size_t(p.rt) * kTileN *
                                              size_t(m) * sizeof(float));
    } else {
        p.ws_counters = 0;
        p.ws_bytes = 0;
    }
    return p;
}

} // namespace w8
