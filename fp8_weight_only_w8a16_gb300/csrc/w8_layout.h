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
// Weight dtypes of the kernels (the register ring reads all five; the
// tensor-memory kernel bf16 and FP8).  kDtFp8B is an FP8 plane with one fp32
// factor per kBlockB x kBlockB block instead of row scales: the FP8 codes and
// packed layout, each block's partial sum multiplied by its factor.  kDtFp4
// and kDtFp4Wide are MXFP4 planes in one packed layout; they differ in the
// bf16 factor stored beside each block's codes: 2^126 times the E8M0 scale
// (one multiply per code pair) when every scale of the plane is at most 2^1,
// else the scale alone (kDtFp4Wide: times 2^126 first, a second multiply).
constexpr int kDtBf16 = 0, kDtFp8 = 1, kDtFp4 = 2, kDtFp8B = 3, kDtFp4Wide = 4;
W8_HD constexpr bool is_fp4(int dt) { return dt == kDtFp4 || dt == kDtFp4Wide; }
constexpr int kBlockB = 128;      // rows and columns one block factor covers
constexpr int kMaxM = 256;        // tokens per call (decode steps, draft rows, prefill chunks)
constexpr int kMaxRingM = 64;     // the register-ring kernel's limit (8 token groups of 8)

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

// MXFP4 (w4a16): a (tile, block) run is 256 bytes of codes, then 8 words of
// block scales (word g = bf16 scale of row g | bf16 scale of row g+8 << 16).
// Lane (g, t) holds 8 bytes: word q for tensor-core step q, whose four A
// registers (row g, cols 8t+4q, +1), (row g+8, same), (row g, cols 8t+4q+2,
// +3), (row g+8, same) each take 8 bits -- the (low, high) elements'
// magnitude bits (mantissa, exponent low, exponent high) and sign bits -- at
// places that one shift and one mask carry to their bf16 positions (6..8 and
// 15 for the low element, 22..24 and 31 for the high one): registers 0, 1, 2
// at bit o = 0, 3, 6 (magnitude at o..o+2 and o+16..o+18, signs at o+9 and
// o+25), register 3 in the remaining bits 10, 11, 13 (magnitude), 14 (sign)
// and 26, 27, 29, 30.
constexpr int kRunFp4 = 288;
constexpr int kRunFp4Codes = 256;

// Bit offsets, inside a plane's packed MXFP4 runs, of element (row, col)'s
// mantissa, exponent-low, exponent-high and sign bits.
W8_HD void mxfp4_code_bits(int64_t k_blocks, int64_t row, int64_t col, int64_t (&bits)[4])
{
    const int64_t rt = row >> 4, kb = col >> 5;
    const int r = int(row & 15), c = int(col & 31);
    const int g = r & 7, hi = r >> 3, t = c >> 3, j = c & 7;
    const int lane = g * 4 + t;
    const int q = j >> 2, jj = j & 3;
    const int reg = (jj >> 1) * 2 + hi, half = jj & 1;
    const int64_t base = ((rt * k_blocks + kb) * kRunFp4 + lane * 8 + q * 4) * 8;
    if (reg < 3) {
        const int o = 3 * reg + 16 * half;
        bits[0] = base + o;
        bits[1] = base + o + 1;
        bits[2] = base + o + 2;
        bits[3] = base + o + 9;
    } else {
        const int o = 16 * half;
        bits[0] = base + o + 10;
        bits[1] = base + o + 11;
        bits[2] = base + o + 13;
        bits[3] = base + o + 14;
    }
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
// A CTA has kWarps warps arranged as wt tile groups x wk K parts (wt*wk = 8).
// It owns wt*R row tiles (tile group tg takes tiles tg, tg+wt, ...; each warp
// of the group holds R of them) and one range of K blocks (split sp of
// `splits`), which the wk warps of a group cut into wk contiguous parts.  Each
// warp streams its (R tiles x K part) straight from HBM into registers, D
// blocks ahead, with the matching activations from L2/L1.  The wk partial
// sums of a tile meet in shared memory and are added in K-part order.  With
// splits > 1 (only for planes with few row tiles) the CTA partials go to the
// workspace and the last CTA of a row group to arrive (an atomic counter; no
// CTA waits on another) adds them in split order.  Every sum therefore has a
// fixed order that depends only on the plan.
// ---------------------------------------------------------------------------
struct Plan {
    bool tc;         // the tensor-memory kernel (w8_tc.cu) instead of the register ring
    int npad;        // tc: tokens rounded up to 16 (the tensor-core N)
    int nt;          // 8-token groups (tensor-core N = 8): 1, 2, 4 or 8
    int r;           // row tiles per warp
    int dw;          // weight prefetch depth in K blocks (FP8 instance; see depth_w)
    int occ;         // CTAs per SM of the chosen kernel instance
    int wk;          // warps of a tile group along K: 1, 2, 4 or 8
    int64_t rt;      // row tiles of the plane
    int64_t kb;      // K blocks of the plane
    int row_groups;
    int splits;
    int cluster;     // tc: CTAs of a thread-block cluster -- the splits of a row
                     // block, whose partial tiles meet in distributed shared
                     // memory; 1 with splits > 1: they meet in the workspace
    int kbs_max;     // most K blocks one warp streams
    bool long_k;     // ring: K parts of at least four ring groups (the kernel copy
                     // with a predicate-free steady loop)
    int grid;
    int smem;        // dynamic shared memory bytes (the K-part reduction)
    size_t ws_counters; // bytes of the counter head of the workspace: one counter
                        // per row tile of the plane, whatever the plan, so that
                        // every plan of a build finds its counters in one place
    size_t ws_bytes;    // total workspace bytes (0 when splits == 1)
};

W8_HD int nt_for_m(int m) { return m <= 8 ? 1 : m <= 16 ? 2 : m <= 32 ? 4 : 8; }

// The kernel instances: a table of (token groups NT, row tiles per warp R,
// CTAs per SM OCC) with, per weight dtype, the weight ring depth DW and the
// activation ring depth DX in K blocks (DX divides DW).  Deep rings give the
// most bytes in flight per warp, higher occupancy gives more warps per SM; the
// planner picks per shape.  The depths are the only dtype-dependent choice --
// a bf16 block takes twice the registers of an FP8 block, so its ring holds
// about half the blocks and the same bytes -- and no depth changes a
// summation order.  Activations come from L2/L1; with one token group their
// ring is as deep as, or half, the weight ring: the ring refills wait an L2
// round trip, so the ring's depth, not the bandwidth, sets the pace there
// (measured: depths 16/8 -> 12/6 took fused_qkv_a_proj from 5.8 to 5.4 us).
struct Inst {
    int nt, r, occ;
    int dw_fp8, dx_fp8, dw_bf16, dx_bf16, dw_fp4, dx_fp4, dw_b128, dx_b128;
};
// (MXFP4 fragments hold 12 bytes a block against FP8's 16 but widen through
// more temporaries: the FP8 depths, except where they spill.  Block-scaled
// FP8 keeps a second set of accumulators, the open column block's sum, and
// its weight ring holds whole column blocks (a multiple of 4 K blocks): the
// nearest such depth the registers hold, or 0 -- no such instance -- where
// none does.)
constexpr int kNumInst = 10;
constexpr Inst kInst[kNumInst] = {
    {1, 1, 2, 12, 6, 8, 4, 12, 6, 12, 6}, {1, 2, 2, 6, 6, 4, 2, 6, 6, 4, 4},
    {1, 1, 3, 6, 6, 4, 2, 6, 6, 8, 2},    {1, 2, 3, 4, 4, 2, 2, 4, 4, 0, 0},
    {2, 1, 2, 10, 5, 6, 3, 8, 4, 8, 4},   {2, 2, 2, 6, 3, 2, 2, 6, 3, 4, 2},
    {4, 1, 2, 6, 2, 4, 2, 6, 2, 4, 1},    {4, 2, 1, 8, 4, 4, 2, 8, 4, 8, 4},
    {8, 1, 1, 6, 2, 4, 2, 6, 2, 4, 2},    {8, 2, 1, 6, 2, 4, 2, 6, 2, 0, 0},
};
constexpr int inst_index(int nt, int r, int occ)
{
    for (int i = 0; i < kNumInst; ++i)
        if (kInst[i].nt == nt && kInst[i].r == r && kInst[i].occ == occ)
            return i;
    return -1;
}
constexpr int depth_w(int nt, int r, bool fp8, int occ)
{
    return fp8 ? kInst[inst_index(nt, r, occ)].dw_fp8 : kInst[inst_index(nt, r, occ)].dw_bf16;
}
constexpr int depth_x(int nt, int r, bool fp8, int occ)
{
    return fp8 ? kInst[inst_index(nt, r, occ)].dx_fp8 : kInst[inst_index(nt, r, occ)].dx_bf16;
}
// The depths of one kernel dtype (kDtBf16, kDtFp8, kDtFp4, kDtFp4Wide, kDtFp8B); 0 for a
// block-scaled instance that does not exist.
constexpr int depth_w_dt(int nt, int r, int dt, int occ)
{
    return is_fp4(dt)      ? kInst[inst_index(nt, r, occ)].dw_fp4
           : dt == kDtFp8B ? kInst[inst_index(nt, r, occ)].dw_b128
                           : depth_w(nt, r, dt == kDtFp8, occ);
}
constexpr int depth_x_dt(int nt, int r, int dt, int occ)
{
    return is_fp4(dt)      ? kInst[inst_index(nt, r, occ)].dx_fp4
           : dt == kDtFp8B ? kInst[inst_index(nt, r, occ)].dx_b128
                           : depth_x(nt, r, dt == kDtFp8, occ);
}

inline int64_t plan_ctas(int64_t rt, int r, int wk, int splits)
{
    const int64_t tiles_per_cta = int64_t(kWarps / wk) * r;
    return ceil_div(rt, tiles_per_cta) * splits;
}

// Choose (occupancy, wk, R): the fewest waves, then the most weight bytes in
// flight, then the most resident warps, then the higher occupancy, then R = 2
// (activations reused over two tiles), then the longest K parts.  Every warp keeps at least kMinBlocks
// K blocks when K allows it.  K is split across CTAs only for planes whose
// row tiles leave most SMs idle.
// The tensor-memory kernel (w8_tc.cu): CTAs of 128 rows x a K range, eleven
// warps.  Up to 64 tokens: 2 CTAs per SM (256 tensor-memory columns and about
// 100 KB of shared memory each), or at 49..64 tokens 1 CTA per SM with deeper
// rings where one wave of such CTAs fills the SMs; from 65 to 256 tokens
// (padded to 96, 128, 192 or 256): 1 CTA per SM (512 columns: the
// accumulator, then A stages; about 200 KB).  K is split across the CTAs of
// a cluster (up to 8) until about the resident CTAs are busy, keeping at
// least one stage of K blocks per split; the partial sums meet in
// distributed shared memory -- or, on planes of few row blocks up to 64
// tokens, K is split into more ranges whose partial sums meet in the
// workspace.
constexpr int kTcMinM = 17;       // decode tokens from which the tc kernel may run
constexpr int kTcMinRowBlocks = 48; // ... on planes of at least this many 128-row blocks
constexpr int kTcStageBlocks = 4; // K blocks per stage of the tc kernel
constexpr int kTcCtasPerSm = 2;
constexpr int kTcThreadsPerCta = 352;

// Token paddings of the tensor-memory kernel (its MMA N): steps of 16 up to
// 64, then 96, 128, 192, 256.
W8_HD constexpr int tc_npad(int m)
{
    return m <= 64 ? int((m + 15) / 16) * 16 : m <= 96 ? 96 : m <= 128 ? 128 : m <= 192 ? 192 : 256;
}
W8_HD constexpr int tc_occ(int npad) { return npad <= 64 ? kTcCtasPerSm : 1; }

// Stage slots of the tensor-memory kernel in shared memory: nw weight stages
// (8 row tiles x 4 K blocks of packed runs, filled by bulk copies) and nb
// activation stages (4 K blocks x npad tokens): about 100 KB per CTA up to 64
// tokens (two CTAs share an SM), about 200 KB above.  At 64 tokens a second
// instance runs one CTA per SM (occ 1) with deeper rings, 192 KB: 8 FP8 or 4
// bf16 weight stages of 4 K blocks, and 4 activation stages (measured on
// o_proj bf16 at 64 tokens: 56.1 us with 2 + 2 bf16 stages, 52.6 with 4 + 4,
// 51.6 with 3 + 4; q_b 20.2, 19.6, 19.9).
struct TcStages {
    int nw, nb;
};
W8_HD constexpr TcStages tc_stages(bool fp8, int npad, int occ)
{
    return (occ == 1 && npad == 64) ? (fp8 ? TcStages{8, 4} : TcStages{4, 4})
         : fp8 ? (npad <= 16 ? TcStages{5, 6} : npad <= 32 ? TcStages{4, 5}
                  : npad <= 48 ? TcStages{4, 3} : npad <= 64 ? TcStages{3, 3}
                  : npad <= 96 ? TcStages{5, 5} : npad <= 128 ? TcStages{5, 4}
                  : npad <= 192 ? TcStages{4, 3} : TcStages{4, 2})
               : (npad <= 16 ? TcStages{3, 2} : npad <= 32 ? TcStages{2, 4}
                  : npad <= 48 ? TcStages{2, 3} : npad <= 64 ? TcStages{2, 2}
                  : npad <= 96 ? TcStages{3, 4} : npad <= 128 ? TcStages{3, 3}
                  : npad <= 192 ? TcStages{2, 3} : TcStages{2, 2});
}
// Dynamic shared memory of a CTA: the stages, plus room to start them on a
// 1024-byte boundary (the activation stages' swizzle atoms).
constexpr int kTcSmemAlign = 1024;
W8_HD constexpr int tc_smem_bytes(bool fp8, int npad, int occ)
{
    return tc_stages(fp8, npad, occ).nw * 8 * 4 * (fp8 ? kRunFp8 : kRunBf16) +
           tc_stages(fp8, npad, occ).nb * 4 * npad * 64 + kTcSmemAlign;
}
constexpr int kTcMaxSplits = 8;  // CTAs per cluster (the portable cluster size)
constexpr int kTcMaxGlobalSplits = 8; // K ranges of a row block that meet in the workspace
constexpr int kTcMinGlobalSplitBlocks = 32; // ... each at least this many K blocks (8 stages),
                                            // so that the stream outweighs the reduction

// The tensor-memory plan for occ CTAs per SM.
inline Plan make_tc_plan_occ(int64_t n, int64_t k, int m, int sm_count, int occ)
{
    Plan p{};
    p.tc = true;
    p.npad = tc_npad(m);
    p.nt = p.npad / 8;
    p.r = 8;  // row tiles per CTA
    p.dw = tc_stages(true, p.npad, occ).nw * kTcStageBlocks; // weight blocks staged ahead (FP8)
    p.occ = occ;
    p.wk = 1;
    p.rt = ceil_div(n, kTileN);
    p.kb = ceil_div(k, kTileK);
    const int64_t rbs = ceil_div(n, 128);
    const int64_t target = int64_t(sm_count > 0 ? sm_count : 1) * p.occ;
    // the splits of a row block form one thread-block cluster: a power of two
    // up to 8 (the portable cluster size) that keeps one stage per split
    // Powers of two until about the resident CTAs are busy.  (Counts of 3 or
    // 6 that would fill every SM with one CTA each measured slower: o_proj at
    // 96 tokens 49.5 -> 68.8 us with clusters of 6, the clusters not all
    // resident at once.)
    int splits = 1;
    while (splits < kTcMaxSplits && rbs * splits * 2 <= target &&
           p.kb / (int64_t(splits) * 2) >= kTcStageBlocks)
        splits *= 2;
    p.cluster = splits;
    p.ws_counters = p.ws_bytes = 0; // partial sums stay on chip (cluster exchange)
    // Planes of few row blocks (o_proj's 48): the power-of-two cluster splits
    // leave SMs idle (96 CTAs on 152 SMs) or some SMs with one CTA more than
    // the rest (192), which end long after the others.  Where more K ranges
    // fit the resident slots, split K into that many instead and add the
    // partial tiles through the workspace (the last CTA of a row block to
    // arrive), so that no cluster has to be placed whole: up to
    // kTcMaxGlobalSplits, each range at least kTcMinGlobalSplitBlocks; up to
    // 64 tokens only, where the last CTA's reduction (128 rows x the tokens x
    // the splits) stays short.  Measured: o_proj 36.4 -> 28.8 us at 17 tokens,
    // 38.1 -> 31.8 at 32, 53.7 -> 52.3 at 64; above 64 tokens the reduction
    // cost more than the balance gained (6144 x 4096 at 96 tokens 21.3 ->
    // 32.0 us).
    int64_t sg = target / rbs;
    if (sg > kTcMaxGlobalSplits)
        sg = kTcMaxGlobalSplits;
    while (sg > 1 && p.kb / sg < kTcMinGlobalSplitBlocks)
        --sg;
    if (sg > splits && p.npad <= 64) {
        splits = int(sg);
        p.cluster = 1;
        p.ws_counters = align256(size_t(p.rt) * sizeof(int));
        p.ws_bytes = p.ws_counters + align256(size_t(splits) * size_t(p.rt) * kTileN *
                                              size_t((m + 3) & ~3) * sizeof(float));
    }
    p.splits = splits;
    p.row_groups = int(rbs);
    p.grid = int(rbs * splits);
    p.kbs_max = int(ceil_div(p.kb, splits));
    p.smem = tc_smem_bytes(true, p.npad, occ); // the FP8 instance (bf16: its own table)
    return p;
}

// At 49..64 tokens, one CTA per SM with the deeper ring where one wave of
// those CTAs, each on its own K range with no cluster, covers at least 3/4
// of the SMs (o_proj's 48 row blocks x 3 K ranges = 144 CTAs, q_b's 128 row
// blocks); two CTAs per SM otherwise.  Measured on 152 SMs: o_proj FP8 at 64
// tokens 52.4 -> 46.7 us, bf16 59.5 -> 52.6, q_b 18.6 -> 17.3; the same
// instance below 49 tokens was slower (o_proj at 32 tokens 31.9 -> 36.4), and
// on planes of more row blocks than SMs (kv_b's 224: two waves) much slower.
inline Plan make_tc_plan(int64_t n, int64_t k, int m, int sm_count)
{
    if (tc_npad(m) == 64) {
        const Plan d = make_tc_plan_occ(n, k, m, sm_count, 1);
        const int64_t sms = sm_count > 0 ? sm_count : 1;
        if (d.cluster == 1 && d.grid <= sms && 4 * int64_t(d.grid) >= 3 * sms)
            return d;
    }
    return make_tc_plan_occ(n, k, m, sm_count, tc_occ(tc_npad(m)));
}

// Which kernel a shape gets (measured on GB300 over the GLM-5.2 projections):
// the tensor-memory kernel wins from 17 tokens on planes with many row blocks
// (o_proj, q_b, kv_b), where one activation tile serves 128 rows; the register
// ring wins below that and on planes with few rows, where the tc kernel's
// fixed cost per CTA and its cluster reduction dominate.  Above 64 tokens
// only the tensor-memory kernel runs.
inline bool use_tc(int64_t n, int m)
{
    return m > kMaxRingM || (m >= kTcMinM && ceil_div(n, 128) >= kTcMinRowBlocks);
}

// The register-ring plan (1..64 tokens), for every dtype; MXFP4 and
// block-scaled planes run only this kernel.  The plan is the same for every
// dtype, except that block-scaled planes (b128) choose among the instances
// that exist for them, scored with their own ring depths.
inline Plan make_ring_plan(int64_t n, int64_t k, int m, int sm_count, bool b128 = false)
{
    Plan p{};
    p.nt = nt_for_m(m);
    p.rt = ceil_div(n, kTileN);
    p.kb = ceil_div(k, kTileK);
    const int sms = sm_count > 0 ? sm_count : 1;
    const int64_t kMinBlocks = 8;

    bool have = false;
    int64_t best_waves = 0, best_inflight = 0, best_warps = 0, best_bpw = 0;
    int best_r = 1, best_wk = 1, best_occ = 1;
    for (int ii = 0; ii < kNumInst; ++ii) {
        if (kInst[ii].nt != p.nt || (b128 && kInst[ii].dw_b128 == 0))
            continue;
        const int occ = kInst[ii].occ, r = kInst[ii].r;
        const int64_t slots = int64_t(sms) * occ;
        {
            for (int wk = 8; wk >= 1; wk /= 2) {
                const int64_t bpw = p.kb / wk;
                if (wk > 1 && bpw < kMinBlocks)
                    continue;
                const int64_t ctas = plan_ctas(p.rt, r, wk, 1);
                const int64_t waves = ceil_div(ctas, slots);
                const int64_t resident = ctas < slots ? ctas : slots;
                const int64_t dw = b128 ? kInst[ii].dw_b128 : depth_w(p.nt, r, true, occ);
                // only row tiles that exist are streamed: a plane with fewer
                // tiles than its CTAs hold leaves the other warps idle
                const int64_t cta_tiles = int64_t(kWarps / wk) * r;
                const int64_t tiles = resident * cta_tiles < p.rt ? resident * cta_tiles : p.rt;
                const int64_t inflight = tiles * wk * (bpw < dw ? bpw : dw) * kRunFp8;
                const int64_t warps = ceil_div(tiles, r) * wk;
                bool better;
                if (!have)
                    better = true;
                else if (waves != best_waves)
                    better = waves < best_waves;
                else if (inflight != best_inflight)
                    better = inflight > best_inflight;
                else if (warps != best_warps)
                    better = warps > best_warps;
                else if (occ != best_occ)
                    better = occ > best_occ;
                else if (r != best_r)
                    better = r > best_r;
                else
                    better = bpw > best_bpw;
                if (better) {
                    have = true;
                    best_waves = waves;
                    best_inflight = inflight;
                    best_warps = warps;
                    best_bpw = bpw;
                    best_r = r;
                    best_wk = wk;
                    best_occ = occ;
                }
            }
        }
    }
    p.r = best_r;
    p.wk = best_wk;
    p.occ = best_occ;
    p.dw = depth_w_dt(p.nt, p.r, b128 ? kDtFp8B : kDtFp8, p.occ);
    int splits = 1;
    while (plan_ctas(p.rt, p.r, p.wk, splits) * 2 <= sms &&
           p.kb / (int64_t(p.wk) * splits * 2) >= 4)
        splits *= 2;
    p.splits = splits;
    p.row_groups = int(ceil_div(p.rt, int64_t(kWarps / p.wk) * p.r));
    p.grid = p.row_groups * p.splits;
    p.kbs_max = int(ceil_div(ceil_div(p.kb, p.splits), p.wk));
    p.long_k = p.kbs_max >= 4 * p.dw;
    p.smem = kWarps * p.r * p.nt * 4 * 32 * int(sizeof(float));
    if (p.splits > 1) {
        p.ws_counters = align256(size_t(p.rt) * sizeof(int));
        p.ws_bytes = p.ws_counters + align256(size_t(p.splits) * size_t(p.rt) * kTileN *
                                              size_t(m) * sizeof(float));
    } else {
        p.ws_counters = 0;
        p.ws_bytes = 0;
    }
    return p;
}

inline Plan make_plan(int64_t n, int64_t k, int m, int sm_count)
{
    return use_tc(n, m) ? make_tc_plan(n, k, m, sm_count) : make_ring_plan(n, k, m, sm_count);
}

} // namespace w8
