// w8_internal.h -- what the C-ABI layer (w8_api.cu) hands to the kernels.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "w8.h"
#include "w8_layout.h"

// The library-owned host handle behind the opaque w8_build of include/w8.h.
struct w8_build {
    int device;
    int sm_count;
    int32_t dtype;
    size_t ws_counters; // the workspace's counter head for every call of the build:
                        // one counter per row tile of its largest plane
    std::vector<w8_plane_info> planes;
    std::vector<int> kdt; // each plane's kernel dtype (w8_layout.h)
};

// Workspace bytes a call with this plan needs on this build: the build's
// counter head, then the plan's partial sums (0 when the plan needs none).
inline size_t build_ws_bytes(const w8_build *b, size_t plan_ws_bytes, size_t plan_ws_counters)
{
    return plan_ws_bytes == 0 ? 0 : b->ws_counters + (plan_ws_bytes - plan_ws_counters);
}

namespace w8 {

// What a gemv call writes (GemvArgs::act).  A gate_up plane is a merged
// [2I, K] projection whose source rows 0..I-1 are the gate and I..2I-1 the
// up projection; bind interleaves them so that packed 16-row tile t holds
// gate rows 8t..8t+7 followed by up rows 8t..8t+7.
constexpr int kActPlain = 0;   // y[:, n] for packed row n (a plain plane)
constexpr int kActGateUp = 1;  // a gate_up plane's plain GEMV, y in source row order
constexpr int kActSiluMul = 2; // a gate_up plane: y[:, j] = bf16(silu(g_j) * u_j), j < I

struct GemvArgs {
    const uint8_t *wp;      // packed weights of the plane (device)
    const float *scale;     // the build's row scales (FP8) or nullptr (bf16)
    const uint16_t *x;      // [m][ldx] bf16
    int64_t ldx;
    uint16_t *y;            // [m][ldy] bf16
    int64_t ldy;
    int n, k, m;
    int kb;                 // K blocks
    int rt;                 // row tiles
    int splits;
    int wk;                 // warps of a tile group along K
    int *counters;          // workspace head (splits > 1)
    float *partial;         // workspace body: [splits][rt*16][m] fp32 (splits > 1)
    int act;                // kActPlain, kActGateUp or kActSiluMul
    int half;               // gate_up planes: I = n / 2
    const float *bfac;      // block-scaled FP8: the build's factors [ceil(n/128)][nbf]
    int nbf;                // block-scaled FP8: column blocks, ceil(k / 128)
    int gsplit;             // tc, splits > 1: the partial tiles meet in the workspace
                            // (counters, partial) instead of a cluster's shared memory
};

// The output mapping of a plane: gate_up planes (bound with W8_SRC_GATE_UP)
// store in source row order, or apply SiLU-and-multiply when silu is set.
inline void set_output_map(GemvArgs &a, const w8_plane_info &p, bool silu)
{
    const bool gated = p.layout == W8_LAYOUT_MMA_16x32_GATE_UP;
    a.act = gated ? (silu ? kActSiluMul : kActGateUp) : kActPlain;
    a.half = gated ? int(p.n / 2) : 0;
}

// One launch of the GEMV kernel chosen by the plan; dt is the weight dtype
// (kDtBf16, kDtFp8, kDtFp4, kDtFp4Wide or kDtFp8B of w8_layout.h; MXFP4 and
// block-scaled plans are register-ring plans).
cudaError_t launch_gemv(int dt, const Plan &plan, const GemvArgs &a, cudaStream_t s);

// Raise the dynamic shared-memory limit of every GEMV kernel instance on the
// current device (called once per device before the first launch).
cudaError_t prepare_gemv_kernels();

// The tensor-memory kernel (w8_tc.cu), which launch_gemv runs for plan.tc.
cudaError_t launch_tc(bool fp8, const Plan &plan, const GemvArgs &a, cudaStream_t s);
cudaError_t prepare_tc_kernels();
// Read (and optionally clear) the tc kernel's device status word.
cudaError_t tc_status(int *out, bool reset);

struct RepackArgs {
    const uint8_t *src;     // source plane (device), row-major
    int64_t ld_bytes;       // source row stride in bytes
    int64_t n, k;
    int64_t kb, rt;
    uint8_t *dst;           // packed weights (device)
    const float *scale_src; // FP8: caller's row scales (device); NULL for block-scaled
                            // FP8, whose row scales are 1
    float *scale_dst;       // FP8 and block-scaled FP8: the build's copy, rt*16 entries
    int64_t half;           // 0, or I for a gate_up plane (n = 2I, I % 8 == 0):
                            // packed row 16t+i reads source row 8t+i (i < 8)
                            // or I + 8t + i - 8 (i >= 8)
    const uint8_t *bscale_src; // MXFP4: caller's E8M0 block scales [n][ldb] (device)
    int64_t ldb;            // row stride of the block scales (MXFP4: bytes; block-scaled
                            // FP8: floats)
    const float *bfac_src;  // block-scaled FP8: caller's factors [ceil(n/128)][ldb] (device)
    float *bfac_dst;        // block-scaled FP8: the build's copy [ceil(n/128)][ceil(k/128)]
    bool fp4_fold;          // MXFP4: store 2^126 x each scale (kDtFp4), else the scale
                            // (kDtFp4Wide)
};

// MXFP4: whether any block scale of the plane is past 2^1 (E8M0 129..254), so
// that the plane needs kDtFp4Wide.  Uses 4 bytes of device scratch and
// synchronises s (bind time).
cudaError_t fp4_scales_wide(const RepackArgs &a, unsigned *scratch, bool *wide, cudaStream_t s);

// The repack of one plane (dt: kDtBf16, kDtFp8, kDtFp4, kDtFp4Wide or kDtFp8B).
cudaError_t launch_repack(int dt, const RepackArgs &a, cudaStream_t s);

} // namespace w8
