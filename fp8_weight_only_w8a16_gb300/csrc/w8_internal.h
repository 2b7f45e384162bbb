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
    std::vector<w8_plane_info> planes;
};

namespace w8 {

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
};

// One launch of the GEMV kernel chosen by the plan (FP8 or bf16 weights).
cudaError_t launch_gemv(bool fp8, const Plan &plan, const GemvArgs &a, cudaStream_t s);

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
    const float *scale_src; // FP8: caller's row scales (device)
    float *scale_dst;       // FP8: the build's copy, rt*16 entries (device)
};

cudaError_t launch_repack(bool fp8, const RepackArgs &a, cudaStream_t s);

} // namespace w8
