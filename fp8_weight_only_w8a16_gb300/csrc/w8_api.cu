// w8_api.cu -- the C ABI of libw8 (declared and documented in include/w8.h).
//
// Host-side validation and binding follow the refusals of ATOM PR #2980
// (Changes and Limitations): a plane in any 8-bit format other than E4M3fn,
// a row stride or base that is not 16-byte aligned, a bias, and a build that
// mixes bf16 with FP8 are turned away at bind.  The gemv entry points take
// the same arguments for every weight dtype; the FP8 row scales travel with
// the build and reach the kernel after the other arguments, so the bf16
// call's arguments are those of the FP8 one without them (the PR appends the
// scales in the same way).
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <new>
#include <vector>

#include "w8.h"
#include "w8_internal.h"

namespace {

constexpr int64_t kMaxDim = int64_t(1) << 30;

int elem_bytes(int32_t dtype) { return dtype == W8_DT_BF16 ? 2 : 1; }

// Bytes of a row of ldw elements (MXFP4: two elements a byte).
int64_t row_bytes(int32_t dtype, int64_t ldw)
{
    return dtype == W8_DT_MXFP4 ? ldw / 2 : ldw * elem_bytes(dtype);
}

// The kernels' dtype of a plane dtype.
int kernel_dt(int32_t dtype)
{
    return dtype == W8_DT_E4M3FN        ? w8::kDtFp8
           : dtype == W8_DT_MXFP4       ? w8::kDtFp4
           : dtype == W8_DT_E4M3FN_B128 ? w8::kDtFp8B
                                        : w8::kDtBf16;
}

// Planes whose factors vary along K (MXFP4, block-scaled FP8) run the
// register ring only.
bool ring_only(int32_t dtype) { return dtype == W8_DT_MXFP4 || dtype == W8_DT_E4M3FN_B128; }

// The launch plan of a plane's dtype.
w8::Plan plan_for(int32_t dtype, int64_t n, int64_t k, int m, int sms)
{
    return ring_only(dtype) ? w8::make_ring_plan(n, k, m, sms, dtype == W8_DT_E4M3FN_B128)
                            : w8::make_plan(n, k, m, sms);
}

int max_m(int32_t dtype) { return ring_only(dtype) ? w8::kMaxRingM : w8::kMaxM; }

// FP8 planes with row scales (E4M3FN) or block factors (E4M3FN_B128): both
// carry fp32 factors in `scale` and run through w8_gemv.
bool fp8_codes(int32_t dtype) { return dtype == W8_DT_E4M3FN || dtype == W8_DT_E4M3FN_B128; }

w8_status check_plane(const w8_plane_desc &d)
{
    if (!d.w)
        return W8_ERR_NULL;
    if (d.dtype != W8_DT_E4M3FN && d.dtype != W8_DT_BF16 && d.dtype != W8_DT_MXFP4 &&
        d.dtype != W8_DT_E4M3FN_B128)
        return W8_ERR_DTYPE;
    if (d.layout != W8_SRC_ROW_MAJOR && d.layout != W8_SRC_GATE_UP)
        return W8_ERR_LAYOUT;
    if (d.layout == W8_SRC_GATE_UP && d.dtype == W8_DT_E4M3FN_B128)
        return W8_ERR_LAYOUT; // a tile would hold gate and up rows of two row blocks
    if (d.bias)
        return W8_ERR_BIAS;
    if (d.n < 1 || d.k < 1 || d.n > kMaxDim || d.k > kMaxDim || d.ldw < d.k ||
        d.ldw > 4 * kMaxDim)
        return W8_ERR_SHAPE;
    if (d.layout == W8_SRC_GATE_UP && d.n % (2 * 8) != 0)
        return W8_ERR_SHAPE; // I = n / 2 gate rows, a multiple of 8
    if (fp8_codes(d.dtype) && !d.scale)
        return W8_ERR_SCALE;
    if (!fp8_codes(d.dtype) && d.scale)
        return W8_ERR_SCALE;
    if (d.dtype == W8_DT_E4M3FN_B128 && d.ldb < w8::ceil_div(d.k, w8::kBlockB))
        return W8_ERR_SCALE;
    if (d.dtype == W8_DT_MXFP4 && (!d.block_scale || d.ldb < w8::ceil_div(d.k, 32)))
        return W8_ERR_SCALE;
    if (d.dtype != W8_DT_MXFP4 && d.block_scale)
        return W8_ERR_SCALE;
    if ((reinterpret_cast<uintptr_t>(d.w) & 15u) != 0 || (d.dtype == W8_DT_MXFP4 && (d.ldw & 1)) ||
        (row_bytes(d.dtype, d.ldw) & 15) != 0)
        return W8_ERR_UNPADDED;
    return W8_OK;
}

size_t plane_packed_bytes(int32_t dtype, int64_t n, int64_t k)
{
    const int64_t rt = w8::ceil_div(n, w8::kTileN), kb = w8::ceil_div(k, w8::kTileK);
    return size_t(rt) * size_t(kb) *
           size_t(dtype == W8_DT_BF16 ? w8::kRunBf16 : dtype == W8_DT_MXFP4 ? w8::kRunFp4 : w8::kRunFp8);
}

size_t plane_scale_bytes(int32_t dtype, int64_t n)
{
    if (!fp8_codes(dtype))
        return 0;
    return size_t(w8::ceil_div(n, w8::kTileN)) * w8::kTileN * sizeof(float);
}

// The build's copy of a block-scaled plane's factors: [ceil(n/128)][ceil(k/128)].
size_t plane_factor_bytes(int32_t dtype, int64_t n, int64_t k)
{
    if (dtype != W8_DT_E4M3FN_B128)
        return 0;
    return size_t(w8::ceil_div(n, w8::kBlockB)) * size_t(w8::ceil_div(k, w8::kBlockB)) *
           sizeof(float);
}

// want_dtype 0: either dtype (SiLU-and-multiply serves both).
w8_status gemv_common(const w8_build *b, int plane, int32_t want_dtype, bool silu,
                      const uint16_t *x, int64_t ldx, int m, uint16_t *y, int64_t ldy, void *ws,
                      size_t ws_bytes, w8_stream s)
{
    if (!b)
        return W8_ERR_NULL;
    if (plane < 0 || plane >= int(b->planes.size()))
        return W8_ERR_PLANE;
    const w8_plane_info &p = b->planes[size_t(plane)];
    if (want_dtype != 0 && p.dtype != want_dtype &&
        !(want_dtype == W8_DT_E4M3FN && p.dtype == W8_DT_E4M3FN_B128))
        return W8_ERR_DTYPE;
    if (silu && p.layout != W8_LAYOUT_MMA_16x32_GATE_UP)
        return W8_ERR_LAYOUT;
    if (m < 0 || m > max_m(p.dtype))
        return W8_ERR_SHAPE;
    if (m == 0)
        return W8_OK;
    if (!x || !y)
        return W8_ERR_NULL;
    if (ldx < p.k || ldy < (silu ? p.n / 2 : p.n))
        return W8_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (ldx & 7) || (reinterpret_cast<uintptr_t>(y) & 1u))
        return W8_ERR_ALIGN;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return W8_ERR_CUDA;
    if (dev != b->device)
        return W8_ERR_DEVICE;

    const w8::Plan plan = plan_for(p.dtype, p.n, p.k, m, b->sm_count);
    w8::GemvArgs a{};
    a.wp = static_cast<const uint8_t *>(p.packed);
    a.scale = p.scale;
    a.x = x;
    a.ldx = ldx;
    a.y = y;
    a.ldy = ldy;
    a.n = int(p.n);
    a.k = int(p.k);
    a.m = m;
    a.kb = int(plan.kb);
    a.rt = int(plan.rt);
    a.splits = plan.splits;
    a.wk = plan.wk;
    a.bfac = p.block_factors;
    a.nbf = int(w8::ceil_div(p.k, w8::kBlockB));
    w8::set_output_map(a, p, silu);
    if (plan.ws_bytes > 0) { // register-ring split-K plans (tensor-memory plans need none)
        if (!ws)
            return W8_ERR_NULL;
        if (reinterpret_cast<uintptr_t>(ws) & 255u)
            return W8_ERR_ALIGN;
        if (ws_bytes < build_ws_bytes(b, plan.ws_bytes, plan.ws_counters))
            return W8_ERR_CAPACITY;
        // the counters at the head, in the same place for every plan of the
        // build (each call leaves them zero); the partial sums after them
        a.counters = static_cast<int *>(ws);
        a.partial = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + b->ws_counters);
    }
    if (w8::launch_gemv(b->kdt[size_t(plane)], plan, a, reinterpret_cast<cudaStream_t>(s)) !=
        cudaSuccess)
        return W8_ERR_CUDA;
    return W8_OK;
}

// The checks of a w8_mlp call on the two planes: a gate_up plane and a
// row-major down plane whose K is the gate_up plane's I.
w8_status mlp_check(const w8_build *b, int gate_up, int down, int m)
{
    if (!b)
        return W8_ERR_NULL;
    if (gate_up < 0 || gate_up >= int(b->planes.size()) || down < 0 ||
        down >= int(b->planes.size()))
        return W8_ERR_PLANE;
    const w8_plane_info &u = b->planes[size_t(gate_up)], &d = b->planes[size_t(down)];
    if (u.layout != W8_LAYOUT_MMA_16x32_GATE_UP || d.layout != W8_LAYOUT_MMA_16x32)
        return W8_ERR_LAYOUT;
    if (d.k != u.n / 2 || m < 0 || m > max_m(u.dtype))
        return W8_ERR_SHAPE;
    return W8_OK;
}

} // namespace

extern "C" {

const char *w8_status_str(w8_status s)
{
    switch (s) {
    case W8_OK: return "ok";
    case W8_ERR_NULL: return "a required pointer is NULL";
    case W8_ERR_DTYPE: return "weight dtype the kernels cannot read (only E4M3FN, E4M3FN_B128, "
                              "BF16 and MXFP4), or a gemv call of another dtype";
    case W8_ERR_UNPADDED: return "unpadded plane: base not 16-byte aligned or row stride not a "
                                 "multiple of 16 bytes";
    case W8_ERR_BIAS: return "a bias was given; the GEMV has none";
    case W8_ERR_MIXED: return "bf16 and FP8 planes mixed in one build";
    case W8_ERR_SHAPE: return "bad shape: N, K >= 1, ldw >= K, 0 <= m <= 256, ldx >= K, ldy >= N "
                              "(N/2 for SiLU-and-multiply); a gate_up plane needs N % 16 == 0";
    case W8_ERR_SCALE: return "FP8 planes need fp32 row scales, block-scaled FP8 planes fp32 block "
                              "factors (ldb >= ceil(K/128)), MXFP4 planes E8M0 block scales "
                              "(ldb >= ceil(K/32)); no other plane takes either";
    case W8_ERR_LAYOUT: return "unknown source layout (row-major or gate_up), a block-scaled plane "
                               "bound as gate_up, or SiLU-and-multiply on a plane not bound as "
                               "gate_up";
    case W8_ERR_CAPACITY: return "packed buffer or workspace too small";
    case W8_ERR_ALIGN: return "misaligned buffer (packed/workspace: 256 B; x: 16 B with ldx % 8 == 0; y: 2 B)";
    case W8_ERR_PLANE: return "plane index outside the build";
    case W8_ERR_DEVICE: return "current device is not the device the build was bound on";
    case W8_ERR_CUDA: return "CUDA runtime error";
    case W8_ERR_SCRATCH: return "w8_gemv_noalloc: the call needs more scratch than the library's "
                                "fixed W8_NOALLOC_SCRATCH_BYTES";
    }
    return "unknown status";
}

int w8_abi_version(void) { return W8_ABI_VERSION; }

w8_status w8_device_status(int *status, int reset)
{
    if (!status)
        return W8_ERR_NULL;
    if (w8::tc_status(status, reset != 0) != cudaSuccess)
        return W8_ERR_CUDA;
    return W8_OK;
}

w8_status w8_validate(const w8_plane_desc *d, int n_planes)
{
    if (!d || n_planes < 1)
        return W8_ERR_NULL;
    for (int i = 0; i < n_planes; ++i) {
        const w8_status st = check_plane(d[i]);
        if (st != W8_OK)
            return st;
    }
    for (int i = 1; i < n_planes; ++i)
        if (d[i].dtype != d[0].dtype)
            return W8_ERR_MIXED;
    return W8_OK;
}

w8_status w8_packed_bytes(const w8_plane_desc *d, int n_planes, size_t *bytes)
{
    const w8_status st = w8_validate(d, n_planes);
    if (st != W8_OK)
        return st;
    if (!bytes)
        return W8_ERR_NULL;
    size_t total = 0;
    for (int i = 0; i < n_planes; ++i) {
        total += w8::align256(plane_scale_bytes(d[i].dtype, d[i].n));
        total += w8::align256(plane_factor_bytes(d[i].dtype, d[i].n, d[i].k));
        total += w8::align256(plane_packed_bytes(d[i].dtype, d[i].n, d[i].k));
    }
    *bytes = total;
    return W8_OK;
}

w8_status w8_bind(const w8_plane_desc *d, int n_planes, void *dst, size_t dst_bytes,
                  w8_stream s, w8_build **out)
{
    if (!out)
        return W8_ERR_NULL;
    *out = nullptr;
    size_t need = 0;
    w8_status st = w8_packed_bytes(d, n_planes, &need);
    if (st != W8_OK)
        return st;
    if (!dst)
        return W8_ERR_NULL;
    if (reinterpret_cast<uintptr_t>(dst) & 255u)
        return W8_ERR_ALIGN;
    if (dst_bytes < need)
        return W8_ERR_CAPACITY;

    int dev = -1, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return W8_ERR_CUDA;
    if (w8::prepare_gemv_kernels() != cudaSuccess)
        return W8_ERR_CUDA;

    w8_build *b = new (std::nothrow) w8_build;
    if (!b)
        return W8_ERR_CAPACITY;
    b->device = dev;
    b->sm_count = sms;
    b->dtype = d[0].dtype;
    b->ws_counters = 0;
    for (int i = 0; i < n_planes; ++i) {
        const size_t c = w8::align256(size_t(w8::ceil_div(d[i].n, w8::kTileN)) * sizeof(int));
        b->ws_counters = c > b->ws_counters ? c : b->ws_counters;
    }
    uint8_t *cursor = static_cast<uint8_t *>(dst);
    for (int i = 0; i < n_planes; ++i) {
        const w8_plane_desc &pd = d[i];
        w8_plane_info info{};
        info.dtype = pd.dtype;
        const bool gated = pd.layout == W8_SRC_GATE_UP;
        info.layout = gated ? W8_LAYOUT_MMA_16x32_GATE_UP : W8_LAYOUT_MMA_16x32;
        info.n = pd.n;
        info.k = pd.k;
        info.row_tiles = w8::ceil_div(pd.n, w8::kTileN);
        info.k_blocks = w8::ceil_div(pd.k, w8::kTileK);
        float *scale_copy = nullptr;
        const size_t sb = plane_scale_bytes(pd.dtype, pd.n);
        if (sb) {
            scale_copy = reinterpret_cast<float *>(cursor);
            cursor += w8::align256(sb);
        }
        info.scale = scale_copy;
        float *factor_copy = nullptr;
        const size_t fb = plane_factor_bytes(pd.dtype, pd.n, pd.k);
        if (fb) {
            factor_copy = reinterpret_cast<float *>(cursor);
            cursor += w8::align256(fb);
        }
        info.block_factors = factor_copy;
        info.packed = cursor;
        info.packed_bytes = plane_packed_bytes(pd.dtype, pd.n, pd.k);
        cursor += w8::align256(info.packed_bytes);

        w8::RepackArgs ra{};
        ra.src = static_cast<const uint8_t *>(pd.w);
        ra.ld_bytes = row_bytes(pd.dtype, pd.ldw);
        ra.bscale_src = pd.block_scale;
        ra.ldb = pd.ldb;
        ra.n = pd.n;
        ra.k = pd.k;
        ra.kb = info.k_blocks;
        ra.rt = info.row_tiles;
        ra.dst = static_cast<uint8_t *>(const_cast<void *>(info.packed));
        const bool b128 = pd.dtype == W8_DT_E4M3FN_B128;
        ra.scale_src = b128 ? nullptr : pd.scale;
        ra.scale_dst = scale_copy;
        ra.bfac_src = b128 ? pd.scale : nullptr;
        ra.bfac_dst = factor_copy;
        ra.half = gated ? pd.n / 2 : 0;
        int kdt = kernel_dt(pd.dtype);
        if (pd.dtype == W8_DT_MXFP4) {
            // the plane's first 4 packed bytes hold the scan's flag until the
            // repack writes them
            bool wide = false;
            if (w8::fp4_scales_wide(ra, static_cast<unsigned *>(const_cast<void *>(info.packed)),
                                    &wide, reinterpret_cast<cudaStream_t>(s)) != cudaSuccess) {
                delete b;
                return W8_ERR_CUDA;
            }
            ra.fp4_fold = !wide;
            kdt = wide ? w8::kDtFp4Wide : w8::kDtFp4;
            info.mxfp4_wide_scales = wide ? 1 : 0;
        }
        if (w8::launch_repack(kdt, ra, reinterpret_cast<cudaStream_t>(s)) != cudaSuccess) {
            delete b;
            return W8_ERR_CUDA;
        }
        b->planes.push_back(info);
        b->kdt.push_back(kdt);
    }
    // The GEMV kernels start reading the packed weights before they wait for
    // the previous kernel of their stream (programmatic dependent launch), so
    // the repack must be complete before any GEMV can be enqueued.
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(s)) != cudaSuccess) {
        delete b;
        return W8_ERR_CUDA;
    }
    *out = b;
    return W8_OK;
}

void w8_release(w8_build *b) { delete b; }

int w8_build_planes(const w8_build *b) { return b ? int(b->planes.size()) : 0; }

w8_status w8_build_info(const w8_build *b, int plane, w8_plane_info *info)
{
    if (!b || !info)
        return W8_ERR_NULL;
    if (plane < 0 || plane >= int(b->planes.size()))
        return W8_ERR_PLANE;
    *info = b->planes[size_t(plane)];
    return W8_OK;
}

static void fill_plan(const w8::Plan &pl, w8_plan *out)
{
    out->kernel = pl.tc ? 1 : 0;
    out->grid = pl.grid;
    out->block = pl.tc ? w8::kTcThreadsPerCta : w8::kThreads;
    out->smem_bytes = pl.smem;
    out->n_tiles = pl.nt;
    out->row_tiles_per_warp = pl.r;
    out->warps_k = pl.wk;
    out->depth = pl.dw;
    out->row_groups = pl.row_groups;
    out->splits = pl.splits;
    out->k_blocks_per_warp_max = pl.kbs_max;
    out->workspace_bytes = pl.ws_bytes;
    out->cluster = pl.tc ? pl.cluster : 1;
    out->ctas_per_sm = pl.occ;
}

w8_status w8_plan_shape(int64_t n, int64_t k, int m, int sm_count, w8_plan *out)
{
    if (!out)
        return W8_ERR_NULL;
    if (n < 1 || k < 1 || n > kMaxDim || k > kMaxDim || m < 1 || m > w8::kMaxM || sm_count < 1)
        return W8_ERR_SHAPE;
    fill_plan(w8::make_plan(n, k, m, sm_count), out);
    return W8_OK;
}

// The plan a gemv call on a plane of this dtype and shape makes, with the
// dtype's own ring depth.
static void fill_plan_dt(int32_t dtype, int64_t n, int64_t k, int m, int sms, w8_plan *out)
{
    const w8::Plan pl = plan_for(dtype, n, k, m, sms);
    fill_plan(pl, out);
    if (dtype == W8_DT_BF16)
        out->depth = pl.tc ? w8::tc_stages(false, pl.npad, pl.occ).nw * w8::kTcStageBlocks
                           : w8::depth_w(pl.nt, pl.r, false, pl.occ);
    if (dtype == W8_DT_MXFP4)
        out->depth = w8::depth_w_dt(pl.nt, pl.r, w8::kDtFp4, pl.occ);
    if (dtype == W8_DT_E4M3FN_B128 && !pl.tc) {
        // the kernel splits K among CTAs and warps in whole column blocks
        // (units of 4 K blocks, floor boundaries, the last unit cut at kb)
        const int64_t u = w8::kBlockB / w8::kTileK, nu = w8::ceil_div(pl.kb, u);
        int64_t most = 0;
        for (int sp = 0; sp < pl.splits; ++sp) {
            const int64_t c0 = sp * nu / pl.splits, c1 = (sp + 1) * nu / pl.splits;
            for (int q = 0; q < pl.wk; ++q) {
                const int64_t k0 = (c0 + q * (c1 - c0) / pl.wk) * u;
                const int64_t k1 = (c0 + (q + 1) * (c1 - c0) / pl.wk) * u;
                const int64_t len = (k1 < pl.kb ? k1 : pl.kb) - k0;
                most = len > most ? len : most;
            }
        }
        out->k_blocks_per_warp_max = int32_t(most);
    }
}

w8_status w8_plan_shape_dtype(int64_t n, int64_t k, int m, int sm_count, int32_t dtype,
                              w8_plan *out)
{
    if (!out)
        return W8_ERR_NULL;
    if (dtype != W8_DT_E4M3FN && dtype != W8_DT_E4M3FN_B128 && dtype != W8_DT_BF16 &&
        dtype != W8_DT_MXFP4)
        return W8_ERR_DTYPE;
    if (n < 1 || k < 1 || n > kMaxDim || k > kMaxDim || m < 1 || m > max_m(dtype) ||
        sm_count < 1)
        return W8_ERR_SHAPE;
    fill_plan_dt(dtype, n, k, m, sm_count, out);
    return W8_OK;
}

w8_status w8_plan_info(const w8_build *b, int plane, int m, w8_plan *out)
{
    if (!b || !out)
        return W8_ERR_NULL;
    if (plane < 0 || plane >= int(b->planes.size()))
        return W8_ERR_PLANE;
    const w8_plane_info &p = b->planes[size_t(plane)];
    if (m < 1 || m > max_m(p.dtype))
        return W8_ERR_SHAPE;
    fill_plan_dt(p.dtype, p.n, p.k, m, b->sm_count, out);
    const w8::Plan pl = plan_for(p.dtype, p.n, p.k, m, b->sm_count);
    out->workspace_bytes = build_ws_bytes(b, pl.ws_bytes, pl.ws_counters);
    return W8_OK;
}

w8_status w8_workspace_bytes(const w8_build *b, int plane, int m, size_t *bytes)
{
    if (!b || !bytes)
        return W8_ERR_NULL;
    if (plane < -1 || plane >= int(b->planes.size()))
        return W8_ERR_PLANE;
    if (m < 0 || m > w8::kMaxM)
        return W8_ERR_SHAPE;
    size_t best = 0;
    const int p0 = plane < 0 ? 0 : plane;
    const int p1 = plane < 0 ? int(b->planes.size()) : plane + 1;
    for (int pi = p0; pi < p1; ++pi) {
        const w8_plane_info &p = b->planes[size_t(pi)];
        const int m0 = m == 0 ? 1 : m, m1 = m == 0 ? max_m(p.dtype) : m;
        for (int mm = m0; mm <= m1 && mm <= max_m(p.dtype); ++mm) {
            const w8::Plan pl = plan_for(p.dtype, p.n, p.k, mm, b->sm_count);
            const size_t ws = build_ws_bytes(b, pl.ws_bytes, pl.ws_counters);
            if (ws > best)
                best = ws;
        }
    }
    *bytes = best;
    return W8_OK;
}

w8_status w8_gemv(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                  uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes, w8_stream s)
{
    return gemv_common(b, plane, W8_DT_E4M3FN, false, x, ldx, m, y, ldy, workspace,
                       workspace_bytes, s);
}

w8_status bf16_gemv(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                    uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes, w8_stream s)
{
    return gemv_common(b, plane, W8_DT_BF16, false, x, ldx, m, y, ldy, workspace,
                       workspace_bytes, s);
}

w8_status mxfp4_gemv(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                     uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes, w8_stream s)
{
    return gemv_common(b, plane, W8_DT_MXFP4, false, x, ldx, m, y, ldy, workspace,
                       workspace_bytes, s);
}

w8_status w8_gemv_silu_mul(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                           uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes,
                           w8_stream s)
{
    return gemv_common(b, plane, 0, true, x, ldx, m, y, ldy, workspace, workspace_bytes, s);
}

w8_status w8_mlp_workspace_bytes(const w8_build *b, int gate_up, int down, int m, size_t *bytes)
{
    if (!bytes)
        return W8_ERR_NULL;
    const w8_status st = mlp_check(b, gate_up, down, m);
    if (st != W8_OK)
        return st;
    size_t wu = 0, wd = 0;
    w8_workspace_bytes(b, gate_up, m, &wu);
    w8_workspace_bytes(b, down, m, &wd);
    *bytes = wu > wd ? wu : wd;
    return W8_OK;
}

w8_status w8_mlp(const w8_build *b, int gate_up, int down, const uint16_t *x, int64_t ldx, int m,
                 uint16_t *h, int64_t ldh, uint16_t *y, int64_t ldy, void *workspace,
                 size_t workspace_bytes, w8_stream s)
{
    w8_status st = mlp_check(b, gate_up, down, m);
    if (st != W8_OK || m == 0)
        return st;
    // The down launch's host checks before the first launch is enqueued, so
    // that a refused call enqueues nothing: h as its x (16-byte loads), y,
    // and the workspace of either projection (x and the device are checked
    // by the gate_up launch, before it is enqueued).
    const w8_plane_info &pd = b->planes[size_t(down)];
    if (!h || !y)
        return W8_ERR_NULL;
    if (ldh < pd.k || ldy < pd.n)
        return W8_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(h) & 15u) || (ldh & 7) || (reinterpret_cast<uintptr_t>(y) & 1u))
        return W8_ERR_ALIGN;
    size_t need = 0;
    w8_mlp_workspace_bytes(b, gate_up, down, m, &need);
    if (need > 0 && !workspace)
        return W8_ERR_NULL;
    if (workspace_bytes < need)
        return W8_ERR_CAPACITY;
    st = gemv_common(b, gate_up, 0, true, x, ldx, m, h, ldh, workspace, workspace_bytes, s);
    if (st != W8_OK)
        return st;
    // the down projection of h: it may begin streaming its weights while the
    // gate_up kernel drains, and reads h once that kernel has completed
    return gemv_common(b, down, 0, false, h, ldh, m, y, ldy, workspace, workspace_bytes, s);
}

int64_t w8_packed_offset(int dtype, int64_t k_blocks, int64_t row, int64_t col)
{
    if (k_blocks < 1 || row < 0 || col < 0 || col >= k_blocks * w8::kTileK)
        return -1;
    if (dtype == W8_DT_E4M3FN || dtype == W8_DT_E4M3FN_B128)
        return w8::packed_offset_fp8(k_blocks, row, col);
    if (dtype == W8_DT_BF16)
        return w8::packed_offset_bf16(k_blocks, row, col);
    return -1; // MXFP4: w8_mxfp4_code_bits
}

w8_status w8_mxfp4_code_bits(int64_t k_blocks, int64_t row, int64_t col, int64_t *bits)
{
    if (!bits)
        return W8_ERR_NULL;
    if (k_blocks < 1 || row < 0 || col < 0 || col >= k_blocks * w8::kTileK)
        return W8_ERR_SHAPE;
    int64_t b[4];
    w8::mxfp4_code_bits(k_blocks, row, col, b);
    for (int i = 0; i < 4; ++i)
        bits[i] = b[i];
    return W8_OK;
}

int64_t w8_gate_up_packed_row(int64_t n, int64_t row)
{
    if (n < 16 || n % 16 != 0 || row < 0 || row >= n)
        return -1;
    const int64_t half = n / 2;
    // gate row j sits at 16 (j / 8) + j % 8, up row j at 16 (j / 8) + 8 + j % 8
    return row < half ? 16 * (row / 8) + row % 8 : 16 * ((row - half) / 8) + 8 + (row - half) % 8;
}

} // extern "C"
