/*
 * w8.h -- C ABI of libw8: the FP8 weight-only (w8a16) decode GEMV for one
 * GB300 GPU (sm_103a).
 *
 * What the library computes (ATOM pull request #2980,
 * sections Summary and Changes): for a bound weight plane W [N, K] and M
 * decode tokens x [M, K] (bf16),
 *
 *     y[m, n] = bf16_rne( scale[n] * sum_k bf16(W[n, k]) * x[m, k] )
 *
 * W is an E4M3fn plane carrying a single fp32 factor for every output row;
 * each of its codes converts to a bf16 value with no rounding; the products
 * are summed in fp32, and the row's factor is applied to that finished sum
 * just before the one conversion to bf16.  A bf16 plane takes the same path
 * with no factor at all (the PR keeps bf16 weights on their existing path).
 * Three more plane kinds share the entry points' shape: block-scaled FP8
 * (W8_DT_E4M3FN_B128, through w8_gemv), w4a16 MXFP4 (W8_DT_MXFP4,
 * mxfp4_gemv) and merged gate_up planes whose call applies SiLU-and-multiply
 * (W8_SRC_GATE_UP, w8_gemv_silu_mul, and w8_mlp: gate_up, SiLU-and-multiply
 * and the down projection in one call); each is defined where it is
 * declared.
 *
 * Conventions for every function below:
 *  - Pointers named "device" point into CUDA device memory of the device that
 *    is current when the call is made; pointers named "host" point into host
 *    memory.  The caller owns all device memory: source planes, scales, the
 *    packed buffer, activations, outputs and workspace.  The library owns
 *    only the small host-side w8_build handle.
 *  - Every function returns a w8_status.  Arguments are checked on the host
 *    before anything is enqueued; nothing traps on the device and no function
 *    exits the process.  A failed launch or CUDA call returns W8_ERR_CUDA.
 *  - The gemv calls (w8_gemv, bf16_gemv, mxfp4_gemv, w8_gemv_silu_mul,
 *    w8_gemv_noalloc) are asynchronous on the caller's stream, never
 *    synchronise and launch exactly one kernel, with programmatic dependent
 *    launch: the kernel may begin streaming weights while the previous kernel
 *    of the stream drains, and reads activations and writes outputs only
 *    after that kernel has completed.  w8_mlp is asynchronous in the same
 *    way and launches two such kernels, the second dependent on the first.  w8_bind runs its repack kernels on the
 *    caller's stream and synchronises that stream before it returns (load
 *    time; it must not be captured in a CUDA graph).
 *  - A stream argument is a cudaStream_t (NULL is the legacy default stream).
 */
#ifndef W8_H
#define W8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define W8_ABI_VERSION 8

/* A cudaStream_t: the runtime's stream type is this same pointer type. */
typedef struct CUstream_st *w8_stream;

typedef enum {
    W8_OK = 0,
    W8_ERR_NULL = 1,      /* a required pointer is NULL, or no planes given */
    W8_ERR_DTYPE = 2,     /* plane dtype the kernels cannot read (e4m3fnuz, e5m2, fp16,
                             unknown), or a gemv call whose dtype is not the build's */
    W8_ERR_UNPADDED = 3,  /* plane base not 16-byte aligned, or row stride not a multiple
                             of 16 bytes */
    W8_ERR_BIAS = 4,      /* a bias pointer was given: the GEMV has no bias */
    W8_ERR_MIXED = 5,     /* planes of different dtypes in one build (bf16 and FP8 among
                             them) */
    W8_ERR_SHAPE = 6,     /* N or K < 1 or too large, ldw < K, M outside 0..256,
                             ldx < K, ldy < N (< N/2 for w8_gemv_silu_mul), or a
                             W8_SRC_GATE_UP plane whose N is not a multiple of 16 */
    W8_ERR_SCALE = 7,     /* an FP8 plane without row scales, a block-scaled FP8 plane
                             without factors or ldb < ceil(k / 128), a bf16 or MXFP4
                             plane with scale set, an MXFP4 plane without block scales
                             or ldb too short, or another plane with block_scale set */
    W8_ERR_LAYOUT = 8,    /* unknown source layout, a block-scaled FP8 plane given as
                             W8_SRC_GATE_UP, or w8_gemv_silu_mul on a plane not bound as
                             W8_SRC_GATE_UP */
    W8_ERR_CAPACITY = 9,  /* packed buffer or workspace smaller than required */
    W8_ERR_ALIGN = 10,    /* packed buffer or workspace not 256-byte aligned, x not 16-byte
                             aligned or ldx not a multiple of 8, or y not 2-byte aligned */
    W8_ERR_PLANE = 11,    /* plane index outside the build */
    W8_ERR_DEVICE = 12,   /* the current device is not the one the build was bound on */
    W8_ERR_CUDA = 13,     /* a CUDA runtime call or kernel launch failed */
    W8_ERR_SCRATCH = 14   /* w8_gemv_noalloc: the call needs more scratch than the
                             library's fixed W8_NOALLOC_SCRATCH_BYTES */
} w8_status;

/* Source element types.  Bind accepts E4M3FN, E4M3FN_B128, BF16 and (w4a16)
 * MXFP4 and refuses every other format, e4m3fnuz among them (the PR page,
 * Changes and Limitations: bind turns away planes its kernels cannot
 * decode). */
typedef enum {
    W8_DT_E4M3FN = 1,
    W8_DT_BF16 = 2,
    W8_DT_E4M3FNUZ = 3,
    W8_DT_E5M2 = 4,
    W8_DT_FP16 = 5,
    /* w4a16: MXFP4 weights (ATOM Model Support Guide, Model-specific
     * optimizations, DeepSeek V2/V3: FP4 support names MXFP4 GEMMs with
     * 16-bit activations; the GLM-5.2 anatomy page deploys a GLM-5.2-MXFP4
     * checkpoint).  The OCP microscaling format: E2M1 elements, two per
     * byte (the even column in the low nibble), 32 consecutive elements
     * along K sharing one E8M0 scale 2^(e - 127) (255 = NaN). */
    W8_DT_MXFP4 = 6,
    /* Block-scaled FP8: E4M3fn codes with one fp32 factor per block of 128
     * rows x 128 columns instead of row scales (the GLM-5.2 anatomy page runs
     * fused_qkv_a_proj through a blockscale GEMM; the ATOM Model Support
     * Guide, Weight loading, loads a checkpoint's weight_scale_inv tensors as
     * the weight scales).  The pages fix neither the block shape nor where
     * the factor enters; this library takes 128 x 128 and applies each
     * factor to the finished sum of its block's 128 columns:
     *   y[m, n] = bf16( sum_j f[n/128, j] * sum_{k in block j} W[n, k] x[m, k] ),
     * the inner sums and the total in fp32.  Register-ring kernel only
     * (m <= 64); not with W8_SRC_GATE_UP. */
    W8_DT_E4M3FN_B128 = 7
} w8_dtype;

/* Source layouts: row-major [n][ldw] planes (K contiguous).
 * W8_SRC_GATE_UP is a merged MLP projection of n = 2I rows: rows 0..I-1 are
 * the gate projection and rows I..2I-1 the up projection (ATOM Model Support
 * Guide: the Llama MLP merges gate and up into one column-parallel
 * projection, followed by SiLU-and-multiply and the down projection; Adding
 * a new model, Step 5: gate_proj is shard 0 and up_proj shard 1 of
 * gate_up_proj).  I must be a multiple of 8 (n a multiple of 16). */
#define W8_SRC_ROW_MAJOR 0
#define W8_SRC_GATE_UP 1

/* Packed layout the kernels read (recorded in every build; the PR page,
 * Limitations, says its own tensors do not carry their layout):
 * rows in tiles of 16, K in blocks of 32, each (tile, block) a 512-byte
 * (FP8) or 1024-byte (bf16) run holding the 16x32 weights in the order of
 * the tensor-core A operand, one 16-byte vector per lane.  The K tail and
 * the row tail are zero-filled.  MXFP4: 288-byte runs, 256 bytes of codes
 * (lane (g, t): 8 bytes, one 32-bit word per tensor-core step, bit places of
 * w8_mxfp4_code_bits) then 8 words of block scales, word g = bf16 scale of
 * row g | bf16 scale of row g+8 << 16 (E8M0 0 -> bf16 2^-127, 255 -> NaN). */
#define W8_LAYOUT_MMA_16x32 1
/* The same layout for a W8_SRC_GATE_UP plane, with the rows interleaved:
 * packed 16-row tile t holds gate rows 8t..8t+7, then up rows 8t..8t+7 (the
 * source rows 8t..8t+7 and I+8t..I+8t+7), so that one tensor-core tile
 * holds a gate row and its up row eight rows apart.  The scales follow their
 * rows.  Both gemv calls still write y in source row order. */
#define W8_LAYOUT_MMA_16x32_GATE_UP 2

/* One source weight plane: W[n][ldw] in device memory, row-major. */
typedef struct {
    const void *w;        /* device; E4M3 codes (1 byte), bf16 bits (2 bytes) or MXFP4
                             codes (two per byte); 16-byte aligned */
    int32_t dtype;        /* w8_dtype */
    int32_t layout;       /* W8_SRC_ROW_MAJOR or W8_SRC_GATE_UP */
    int64_t n;            /* output rows, >= 1 */
    int64_t k;            /* logical reduction columns, >= 1; columns k..ldw-1 are ignored */
    int64_t ldw;          /* row stride in elements, >= k, ldw * element bytes % 16 == 0
                             (MXFP4: ldw % 32 == 0) */
    const float *scale;   /* device fp32: E4M3FN [n] row scales; E4M3FN_B128
                             [ceil(n / 128)][ldb] block factors, entry (i, j) covering
                             rows 128i .. 128i+127 and columns 128j .. 128j+127;
                             NULL for the other dtypes */
    const void *bias;     /* must be NULL */
    const uint8_t *block_scale; /* device, MXFP4 only: [n][ldb] E8M0 scales, block j covering
                             columns 32j .. 32j+31; NULL for the other dtypes */
    int64_t ldb;          /* MXFP4: row stride of block_scale in bytes, >= ceil(k / 32);
                             E4M3FN_B128: row stride of scale in floats, >= ceil(k / 128) */
} w8_plane_desc;

/* What a build records about one bound plane. */
typedef struct {
    int32_t dtype;           /* W8_DT_E4M3FN, W8_DT_E4M3FN_B128, W8_DT_BF16 or W8_DT_MXFP4 */
    int32_t layout;          /* W8_LAYOUT_MMA_16x32 or W8_LAYOUT_MMA_16x32_GATE_UP */
    int64_t n, k;
    int64_t row_tiles;       /* ceil(n / 16) */
    int64_t k_blocks;        /* ceil(k / 32) */
    const void *packed;      /* device, inside the caller's packed buffer */
    const float *scale;      /* device, the build's copy of the row scales (FP8; 1 for
                                block-scaled FP8), else NULL */
    size_t packed_bytes;     /* bytes of the packed weights (MXFP4: with the block scales) */
    const float *block_factors; /* device, block-scaled FP8: the build's copy of the factors,
                                [ceil(n / 128)][ceil(k / 128)]; else NULL */
    int32_t mxfp4_wide_scales; /* MXFP4: 1 when a block scale of the plane is above 2^1
                                (E8M0 129..254), so its codes take two multiplies (2^126,
                                then the scale) instead of one by 2^126 x the scale folded
                                at bind; the result is the same.  0 otherwise. */
} w8_plane_info;

/* The launch a gemv call makes for one (plane, m); returned for inspection.
 * kernel 0 (m <= 16, or m <= 64 on a plane of fewer than 48 blocks of 128
 *   rows): the register-ring kernel, 8 warps per CTA.
 * kernel 1 (m >= 17 on a plane of at least 48 blocks of 128 rows, and every
 *   m >= 65): the tensor-memory kernel, 128 rows x one K range per CTA;
 *   there n_tiles = tokens rounded up to 16 (to 96, 128, 192 or 256 above
 *   64), over 8; row_tiles_per_warp = the CTA's 8 row tiles; warps_k = 1;
 *   depth = the weight blocks staged ahead. */
typedef struct {
    int32_t kernel;          /* 0: register ring (mma.sync), 1: tensor memory (tcgen05) */
    int32_t grid;            /* CTAs */
    int32_t block;           /* threads per CTA */
    int32_t smem_bytes;      /* dynamic shared memory per CTA */
    int32_t n_tiles;         /* 8-token groups of the tensor-core N dimension */
    int32_t row_tiles_per_warp;
    int32_t warps_k;         /* warps that share one row tile, each on its own K part */
    int32_t depth;           /* K blocks each warp keeps in flight (w8_plan_shape gives
                                the FP8 depth; bf16 rings hold fewer, larger blocks;
                                the depth never changes a summation order) */
    int32_t row_groups;      /* CTAs along N */
    int32_t splits;          /* CTAs along K */
    int32_t k_blocks_per_warp_max; /* most 32-column K blocks one warp streams */
    size_t workspace_bytes;  /* 0 unless the splits add their partial sums through the
                                workspace (every kernel-0 plan with splits > 1; kernel 1
                                when cluster is 1) */
    int32_t cluster;         /* kernel 1: CTAs of a thread-block cluster, the splits of a
                                row block when they add their partial sums on chip
                                (cluster == splits, no workspace), or 1 when K is split
                                into more ranges than a power of two that fill the SMs
                                evenly (up to 8) and the last CTA of a row block adds
                                them from the workspace; kernel 0: 1 */
    int32_t ctas_per_sm;     /* CTAs one SM holds at once (the occupancy the launch is
                                built for): kernel 1 two up to 64 tokens, except one
                                (with a deeper weight ring) at 49..64 tokens where one
                                wave of unclustered CTAs covers at least 3/4 of the SMs;
                                one above 64 tokens */
} w8_plan;

typedef struct w8_build w8_build; /* opaque, host-side, library-owned */

/* The tensor-memory kernel's status word on the current device: 0 when every
 * wait of every launch so far ended normally; bit 0 = a pipeline-stage wait
 * gave up, bit 1 = the accumulator wait gave up (each wait polls a bounded
 * number of times, then the kernel runs to its end with that output wrong and
 * flags it here).  Synchronous (reads device memory); reset != 0 clears it.
 * No counterpart on the pages: it reports this library's own safety bound. */
w8_status w8_device_status(int *status, int reset);

/* Text for a status code (static storage; never NULL). */
const char *w8_status_str(w8_status s);

/* W8_ABI_VERSION of the loaded library. */
int w8_abi_version(void);

/* Host-only check of n_planes descriptors, as w8_bind makes them: dtype, layout,
 * bias, shape, scale presence, 16-byte padding and alignment, and that all
 * planes share one dtype (W8_ERR_MIXED).  Touches no device memory and calls
 * no CUDA API. */
w8_status w8_validate(const w8_plane_desc *d, int n_planes);

/* Bytes of the packed buffer w8_bind needs for these planes (host-only).
 * *bytes is set on W8_OK. */
w8_status w8_packed_bytes(const w8_plane_desc *d, int n_planes, size_t *bytes);

/* Validate the planes, then repack each into the caller's device buffer dst
 * (256-byte aligned, at least w8_packed_bytes) on stream s: the weights in
 * W8_LAYOUT_MMA_16x32 and, for FP8, a copy of the row scales (all 1 for a
 * block-scaled plane, which also gets a copy of its block factors).  An FP8
 * row holding a NaN code (0x7F / 0xFF) gets a NaN scale in that copy, so its
 * outputs are NaN, as the definition gives.  On W8_OK *out is a new handle
 * for the device current at the call, the repack has completed (the stream
 * is synchronised) and the source planes and scales may be freed.  dst must
 * outlive the handle and must not be written while gemv calls may read it. */
w8_status w8_bind(const w8_plane_desc *d, int n_planes, void *dst, size_t dst_bytes,
                  w8_stream s, w8_build **out);

/* Free a handle (host memory only; NULL is ignored).  The caller's buffers
 * are untouched. */
void w8_release(w8_build *b);

/* Number of planes in a build, and what one of them holds. */
int w8_build_planes(const w8_build *b);
w8_status w8_build_info(const w8_build *b, int plane, w8_plane_info *info);

/* The launch plan of a gemv call on this plane with m tokens (1..256). */
w8_status w8_plan_info(const w8_build *b, int plane, int m, w8_plan *plan);

/* The same plan for a plane of n rows and k columns on a GPU with sm_count
 * SMs, computed on the host without a build (no CUDA call).  The plan depends
 * on (n, k, m, sm_count) only, not on the weight dtype, except that MXFP4 and
 * block-scaled FP8 planes always run the register ring, block-scaled ones on
 * the instances that hold their second set of accumulators (w8_plan_info
 * gives a bound plane's own plan). */
w8_status w8_plan_shape(int64_t n, int64_t k, int m, int sm_count, w8_plan *plan);

/* The plan, with the dtype's own ring depth, that a gemv call makes on a
 * bound plane of this dtype (W8_DT_E4M3FN, W8_DT_E4M3FN_B128, W8_DT_BF16 or
 * W8_DT_MXFP4), n rows and k columns on a GPU of sm_count SMs: what
 * w8_plan_info returns for such a plane, computed on the host without a
 * build (no CUDA call).  m: 1..256, or 1..64 for the register-ring-only
 * dtypes (MXFP4, block-scaled FP8); W8_ERR_SHAPE otherwise, W8_ERR_DTYPE
 * for another dtype.  No counterpart on the pages: it reports this
 * library's own launch plan. */
w8_status w8_plan_shape_dtype(int64_t n, int64_t k, int m, int sm_count, int32_t dtype,
                              w8_plan *plan);

/* Workspace bytes a gemv call on `plane` with `m` tokens needs (0 if none).
 * plane = -1 takes the largest over all planes, m = 0 the largest over
 * m = 1..256, so one workspace can serve every call of a build.
 *
 * Workspace contract: 256-byte aligned device memory, zero-filled once by the
 * caller before its first use.  Its head holds one arrival counter per row
 * tile of the build's largest plane, in the same place for every call of the
 * build, and every call leaves them at zero again; the partial sums follow.
 * Calls that share a workspace must not overlap on the GPU: order them on one
 * stream or synchronise between them. */
w8_status w8_workspace_bytes(const w8_build *b, int plane, int m, size_t *bytes);

/* The FP8 (w8a16) GEMV on an E4M3FN build:
 *   y[i*ldy + n] = bf16(scale[n] * sum_k W[n,k] * x[i*ldx + k]),  0 <= i < m, 0 <= n < N;
 * on an E4M3FN_B128 build the block-factor form of that dtype's comment
 * (m: 0..64, W8_ERR_SHAPE above).
 * x: device bf16 [m][ldx], ldx >= K, ldx % 8 == 0, 16-byte aligned (every
 *    row is read with 16-byte loads; columns K..ldx-1 are never read);
 * y: device bf16 [m][ldy], ldy >= N, written for n < N only;
 * m: tokens, 0..256 (0 is a no-op): decode steps up to 64, draft rows and
 *    prefill chunks above (the tensor-memory kernel runs every call of 65..256);
 * workspace / workspace_bytes: see w8_workspace_bytes (may be NULL / 0 when
 *    that returns 0).
 * Returns W8_ERR_DTYPE on a bf16 build.  One kernel launch on s. */
w8_status w8_gemv(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                  uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes,
                  w8_stream s);

/* The bf16-weight GEMV on a BF16 build: the same call without the scale,
 *   y[i*ldy + n] = bf16(sum_k W[n,k] * x[i*ldx + k]).
 * Same summation order as w8_gemv for the same (N, K, m), so a bf16 plane of
 * widened codes gives bit for bit the FP8 result with unit scales.
 * Returns W8_ERR_DTYPE on an FP8 build.  One kernel launch on s. */
w8_status bf16_gemv(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                    uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes,
                    w8_stream s);

/* The merged gate_up projection followed by SiLU-and-multiply, in one kernel
 * (ATOM Model Support Guide, Model architecture details, Llama MLP: one
 * merged projection for gate and up, the SiLU-and-multiply activation, then
 * the down projection; Model-specific optimizations: the activation fused
 * into a neighbouring kernel).  On a plane bound as
 * W8_SRC_GATE_UP (n = 2I), for 0 <= i < m and 0 <= j < I:
 *   g = the GEMV's output for source row j (what w8_gemv / bf16_gemv give),
 *   u = the GEMV's output for source row I + j,
 *   y[i*ldy + j] = bf16(silu(g) * u),  silu(v) = v / (1 + exp(-v)),
 * with g and u rounded to bf16 first and the SiLU and the product in fp32
 * (expf and a correctly rounded division), so the result is what the two
 * separate steps give.  Either dtype (FP8 with row scales, or bf16).
 * y: device bf16 [m][ldy], ldy >= I, written for j < I only.  x, m and the
 * workspace as for w8_gemv (the plan is that of the [2I, K] plane).
 * Returns W8_ERR_LAYOUT on a plane not bound as W8_SRC_GATE_UP.  One kernel
 * launch on s. */
w8_status w8_gemv_silu_mul(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                           uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes,
                           w8_stream s);

/* The w4a16 GEMV on an MXFP4 build: the same call with each weight dequantized
 * as its E2M1 value times its block's E8M0 scale (exact in bf16),
 *   y[i*ldy + n] = bf16(sum_k e2m1(W[n,k]) * 2^(bs[n, k/32] - 127) * x[i*ldx + k]),
 * fp32 accumulation.  m: 0..64 (the register-ring kernel); W8_ERR_SHAPE above.
 * A row holding a NaN scale, or a weight past fp32's range, gives NaN (the
 * plain definition: NaN or inf times a zero token).  The same summation order
 * as bf16_gemv for the same (N, K, m): with every scale 1 the result equals
 * the bf16 plane of the dequantized weights bit for bit.
 * Returns W8_ERR_DTYPE on another build.  One kernel launch on s. */
w8_status mxfp4_gemv(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                     uint16_t *y, int64_t ldy, void *workspace, size_t workspace_bytes,
                     w8_stream s);

/* The MLP block in one call (ATOM Model Support Guide, Model architecture
 * details, Llama MLP: the merged gate and up projection, SiLU-and-multiply,
 * then the down projection), on two planes of one build:
 *   gate_up: bound as W8_SRC_GATE_UP, [2I, K];  down: row-major, [N, I];
 *   h[i*ldh + j] = w8_gemv_silu_mul's output on gate_up and x,  j < I,
 *   y[i*ldy + n] = the gemv's output on down and h,            n < N,
 * for 0 <= i < m, on any build that can hold a gate_up plane (E4M3FN, BF16,
 * MXFP4; the gemv of the build's dtype).  Exactly the two calls in sequence,
 * bit for bit.
 * x: device bf16 [m][ldx], ldx >= K, ldx % 8 == 0, 16-byte aligned;
 * h: device bf16 [m][ldh], ldh >= I, ldh % 8 == 0, 16-byte aligned (the down
 *    projection reads it as its x), written for j < I only;
 * y: device bf16 [m][ldy], ldy >= N, written for n < N only;
 * x, h and y must not overlap.  m: as the build's gemv (0 is a no-op);
 * W8_ERR_SHAPE above, or when down's K is not I.
 * workspace: w8_mlp_workspace_bytes bytes (0 when neither plan splits K),
 *    the contract of w8_workspace_bytes.
 * W8_ERR_LAYOUT when gate_up is not a gate_up plane or down is one.  Every
 * check of both launches is made before the first is enqueued.
 * Two kernel launches on s: gate_up with SiLU-and-multiply into h, then the
 * down projection, which may stream its weights while the first drains
 * (programmatic dependent launch) and reads h once it has completed.  (A
 * single kernel for both, its down items waiting inside the launch for every
 * gate_up item, measured 40-50 % slower on GB300: a down item cannot stream
 * its weights before knowing its item, and its CTA slot opens only when a
 * gate_up CTA ends.) */
w8_status w8_mlp(const w8_build *b, int gate_up, int down, const uint16_t *x, int64_t ldx, int m,
                 uint16_t *h, int64_t ldh, uint16_t *y, int64_t ldy, void *workspace,
                 size_t workspace_bytes, w8_stream s);

/* Workspace bytes of w8_mlp on (gate_up, down) with m tokens (m = 0: the
 * largest over every m): the larger of the two projections'
 * w8_workspace_bytes.  Same checks as w8_mlp's on the planes and m. */
w8_status w8_mlp_workspace_bytes(const w8_build *b, int gate_up, int down, int m, size_t *bytes);

/* The FP8 GEMV for callers that cannot allocate device memory.
 *
 * The pages have no counterpart of this entry point; it serves callers that
 * cannot call cudaMalloc where they run the GEMV (a host callback, an
 * allocator or memory-pool hook, a framework that forbids device allocations
 * while it records or replays a step) and so cannot provide the workspace
 * w8_gemv asks for when a plan splits K across CTAs.
 *
 * It serves row-scaled FP8 builds (W8_DT_E4M3FN) only, plain or gate_up
 * planes; on such a build it takes w8_gemv's arguments without the workspace
 * and gives w8_gemv's result.  Every other build (bf16, block-scaled FP8,
 * MXFP4) returns W8_ERR_DTYPE.  The scratch
 * comes from a fixed array of W8_NOALLOC_SCRATCH_BYTES (64 KiB) inside the
 * library, which every GPU that loads the library holds until the process
 * exits: its first 4 KiB hold the arrival counters (one per row tile) of
 * every call and every build, the rest the partial sums.  A call whose plan
 * needs more (more than 1024 row tiles with K split, or partial sums past the
 * array's end) returns W8_ERR_SCRATCH before any launch.  It allocates nothing: no
 * cudaMalloc, no cudaFree, no allocating library routine.
 *
 * The first call on each device sets the array up, whatever the shape of
 * that call: with that device current it looks up the array's device address
 * and zeroes the array, which synchronises the device, so that first call
 * must come before any stream capture.  Every call leaves the array's
 * counters at zero again.  All calls on a device share the one array, so
 * calls that could overlap on the GPU (different streams without ordering
 * between them) race and must not be made; calls in order on one stream are
 * fine, with no synchronisation between them.  One kernel launch on s. */
#define W8_NOALLOC_SCRATCH_BYTES (64u << 10)
w8_status w8_gemv_noalloc(const w8_build *b, int plane, const uint16_t *x, int64_t ldx, int m,
                          uint16_t *y, int64_t ldy, w8_stream s);

/* Host-side address map of W8_LAYOUT_MMA_16x32: byte offset, inside one
 * plane's packed weights, of element (row, col) of a plane with k_blocks
 * blocks of 32 columns (row is the packed row: for a gate_up plane, see
 * w8_gate_up_packed_row).  dtype is W8_DT_E4M3FN, W8_DT_E4M3FN_B128 (the
 * same layout) or W8_DT_BF16 (MXFP4 codes are not byte-addressable: see
 * w8_mxfp4_code_bits); returns -1 on a bad argument.  The repack kernel places every element at this offset. */
int64_t w8_packed_offset(int dtype, int64_t k_blocks, int64_t row, int64_t col);

/* Host-side address map of an MXFP4 plane's packed runs: the BIT offsets of
 * element (row, col)'s mantissa, exponent-low, exponent-high and sign bits
 * (bits[0..3]; bit b is bit b % 8 of byte b / 8).  In each 16 x 32 run,
 * lane (g, t)'s 8 bytes hold one 32-bit word per tensor-core step whose four
 * A registers each keep their two elements' bits where one shift and one
 * mask put them at bf16 bits 6..8 / 15 and 22..24 / 31.  W8_ERR_SHAPE on a
 * bad argument.  Host-only. */
w8_status w8_mxfp4_code_bits(int64_t k_blocks, int64_t row, int64_t col, int64_t *bits);

/* The packed row that holds source row `row` of a W8_SRC_GATE_UP plane of n
 * rows (W8_LAYOUT_MMA_16x32_GATE_UP); -1 on a bad argument (n not a positive
 * multiple of 16, row outside 0..n-1).  Host-only. */
int64_t w8_gate_up_packed_row(int64_t n, int64_t row);

#ifdef __cplusplus
}
#endif

#endif /* W8_H */
