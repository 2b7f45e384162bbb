// w8_tc.cu -- the w8a16 / bf16 GEMV on the fifth-generation tensor cores
// (tcgen05, tensor memory), for calls with 9..64 decode tokens.
//
// Computes, per output row n and decode token m (ATOM pull request #2980,
// Summary and Changes),
//     y[m,n] = bf16_rne( scale[n] * sum_k widen(W[n,k]) * x[m,k] )
// with fp32 accumulation, like the register-ring kernel in w8_gemv.cu, but
// with the tokens as the N dimension of a 128 x NPAD x 16 tensor-core step
// (NPAD = tokens rounded up to 16), so that one activation tile in shared
// memory serves 128 weight rows instead of 16.
//
// One CTA = 128 output rows (8 row tiles of the packed layout) x one range of
// K blocks, eleven warps:
//   warp 10 (weights): one thread copies the CTA's packed runs into shared
//     memory with bulk asynchronous copies (one per row tile and stage of 4 K
//     blocks: a tile's runs are contiguous), filling every weight stage
//     before the dependency wait -- the plane is bind-time data;
//   warps 0-7 (converters): warp w reads row tile 2 (w % 4) + w / 4 of each
//     stage from shared memory, widens E4M3 to bf16 exactly (bf16 planes pass
//     through) and stores the stage's A operand into tensor memory with one
//     tcgen05.st (TMEM lanes 32 (w % 4) + 16 (w / 4) .., the lane quarter warp
//     w may reach), in natural K order (below);
//   warp 8 (activations): after the dependency wait, one thread copies the
//     activation tiles with tensor-map bulk copies (TMA): one 64-column x
//     tokens box per half stage, each token's 128 bytes a row of the
//     tensor cores' 128-byte-swizzled K-major layout (8-row x 128-byte
//     atoms); columns past K arrive as zeros, rows past the tokens are not
//     copied (their accumulator columns are never stored);
//   warp 9 (issuer): one thread issues the tensor-core steps
//     D[128 x NPAD] += A[128 x 16] (TMEM) * B[16 x NPAD] (shared memory) and
//     commits them to the stages' "empty" barriers.
// Weight, A and activation stages rotate through their slots with mbarriers
// ("full": the producers arrive or the copies complete; "empty": the
// consumers arrive or the issuer commits).  After the last step the
// accumulator D (TMEM columns [0, NPAD)) is read by warps 0-3, one row per
// thread: scale, round, store.  With K split across CTAs, the splits
// of a row block form a thread-block cluster: each CTA parks its partial tile
// in its shared memory and rank r adds rows [r R, (r+1) R) of all the tiles
// in split order through distributed shared memory.  On a gate_up plane
// (packed tile rows g and g+8 are a gate row and its up row) the store maps
// each row to its source row; SiLU-and-multiply pairs TMEM lane l with lane
// l + 8 of the same warp (a shuffle), or row r with row r + 8 of the
// cluster's tiles, and stores one bf16 h per gate row.
//
// K order.  Tensor-core step s of a 32-column block covers columns
// 16s..16s+15 in order: TMEM column c of the step holds columns 16s+2c,
// 16s+2c+1.  tcgen05.st 16x256b.x2 gives lane (g, t) columns 2t, 2t+1 of
// each step for rows g and g+8, i.e. the 4-column units t (step 0) and t+4
// (step 1).  In the packed layout, unit u of a tile lives in packed lane
// 4g + u/2: for FP8 in its words 2(u%2), 2(u%2)+1 (8 bytes), for bf16 in half
// u%2 (16 bytes); the converter reads exactly those from shared memory.
//
// Every mbarrier wait is bounded; on timeout the kernel sets a bit in the
// library's device status word (w8_device_status) and runs to its end, where
// tensor memory is always released.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "w8_device.cuh"
#include "w8_internal.h"

namespace w8 {

// Status word of the tensor-core kernel on each device: bit 0 = a stage
// barrier wait timed out, bit 1 = the accumulator wait timed out.
__device__ int g_tc_status;

namespace {

constexpr int kTcKs = 4;         // K blocks per stage
// Tensor memory of one CTA: the accumulator D in columns [0, NPAD) -- 64
// columns reserved up to 64 tokens -- then A stages of 64 columns (4 K
// blocks x 16): 3 in 256 columns where two CTAs share an SM's 512 columns,
// up to 4 in 512 columns where one CTA has the SM.
W8_HD constexpr int tc_tmem_cols(int occ) { return occ == 2 ? 256 : 512; }
W8_HD constexpr int tc_acol(int npad) { return npad <= 64 ? 64 : npad; }
W8_HD constexpr int tc_a_stages(int npad, int occ)
{
    return (tc_tmem_cols(occ) - tc_acol(npad)) / 64 < 4 ? (tc_tmem_cols(occ) - tc_acol(npad)) / 64 : 4;
}
constexpr int kTcThreads = kTcThreadsPerCta; // 8 converters, activations, issuer, weights
static_assert(kTcThreads == 352, "eleven warps");
constexpr int kWarpAct = 8, kWarpIssue = 9, kWarpW = 10;
static_assert(kTcKs == kTcStageBlocks, "the planner's stage size");
constexpr uint32_t kSpinLimit = 1u << 24;

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return uint32_t(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Wait for the phase with the given parity to complete; false after
// kSpinLimit polls (each poll may itself suspend for a short while).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity)
{
    const uint32_t addr = smem_u32(bar);
    for (uint32_t it = 0; it < kSpinLimit; ++it) {
        uint32_t done;
        asm volatile("{\n\t.reg .pred p;\n\t"
                     "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                     "selp.u32 %0, 1, 0, p;\n\t}"
                     : "=r"(done)
                     : "r"(addr), "r"(parity)
                     : "memory");
        if (done)
            return true;
    }
    return false;
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tm_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tm_load16(uint32_t taddr, float *d)
{
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i)
        d[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tm_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand in the 128-byte
// swizzle layout: rows of 128 bytes (64 bf16 along K) in atoms of 8 rows
// (1024 bytes, 1024-byte aligned), sbo = the byte stride between atoms along
// N; the leading-byte offset is unused in this layout (field 1).  A step of
// 16 columns starts 32 bytes further into the row; the swizzle is applied to
// the absolute address, as the tensor-map copy that wrote the rows did.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t addr, uint32_t sbo)
{
    return uint64_t((addr >> 4) & 0x3FFFu) | (uint64_t(1) << 16) | (uint64_t((sbo >> 4) & 0x3FFFu) << 32) |
           (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// D[tmem] (+)= A[tmem] * B[smem]: bf16 inputs, fp32 accumulate, M = 128.
__device__ __forceinline__ void umma_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_taddr),
                 "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate)
                 : "memory");
}
// Arrive on `bar` once every tensor-core step this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// An L2 policy that marks the lines it fetches first to leave: the weights
// stream through once, and the activations and partial sums they would
// otherwise push out of L2 are read again (measured: 2-4 % on FP8 planes at
// 17-64 tokens, 8 % on bf16 o_proj at 32 tokens).
__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
// Bulk asynchronous copy global -> shared (16-byte aligned, a multiple of 16
// bytes) whose completion counts `bytes` on the barrier's transaction count;
// its lines leave L2 first.
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy_evict_first())
                 : "memory");
}
// 16 bytes of fp32 through L2 only (partial sums other CTAs wrote).
__device__ __forceinline__ float4 ld_cg_f32x4(const float4 *p)
{
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint4 ld_shared16(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Tensor-map bulk copy of a 2-D box (inner coordinate c0, outer c1) into
// shared memory; its bytes count on the barrier's transaction count.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
                     dst),
                 "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
                 : "memory");
}
// The A operand of a whole stage (4 blocks = 64 columns) for 16 rows:
// tcgen05.st 16x256b.x8, registers 8j..8j+7 = block j in tm_store_a's order.
__device__ __forceinline__ void tm_store_stage(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.16x256b.x8.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
                 "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
                 "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
                 "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]),
                 "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

// Units t and t+4 of rows g and g+8 of one staged run (see "K order") as the
// eight A registers of lane (g, t).
template <bool kFp8>
__device__ __forceinline__ void a_units(uint32_t *r, uint32_t run, int g, int t)
{
    if constexpr (kFp8) {
        // 8 bytes = words (row g, g+8 at cols +0,+1), (row g, g+8 at cols +2,+3)
        const uint32_t o0 = run + uint32_t((4 * g + (t >> 1)) * 16 + (t & 1) * 8);
        uint32_t u0, u1, v0, v1;
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(u0), "=r"(u1) : "r"(o0));
        asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(o0 + 32));
        r[0] = widen_e4m3x2<kSelRowG>(u0);
        r[1] = widen_e4m3x2<kSelRowG>(u1);
        r[2] = widen_e4m3x2<kSelRowG8>(u0);
        r[3] = widen_e4m3x2<kSelRowG8>(u1);
        r[4] = widen_e4m3x2<kSelRowG>(v0);
        r[5] = widen_e4m3x2<kSelRowG>(v1);
        r[6] = widen_e4m3x2<kSelRowG8>(v0);
        r[7] = widen_e4m3x2<kSelRowG8>(v1);
    } else {
        // 16 bytes = (row g, cols +0,+1), (row g+8, +0,+1), (row g, +2,+3), (row g+8, +2,+3)
        const uint32_t o0 = run + uint32_t((t & 1) * 512 + (4 * g + (t >> 1)) * 16);
        const uint4 u = ld_shared16(o0), v = ld_shared16(o0 + 32);
        r[0] = u.x;
        r[1] = u.z;
        r[2] = u.y;
        r[3] = u.w;
        r[4] = v.x;
        r[5] = v.z;
        r[6] = v.y;
        r[7] = v.w;
    }
}

// The fp32 sums of one row's four tokens over the splits of a row block
// (cluster ranks 0 .. splits - 1): every split CTA's tile at the same
// shared-memory offset, loaded first (all independent), then added in split
// order.
__device__ __forceinline__ float4 cluster_sum4(uint32_t off, int splits)
{
    float4 p[kTcMaxSplits];
#pragma unroll
    for (int r = 0; r < kTcMaxSplits; ++r) {
        p[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (r < splits) {
            uint32_t remote;
            asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(off), "r"(r));
            asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
                         : "=f"(p[r].x), "=f"(p[r].y), "=f"(p[r].z), "=f"(p[r].w)
                         : "r"(remote)
                         : "memory");
        }
    }
    float4 v = p[0];
#pragma unroll
    for (int r = 1; r < kTcMaxSplits; ++r) {
        if (r < splits) {
            v.x += p[r].x;
            v.y += p[r].y;
            v.z += p[r].z;
            v.w += p[r].w;
        }
    }
    return v;
}

template <bool kFp8, int NPAD, int OCC>
__global__ void __launch_bounds__(kTcThreads, OCC)
    tc_gemv_kernel(const GemvArgs a, const __grid_constant__ CUtensorMap tmx)
{
    constexpr int kRun = kFp8 ? kRunFp8 : kRunBf16;
    constexpr int kNW = tc_stages(kFp8, NPAD, OCC).nw; // weight stages (shared memory)
    constexpr int kNB = tc_stages(kFp8, NPAD, OCC).nb; // activation stages (shared memory)
    constexpr int kNA = tc_a_stages(NPAD, OCC);        // A stages (tensor memory)
    constexpr uint32_t kTmemCols = tc_tmem_cols(OCC);
    constexpr int kACol = tc_acol(NPAD);
    static_assert(kNA >= 3 && kACol + kNA * 64 <= int(kTmemCols) && kACol >= NPAD, "tensor memory map");
    constexpr int kTileW = kTcKs * kRun;          // one row tile's runs of a stage
    constexpr int kStageW = 8 * kTileW;
    constexpr int kHalfB = NPAD * 128;            // activation bytes of 64 columns (2 K blocks)
    constexpr int kStageB = 2 * kHalfB;           // ... of a stage (4 K blocks)
    static_assert(kTcKs * kTileK == 128 && kHalfB % 1024 == 0 && kStageW % 1024 == 0,
                  "swizzle atoms stay 1024-byte aligned");
    constexpr int kRedPitch = NPAD + 4;           // floats per row of the split-K exchange tile
    // instruction descriptor: D f32, A and B bf16, both K-major, N = NPAD, M = 128
    constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(NPAD >> 3) << 17) |
                                (uint32_t(128 >> 4) << 24);
    static_assert(NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 256, "M = 128 needs N in 16..256, step 16");
    static_assert(OCC == tc_occ(NPAD) || (OCC == 1 && NPAD == 64), "the planner's instances");
    static_assert(128 * kRedPitch * 4 <= tc_smem_bytes(kFp8, NPAD, OCC),
                  "the exchange tile reuses the stages' shared memory");
    static_assert(kNW * kStageW + kNB * kStageB + kTcSmemAlign == tc_smem_bytes(kFp8, NPAD, OCC),
                  "stage geometry");

    extern __shared__ __align__(16) uint8_t s_dyn[]; // kNW weight stages, then kNB B stages
    __shared__ __align__(8) uint64_t bar_full_w[kNW], bar_empty_w[kNW];
    __shared__ __align__(8) uint64_t bar_full_a[kNA], bar_empty_a[kNA];
    __shared__ __align__(8) uint64_t bar_full_b[kNB], bar_empty_b[kNB];
    __shared__ __align__(8) uint64_t bar_done;
    __shared__ uint32_t s_tmem;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // The splits of a row block form one cluster: cluster rank = K range.
    const int sp = int(blockIdx.x) % a.splits;          // K range (split)
    const int rb = int(blockIdx.x) / a.splits;          // row block: rows rb*128 ..
    const int cb0 = int((int64_t(sp) * a.kb) / a.splits); // this CTA's K blocks
    const int cnb = int((int64_t(sp + 1) * a.kb) / a.splits) - cb0;
    const int nst = (cnb + kTcKs - 1) / kTcKs;          // stages
    const int row0 = rb * 128;
    const int tile0 = rb * 8;
    // the stages start at the first 1024-byte boundary of the dynamic shared
    // memory (the swizzle atoms of the activation stages need it; the launch
    // adds kTcSmemAlign bytes for the shift)
    uint8_t *const s_w = s_dyn + ((1024u - (smem_u32(s_dyn) & 1023u)) & 1023u);
    uint8_t *const s_b = s_w + kNW * kStageW;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNW; ++s) {
            mbar_init(&bar_full_w[s], 1);
            mbar_init(&bar_empty_w[s], 8);
        }
        for (int s = 0; s < kNA; ++s) {
            mbar_init(&bar_full_a[s], 8);
            mbar_init(&bar_empty_a[s], 1);
        }
        for (int s = 0; s < kNB; ++s) {
            mbar_init(&bar_full_b[s], 1);
            mbar_init(&bar_empty_b[s], 1);
        }
        mbar_init(&bar_done, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&s_tmem)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = s_tmem;
    pdl_launch_dependents();

    if (warp == kWarpW) {
        // ---- weights: packed runs -> shared memory (bulk copies) --------------
        // The packed plane is written only by w8_bind, which finishes before any
        // GEMV is launched, so this runs ahead of the dependency wait.  Lane h
        // copies row tile h's runs of the stage (the copies go out in parallel).
        int tiles = a.rt - tile0;
        tiles = tiles > 8 ? 8 : tiles;
        bool ok = true;
        for (int st = 0; st < nst && ok; ++st) {
            const int s = st % kNW;
            if (st >= kNW)
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_empty_w[s], uint32_t((st / kNW - 1) & 1)));
            if (!ok)
                break;
            const int nb = cnb - st * kTcKs < kTcKs ? cnb - st * kTcKs : kTcKs;
            if (lane == 0)
                mbar_expect_tx(&bar_full_w[s], uint32_t(tiles * nb * kRun));
            __syncwarp();
            if (lane < tiles)
                bulk_copy(smem_u32(s_w + s * kStageW + lane * kTileW),
                          a.wp + (int64_t(tile0 + lane) * a.kb + cb0 + st * kTcKs) * kRun,
                          uint32_t(nb * kRun), &bar_full_w[s]);
        }
        if (!ok && lane == 0)
            atomicOr(&g_tc_status, 1);
    } else if (warp < 8) {
        // ---- converters: staged weights -> widened A in tensor memory ---------
        // warp w widens row tile 2 (w % 4) + w / 4 into TMEM lanes
        // 32 (w % 4) + 16 (w / 4) .. + 15 (a warp reaches lane quarter w % 4).
        const int h = 2 * (warp & 3) + (warp >> 2);
        const uint32_t okt = tile0 + h < a.rt;
        const uint32_t lanes = uint32_t(32 * (warp & 3) + 16 * (warp >> 2)) << 16;
        const int g = lane >> 2, t = lane & 3;
        bool ok = true;
        for (int st = 0; st < nst && ok; ++st) {
            const int sw = st % kNW, sa_ = st % kNA;
            ok = __all_sync(0xffffffffu, mbar_wait(&bar_full_w[sw], uint32_t((st / kNW) & 1)));
            if (ok && st >= kNA)
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_empty_a[sa_], uint32_t((st / kNA - 1) & 1)));
            if (!ok)
                break;
            const uint32_t w0 = smem_u32(s_w + sw * kStageW + h * kTileW);
            const int nb = cnb - st * kTcKs < kTcKs ? cnb - st * kTcKs : kTcKs;
            uint32_t r[32];
#pragma unroll
            for (int j = 0; j < kTcKs; ++j) {
                if (okt && j < nb) {
                    a_units<kFp8>(r + 8 * j, w0 + j * kRun, g, t);
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e)
                        r[8 * j + e] = 0; // blocks past the stage's end are never read
                }
            }
            tm_store_stage(tbase + lanes + uint32_t(kACol + sa_ * kTcKs * 16), r);
            tm_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&bar_empty_w[sw]); // the stage's weights are in TMEM now
                mbar_arrive(&bar_full_a[sa_]);
            }
        }
        if (!ok && lane == 0)
            atomicOr(&g_tc_status, 1);
    } else if (warp == kWarpAct) {
        // ---- activations: x -> B tiles in shared memory (tensor-map copies) -----
        // Lane h < 2 copies columns 64h..64h+63 of the stage (K blocks 2h,
        // 2h+1) as one 64-column x min(m, NPAD)-row box into its half of the
        // slot (rows past m keep whatever the slot held: they meet only the
        // accumulator columns of tokens >= m, which are never stored); a
        // last stage of one or three blocks copies a whole half, whose
        // columns past the CTA's range no step reads.
        pdl_wait(); // x may be the previous kernel's output
        bool ok = true;
        for (int st = 0; st < nst && ok; ++st) {
            const int s = st % kNB;
            if (st >= kNB)
                ok = __all_sync(0xffffffffu, mbar_wait(&bar_empty_b[s], uint32_t((st / kNB - 1) & 1)));
            if (!ok)
                break;
            const int nb = cnb - st * kTcKs < kTcKs ? cnb - st * kTcKs : kTcKs;
            const int nh = (nb + 1) >> 1; // 64-column halves to copy
            if (lane == 0)
                mbar_expect_tx(&bar_full_b[s], uint32_t(nh * 128 * (a.m < NPAD ? a.m : NPAD)));
            __syncwarp();
            if (lane < nh) {
                const uint32_t dst = smem_u32(s_b + s * kStageB + lane * kHalfB);
                const int c0 = (cb0 + st * kTcKs) * kTileK + 64 * lane;
                tma_load_2d(dst, &tmx, c0, 0, &bar_full_b[s]);
            }
        }
        if (!ok && lane == 0)
            atomicOr(&g_tc_status, 1);
    } else if (warp == kWarpIssue && lane == 0) {
        // ---- issuer: one thread drives the tensor cores --------------------------
        // The descriptors of a stage are its slot's base plus compile-time
        // offsets (the address field holds addr >> 4, and every shared-memory
        // address stays below 256 KB, so adding never carries out of it); a
        // full stage is issued unrolled, a partial last stage block by block.
        const uint64_t bdesc0 = smem_desc_sw128(smem_u32(s_b), 1024);
        bool ok = true;
        for (int st = 0; st < nst && ok; ++st) {
            const int sa_ = st % kNA, sb = st % kNB;
            ok = mbar_wait(&bar_full_a[sa_], uint32_t((st / kNA) & 1)) &&
                 mbar_wait(&bar_full_b[sb], uint32_t((st / kNB) & 1));
            if (!ok)
                break;
            tc_fence_after();
            const uint64_t bd = bdesc0 + uint64_t((sb * kStageB) >> 4);
            const uint32_t at = tbase + uint32_t(kACol + sa_ * kTcKs * 16);
            const int nb = cnb - st * kTcKs < kTcKs ? cnb - st * kTcKs : kTcKs;
            if (nb == kTcKs) {
#pragma unroll
                for (int j = 0; j < kTcKs; ++j)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        umma_ts(tbase, at + uint32_t(j * 16 + q * 8),
                                bd + uint64_t(((j >> 1) * kHalfB + ((j & 1) * 2 + q) * 32) >> 4), kIdesc,
                                uint32_t(st | j | q));
            } else {
                for (int j = 0; j < nb; ++j)
#pragma unroll
                    for (int q = 0; q < 2; ++q)
                        umma_ts(tbase, at + uint32_t(j * 16 + q * 8),
                                bd + uint64_t(((j >> 1) * kHalfB + ((j & 1) * 2 + q) * 32) >> 4), kIdesc,
                                uint32_t(st | j | q));
            }
            umma_commit(&bar_empty_a[sa_]);
            umma_commit(&bar_empty_b[sb]);
        }
        umma_commit(&bar_done);
        if (!ok)
            atomicOr(&g_tc_status, 1);
    }

    // ---- epilogue: D (128 rows x NPAD tokens) from tensor memory -------------
    // Warps 0-3 read their lane quarter, 16 token columns at a time.
    if (warp < 4) {
        if (!mbar_wait(&bar_done, 0) && lane == 0)
            atomicOr(&g_tc_status, 2);
        tc_fence_after();
    }
    const int row = row0 + 32 * warp + lane;
    const uint32_t dq = tbase + (uint32_t(32 * (warp & 3)) << 16);
    if (a.splits == 1) {
        pdl_wait(); // every global write comes after the previous kernel
        if (warp < 4) {
            const float sc = (kFp8 && row < a.n) ? __ldg(a.scale + row) : 1.0f;
            const int col = out_col(row, a.act != kActPlain, a.half);
            // SiLU-and-multiply: lane l (l & 8 == 0, a gate row) takes the up
            // row's sums from lane l + 8 (row + 8) of the same warp
            const bool gate = a.act == kActSiluMul && (lane & 8) == 0 && row < a.n;
            const float scu = (kFp8 && gate) ? __ldg(a.scale + row + 8) : 1.0f;
#pragma unroll
            for (int c = 0; c < NPAD / 16; ++c) {
                float d[16];
                tm_load16(dq + uint32_t(16 * c), d);
                tm_wait_ld();
                if (a.act == kActSiluMul) {
                    float du[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        du[e] = __shfl_down_sync(0xffffffffu, d[e], 8);
                    if (gate) {
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (16 * c + e < a.m)
                                a.y[int64_t(16 * c + e) * a.ldy + col] =
                                    silu_mul_bf16(kFp8 ? sc * d[e] : d[e], kFp8 ? scu * du[e] : du[e]);
                    }
                } else if (row < a.n) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        if (16 * c + e < a.m)
                            a.y[int64_t(16 * c + e) * a.ldy + col] = to_bf16(kFp8 ? sc * d[e] : d[e]);
                }
            }
        }
    } else if (a.gsplit) {
        // Split K across CTAs that meet in the workspace (no cluster): each
        // CTA stores its partial tile, [split][row][token] with the tokens
        // padded to a multiple of 4 (mq), and counts its arrival; the last CTA
        // of the row block adds the splits in split order (all of a quad's
        // loads in flight at once), then scales, rounds and stores.  Every
        // global write follows the wait for the previous kernel (the
        // workspace may be its too).
        pdl_wait();
        const int mq = (a.m + 3) & ~3;
        const int64_t rows_pad = int64_t(a.rt) * kTileN;
        if (warp < 4) {
            // the tensor-memory loads are warp-collective: the whole warp
            // loads, and only the rows inside the plane are stored
            float4 *dst = reinterpret_cast<float4 *>(a.partial + (int64_t(sp) * rows_pad + row) * mq);
#pragma unroll
            for (int c = 0; c < NPAD / 16; ++c) {
                if (16 * c < mq) { // uniform across the warp
                    float d[16];
                    tm_load16(dq + uint32_t(16 * c), d);
                    tm_wait_ld();
                    if (row < a.n) {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (16 * c + 4 * q < mq)
                                dst[4 * c + q] =
                                    make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
                    }
                }
            }
        }
        __threadfence();
        __syncthreads();
        __shared__ int s_last;
        if (threadIdx.x == 0)
            s_last = atomicAdd(a.counters + rb, 1) == a.splits - 1;
        __syncthreads();
        if (s_last) {
            __threadfence();
            const int row_end = row0 + 128 < a.n ? row0 + 128 : a.n;
            const int quads = mq / 4;
            const int items = (row_end - row0) * quads; // (row, token quad), quads fastest
            const float4 *base = reinterpret_cast<const float4 *>(a.partial + int64_t(row0) * mq);
            const int64_t split_stride = rows_pad * quads; // in float4
            // the splits of one (row, quad), loaded together, added in split order
            auto split_sum = [&](int off) {
                float4 p[kTcMaxGlobalSplits];
#pragma unroll
                for (int q = 0; q < kTcMaxGlobalSplits; ++q) {
                    p[q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (q < a.splits)
                        p[q] = ld_cg_f32x4(base + q * split_stride + off);
                }
                float4 v = p[0];
#pragma unroll
                for (int q = 1; q < kTcMaxGlobalSplits; ++q) {
                    if (q < a.splits) {
                        v.x += p[q].x;
                        v.y += p[q].y;
                        v.z += p[q].z;
                        v.w += p[q].w;
                    }
                }
                return v;
            };
            for (int it = threadIdx.x; it < items; it += kTcThreads) {
                const int rl = it / quads;
                const int q4 = it - rl * quads;
                const int orow = row0 + rl;
                if (a.act == kActSiluMul && (rl & 8))
                    continue; // an up row: added with its gate row (rl - 8)
                const float4 v = split_sum(it);
                const float out[4] = {v.x, v.y, v.z, v.w};
                const float sc = kFp8 ? __ldg(a.scale + orow) : 1.0f;
                const int col = out_col(orow, a.act != kActPlain, a.half);
                if (a.act != kActSiluMul) {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * q4 + e < a.m)
                            a.y[int64_t(4 * q4 + e) * a.ldy + col] = to_bf16(kFp8 ? sc * out[e] : out[e]);
                } else {
                    const float4 vu = split_sum(it + 8 * quads);
                    const float up[4] = {vu.x, vu.y, vu.z, vu.w};
                    const float scu = kFp8 ? __ldg(a.scale + orow + 8) : 1.0f;
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (4 * q4 + e < a.m)
                            a.y[int64_t(4 * q4 + e) * a.ldy + col] =
                                silu_mul_bf16(kFp8 ? sc * out[e] : out[e], kFp8 ? scu * up[e] : up[e]);
                }
            }
            if (threadIdx.x == 0)
                a.counters[rb] = 0; // ready for the next call on this workspace
        }
    } else {
        // Split K across the CTAs of a cluster (rank = split): each CTA parks
        // its partial tile in its own shared memory (the stages are free:
        // every step has completed and every copy has landed), then rank r adds the splits of rows
        // [r R, (r+1) R) in split order, reading the others' tiles directly.
        float *red = reinterpret_cast<float *>(s_dyn);
        if (warp < 4) {
            float4 *dst = reinterpret_cast<float4 *>(red + (32 * warp + lane) * kRedPitch);
#pragma unroll
            for (int c = 0; c < NPAD / 16; ++c) {
                float d[16];
                tm_load16(dq + uint32_t(16 * c), d);
                tm_wait_ld();
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[4 * c + q] = make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
            }
        }
        __syncwarp(); // the cluster barrier is warp-aligned: reconverge first
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
        pdl_wait();
        const int r_lo = (sp * 128) / a.splits; // split sp adds rows [r_lo, r_lo + rows_per)
        const int rows_per = ((sp + 1) * 128) / a.splits - r_lo;
        const int items = rows_per * (NPAD / 4);
        const uint32_t red_local = smem_u32(red);
        for (int it = threadIdx.x; it < items; it += kTcThreads) {
            const int q = it / rows_per;           // token quad
            const int rl = r_lo + (it - q * rows_per);
            const int orow = row0 + rl;
            if (4 * q >= a.m || orow >= a.n)
                continue;
            if (a.act == kActSiluMul && (rl & 8))
                continue; // an up row: added with its gate row (rl - 8), whichever split has it
            const uint32_t off = red_local + uint32_t((rl * kRedPitch + 4 * q) * 4);
            const float4 v = cluster_sum4(off, a.splits);
            const float sc = kFp8 ? __ldg(a.scale + orow) : 1.0f;
            const float out[4] = {v.x, v.y, v.z, v.w};
            const int col = out_col(orow, a.act != kActPlain, a.half);
            if (a.act != kActSiluMul) {
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q + e < a.m)
                        a.y[int64_t(4 * q + e) * a.ldy + col] = to_bf16(kFp8 ? sc * out[e] : out[e]);
            } else {
                const float4 vu = cluster_sum4(off + uint32_t(8 * kRedPitch * 4), a.splits);
                const float scu = kFp8 ? __ldg(a.scale + orow + 8) : 1.0f;
                const float up[4] = {vu.x, vu.y, vu.z, vu.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (4 * q + e < a.m)
                        a.y[int64_t(4 * q + e) * a.ldy + col] =
                            silu_mul_bf16(kFp8 ? sc * out[e] : out[e], kFp8 ? scu * up[e] : up[e]);
            }
        }
        // no CTA leaves while another may still read its tile
        __syncwarp();
        asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
    }

    // ---- release tensor memory -------------------------------------------------
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tbase), "r"(kTmemCols)
                     : "memory");
    }
}

template <bool kFp8>
void *tc_instance(int npad, int occ)
{
    if (occ != tc_occ(npad))
        return npad == 64 && occ == 1 ? reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 64, 1>) : nullptr;
    switch (npad) {
    case 16: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 16, tc_occ(16)>);
    case 32: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 32, tc_occ(32)>);
    case 48: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 48, tc_occ(48)>);
    case 64: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 64, tc_occ(64)>);
    case 96: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 96, tc_occ(96)>);
    case 128: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 128, tc_occ(128)>);
    case 192: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 192, tc_occ(192)>);
    case 256: return reinterpret_cast<void *>(&tc_gemv_kernel<kFp8, 256, tc_occ(256)>);
    default: return nullptr;
    }
}
constexpr int kTcNpads[] = {16, 32, 48, 64, 96, 128, 192, 256};

} // namespace

cudaError_t prepare_tc_kernels()
{
    for (int npad : kTcNpads) {
        for (int occ = 1; occ <= 2; ++occ) {
            for (int f = 0; f < 2; ++f) {
                void *fn = f ? tc_instance<true>(npad, occ) : tc_instance<false>(npad, occ);
                if (!fn)
                    continue;
                cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     tc_smem_bytes(f == 1, npad, occ));
                if (e != cudaSuccess)
                    return e;
            }
        }
    }
    return cudaSuccess;
}

namespace {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The activations x [m][ldx] bf16 as a 2-D tensor (K columns, m rows) read in
// 64-column (128-byte) x min(m, npad)-row boxes with the 128-byte swizzle;
// outside K the boxes are zero.
bool encode_x_map(CUtensorMap *map, const GemvArgs &a, int npad)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc)
        return false;
    const cuuint64_t dims[2] = {cuuint64_t(a.k), cuuint64_t(a.m)};
    const cuuint64_t strides[1] = {cuuint64_t(a.ldx) * 2};
    // m rows, not npad: the stage rows of tokens m..npad-1 are never written
    // (they feed only accumulator columns that are never stored), so no copy
    // reads past the tensor's last row (measured: boxes with out-of-range
    // rows, filled by the copy engine, made 17..31 tokens slower than 32)
    const cuuint32_t box[2] = {64, cuuint32_t(a.m < npad ? a.m : npad)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t *>(a.x), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

} // namespace

cudaError_t launch_tc(bool fp8, const Plan &plan, const GemvArgs &a, cudaStream_t s)
{
    void *fn = fp8 ? tc_instance<true>(plan.npad, plan.occ) : tc_instance<false>(plan.npad, plan.occ);
    if (!fn)
        return cudaErrorInvalidValue;
    alignas(64) CUtensorMap tmx;
    if (!encode_x_map(&tmx, a, plan.npad))
        return cudaErrorInvalidValue;
    GemvArgs aa = a;
    aa.gsplit = plan.splits > 1 && plan.cluster == 1; // the splits meet in the workspace
    void *args[] = {&aa, &tmx};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(unsigned(plan.grid));
    cfg.blockDim = dim3(kTcThreads);
    cfg.dynamicSmemBytes = size_t(tc_smem_bytes(fp8, plan.npad, plan.occ));
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // a cluster: the splits of one row block (they exchange partial tiles),
    // unless they meet in the workspace
    const int csz = plan.cluster;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = unsigned(csz);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = csz > 1 ? 2 : 1;
    return cudaLaunchKernelExC(&cfg, fn, args);
}

cudaError_t tc_status(int *out, bool reset)
{
    cudaError_t e = cudaMemcpyFromSymbol(out, g_tc_status, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_tc_status, &zero, sizeof(int));
    }
    return e;
}

} // namespace w8
