// w8_noalloc.cu -- w8_gemv_noalloc: the FP8 (w8a16) GEMV for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run a GEMV: code
// that runs inside a host callback, inside a custom allocator or memory-pool
// hook, or under a framework that forbids device allocations while it records
// or replays a step.  w8_gemv needs a caller-provided workspace only when the
// plan splits K across CTAs (planes with few row tiles); this entry point runs
// the same kernel with that scratch taken from a fixed array in the library
// instead, so the caller passes only the build, the activations and the
// output.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kScratchBytes of it until the process exits.  Host code cannot
// use the array's name as a device address (it is a host-side stand-in), so
// the first call on each device looks up the real address with
// cudaGetSymbolAddress, with that device current, zeroes the array (its head
// holds the arrival counters, which every call leaves at zero again) and
// caches the address -- every first call on a device does this, whether or
// not its own plan needs the scratch, so which call pays for it never depends
// on the shape.  That first call therefore synchronises the device and must
// come before any stream capture.  All calls on a device share the array:
// calls that overlap on the GPU (different streams without ordering) race on
// it and must not be issued.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "w8.h"
#include "w8_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(64) << 10; // W8_NOALLOC_SCRATCH_BYTES
static_assert(kScratchBytes == W8_NOALLOC_SCRATCH_BYTES, "keep w8.h in step");
// The arrival counters live in the first kCounterBytes of the array for every
// call and every build (each call leaves them zero), the partial sums after:
// a call's partials never land where another call's counters are.
constexpr size_t kCounterBytes = size_t(4) << 10;

static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices];

// The device address of g_scratch on the current device (set up once).
w8_status scratch_on(int dev, void **out)
{
    if (dev < 0 || dev >= kMaxDevices)
        return W8_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p)
            return W8_ERR_CUDA;
        if (cudaMemset(p, 0, kScratchBytes) != cudaSuccess ||
            cudaDeviceSynchronize() != cudaSuccess)
            return W8_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return W8_OK;
}

} // namespace

extern "C" w8_status w8_gemv_noalloc(const w8_build *b, int plane, const uint16_t *x,
                                     int64_t ldx, int m, uint16_t *y, int64_t ldy, w8_stream s)
{
    if (!b)
        return W8_ERR_NULL;
    if (plane < 0 || plane >= int(b->planes.size()))
        return W8_ERR_PLANE;
    const w8_plane_info &p = b->planes[size_t(plane)];
    if (p.dtype != W8_DT_E4M3FN)
        return W8_ERR_DTYPE;
    if (m < 0 || m > w8::kMaxM)
        return W8_ERR_SHAPE;
    if (m == 0)
        return W8_OK;
    if (!x || !y)
        return W8_ERR_NULL;
    if (ldx < p.k || ldy < p.n)
        return W8_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (ldx & 7) || (reinterpret_cast<uintptr_t>(y) & 1u))
        return W8_ERR_ALIGN;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess)
        return W8_ERR_CUDA;
    if (dev != b->device)
        return W8_ERR_DEVICE;
    // the first call on this device sets the scratch up, whatever its plan
    void *ws = nullptr;
    const w8_status st = scratch_on(dev, &ws);
    if (st != W8_OK)
        return st;

    const w8::Plan plan = w8::make_plan(p.n, p.k, m, b->sm_count);
    if (plan.ws_bytes > 0 && (plan.ws_counters > kCounterBytes ||
                              kCounterBytes + (plan.ws_bytes - plan.ws_counters) > kScratchBytes))
        return W8_ERR_SCRATCH;
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
    w8::set_output_map(a, p, false);
    if (plan.ws_bytes > 0) {
        a.counters = static_cast<int *>(ws);
        a.partial = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kCounterBytes);
    }
    if (w8::launch_gemv(w8::kDtFp8, plan, a, reinterpret_cast<cudaStream_t>(s)) != cudaSuccess)
        return W8_ERR_CUDA;
    return W8_OK;
}
