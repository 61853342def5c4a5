// k_noalloc.cu -- code3 encode whose scratch memory is a fixed device array
// of this library, so that the call allocates nothing.
//
// Who needs it: a caller that compresses on a communication runtime's send
// path, from a host thread that must not block, or inside an application
// whose device memory is owned by a pooling allocator it cannot call into.
// cudaMalloc and cudaFree may synchronize the whole device and take driver
// locks, which can stall or deadlock against communication kernels that are
// still waiting on peers; and a pooled application has no raw cudaMalloc
// budget to spare.  Such a caller cannot hand the ordinary encoder a
// workspace, so this variant uses the array below instead.
//
// The array is shared by every call on a device and keeps the previous
// call's contents; each call clears the part that must start at zero (tile
// counters, per-chunk tile counters and look-back state) on its own stream
// before the launch.  Two calls on one device whose work overlaps on the GPU
// (different streams, no ordering between them) race on the array and give
// undefined results.
#include <atomic>
#include <cstdint>
#include <mutex>

#include "ez_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[EZ_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

std::atomic<void*> g_scratch_ptr[kMaxDevices];
std::mutex g_setup_mutex;

bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Bytes of scratch a code3 encode of `count` chunks touches: the plan's
// workspace prefix up to the end of the look-back state of those chunks.
uint64_t scratch_needed(const ez_plan_s* p, uint32_t count)
{
    return p->off_state_a + (uint64_t)count * p->tpc * 8;
}

// Device address of this device's array; looked up once per device, with
// that device current, on its first call.
ez_status scratch_of(int dev, void** out)
{
    void* ptr = g_scratch_ptr[dev].load(std::memory_order_acquire);
    if (!ptr) {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        ptr = g_scratch_ptr[dev].load(std::memory_order_relaxed);
        if (!ptr) {
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
                return EZ_ERR_CUDA;
            g_scratch_ptr[dev].store(ptr, std::memory_order_release);
        }
    }
    *out = ptr;
    return EZ_OK;
}

}  // namespace

extern "C" ez_status ez_encode_code3_noalloc(ez_plan p, const uint16_t* d_x, uint32_t first,
                                             uint32_t count, const ez_stats_t* d_stats,
                                             uint8_t* d_out, uint64_t out_bytes,
                                             uint64_t* d_sizes, uint32_t* d_status, void* stream)
{
    if (!p || p->codec != EZ_CODEC_CODE3) return EZ_ERR_ARG;
    if (count == 0 || first >= p->W || count > p->W - first) return EZ_ERR_ARG;
    if (!d_stats || !al(d_stats, 8) || !d_out || !al(d_out, 16) || !d_sizes || !al(d_sizes, 8) ||
        !d_status || !al(d_status, 4))
        return EZ_ERR_ARG;
    if (p->n && (!d_x || !al(d_x, 16))) return EZ_ERR_ARG;
    if (out_bytes / p->slot_bytes < count) return EZ_ERR_CAPACITY;
    const uint64_t need = scratch_needed(p, count);
    if (need > (uint64_t)EZ_NOALLOC_SCRATCH_BYTES) return EZ_ERR_CAPACITY;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return EZ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EZ_ERR_UNSUPPORTED;
    void* ws = nullptr;
    ez_status s = scratch_of(dev, &ws);
    if (s != EZ_OK) return s;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, need, st) != cudaSuccess) return EZ_ERR_CUDA;
    const cudaError_t e = ezk::launch_code3_encode(p, d_x, first, count, d_stats, d_out, d_sizes,
                                                   d_status, ezk::ws_view(p, ws), st);
    return e == cudaSuccess ? EZ_OK : EZ_ERR_CUDA;
}
