// k_noalloc.cu -- gather-decode whose scratch memory is a fixed device array
// of this library, so that the call allocates nothing.
//
// Who needs it: a caller that decodes received payloads from inside a
// communication runtime's progress path, a host thread that must not block,
// or an application whose device memory is owned by a pooling allocator it
// cannot call into.  cudaMalloc and cudaFree may synchronize the whole device
// and take driver locks, which can stall or deadlock against communication
// kernels that are still waiting on peers; and a pooled application has no
// raw cudaMalloc budget to spare.  Such a caller cannot hand the ordinary
// gather-decode a workspace, so this variant uses the array below instead.
//
// The array is shared by every call on a device and keeps the previous
// call's contents; each call clears the part that must start at zero (tile
// counters and look-back state) on its own stream before the launch.  Two
// calls on one device whose work overlaps on the GPU (different streams, no
// ordering between them) race on the array and give undefined results.
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

// Bytes of scratch the gather-decode of plan p touches: the zeroed prefix of
// the plan's workspace up to the end of the look-back state it uses.  The
// later regions (encoder-only exponent buffer) are never read by a decoder.
uint64_t scratch_needed(const ez_plan_s* p)
{
    const uint64_t state = (uint64_t)p->W * p->tpc * 8;
    return p->codec == EZ_CODEC_CODE3 ? p->off_state_a + state : p->off_state_b + state;
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

extern "C" ez_status ez_gather_decode_noalloc(ez_plan p, const uint8_t* d_recv,
                                              const uint64_t* d_offsets, uint8_t* d_recv_cache,
                                              uint16_t* d_full_out, uint32_t* d_status,
                                              void* stream)
{
    if (!p) return EZ_ERR_ARG;
    if (!d_recv || !al(d_recv, 16) || !d_offsets || !al(d_offsets, 8) || !d_status ||
        !al(d_status, 4))
        return EZ_ERR_ARG;
    const bool reuse = p->codec != EZ_CODEC_CODE3;
    if (p->n && (!d_full_out || !al(d_full_out, 16))) return EZ_ERR_ARG;
    if (reuse && p->n && (!d_recv_cache || !al(d_recv_cache, 16))) return EZ_ERR_ARG;
    const uint64_t need = scratch_needed(p);
    if (need > (uint64_t)EZ_NOALLOC_SCRATCH_BYTES) return EZ_ERR_CAPACITY;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return EZ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EZ_ERR_UNSUPPORTED;
    void* ws = nullptr;
    ez_status s = scratch_of(dev, &ws);
    if (s != EZ_OK) return s;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(ws, 0, need, st) != cudaSuccess) return EZ_ERR_CUDA;
    const ezk::WsView w = ezk::ws_view(p, ws);
    const cudaError_t e =
        reuse ? ezk::launch_reuse_decode(p, d_recv, d_offsets, 0, 0, p->W, d_recv_cache,
                                         d_full_out, d_status, w, st)
              : ezk::launch_code3_decode(p, d_recv, d_offsets, 0, p->W, d_full_out, d_status, w,
                                         st);
    return e == cudaSuccess ? EZ_OK : EZ_ERR_CUDA;
}
