// ca_decode_attention_static_ws: decode attention for callers that cannot
// allocate device memory at the point of the call.
//
// ca_decode_attention needs a caller-provided device workspace for the
// partial results of the two phases.  Some callers cannot allocate one: a
// component running inside a server that has already reserved the whole
// device memory budget for its own pool, code on a latency-critical path
// where cudaMalloc / cudaFree would synchronise the device, or a plugin whose
// host forbids allocation inside its callbacks.  This entry point takes the
// partials from a fixed buffer that the library itself holds in device
// memory, so the call allocates nothing.
//
// The buffer is a file-scope __device__ array of CA_STATIC_WS_BYTES bytes.
// Every GPU that loads the library keeps it until the process exits.  All
// calls share it and it keeps whatever the last call left there: the kernels
// write every partial before reading it, so nothing has to be cleared, but
// two calls that overlap on the GPU (different streams, or different host
// threads) would overwrite each other's partials.
#include <cuda_runtime.h>

#include <atomic>
#include <mutex>

#include "ca_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[CA_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_lookup_lock;                       // taken only by a device's first call
std::atomic<void*> g_ws_ptr[kMaxDevices] = {};

// Device address of g_static_ws on `device` (which must be current).  Looked
// up once per device: in host code the array's name is only a host-side
// stand-in, not a device address.  After the first call a device's address
// is read without a lock, so host threads driving different GPUs do not
// serialise here.  The address stays valid for the life of the device's
// primary context; a cudaDeviceReset after the first call would leave it
// stale (the entry point does not support that).
int static_ws_address(int device, void** out) {
    if (device < 0 || device >= kMaxDevices) return CA_ERR_INVALID;
    void* ptr = g_ws_ptr[device].load(std::memory_order_acquire);
    if (!ptr) {
        std::lock_guard<std::mutex> guard(g_lookup_lock);
        ptr = g_ws_ptr[device].load(std::memory_order_relaxed);
        if (!ptr) {
            if (cudaGetSymbolAddress(&ptr, g_static_ws) != cudaSuccess || !ptr) return CA_ERR_CUDA;
            g_ws_ptr[device].store(ptr, std::memory_order_release);
        }
    }
    *out = ptr;
    return CA_OK;
}

}  // namespace

extern "C" int ca_decode_attention_static_ws(const ca_pool* pool_, const ca_sched* sched_,
                                             int32_t layer, const void* q_dev, void* out_dev,
                                             float scale, void* stream) {
    const ca::Pool* pool = reinterpret_cast<const ca::Pool*>(pool_);
    const ca::Sched* s = reinterpret_cast<const ca::Sched*>(sched_);
    if (!pool || !s || !pool->kv || s->pool != pool || !s->dev) return CA_ERR_INVALID;
    if (s->generation != pool->generation) return CA_ERR_STALE;
    if (layer < 0 || layer >= pool->cfg.n_layers) return CA_ERR_INVALID;
    if (!q_dev || !out_dev || (reinterpret_cast<uintptr_t>(q_dev) & 15) ||
        (reinterpret_cast<uintptr_t>(out_dev) & 15))
        return CA_ERR_INVALID;
    if (s->ws.total > (size_t)CA_STATIC_WS_BYTES) return CA_ERR_SCRATCH_LIMIT;
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return CA_ERR_CUDA;
    if (device != pool->device) return CA_ERR_INVALID;
    void* ws = nullptr;
    int st = static_ws_address(device, &ws);
    if (st) return st;
    const ca::AttnParams a = ca::attn_params(*pool, *s, layer, q_dev, out_dev, scale, ws);
    return ca::launch_attention(*pool, *s, a, stream);
}
