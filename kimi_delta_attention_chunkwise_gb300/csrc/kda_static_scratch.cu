// kda_static_scratch.cu -- chunkwise prefill for callers that must not
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run prefill: code that runs inside a host framework that owns all
// device memory and forbids other allocations, code on a latency-critical
// path where an allocation can synchronise the device, or long-running
// services that must not grow their memory footprint after start-up.  For
// them, kda_chunk_fwd_static runs the same kernels as kda_chunk_fwd_ws but
// takes its scratch from a fixed array that the library reserves in device
// memory when it is loaded.
//
// Costs of that choice, stated once here and in include/kda.h:
//   * the array (KDA_STATIC_SCRATCH_BYTES) is held on every GPU that loads
//     the library, until the process exits, whether or not this entry point
//     is ever called;
//   * every call shares it, so two calls whose work overlaps on the GPU
//     (different streams, or different host threads) race on it and give
//     wrong results -- serialise them;
//   * the array keeps whatever the previous call left in it.  Nothing in it
//     has to start at zero: the kernels write every scratch byte before they
//     read it, so no clearing is done;
//   * problems needing more scratch than the array holds are rejected.
//
// In host code the array's name is only a host-side stand-in, not a device
// address.  Its device address is looked up once per device, with that device
// current, by the first call made on the device; make that first call before
// any stream capture begins.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "kda_internal.cuh"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[KDA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_static_scratch on the current device (set-up on first
// use per device).  Returns nullptr if the lookup fails.
void *static_scratch_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr) {
            (void)cudaGetLastError();
            return nullptr;
        }
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" kdaStatus_t kda_chunk_fwd_static(const void *q, const void *k, const void *v,
                                            const float *log_alpha, const float *beta,
                                            float scale, const float *initial_state,
                                            const int32_t *cu_seqlens, void *out,
                                            float *final_state, const kdaShape_t *shape,
                                            cudaStream_t stream) {
    size_t need = 0;
    kdaStatus_t st = kda_chunk_fwd_workspace_size(shape, &need);
    if (st != KDA_SUCCESS) return st;
    if (need > (size_t)KDA_STATIC_SCRATCH_BYTES) return KDA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    if (need > 0) {
        scratch = static_scratch_address();
        if (!scratch) return KDA_ERR_CUDA;
    }
    return kda_chunk_fwd_ws(q, k, v, log_alpha, beta, scale, initial_state, cu_seqlens, out,
                            final_state, shape, scratch, (size_t)KDA_STATIC_SCRATCH_BYTES, stream);
}
