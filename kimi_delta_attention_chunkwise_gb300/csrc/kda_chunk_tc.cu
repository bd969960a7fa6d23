// kda_chunk_tc.cu -- tensor-core chunk engine (placeholder until the
// tcgen05 kernels land).
#include "kda_internal.cuh"

namespace kda {

size_t chunk_tc_workspace_bytes(int32_t, int32_t, int32_t) { return 0; }

cudaError_t launch_chunk_tc(const ChunkArgs &a, void *, size_t, cudaStream_t stream) {
    return launch_chunk_simt(a, stream);
}

}  // namespace kda
