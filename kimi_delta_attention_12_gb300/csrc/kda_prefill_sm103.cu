// kda_prefill_sm103.cu -- chunked KDA prefill on tcgen05/TMEM (placeholder
// until the tensor-core kernel lands; the API does not route here yet).
#include <cuda_runtime.h>

#include "kda_internal.h"

namespace kda {

size_t chunked_workspace_bytes(int32_t N, int32_t H) {
    return 256 + (size_t)N * H * sizeof(int32_t);
}

cudaError_t launch_chunked_prefill(const ChunkedParams& p, cudaStream_t stream) {
    (void)p; (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace kda
