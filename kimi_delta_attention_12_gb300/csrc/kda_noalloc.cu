// kda_noalloc.cu -- kda_prefill for callers that cannot allocate device memory.
//
// Some callers of this library are not allowed to allocate device memory
// themselves: a plugin running inside a host framework that owns every byte
// of device memory and hands the plugin only its input and output buffers,
// or a latency-critical loop that must never call into the CUDA allocator
// after start-up.  kda_prefill needs a small device workspace (a status
// word, a work counter and a per-(sequence, head) schedule); for those
// callers this file provides that workspace from a fixed array in the
// library's own device memory instead of asking the caller for one.
//
// The array below is a file-scope __device__ variable: every GPU that loads
// the library holds it until the process exits.  In host code its name is
// only a host-side stand-in, so its device address is looked up once per
// device (cudaGetSymbolAddress, with that device current) and cached.
#include "../../include/kda.h"

#include <cuda_runtime.h>

#include "kda_internal.h"

#include <mutex>

namespace {

// 256-byte header + one int32 per (sequence, head): up to 16384 pairs.
constexpr size_t kNoAllocScratchBytes = 256 + 16384 * sizeof(int32_t);

__device__ __align__(256) unsigned char g_kda_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device (looked up on
// the first call for that device).  Returns nullptr on failure.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void* addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_kda_noalloc_scratch) != cudaSuccess || !addr) {
            return nullptr;
        }
        g_scratch_addr[dev] = addr;
    }
    return g_scratch_addr[dev];
}

}  // namespace

extern "C" KDA_API int kda_prefill_noalloc(const void* q, const void* k, const void* v,
                                           const void* z, const void* beta, const float* A,
                                           const float* initial_state,
                                           const int32_t* cu_seqlens,
                                           const int32_t* cu_seqlens_host, int32_t N,
                                           int32_t total_T, int32_t H, int32_t d_k,
                                           int32_t d_v, kda_dtype dt, float scale,
                                           uint32_t flags, void* o, float* final_state,
                                           void* stream) {
    // the array always holds the smallest workspace kda_prefill accepts for
    // up to 16384 (sequence, head) pairs (which then runs its single-pass kernel)
    if (N < 0 || H < 0 || kda::min_prefill_workspace_bytes(N, H) > kNoAllocScratchBytes) {
        return KDA_ERR_WORKSPACE;
    }
    void* scratch = scratch_on_current_device();
    if (!scratch) {
        return KDA_ERR_CUDA;
    }
    return kda_prefill(q, k, v, z, beta, A, initial_state, cu_seqlens, cu_seqlens_host, N,
                       total_T, H, d_k, d_v, dt, scale, flags, o, final_state, scratch,
                       kNoAllocScratchBytes, stream);
}
