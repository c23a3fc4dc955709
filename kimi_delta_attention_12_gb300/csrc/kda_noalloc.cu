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
// only a host-side stand-in, so its device address is looked up per device
// (cudaGetSymbolAddress, with that device current) and cached together with
// the unique id of the CUDA context it belongs to; a call from a different
// context (for example after cudaDeviceReset recreated the primary context)
// looks it up again instead of using a stale address.
#include "../../include/kda.h"

#include <cuda.h>
#include <cuda_runtime.h>

#include "kda_internal.h"

#include <mutex>

namespace {

// 256-byte header + one int32 per (sequence, head): up to 16384 pairs.
constexpr size_t kNoAllocScratchBytes = 256 + 16384 * sizeof(int32_t);

__device__ __align__(256) unsigned char g_kda_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchAddr {
    unsigned long long ctx_id;  // unique id of the context the address belongs to
    void* addr;
};
ScratchAddr g_scratch[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess) {
        return nullptr;
    }
    return reinterpret_cast<Fn>(f);
}

// Unique id of the calling thread's current CUDA context; false if there is
// none (or the driver cannot say).
bool current_ctx_id(unsigned long long* id) {
    static const CtxGetCurrentFn get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
    static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
    CUcontext ctx = nullptr;
    return get_current && get_id && get_current(&ctx) == CUDA_SUCCESS && ctx &&
           get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch array in the current context (looked up on
// the first call in that context).  Returns nullptr on failure.
void* scratch_on_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long id = 0;
    if (g_scratch[dev].addr && current_ctx_id(&id) && id == g_scratch[dev].ctx_id) {
        return g_scratch[dev].addr;
    }
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_kda_noalloc_scratch) != cudaSuccess || !addr) {
        cudaGetLastError();
        return nullptr;
    }
    // the lookup made the device's context current if it was not
    if (!current_ctx_id(&id)) {
        id = 0;   // no id: the address is looked up again on every call
        g_scratch[dev].addr = nullptr;
        return addr;
    }
    g_scratch[dev].ctx_id = id;
    g_scratch[dev].addr = addr;
    return addr;
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

extern "C" KDA_API int kda_prefill_noalloc_status(void* stream) {
    void* scratch = scratch_on_current_device();
    if (!scratch) {
        return KDA_ERR_CUDA;
    }
    return kda_workspace_status(scratch, stream);
}
