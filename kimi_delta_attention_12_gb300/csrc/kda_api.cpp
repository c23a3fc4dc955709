// kda_api.cpp -- the C ABI declared in include/kda.h: argument validation,
// kernel selection and launch on the caller's stream.  No allocation, no
// exceptions across the boundary.
#include "../../include/kda.h"

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include "kda_internal.h"

namespace {

inline bool aligned(const void* p, uintptr_t a) {
    return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

inline bool supported_dim(int32_t d) { return d == 32 || d == 64 || d == 128; }

inline size_t elem_bytes(kda_dtype dt) { return dt == KDA_F32 ? 4 : 2; }

constexpr uint32_t kKnownFlags = KDA_FLAG_L2NORM_QK | KDA_FLAG_RECURRENT |
                                 KDA_FLAG_SOFTPLUS_GATE | KDA_FLAG_SHORT_PEER_WAITS;
// polls of a split-kernel wait on another CTA before it gives up (~2^25, far
// longer than any legitimate wait); one poll with KDA_FLAG_SHORT_PEER_WAITS
constexpr uint32_t kPeerWaitPolls = 1u << 25;
constexpr uint32_t kFlagRecurrent = KDA_FLAG_RECURRENT;
constexpr int32_t kCheckpointGrain = 64;  // checkpoints fall on chunk boundaries

// status word + work counter, then the optional schedule (one int per unit)
constexpr size_t kWsHeader = 256;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Whether the byte ranges [a, a + na) and [b, b + nb) share a byte.
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    if (!a || !b || na == 0 || nb == 0) return false;
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

constexpr int32_t kMaxConvWidth = 4;

// Minimum workspace: the header and one int per (sequence, head) unit.
size_t basic_workspace_bytes(int32_t N, int32_t H) {
    const size_t units = (N > 0 && H > 0) ? (size_t)N * (size_t)H : 0;
    return kWsHeader + round_up(units * sizeof(int32_t), 256);
}

// SMs of the current device, 0 if there is none.
int current_sm_count() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return sms;
}

// bf16 at d = 128 runs the split kernel when its tables can describe the
// sizes (the single-pass kernel otherwise, or with a minimal workspace).
bool split_eligible(int32_t N, int32_t H, kda_dtype dt, int32_t d_k, int32_t d_v, int sms,
                    kda::SplitPlan* plan) {
    return dt == KDA_BF16 && d_k == 128 && d_v == 128 && kda::split_plan(N, H, sms, plan);
}

}  // namespace

namespace kda {
size_t min_prefill_workspace_bytes(int32_t N, int32_t H) { return basic_workspace_bytes(N, H); }
}  // namespace kda

extern "C" {

const char* kda_status_string(int status) {
    switch (status) {
        case KDA_OK: return "KDA_OK";
        case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
        case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
        case KDA_ERR_ALIGNMENT: return "KDA_ERR_ALIGNMENT";
        case KDA_ERR_WORKSPACE: return "KDA_ERR_WORKSPACE";
        case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
        case KDA_ERR_TIMEOUT: return "KDA_ERR_TIMEOUT";
        default: return "KDA_ERR_UNKNOWN";
    }
}

int kda_version(void) { return 100; }

size_t kda_prefill_workspace_bytes(int32_t N, int32_t total_T, int32_t H, int32_t d_k,
                                   int32_t d_v, kda_dtype dt) {
    const size_t basic = basic_workspace_bytes(N, H);
    kda::SplitPlan plan;
    if (N > 0 && H > 0 && total_T > 0 &&
        split_eligible(N, H, dt, d_k, d_v, current_sm_count(), &plan)) {
        const size_t split = kda::split_workspace_bytes(plan);
        return split > basic ? split : basic;
    }
    return basic;
}

int kda_workspace_status(const void* workspace, void* stream) {
    if (!workspace) {
        return KDA_ERR_INVALID_ARG;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) {
        return KDA_ERR_CUDA;
    }
    int32_t st = 0;
    if (cudaMemcpy(&st, workspace, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) {
        return KDA_ERR_CUDA;
    }
    return st == 0 ? KDA_OK : KDA_ERR_TIMEOUT;
}

int kda_prefill(const void* q, const void* k, const void* v, const void* z,
                const void* beta, const float* A, const float* initial_state,
                const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                kda_dtype dt, float scale, uint32_t flags,
                void* o, float* final_state,
                void* workspace, size_t workspace_bytes, void* stream) {
    return kda_prefill_checkpointed(q, k, v, z, beta, A, initial_state, cu_seqlens,
                                    cu_seqlens_host, N, total_T, H, d_k, d_v, dt, scale, flags,
                                    o, final_state, 0, nullptr, nullptr, 0, workspace,
                                    workspace_bytes, stream);
}

int64_t kda_checkpoint_count(const int32_t* cu_seqlens_host, int32_t N, int32_t total_T,
                             int32_t ckpt_interval) {
    if (N < 1 || total_T < 0 || ckpt_interval <= 0) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens_host) {
        if (total_T % N != 0) return KDA_ERR_INVALID_ARG;
        return (int64_t)N * ((total_T / N) / ckpt_interval);
    }
    if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INVALID_ARG;
    int64_t count = 0;
    for (int32_t n = 0; n < N; ++n) {
        const int32_t len = cu_seqlens_host[n + 1] - cu_seqlens_host[n];
        if (len < 0) return KDA_ERR_INVALID_ARG;
        count += len / ckpt_interval;
    }
    return count;
}

int kda_prefill_checkpointed(const void* q, const void* k, const void* v, const void* z,
                             const void* beta, const float* A, const float* initial_state,
                             const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                             int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                             kda_dtype dt, float scale, uint32_t flags, void* o,
                             float* final_state, int32_t ckpt_interval, float* ckpt_pool,
                             const int32_t* ckpt_slots, int32_t ckpt_pool_size,
                             void* workspace, size_t workspace_bytes, void* stream) {
    if (ckpt_interval < 0 || ckpt_interval % kCheckpointGrain != 0) return KDA_ERR_INVALID_ARG;
    if (ckpt_interval > 0 && (!ckpt_pool || ckpt_pool_size < 1)) return KDA_ERR_INVALID_ARG;
    if (ckpt_interval > 0 && (!aligned(ckpt_pool, 16) || !aligned(ckpt_slots, 4))) {
        return KDA_ERR_ALIGNMENT;
    }
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dim(d_k) || !supported_dim(d_v)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || H < 1 || total_T < 0) return KDA_ERR_INVALID_ARG;
    if ((flags & ~kKnownFlags) != 0) return KDA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (!A) return KDA_ERR_INVALID_ARG;
    if (total_T > 0 && (!q || !k || !v || !z || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && total_T % N != 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INVALID_ARG;
        for (int32_t n = 0; n < N; ++n) {
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
        }
    }
    if (!workspace || workspace_bytes < basic_workspace_bytes(N, H)) {
        return KDA_ERR_WORKSPACE;
    }
    const size_t eb = elem_bytes(dt);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) ||
        !aligned(o, 16) || !aligned(beta, eb) || !aligned(A, 4) ||
        !aligned(initial_state, 16) || !aligned(final_state, 16) ||
        !aligned(cu_seqlens, 4) || !aligned(workspace, 256)) {
        return KDA_ERR_ALIGNMENT;
    }

    // Checkpoints (and reads of ckpt_slots) stop at the count the host can
    // vouch for: from the host mirror, from the equal split, or -- with only
    // a device cu_seqlens -- floor(total_T / interval), which bounds the count
    // of every valid array.
    int64_t ckpt_count = 0;
    if (ckpt_interval > 0) {
        ckpt_count = (cu_seqlens_host || !cu_seqlens)
                         ? kda_checkpoint_count(cu_seqlens_host, N, total_T, ckpt_interval)
                         : (int64_t)total_T / ckpt_interval;
        if (ckpt_count < 0) return KDA_ERR_INVALID_ARG;
    }

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t* ws = static_cast<int32_t*>(workspace);
    const bool use_chunked = kda::kChunkedPrefillBuilt && dt == KDA_BF16 && d_k == 128 && d_v == 128 &&
                             (flags & (kFlagRecurrent | KDA_FLAG_SOFTPLUS_GATE)) == 0 &&
                             total_T > 0;
    const int sms = use_chunked ? current_sm_count() : 0;
    kda::SplitPlan plan;
    const bool use_split = use_chunked && split_eligible(N, H, dt, d_k, d_v, sms, &plan) &&
                           workspace_bytes >= kda::split_workspace_bytes(plan);
    // the header (status, work counter) and, for the split kernel, the ring
    // flags and consumer counters that follow it start at zero on every call
    const size_t zero_bytes = use_split ? kda::split_zeroed_bytes(plan) : kWsHeader;
    if (cudaMemsetAsync(ws, 0, zero_bytes, s) != cudaSuccess) return KDA_ERR_CUDA;

    cudaError_t err;
    if (use_chunked) {
        kda::ChunkedParams p;
        memset(&p, 0, sizeof(p));
        p.q = q; p.k = k; p.v = v; p.z = z; p.beta = beta; p.A = A;
        p.initial_state = initial_state; p.final_state = final_state;
        p.cu_seqlens = cu_seqlens; p.o = o;
        p.status = ws; p.work_counter = ws + 1; p.schedule = nullptr;
        p.N = N; p.total_T = total_T; p.H = H; p.scale = scale;
        p.l2norm = (flags & KDA_FLAG_L2NORM_QK) ? 1 : 0;
        p.ckpt_interval = ckpt_interval; p.ckpt_pool = ckpt_pool;
        p.ckpt_slots = ckpt_slots; p.ckpt_pool_size = ckpt_pool_size;
        p.ckpt_count = ckpt_count;
        p.peer_wait_polls = (flags & KDA_FLAG_SHORT_PEER_WAITS) ? 1u : kPeerWaitPolls;
        err = cudaErrorCooperativeLaunchTooLarge;
        if (use_split) {
            kda::split_bind(plan, workspace, &p);
            err = kda::launch_split_prefill(p, sms, s);
        }
        // the split kernel needs every SM at once; where a cooperative launch
        // cannot promise that, the single-pass kernel runs instead
        if (err == cudaErrorCooperativeLaunchTooLarge) {
            err = kda::launch_chunked_prefill(p, s);
        }
    } else {
        kda::RecurrentParams p;
        memset(&p, 0, sizeof(p));
        p.q = q; p.k = k; p.v = v; p.z = z; p.beta = beta; p.A = A;
        p.state_in = initial_state; p.state_out = final_state;
        p.slots = nullptr; p.cu_seqlens = cu_seqlens; p.o = o;
        p.rows = N; p.total_T = total_T; p.H = H; p.pool_size = 0;
        p.scale = scale; p.l2norm = (flags & KDA_FLAG_L2NORM_QK) ? 1 : 0; p.decode = 0;
        p.softplus_gate = (flags & KDA_FLAG_SOFTPLUS_GATE) ? 1 : 0;
        p.ckpt_interval = ckpt_interval; p.ckpt_pool = ckpt_pool;
        p.ckpt_slots = ckpt_slots; p.ckpt_pool_size = ckpt_pool_size;
        p.ckpt_count = ckpt_count;
        if (total_T == 0 && !final_state) {
            return KDA_OK;
        }
        err = kda::launch_recurrent(p, d_k, d_v, dt == KDA_F32 ? 0 : 1, s);
    }
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_short_conv(const void* q, const void* k, const void* v, const float* conv_w,
                   const void* conv_state_in, void* conv_state_out,
                   const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                   int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                   int32_t W, kda_dtype dt, uint32_t flags,
                   void* q_out, void* k_out, void* v_out, void* stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dim(d_k) || !supported_dim(d_v)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || H < 1 || total_T < 0) return KDA_ERR_INVALID_ARG;
    if (W < 1 || W > kMaxConvWidth) return KDA_ERR_INVALID_ARG;
    if ((flags & ~(uint32_t)KDA_FLAG_CONV_SILU) != 0) return KDA_ERR_INVALID_ARG;
    if (!conv_w) return KDA_ERR_INVALID_ARG;
    if (total_T > 0 && (!q || !k || !v || !q_out || !k_out || !v_out)) {
        return KDA_ERR_INVALID_ARG;
    }
    if (!cu_seqlens && total_T % N != 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INVALID_ARG;
        for (int32_t n = 0; n < N; ++n) {
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
        }
    }
    const size_t eb = elem_bytes(dt);
    const size_t nqk = (size_t)total_T * H * d_k * eb, nv = (size_t)total_T * H * d_v * eb;
    const size_t nst = (size_t)N * H * (W - 1) * (2 * d_k + d_v) * eb;
    const void* ins[3] = {q, k, v};
    const void* outs[3] = {q_out, k_out, v_out};
    const size_t sz[3] = {nqk, nqk, nv};
    for (int i = 0; i < 3; ++i) {
        for (int j = 0; j < 3; ++j) {
            if (overlaps(outs[i], sz[i], ins[j], sz[j])) return KDA_ERR_INVALID_ARG;
            if (j != i && overlaps(outs[i], sz[i], outs[j], sz[j])) return KDA_ERR_INVALID_ARG;
        }
        if (overlaps(outs[i], sz[i], conv_state_out, nst) ||
            overlaps(outs[i], sz[i], conv_state_in, nst)) {
            return KDA_ERR_INVALID_ARG;
        }
    }
    if (overlaps(conv_state_in, nst, conv_state_out, nst)) return KDA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(q_out, 16) ||
        !aligned(k_out, 16) || !aligned(v_out, 16) || !aligned(conv_w, 16) ||
        !aligned(conv_state_in, 16) || !aligned(conv_state_out, 16) ||
        !aligned(cu_seqlens, 4)) {
        return KDA_ERR_ALIGNMENT;
    }
    kda::ShortConvParams p;
    memset(&p, 0, sizeof(p));
    p.x[0] = q; p.x[1] = k; p.x[2] = v;
    p.y[0] = q_out; p.y[1] = k_out; p.y[2] = v_out;
    p.w = conv_w;
    p.state_in = W > 1 ? conv_state_in : nullptr;
    p.state_out = W > 1 ? conv_state_out : nullptr;
    p.cu_seqlens = cu_seqlens;
    p.N = N; p.total_T = total_T; p.H = H; p.d_k = d_k; p.d_v = d_v; p.W = W;
    p.silu = (flags & KDA_FLAG_CONV_SILU) ? 1 : 0;
    const cudaError_t err = kda::launch_short_conv(p, dt == KDA_F32 ? 0 : 1,
                                                   static_cast<cudaStream_t>(stream));
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

// kda_prefill_conv's workspace: the prefill's part (large enough for the split
// kernel with the convolutions fused, whose slots also carry the convolved v)
// then, for the two-pass path, the convolved q, k, v.
static size_t prefill_conv_part(int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                                kda_dtype dt) {
    size_t part = kda_prefill_workspace_bytes(N, total_T, H, d_k, d_v, dt);
    kda::SplitPlan plan;
    if (N > 0 && H > 0 && total_T > 0 &&
        split_eligible(N, H, dt, d_k, d_v, current_sm_count(), &plan)) {
        const size_t fused = kda::split_workspace_bytes(plan, true);
        part = fused > part ? fused : part;
    }
    return round_up(part, 256);
}

size_t kda_prefill_conv_workspace_bytes(int32_t N, int32_t total_T, int32_t H, int32_t d_k,
                                        int32_t d_v, kda_dtype dt) {
    if (N < 1 || H < 1 || total_T < 0 || !supported_dim(d_k) || !supported_dim(d_v) ||
        (dt != KDA_F32 && dt != KDA_BF16)) {
        return 0;
    }
    const size_t eb = elem_bytes(dt);
    return prefill_conv_part(N, total_T, H, d_k, d_v, dt) +
           2 * round_up((size_t)total_T * H * d_k * eb, 256) +
           round_up((size_t)total_T * H * d_v * eb, 256);
}

int kda_prefill_conv(const void* q, const void* k, const void* v, const void* z,
                     const void* beta, const float* A, const float* initial_state,
                     const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                     int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                     kda_dtype dt, float scale, uint32_t flags,
                     const float* conv_w, const void* conv_state_in, void* conv_state_out,
                     int32_t W, void* o, float* final_state,
                     void* workspace, size_t workspace_bytes, void* stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dim(d_k) || !supported_dim(d_v)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || H < 1 || total_T < 0) return KDA_ERR_INVALID_ARG;
    if ((flags & ~(kKnownFlags | (uint32_t)KDA_FLAG_CONV_SILU)) != 0) return KDA_ERR_INVALID_ARG;
    if (W < 1 || W > kMaxConvWidth || !conv_w) return KDA_ERR_INVALID_ARG;
    if (!isfinite(scale) || !A) return KDA_ERR_INVALID_ARG;
    if (total_T > 0 && (!q || !k || !v || !z || !beta || !o)) return KDA_ERR_INVALID_ARG;
    if (!cu_seqlens && total_T % N != 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INVALID_ARG;
        for (int32_t n = 0; n < N; ++n) {
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
        }
    }
    const size_t need = kda_prefill_conv_workspace_bytes(N, total_T, H, d_k, d_v, dt);
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    const size_t eb = elem_bytes(dt);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) ||
        !aligned(o, 16) || !aligned(beta, eb) || !aligned(A, 4) ||
        !aligned(initial_state, 16) || !aligned(final_state, 16) || !aligned(conv_w, 16) ||
        !aligned(conv_state_in, 16) || !aligned(conv_state_out, 16) ||
        !aligned(cu_seqlens, 4) || !aligned(workspace, 256)) {
        return KDA_ERR_ALIGNMENT;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    const size_t part = prefill_conv_part(N, total_T, H, d_k, d_v, dt);
    const uint32_t pflags = flags & ~(uint32_t)KDA_FLAG_CONV_SILU;

    // fused: the split kernel convolves q, k and v in its producers -- where
    // its units fit one batch.  The convolutions add about a third to a
    // producer's work per chunk; with one batch the producers have that slack
    // (4K workload, 32 heads: 0.243 ms fused against 0.275 ms for the two
    // passes, 0.228 ms prefill alone), with several batches they are the
    // binding resource and the two passes are faster (96 heads x 65,536
    // tokens, two batches: 10.8 against 8.45 ms).
    kda::SplitPlan plan;
    const int sms = (dt == KDA_BF16 && d_k == 128 && d_v == 128 && total_T > 0 &&
                     (flags & (kFlagRecurrent | KDA_FLAG_SOFTPLUS_GATE)) == 0)
                        ? current_sm_count()
                        : 0;
    if (sms > 0 && split_eligible(N, H, dt, d_k, d_v, sms, &plan) && plan.batches == 1 &&
        part >= kda::split_workspace_bytes(plan, true)) {
        if (cudaMemsetAsync(ws, 0, kda::split_zeroed_bytes(plan), s) != cudaSuccess) {
            return KDA_ERR_CUDA;
        }
        kda::ChunkedParams p;
        memset(&p, 0, sizeof(p));
        p.q = q; p.k = k; p.v = v; p.z = z; p.beta = beta; p.A = A;
        p.initial_state = initial_state; p.final_state = final_state;
        p.cu_seqlens = cu_seqlens; p.o = o;
        p.status = reinterpret_cast<int32_t*>(ws);
        p.work_counter = reinterpret_cast<int32_t*>(ws) + 1;
        p.N = N; p.total_T = total_T; p.H = H; p.scale = scale;
        p.l2norm = (flags & KDA_FLAG_L2NORM_QK) ? 1 : 0;
        p.peer_wait_polls = (flags & KDA_FLAG_SHORT_PEER_WAITS) ? 1u : kPeerWaitPolls;
        p.conv_w = conv_w;
        p.conv_state_in = W > 1 ? conv_state_in : nullptr;
        p.conv_state_out = W > 1 ? conv_state_out : nullptr;
        p.conv_W = W;
        p.conv_silu = (flags & KDA_FLAG_CONV_SILU) ? 1 : 0;
        kda::split_bind(plan, ws, &p);
        const cudaError_t err = kda::launch_split_prefill(p, sms, s);
        if (err == cudaSuccess) return KDA_OK;
        if (err != cudaErrorCooperativeLaunchTooLarge) return KDA_ERR_CUDA;
    }
    // two passes: the convolutions into the workspace, then the prefill on them
    char* qc = ws + part;
    char* kc = qc + round_up((size_t)total_T * H * d_k * eb, 256);
    char* vc = kc + round_up((size_t)total_T * H * d_k * eb, 256);
    int st = kda_short_conv(q, k, v, conv_w, conv_state_in, conv_state_out, cu_seqlens,
                            cu_seqlens_host, N, total_T, H, d_k, d_v, W, dt,
                            flags & (uint32_t)KDA_FLAG_CONV_SILU, qc, kc, vc, stream);
    if (st != KDA_OK) return st;
    return kda_prefill(qc, kc, vc, z, beta, A, initial_state, cu_seqlens, cu_seqlens_host, N,
                       total_T, H, d_k, d_v, dt, scale, pflags, o, final_state, ws, part,
                       stream);
}

// One of the three convolved tensors in the decode-conv workspace.
static size_t conv_ws_part(int32_t B, int32_t H, int32_t d, kda_dtype dt) {
    return round_up((size_t)B * H * d * elem_bytes(dt), 256);
}

size_t kda_decode_conv_workspace_bytes(int32_t B, int32_t H, int32_t d_k, int32_t d_v,
                                       kda_dtype dt) {
    if (B < 0 || H < 0 || d_k < 0 || d_v < 0) return 0;
    return 2 * conv_ws_part(B, H, d_k, dt) + conv_ws_part(B, H, d_v, dt);
}

// kda_decode_step and kda_decode_step_conv (W = 0: no convolution)
static int decode_step_impl(const void* q, const void* k, const void* v, const void* z,
                     const void* beta, const float* A, float* state,
                     const int32_t* slots, int32_t pool_size, const float* conv_w,
                     void* conv_state, int32_t W, int32_t B, int32_t H, int32_t d_k,
                     int32_t d_v, kda_dtype dt, float scale, uint32_t flags, void* o,
                     void* workspace, size_t workspace_bytes, void* stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dim(d_k) || !supported_dim(d_v)) return KDA_ERR_UNSUPPORTED;
    if (B < 0 || H < 1 || pool_size < 0) return KDA_ERR_INVALID_ARG;
    const uint32_t known = KDA_FLAG_L2NORM_QK | KDA_FLAG_SOFTPLUS_GATE |
                           (W > 0 ? (uint32_t)KDA_FLAG_CONV_SILU : 0u);
    if ((flags & ~known) != 0) return KDA_ERR_INVALID_ARG;
    if (W < 0 || W > kMaxConvWidth) return KDA_ERR_INVALID_ARG;
    if (W > 0 && (!conv_w || (W > 1 && !conv_state))) return KDA_ERR_INVALID_ARG;
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (B == 0) return KDA_OK;
    if (!q || !k || !v || !z || !beta || !A || !state || !o) return KDA_ERR_INVALID_ARG;
    if (W > 0) {
        if (B > 65535) return KDA_ERR_UNSUPPORTED;
        if (!workspace || workspace_bytes < kda_decode_conv_workspace_bytes(B, H, d_k, d_v, dt)) {
            return KDA_ERR_WORKSPACE;
        }
        const size_t wsb = kda_decode_conv_workspace_bytes(B, H, d_k, d_v, dt);
        const size_t eb = elem_bytes(dt);
        const size_t nqk = (size_t)B * H * d_k * eb, nv = (size_t)B * H * d_v * eb;
        const size_t ncs = (size_t)pool_size * H * (W - 1) * (2 * d_k + d_v) * eb;
        if (overlaps(workspace, wsb, q, nqk) || overlaps(workspace, wsb, k, nqk) ||
            overlaps(workspace, wsb, v, nv) || overlaps(workspace, wsb, o, nv) ||
            overlaps(workspace, wsb, conv_state, ncs)) {
            return KDA_ERR_INVALID_ARG;
        }
        if (!aligned(conv_w, 16) || !aligned(workspace, 16)) return KDA_ERR_ALIGNMENT;
        if (W > 1 && !aligned(conv_state, 16)) return KDA_ERR_ALIGNMENT;
    }
    if (!slots && pool_size < B) return KDA_ERR_INVALID_ARG;
    const size_t eb = elem_bytes(dt);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) ||
        !aligned(o, 16) || !aligned(beta, eb) || !aligned(A, 4) || !aligned(state, 16) ||
        !aligned(slots, 4)) {
        return KDA_ERR_ALIGNMENT;
    }
    kda::RecurrentParams p;
    memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v; p.z = z; p.beta = beta; p.A = A;
    p.state_in = state; p.state_out = state; p.slots = slots; p.cu_seqlens = nullptr;
    p.o = o; p.rows = B; p.total_T = B; p.H = H; p.pool_size = pool_size;
    p.scale = scale; p.l2norm = (flags & KDA_FLAG_L2NORM_QK) ? 1 : 0; p.decode = 1;
    p.softplus_gate = (flags & KDA_FLAG_SOFTPLUS_GATE) ? 1 : 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (W > 0) {
        // the token's short convolutions into the workspace, conv state
        // shifted in place; the decode step then reads the convolved q, k, v
        kda::ShortConvDecodeParams c;
        memset(&c, 0, sizeof(c));
        char* ws = static_cast<char*>(workspace);
        c.x[0] = q; c.x[1] = k; c.x[2] = v;
        c.y[0] = ws;
        c.y[1] = ws + conv_ws_part(B, H, d_k, dt);
        c.y[2] = ws + 2 * conv_ws_part(B, H, d_k, dt);
        c.w = conv_w; c.state = conv_state; c.slots = slots;
        c.B = B; c.pool_size = pool_size; c.H = H; c.d_k = d_k; c.d_v = d_v; c.W = W;
        c.silu = (flags & KDA_FLAG_CONV_SILU) ? 1 : 0;
        const cudaError_t ce = kda::launch_short_conv_decode(c, dt == KDA_F32 ? 0 : 1, s);
        if (ce != cudaSuccess) return KDA_ERR_CUDA;
        p.q = c.y[0]; p.k = c.y[1]; p.v = c.y[2];
    }
    const cudaError_t err = kda::launch_recurrent(p, d_k, d_v, dt == KDA_F32 ? 0 : 1, s);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_decode_step(const void* q, const void* k, const void* v, const void* z,
                    const void* beta, const float* A, float* state,
                    const int32_t* slots, int32_t pool_size,
                    int32_t B, int32_t H, int32_t d_k, int32_t d_v,
                    kda_dtype dt, float scale, uint32_t flags,
                    void* o, void* stream) {
    return decode_step_impl(q, k, v, z, beta, A, state, slots, pool_size, nullptr, nullptr, 0,
                            B, H, d_k, d_v, dt, scale, flags, o, nullptr, 0, stream);
}

int kda_decode_step_conv(const void* q, const void* k, const void* v, const void* z,
                         const void* beta, const float* A, float* state,
                         const int32_t* slots, int32_t pool_size,
                         const float* conv_w, void* conv_state, int32_t W,
                         int32_t B, int32_t H, int32_t d_k, int32_t d_v,
                         kda_dtype dt, float scale, uint32_t flags,
                         void* o, void* workspace, size_t workspace_bytes, void* stream) {
    if (W < 1) return KDA_ERR_INVALID_ARG;
    return decode_step_impl(q, k, v, z, beta, A, state, slots, pool_size, conv_w, conv_state, W,
                            B, H, d_k, d_v, dt, scale, flags, o, workspace, workspace_bytes,
                            stream);
}

// Backward workspace, in order: the workspace of the checkpointed prefill
// that provides the chunk-start states (first, so that kda_workspace_status
// reads its status word), that prefill's output o (not used), the checkpoint
// pool (at most floor(total_T / 64) states), one area used by whichever
// backward runs -- the recurrent one's per-pair scratch and per-CTA column
// partials, or the chunked one's chunk records, per-chunk dL/dS tiles and
// chunk map (at most total_T / 64 + N chunks) -- and the per-token dA shares.
struct BackwardLayout {
    size_t prefill, o, pool, scratch, part, records, dsl, map, dA_tok;
    size_t area() const {
        const size_t rec = scratch + part, chk = records + dsl + map;
        return rec > chk ? rec : chk;
    }
    size_t total() const { return prefill + o + pool + area() + dA_tok; }
};

static int64_t bwd_max_chunks(int32_t N, int32_t total_T) {
    return (int64_t)total_T / kda::kBwChunk + N;
}

static BackwardLayout backward_layout(int32_t N, int32_t total_T, int32_t H, int32_t d_k,
                                      int32_t d_v, kda_dtype dt) {
    const size_t SS = (size_t)d_k * d_v * sizeof(float);
    BackwardLayout l;
    l.prefill = round_up(kda_prefill_workspace_bytes(N, total_T, H, d_k, d_v, dt), 256);
    l.o = round_up((size_t)total_T * H * d_v * elem_bytes(dt), 256);
    l.pool = round_up((size_t)(total_T / kda::kBwChunk) * H * SS, 256);
    l.scratch = round_up((size_t)N * H * kda::kBwChunk * SS, 256);
    l.part = round_up((size_t)(d_v / 32) * total_T * H * (3 * d_k + 1) * sizeof(float), 256);
    l.records = l.dsl = l.map = 0;
    if (dt == KDA_BF16 && d_k == 128 && d_v == 128) {
        const size_t mc = (size_t)bwd_max_chunks(N, total_T);
        l.records = round_up(mc * H * kda::kChunkRecordBytes, 1024);
        l.dsl = round_up(mc * H * kda::kBwdDslBytes, 1024);
        l.map = round_up(mc * 4 * sizeof(int32_t), 256);
    }
    l.dA_tok = round_up((size_t)total_T * H * sizeof(float), 256);
    return l;
}

size_t kda_backward_workspace_bytes(int32_t N, int32_t total_T, int32_t H, int32_t d_k,
                                    int32_t d_v, kda_dtype dt) {
    if (N < 1 || H < 1 || total_T < 0 || !supported_dim(d_k) || !supported_dim(d_v) ||
        (dt != KDA_F32 && dt != KDA_BF16)) {
        return 0;
    }
    return backward_layout(N, total_T, H, d_k, d_v, dt).total();
}

int kda_backward(const void* q, const void* k, const void* v, const void* z,
                 const void* beta, const float* A, const float* initial_state,
                 const int32_t* cu_seqlens, const int32_t* cu_seqlens_host,
                 int32_t N, int32_t total_T, int32_t H, int32_t d_k, int32_t d_v,
                 kda_dtype dt, float scale, uint32_t flags,
                 const void* dO, const float* dS_final,
                 float* dq, float* dk, float* dv, float* dz, float* dbeta, float* dA,
                 float* dS0, void* workspace, size_t workspace_bytes, void* stream) {
    if (dt != KDA_F32 && dt != KDA_BF16) return KDA_ERR_UNSUPPORTED;
    if (!supported_dim(d_k) || !supported_dim(d_v)) return KDA_ERR_UNSUPPORTED;
    if (N < 1 || H < 1 || total_T < 0) return KDA_ERR_INVALID_ARG;
    if ((flags & ~(uint32_t)(KDA_FLAG_L2NORM_QK | KDA_FLAG_SOFTPLUS_GATE)) != 0) {
        return KDA_ERR_INVALID_ARG;
    }
    if (!isfinite(scale)) return KDA_ERR_INVALID_ARG;
    if (!A || !dA || !dS0) return KDA_ERR_INVALID_ARG;
    if (total_T > 0 && (!q || !k || !v || !z || !beta || !dO || !dq || !dk || !dv || !dz ||
                        !dbeta)) {
        return KDA_ERR_INVALID_ARG;
    }
    if (!cu_seqlens && total_T % N != 0) return KDA_ERR_INVALID_ARG;
    if (cu_seqlens_host) {
        if (cu_seqlens_host[0] != 0 || cu_seqlens_host[N] != total_T) return KDA_ERR_INVALID_ARG;
        for (int32_t n = 0; n < N; ++n) {
            if (cu_seqlens_host[n + 1] < cu_seqlens_host[n]) return KDA_ERR_INVALID_ARG;
        }
    }
    // one finalize CTA per (token, head) and d_v / 32 main CTAs per (sequence, head)
    if ((int64_t)total_T * H >= ((int64_t)1 << 31) || (int64_t)N * H * (d_v / 32) >= ((int64_t)1 << 31)) {
        return KDA_ERR_UNSUPPORTED;
    }
    const BackwardLayout wl = backward_layout(N, total_T, H, d_k, d_v, dt);
    if (!workspace || workspace_bytes < wl.total()) return KDA_ERR_WORKSPACE;
    const size_t eb = elem_bytes(dt);
    if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(z, 16) ||
        !aligned(beta, eb) || !aligned(dO, 16) || !aligned(A, 4) || !aligned(dq, 4) ||
        !aligned(dk, 4) || !aligned(dv, 4) || !aligned(dz, 4) || !aligned(dbeta, 4) ||
        !aligned(dA, 4) || !aligned(initial_state, 16) || !aligned(dS_final, 16) ||
        !aligned(dS0, 16) || !aligned(cu_seqlens, 4) || !aligned(workspace, 256)) {
        return KDA_ERR_ALIGNMENT;
    }
    char* ws = static_cast<char*>(workspace);
    char* ws_o = ws + wl.prefill;
    float* pool = reinterpret_cast<float*>(ws_o + wl.o);
    char* area = ws_o + wl.o + wl.pool;
    float* dA_tok = reinterpret_cast<float*>(area + wl.area());
    const int32_t pool_rows = total_T / kda::kBwChunk;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    // The chunked backward (bf16, d = 128, the bounded gate, sequence lengths
    // the host has checked or the equal split): the split prefill keeps a
    // chunk record of every chunk (its operand tiles and start state), then
    // the reverse state chain and the chunk-parallel assembly.  Where the split kernel cannot run
    // (its tables, or co-residency) the recurrent backward below runs instead.
    if (dt == KDA_BF16 && d_k == 128 && d_v == 128 && total_T > 0 &&
        (flags & KDA_FLAG_SOFTPLUS_GATE) == 0 && (cu_seqlens_host || !cu_seqlens) &&
        wl.records > 0) {
        const int sms = current_sm_count();
        kda::SplitPlan plan;
        if (split_eligible(N, H, dt, d_k, d_v, sms, &plan) &&
            wl.prefill >= kda::split_workspace_bytes(plan)) {
            const int64_t max_chunks = bwd_max_chunks(N, total_T);
            uint8_t* records = reinterpret_cast<uint8_t*>(area);
            uint8_t* dsl = records + wl.records;
            int32_t* cmap = reinterpret_cast<int32_t*>(dsl + wl.dsl);
            if (cudaMemsetAsync(ws, 0, kda::split_zeroed_bytes(plan), s) != cudaSuccess) {
                return KDA_ERR_CUDA;
            }
            kda::ChunkedParams fp;
            memset(&fp, 0, sizeof(fp));
            fp.q = q; fp.k = k; fp.v = v; fp.z = z; fp.beta = beta; fp.A = A;
            fp.initial_state = initial_state; fp.final_state = nullptr;
            fp.cu_seqlens = cu_seqlens; fp.o = nullptr;   // (the forward's o is not needed)
            fp.status = reinterpret_cast<int32_t*>(ws);
            fp.work_counter = reinterpret_cast<int32_t*>(ws) + 1;
            fp.N = N; fp.total_T = total_T; fp.H = H; fp.scale = scale;
            fp.l2norm = (flags & KDA_FLAG_L2NORM_QK) ? 1 : 0;
            fp.ckpt_interval = 0;   // the records carry the chunk-start states
            fp.peer_wait_polls = kPeerWaitPolls;
            fp.records = records;
            fp.rec_chunks = max_chunks;
            kda::split_bind(plan, ws, &fp);
            cudaError_t err = kda::launch_split_prefill(fp, sms, s);
            if (err == cudaSuccess) {
                if (cudaMemsetAsync(cmap, 0xff, (size_t)max_chunks * 4 * sizeof(int32_t), s) !=
                    cudaSuccess) {
                    return KDA_ERR_CUDA;
                }
                kda::BwdChunkedParams bp;
                memset(&bp, 0, sizeof(bp));
                bp.q = q; bp.k = k; bp.v = v; bp.z = z; bp.beta = beta; bp.A = A; bp.dO = dO;
                bp.dS_final = dS_final;
                bp.cu_seqlens = cu_seqlens; bp.records = records;
                bp.dsl = dsl; bp.chunk_map = cmap; bp.max_chunks = (int32_t)max_chunks;
                bp.dq = dq; bp.dk = dk; bp.dv = dv; bp.dz = dz; bp.dbeta = dbeta;
                bp.dA_tok = dA_tok; bp.dS0 = dS0;
                bp.status = reinterpret_cast<int32_t*>(ws);
                bp.N = N; bp.total_T = total_T; bp.H = H; bp.scale = scale;
                bp.l2norm = fp.l2norm;
                err = kda::launch_bwd_chunked(bp, s);
                if (err == cudaSuccess) {
                    err = kda::launch_backward_dA(dA_tok, dA, total_T, H, s);
                }
                return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
            }
            if (err != cudaErrorCooperativeLaunchTooLarge) {
                return KDA_ERR_CUDA;
            }
        }
    }

    // the states after every 64 tokens of each sequence, from the forward
    if (pool_rows > 0) {
        const int st = kda_prefill_checkpointed(
            q, k, v, z, beta, A, initial_state, cu_seqlens, cu_seqlens_host, N, total_T, H,
            d_k, d_v, dt, scale, flags, ws_o, nullptr, kda::kBwChunk, pool, nullptr, pool_rows,
            ws, wl.prefill, stream);
        if (st != KDA_OK) return st;
    }
    kda::BackwardParams p;
    memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v; p.z = z; p.beta = beta; p.A = A;
    p.initial_state = initial_state; p.cu_seqlens = cu_seqlens;
    p.dO = dO; p.dS_final = dS_final;
    p.dq = dq; p.dk = dk; p.dv = dv; p.dz = dz; p.dbeta = dbeta; p.dA = dA; p.dS0 = dS0;
    p.pool = pool;
    p.pool_rows = pool_rows;
    p.scratch = reinterpret_cast<float*>(area);
    p.part = reinterpret_cast<float*>(area + wl.scratch);
    p.dA_tok = dA_tok;
    p.N = N; p.total_T = total_T; p.H = H; p.scale = scale;
    p.l2norm = (flags & KDA_FLAG_L2NORM_QK) ? 1 : 0;
    p.softplus_gate = (flags & KDA_FLAG_SOFTPLUS_GATE) ? 1 : 0;
    const cudaError_t err = kda::launch_backward(p, d_k, d_v, dt == KDA_F32 ? 0 : 1, s);
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

int kda_state_io(kda_state_op op, float* dst, const float* src,
                 const int32_t* slots, int32_t n, int32_t pool_size,
                 int32_t H, int32_t d_k, int32_t d_v, void* stream) {
    if (!supported_dim(d_k) || !supported_dim(d_v)) return KDA_ERR_UNSUPPORTED;
    if (n < 0 || H < 1 || pool_size < 0) return KDA_ERR_INVALID_ARG;
    if (n == 0) return KDA_OK;
    if (!dst) return KDA_ERR_INVALID_ARG;
    if (!aligned(dst, 16) || !aligned(src, 16) || !aligned(slots, 4)) return KDA_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t state_floats = (size_t)H * d_k * d_v;
    cudaError_t err = cudaSuccess;
    switch (op) {
        case KDA_STATE_ZERO:
            if (slots) {
                err = kda::launch_state_zero_slots(dst, slots, n, pool_size, state_floats, s);
            } else {
                err = cudaMemsetAsync(dst, 0, (size_t)n * state_floats * sizeof(float), s);
            }
            break;
        case KDA_STATE_COPY:
            if (slots || !src) return KDA_ERR_INVALID_ARG;
            err = cudaMemcpyAsync(dst, src, (size_t)n * state_floats * sizeof(float),
                                  cudaMemcpyDefault, s);
            break;
        case KDA_STATE_GATHER:
            if (!slots || !src) return KDA_ERR_INVALID_ARG;
            err = kda::launch_state_gather(dst, src, slots, n, pool_size, state_floats, s);
            break;
        case KDA_STATE_SCATTER:
            if (!slots || !src) return KDA_ERR_INVALID_ARG;
            err = kda::launch_state_scatter(dst, src, slots, n, pool_size, state_floats, s);
            break;
        default:
            return KDA_ERR_INVALID_ARG;
    }
    return err == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}

}  // extern "C"
