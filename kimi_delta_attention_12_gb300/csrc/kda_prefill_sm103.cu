// kda_prefill_sm103.cu -- chunked KDA prefill on tcgen05 tensor cores (sm_103a).
//
// The pages' prefill ("Kimi K3 Open Weights: What Is Actually New In Its 2.8
// Trillion Parameter Architecture", section 1) processes tokens "parallel
// within chunks, recurrent between", with decay products, triangular
// intra-chunk interactions and dense matrix tiles; the bounded gate
// (g >= -5) keeps the reciprocal decay factors of a 16-token tile inside the
// bf16 range (e^80 < 3.4e38), so the diagonal tiles use dense matmuls too.
// The per-chunk algebra and the phases are in kda_chunk_phases.cuh.
//
// Two kernels run those phases:
//
// kda_chunked_kernel (single pass): one CTA of 16 warps per (sequence, head)
//   walks the sequence's 64-token chunks; per chunk
//     P0  TMA: raw q, k, z tiles [64 tok][128 ch]; v as a 128B-swizzled operand
//     P1  prologue on the CUDA cores: L2 norms, gate, per-block cumulative
//         decay, and the bf16 operand tiles (X~, K~^(a), K+, Q+, Kend)
//     P2  tcgen05: Gram Aqk/Akk (two M=128 x N=64 x K=128 products)
//     P3  Gram -> smem (masking, beta);  S^T -> bf16 operand; S^T *= Gamma
//     P4  UT solve in shared memory (fp32): Tm
//     P5  tcgen05: W^T = K+^T Tm^T, U^T = V^T Tm^T
//     P6  W^T -> bf16 operand
//     P7  tcgen05: U^T += S^T (-W^T), O = Q+ S
//     P8  U^T -> bf16 operand
//     P9  tcgen05: O += Aqk U, S^T += U^T Kend
//     P10 O -> o (bf16)
//   with the fp32 state S^T in TMEM for the whole sequence.
//
// kda_split_kernel (few (sequence, head) units, e.g. 32 heads of one
//   sequence on 152 SMs): one launch of one CTA per SM.  CTAs 0..U-1 are
//   consumers, one per unit, and run only the sequential part of every chunk
//   (P3 state half, P5 U', P7..P10).  The other CTAs are producers: they take
//   (chunk, unit) tasks in chunk-major order from an atomic counter and run
//   the state-independent part (P0..P6) of each, then publish the chunk's
//   operand tiles (W^T, Q+, Kend, Aqk, Tm, Gamma) to a workspace slot and
//   raise the slot's flag (release).  A consumer waits for the flag of its
//   next chunk (acquire, bounded), copies the slot into shared memory with
//   one bulk copy and its v tile with TMA, one chunk ahead of use.
//   Producers never wait for consumers, so progress needs only that every
//   CTA is resident: the grid is one CTA per SM.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_chunk_phases.cuh"
#include "kda_internal.h"
#include "sm103_ptx.cuh"

namespace kda {
namespace {

using namespace sm103;
using namespace chunk;

struct ChunkedArgs {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_z;
    CUtensorMap tm_v;
    ChunkedParams p;
};

// ---- split mode: one published chunk (a workspace slot), byte offsets ----
constexpr uint32_t HO_WT = 0;
constexpr uint32_t HO_QP = 16384;
constexpr uint32_t HO_KE = 32768;
constexpr uint32_t HO_AQK = 49152;
constexpr uint32_t HO_TM = 57344;
constexpr uint32_t HO_GAM = 65536;
constexpr uint32_t HO_BYTES = 66048;           // multiple of 256
// consumer shared memory: two buffers of [slot | v tile], then S^T and U^T
constexpr uint32_t CB_V = 66560;               // v tile inside a buffer (1024-aligned)
constexpr uint32_t CB_BYTES = CB_V + 16384;    // 82944
constexpr uint32_t CB_ST = 2 * CB_BYTES;       // 165888
constexpr uint32_t CB_UT = CB_ST + 32768;      // 198656
static_assert(CB_UT + 16384 <= SMEM_USED, "consumer layout exceeds the shared memory budget");

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ Ctx make_ctx(uint8_t* sm, uint32_t tbase) {
    Ctx x;
    x.sm = sm;
    x.smem_base = smem_u32(sm);
    x.tbase = tbase;
    x.tid = threadIdx.x;
    x.warp = x.tid >> 5;
    x.lane = x.tid & 31;
    x.qd = x.warp & 3;
    x.sub = x.warp >> 2;
    x.lane_base = (uint32_t)(32 * x.qd) << 16;
    return x;
}

__device__ __forceinline__ void seq_bounds(const ChunkedParams& p, int n, int64_t& bos,
                                           int64_t& eos) {
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        eos = p.cu_seqlens[n + 1];
    } else {
        const int64_t len = p.total_T / p.N;
        bos = (int64_t)n * len;
        eos = bos + len;
    }
}

// ====================================================================== single pass
__global__ void __launch_bounds__(kThreads, 1)
kda_chunked_kernel(const __grid_constant__ ChunkedArgs args) {
    const ChunkedParams& p = args.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    __shared__ uint64_t bar_raw;   // raw q, k, z of a chunk landed
    __shared__ uint64_t bar_v;     // v of a chunk landed
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    float* s_beta = reinterpret_cast<float*>(sm + OFF_BETA);
    const float* s_gam = reinterpret_cast<const float*>(sm + OFF_GAM);

    const int tid = threadIdx.x;
    const int H = p.H;
    const int unit = blockIdx.x;
    const int n = unit / H;
    const int h = unit % H;
    int64_t bos, eos;
    seq_bounds(p, n, bos, eos);
    const size_t state_off = (size_t)unit * D * D;

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar_raw, 1);
        mbar_init(&bar_v, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&args.tm_q);
        prefetch_tmap(&args.tm_k);
        prefetch_tmap(&args.tm_z);
        prefetch_tmap(&args.tm_v);
    }
    if ((tid >> 5) == 0) {
        tmem_alloc(&tmem_base_s, TMEM_COLS);
        tmem_relinquish();
    }
    cta_sync_tc();
    const Ctx x = make_ctx(sm, tmem_base_s);
    const StateTiles lt = local_tiles();

    load_state(x, p.initial_state ? p.initial_state + state_off : nullptr);
    cta_sync_tc();

    const float eA_log2 = exp2_approx(p.A[h] * kLog2e) * kLog2e;  // e^A log2(e)
    const __nv_bfloat16* beta_g = static_cast<const __nv_bfloat16*>(p.beta);
    __nv_bfloat16* o_g = static_cast<__nv_bfloat16*>(p.o);

    uint32_t ph_raw = 0, ph_v = 0, ph_mma = 0;
    const int64_t len = eos - bos;
    const int nchunks = (int)((len + C - 1) / C);
    // loads issued and not yet waited for (uniform across the CTA); drained
    // before exit if the chunk loop is left early
    bool raw_pending = nchunks > 0, v_pending = nchunks > 0;

    // loads of chunk 0; later chunks are issued one chunk ahead
    if (tid == 0 && nchunks > 0) {
        mbar_arrive_expect_tx(&bar_raw, 3 * 16384);
        tma_load_3d(sm + OFF_RAWQ, &args.tm_q, 0, h, (int)bos, &bar_raw);
        tma_load_3d(sm + OFF_RAWK, &args.tm_k, 0, h, (int)bos, &bar_raw);
        tma_load_3d(sm + OFF_RAWZ, &args.tm_z, 0, h, (int)bos, &bar_raw);
        mbar_arrive_expect_tx(&bar_v, 16384);
        tma_load_3d(sm + OFF_V, &args.tm_v, 0, h, (int)bos, &bar_v);
        tma_load_3d(sm + OFF_V + 8192, &args.tm_v, 64, h, (int)bos, &bar_v);
    }
    // beta of the next chunk is fetched one chunk ahead into a register
    float beta_next = 0.0f;
    if (tid < C && tid < len) {
        beta_next = __bfloat162float(beta_g[(size_t)(bos + tid) * H + h]);
    }

    for (int ci = 0; ci < nchunks; ++ci) {
        const int64_t t0 = bos + (int64_t)ci * C;
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);

        const bool has_next = ci + 1 < nchunks;
        const int t_next = (int)(t0 + C);

        // ---------------- P0: this chunk's raw tiles (issued one chunk ahead) ----------------
        if (tid < C) {
            s_beta[tid] = beta_next;
            beta_next = 0.0f;
            if (has_next && t_next + tid < eos) {
                beta_next = __bfloat162float(beta_g[(size_t)(t_next + tid) * H + h]);
            }
        }
        if (mbar_wait(&bar_raw, ph_raw, &abort_flag)) {
            ph_raw ^= 1;
            raw_pending = false;
        } else {
            record_timeout(p.status, &abort_flag);
        }
        __syncthreads();
        if (abort_flag) {
            break;
        }

        // ---------------- P1a: per-token L2 norms ----------------
        phase_norms(x, L, p.scale, p.l2norm);
        __syncthreads();

        // ---------------- P1b: gate, decay products and operand tiles ----------------
        phase_prologue(x, L, eA_log2);

        // ---------------- P1c: (operand tiles written above) ----------------
        fence_proxy_async();
        cta_sync_tc();

        // ---------------- P2: Gram products ----------------
        raw_pending = has_next;
        if (tid == 0) {
            if (has_next) {  // raw tiles are consumed: fetch the next chunk's
                mbar_arrive_expect_tx(&bar_raw, 3 * 16384);
                tma_load_3d(sm + OFF_RAWQ, &args.tm_q, 0, h, t_next, &bar_raw);
                tma_load_3d(sm + OFF_RAWK, &args.tm_k, 0, h, t_next, &bar_raw);
                tma_load_3d(sm + OFF_RAWZ, &args.tm_z, 0, h, t_next, &bar_raw);
            }
            issue_gram(x);
            mma_commit(&bar_mma);
        }
        if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
            record_timeout(p.status, &abort_flag);
        }
        ph_mma ^= 1;
        tc_fence_after();
        __syncthreads();
        if (abort_flag) {
            break;
        }

        // ---------------- P3: Gram -> Akk, Aqk;  S^T -> bf16, S^T *= Gamma ----------------
        if (x.warp < 8) {
            phase_gram_epilogue(x);
        } else {
            phase_state_epilogue(x, s_gam, lt.st, 2, 2);
        }
        cta_sync_tc();

        // ---------------- P4: UT solve  Tm = (I + Akk)^-1 Diag(beta) ----------------
        phase_solve(x);
        fence_proxy_async();
        cta_sync_tc();

        // ---------------- P5: W^T = K+^T Tm^T,  U^T = V^T Tm^T ----------------
        if (mbar_wait(&bar_v, ph_v, &abort_flag)) {
            ph_v ^= 1;
            v_pending = false;
        } else {
            record_timeout(p.status, &abort_flag);
        }
        if (tid == 0 && !abort_flag) {
            issue_w(x);
            issue_u_prime(x, lt);
            mma_commit(&bar_mma);
        }
        if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
            record_timeout(p.status, &abort_flag);
        }
        ph_mma ^= 1;
        tc_fence_after();
        __syncthreads();
        if (abort_flag) {
            break;
        }
        v_pending = has_next;
        if (tid == 0 && has_next) {  // v tile consumed by the tensor core: fetch the next one
            mbar_arrive_expect_tx(&bar_v, 16384);
            tma_load_3d(sm + OFF_V, &args.tm_v, 0, h, t_next, &bar_v);
            tma_load_3d(sm + OFF_V + 8192, &args.tm_v, 64, h, t_next, &bar_v);
        }

        // ---------------- P6: W^T -> bf16 operand ----------------
        phase_tile_from_tmem(x, TM_W, lt.wt);
        fence_proxy_async();
        cta_sync_tc();

        // ---------------- P7: U^T += S^T (-W^T),  O = Q+ S ----------------
        if (tid == 0) {
            issue_uo(x, lt);
            mma_commit(&bar_mma);
        }
        if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
            record_timeout(p.status, &abort_flag);
        }
        ph_mma ^= 1;
        tc_fence_after();
        __syncthreads();
        if (abort_flag) {
            break;
        }

        // ---------------- P8: U^T -> bf16 operand ----------------
        phase_tile_from_tmem(x, TM_U, lt.ut);
        fence_proxy_async();
        cta_sync_tc();

        // ---------------- P9: O += Aqk U,  S^T += U^T Kend ----------------
        if (tid == 0) {
            issue_os(x, lt);
            mma_commit(&bar_mma);
        }
        if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
            record_timeout(p.status, &abort_flag);
        }
        ph_mma ^= 1;
        tc_fence_after();
        __syncthreads();
        if (abort_flag) {
            break;
        }

        // ---------------- P10: O -> o ----------------
        phase_o_epilogue(x, o_g, t0, L, h, H);
        cta_sync_tc();
    }

    // a loop left early may still have loads in flight into this CTA's smem
    if (raw_pending) {
        mbar_wait(&bar_raw, ph_raw, nullptr);
    }
    if (v_pending) {
        mbar_wait(&bar_v, ph_v, nullptr);
    }
    if (!abort_flag && p.final_state) {
        store_state(x, p.final_state + state_off);
    }
    cta_sync_tc();
    if (x.warp == 0) {
        tmem_dealloc(x.tbase, TMEM_COLS);
    }
}

// ====================================================================== split mode
// Bounded wait for a release-published flag (acquire, one thread).
__device__ __forceinline__ bool wait_flag(const int32_t* flag, const volatile int* abort_flag) {
    for (uint32_t i = 0; i < (1u << 25); ++i) {
        int32_t v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(flag) : "memory");
        if (v != 0) {
            return true;
        }
        if (*abort_flag) {
            return false;
        }
        __nanosleep(128);
    }
    return false;
}

// chunk index base of sequence n: sum over earlier sequences of ceil(len / C)
__device__ __forceinline__ int64_t chunk_base(const ChunkedParams& p, int n) {
    int64_t base = 0;
    for (int m = 0; m < n; ++m) {
        int64_t b, e;
        seq_bounds(p, m, b, e);
        base += (e - b + C - 1) / C;
    }
    return base;
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes,
                                          uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(gsrc)), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

__global__ void __launch_bounds__(kThreads, 1)
kda_split_kernel(const __grid_constant__ ChunkedArgs args) {
    const ChunkedParams& p = args.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    __shared__ uint64_t bar_raw;
    __shared__ uint64_t bar_full[2];
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base_s;
    __shared__ int s_task;
    __shared__ int s_issued;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int H = p.H;
    const int U = p.N * H;

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar_raw, 1);
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&args.tm_q);
        prefetch_tmap(&args.tm_k);
        prefetch_tmap(&args.tm_z);
        prefetch_tmap(&args.tm_v);
    }
    if ((tid >> 5) == 0) {
        tmem_alloc(&tmem_base_s, TMEM_COLS);
        tmem_relinquish();
    }
    cta_sync_tc();
    const Ctx x = make_ctx(sm, tmem_base_s);
    const __nv_bfloat16* beta_g = static_cast<const __nv_bfloat16*>(p.beta);
    uint32_t ph_mma = 0;

    if ((int)blockIdx.x < U) {
        // ------------------------------------------------------------ consumer
        const int unit = blockIdx.x;
        const int n = unit / H;
        const int h = unit % H;
        int64_t bos, eos;
        seq_bounds(p, n, bos, eos);
        const int nchunks = (int)((eos - bos + C - 1) / C);
        const int64_t base = chunk_base(p, n);
        const size_t state_off = (size_t)unit * D * D;
        __nv_bfloat16* o_g = static_cast<__nv_bfloat16*>(p.o);

        load_state(x, p.initial_state ? p.initial_state + state_off : nullptr);
        cta_sync_tc();

        // one thread: wait for chunk c's slot and copy it (and the v tile) into buffer c & 1
        auto fetch = [&](int c) -> bool {
            const int64_t slot = (base + c) * H + h;
            if (!wait_flag(p.flags + slot, &abort_flag)) {
                return false;
            }
            // order the acquire (and this CTA's earlier generic accesses to the
            // buffer) before the async-proxy copies below
            asm volatile("fence.proxy.async.global;" ::: "memory");
            fence_proxy_async();
            uint8_t* buf = sm + (c & 1) * CB_BYTES;
            uint64_t* bar = &bar_full[c & 1];
            const int t0 = (int)(bos + (int64_t)c * C);
            mbar_arrive_expect_tx(bar, HO_BYTES + 16384);
            bulk_load(buf, p.handoff + slot * HO_BYTES, HO_BYTES, bar);
            tma_load_3d(buf + CB_V, &args.tm_v, 0, h, t0, bar);
            tma_load_3d(buf + CB_V + 8192, &args.tm_v, 64, h, t0, bar);
            return true;
        };
        // number of chunks whose copies were issued (thread 0's count)
        int issued = 0;
        if (tid == 0 && nchunks > 0) {
            if (fetch(0)) {
                issued = 1;
            } else {
                record_timeout(p.status, &abort_flag);
            }
        }
        __syncthreads();
        int waited = 0;
        for (int c = 0; c < nchunks && !abort_flag; ++c) {
            const int b = c & 1;
            const int64_t t0 = bos + (int64_t)c * C;
            const int L = (int)((eos - t0) < C ? (eos - t0) : C);
            const uint32_t cb = b * CB_BYTES;
            const StateTiles st{cb + HO_WT, cb + HO_QP, cb + HO_KE, cb + HO_AQK, cb + HO_TM,
                                cb + HO_GAM, cb + CB_V, CB_ST, CB_UT};
            if (!mbar_wait(&bar_full[b], (c >> 1) & 1, &abort_flag)) {
                record_timeout(p.status, &abort_flag);
            }
            waited = c + 1;
            tc_fence_after();
            __syncthreads();
            if (abort_flag) {
                break;
            }
            if (tid == 0) {
                issue_u_prime(x, st);          // U'^T = V^T Tm^T, independent of S
                mma_commit(&bar_mma);
                if (c + 1 < nchunks) {         // buffer b^1 was released by chunk c-1
                    if (fetch(c + 1)) {
                        issued = c + 2;
                    } else {
                        record_timeout(p.status, &abort_flag);
                    }
                }
            }
            // S^T -> bf16 operand, S^T *= Gamma_C (all 16 warps, 32 columns each)
            phase_state_epilogue(x, reinterpret_cast<const float*>(sm + st.gam), st.st, 0, 4);
            fence_proxy_async();
            tc_fence_before();
            if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
                record_timeout(p.status, &abort_flag);
            }
            ph_mma ^= 1;
            tc_fence_after();
            __syncthreads();
            if (abort_flag) {
                break;
            }
            if (tid == 0) {
                issue_uo(x, st);
                mma_commit(&bar_mma);
            }
            if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
                record_timeout(p.status, &abort_flag);
            }
            ph_mma ^= 1;
            tc_fence_after();
            __syncthreads();
            if (abort_flag) {
                break;
            }
            phase_tile_from_tmem(x, TM_U, st.ut);
            fence_proxy_async();
            cta_sync_tc();
            if (tid == 0) {
                issue_os(x, st);
                mma_commit(&bar_mma);
            }
            if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
                record_timeout(p.status, &abort_flag);
            }
            ph_mma ^= 1;
            tc_fence_after();
            __syncthreads();
            if (abort_flag) {
                break;
            }
            phase_o_epilogue(x, o_g, t0, L, h, H);
            cta_sync_tc();
        }
        // drain copies still in flight into this CTA's smem (early exit only)
        if (tid == 0) {
            s_issued = issued;
        }
        __syncthreads();
        for (int c = waited; c < s_issued; ++c) {
            mbar_wait(&bar_full[c & 1], (c >> 1) & 1, nullptr);
        }
        if (!abort_flag && p.final_state) {
            store_state(x, p.final_state + state_off);
        }
    } else {
        // ------------------------------------------------------------ producer
        int max_chunks = 0;
        for (int m = 0; m < p.N; ++m) {
            int64_t b, e;
            seq_bounds(p, m, b, e);
            const int nc = (int)((e - b + C - 1) / C);
            max_chunks = nc > max_chunks ? nc : max_chunks;
        }
        const int ntasks = max_chunks * U;
        float* s_beta = reinterpret_cast<float*>(sm + OFF_BETA);
        // task t = (chunk t / U, unit t % U), chunk-major; tasks past the end of
        // their sequence are skipped.  Thread 0 only.
        auto grab_valid = [&]() -> int {
            for (;;) {
                const int t = atomicAdd(p.work_counter, 1);
                if (t >= ntasks) {
                    return ntasks;
                }
                int64_t b, e;
                seq_bounds(p, (t % U) / H, b, e);
                if (t / U < (int)((e - b + C - 1) / C)) {
                    return t;
                }
            }
        };
        auto issue_raw = [&](int t) {
            const int hh = (t % U) % H;
            int64_t b, e;
            seq_bounds(p, (t % U) / H, b, e);
            const int tt0 = (int)(b + (int64_t)(t / U) * C);
            mbar_arrive_expect_tx(&bar_raw, 3 * 16384);
            tma_load_3d(sm + OFF_RAWQ, &args.tm_q, 0, hh, tt0, &bar_raw);
            tma_load_3d(sm + OFF_RAWK, &args.tm_k, 0, hh, tt0, &bar_raw);
            tma_load_3d(sm + OFF_RAWZ, &args.tm_z, 0, hh, tt0, &bar_raw);
        };
        uint32_t ph_raw = 0;
        bool raw_pending = false;      // a raw load is in flight (uniform after each barrier)
        if (tid == 0) {
            s_task = grab_valid();
            if (s_task < ntasks) {
                issue_raw(s_task);
            }
        }
        __syncthreads();
        int task = s_task;
        raw_pending = task < ntasks;
        while (task < ntasks && !abort_flag) {
            const int c = task / U;
            const int unit = task % U;
            const int n = unit / H;
            const int h = unit % H;
            int64_t bos, eos;
            seq_bounds(p, n, bos, eos);
            const int64_t t0 = bos + (int64_t)c * C;
            const int L = (int)((eos - t0) < C ? (eos - t0) : C);
            const int64_t slot = (chunk_base(p, n) + c) * H + h;
            const float eA_log2 = exp2_approx(p.A[h] * kLog2e) * kLog2e;
            // beta: loaded now, stored to shared memory once the prologue is done
            float beta_r = 0.0f;
            if (tid < L) {
                beta_r = __bfloat162float(beta_g[(size_t)(t0 + tid) * H + h]);
            }
            if (mbar_wait(&bar_raw, ph_raw, &abort_flag)) {
                ph_raw ^= 1;
                raw_pending = false;
            } else {
                record_timeout(p.status, &abort_flag);
            }
            __syncthreads();
            if (abort_flag) {
                break;
            }
            phase_norms(x, L, p.scale, p.l2norm);
            __syncthreads();
            phase_prologue(x, L, eA_log2);
            // every thread has passed the prologue's barrier: the raw tiles are
            // consumed, fetch the next task's
            if (tid == 0) {
                s_task = grab_valid();
                if (s_task < ntasks) {
                    issue_raw(s_task);
                }
            }
            if (tid < C) {
                s_beta[tid] = beta_r;
            }
            fence_proxy_async();
            cta_sync_tc();
            raw_pending = s_task < ntasks;
            if (tid == 0) {
                issue_gram(x);
                mma_commit(&bar_mma);
            }
            if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
                record_timeout(p.status, &abort_flag);
            }
            ph_mma ^= 1;
            tc_fence_after();
            __syncthreads();
            if (abort_flag) {
                break;
            }
            if (x.warp < 8) {
                phase_gram_epilogue(x);
            }
            cta_sync_tc();
            phase_solve(x);
            fence_proxy_async();
            cta_sync_tc();
            if (tid == 0) {
                issue_w(x);
                mma_commit(&bar_mma);
            }
            if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
                record_timeout(p.status, &abort_flag);
            }
            ph_mma ^= 1;
            tc_fence_after();
            __syncthreads();
            if (abort_flag) {
                break;
            }
            phase_tile_from_tmem(x, TM_W, OFF_WT);
            __syncthreads();
            // publish: the slot is an image of the operand tiles
            uint4* dst = reinterpret_cast<uint4*>(p.handoff + slot * HO_BYTES);
            const uint32_t src_off[6] = {OFF_WT, OFF_QP, OFF_KE, OFF_AQK, OFF_TM, OFF_GAM};
            const uint32_t dst_off[6] = {HO_WT, HO_QP, HO_KE, HO_AQK, HO_TM, HO_GAM};
            const uint32_t nbytes[6] = {16384, 16384, 16384, 8192, 8192, 512};
#pragma unroll
            for (int t = 0; t < 6; ++t) {
                const uint4* src = reinterpret_cast<const uint4*>(sm + src_off[t]);
                uint4* d = dst + dst_off[t] / 16;
                for (uint32_t e = tid; e < nbytes[t] / 16; e += kThreads) {
                    d[e] = src[e];
                }
            }
            __threadfence();
            __syncthreads();
            if (tid == 0) {
                asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.flags + slot), "r"(1)
                             : "memory");
            }
            task = s_task;
        }
        // a loop left early may still have a raw load in flight into this CTA's smem
        if (raw_pending) {
            mbar_wait(&bar_raw, ph_raw, nullptr);
        }
    }
    cta_sync_tc();
    if (x.warp == 0) {
        tmem_dealloc(x.tbase, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            return nullptr;
        }
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

bool make_map(CUtensorMap* map, const void* base, int total_T, int H, int box_c,
              CUtensorMapSwizzle swz) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) {
        return false;
    }
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)total_T};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)box_c, 1, (cuuint32_t)C};
    cuuint32_t es[3] = {1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
              box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_args(ChunkedArgs* args, const ChunkedParams& p) {
    memset(args, 0, sizeof(*args));
    args->p = p;
    return make_map(&args->tm_q, p.q, p.total_T, p.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(&args->tm_k, p.k, p.total_T, p.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(&args->tm_z, p.z, p.total_T, p.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) &&
           make_map(&args->tm_v, p.v, p.total_T, p.H, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

size_t chunked_workspace_bytes(int32_t N, int32_t H) {
    return 256 + (size_t)N * H * sizeof(int32_t);
}

size_t split_slots_bound(int32_t N, int32_t total_T, int32_t H) {
    return (size_t)H * ((size_t)(total_T + C - 1) / C + (size_t)N);
}

size_t split_handoff_offset(int32_t N, int32_t total_T, int32_t H) {
    const size_t flags = split_slots_bound(N, total_T, H) * sizeof(int32_t);
    return 256 + (flags + 255) / 256 * 256;
}

size_t split_workspace_bytes(int32_t N, int32_t total_T, int32_t H) {
    return split_handoff_offset(N, total_T, H) + split_slots_bound(N, total_T, H) * HO_BYTES;
}

int split_max_units(int num_sms) {
    // producers need most of the GPU: at most a third of the SMs are consumers
    return num_sms / 3;
}

cudaError_t launch_chunked_prefill(const ChunkedParams& p, cudaStream_t stream) {
    ChunkedArgs args;
    if (!make_args(&args, p)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = cudaFuncSetAttribute(kda_chunked_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) {
        return err;
    }
    const unsigned grid = (unsigned)((int64_t)p.N * p.H);
    if (grid == 0) {
        return cudaSuccess;
    }
    kda_chunked_kernel<<<grid, kThreads, SMEM_BYTES, stream>>>(args);
    return cudaGetLastError();
}

cudaError_t launch_split_prefill(const ChunkedParams& p, int num_sms, cudaStream_t stream) {
    ChunkedArgs args;
    if (!make_args(&args, p)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = cudaFuncSetAttribute(kda_split_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)SMEM_BYTES);
    if (err != cudaSuccess) {
        return err;
    }
    // p.flags was zeroed by the caller on this stream
    kda_split_kernel<<<(unsigned)num_sms, kThreads, SMEM_BYTES, stream>>>(args);
    return cudaGetLastError();
}

}  // namespace kda
