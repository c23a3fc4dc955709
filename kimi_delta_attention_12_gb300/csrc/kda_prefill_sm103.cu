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
//     P7  tcgen05: U^T += S^T (-W^T), O^T = S^T Q+^T
//     P8  U^T -> bf16 operand
//     P9  tcgen05: S^T += U^T Kend, O^T += U^T Aqk^T
//     P10 O -> o (bf16)
//   with the fp32 state S^T in TMEM for the whole sequence.
//
// kda_split_kernel: one launch of one CTA per SM.  The (sequence, head)
//   units are cut into batches of at most a quarter of the SMs.  CTA i < the
//   batch size is a consumer: it carries the state of the i-th unit of each
//   batch in turn and runs only the sequential part of every chunk (the
//   state epilogue, U', U, O, the state update and o).  The other CTAs are
//   producers: they take (chunk, unit) tasks in batch-major, then chunk-major
//   order from an atomic counter, run the state-independent part of each
//   (prologue, Gram, UT solve, W) and store the chunk's operand tiles
//   (Aqk, Tm, W^T, Q+, Kend, Gamma) with bulk copies into a ring of slots
//   that belongs to the chunk's consumer, then raise the slot's flag
//   (release).  A consumer waits for its next chunk's flag (acquire,
//   bounded), copies the slot into shared memory with one bulk copy and the
//   v tile with TMA, one chunk ahead of use, and reports every chunk it has
//   copied out so that producers may refill the slot.  Tasks are taken in
//   the order consumers need them and every CTA is resident (the grid is
//   one CTA per SM), so each wait ends.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_chunk_phases.cuh"
#include "kda_chunked.h"
#include "kda_seqlens.cuh"
#include "kda_split_phases.cuh"
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

// consumer shared memory: two buffers of [slot | v tile] (its bf16 S^T and
// U^T operands live in TMEM)
constexpr uint32_t CB_BYTES = 66560;          // one slot buffer (HO_BYTES, 1024-aligned)
constexpr uint32_t CB_VRING = 2 * CB_BYTES;    // then a ring of v tiles, prefetched ahead
constexpr int kVRing = 4;
// dynamic shared memory of the split kernel: the larger of the consumer's
// and the producer's layouts, plus slack for the 1024-byte alignment
constexpr uint32_t kSplitSmemBytes =
    (CB_VRING + kVRing * 16384 > split::P_END ? CB_VRING + kVRing * 16384 : split::P_END) + 1024;

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
    clamped_seq(p.cu_seqlens, n, p.N, p.total_T, bos, eos);
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
    __shared__ uint64_t bar_fin;   // every MMA of this CTA done
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
        mbar_init(&bar_fin, 1);
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
    __shared__ int s_ck;
    const int64_t ck_base =
        p.ckpt_interval > 0
            ? ckpt_base(n, p.ckpt_interval,
                        [&](int m) {
                            int64_t b, e;
                            seq_bounds(p, m, b, e);
                            return (int)(e - b);
                        },
                        &s_ck)
            : 0;

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
            record_timeout(p.status, &abort_flag, 211);
        }
        __syncthreads();
        if (abort_flag) {
            break;
        }

        // ---------------- P1a: per-token L2 norms ----------------
        phase_norms(x, L, p.scale, p.l2norm);  // published by the prologue's barrier

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
            record_timeout(p.status, &abort_flag, 241);
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
            record_timeout(p.status, &abort_flag, 268);
        }
        if (tid == 0 && !abort_flag) {
            issue_w(x);
            issue_u_prime(x, lt);
            mma_commit(&bar_mma);
        }
        if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
            record_timeout(p.status, &abort_flag, 276);
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

        // ---------------- P7: U^T += S^T (-W^T),  O^T = S^T Q+^T ----------------
        if (tid == 0) {
            issue_uo(x, lt);
            mma_commit(&bar_mma);
        }
        if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
            record_timeout(p.status, &abort_flag, 302);
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

        // ---------------- P9: S^T += U^T Kend,  O^T += U^T Aqk^T ----------------
        if (tid == 0) {
            issue_os(x, lt);
            mma_commit(&bar_mma);
        }
        if (!mbar_wait(&bar_mma, ph_mma, &abort_flag)) {
            record_timeout(p.status, &abort_flag, 322);
        }
        ph_mma ^= 1;
        tc_fence_after();
        __syncthreads();
        if (abort_flag) {
            break;
        }

        // ---------------- P10: O -> o ----------------
        phase_o_epilogue(x, o_g, t0, L, h, H);
        // state checkpoint after this chunk (S^T in TMEM is the state after it)
        if (p.ckpt_interval > 0) {
            const int64_t done = (int64_t)(ci + 1) * C;
            const int64_t idx = ck_base + done / p.ckpt_interval - 1;
            if (done % p.ckpt_interval == 0 && done <= len && idx < p.ckpt_count) {
                const int64_t row = p.ckpt_slots ? (int64_t)p.ckpt_slots[idx] : idx;
                if (row >= 0 && row < p.ckpt_pool_size) {
                    store_state(x, p.ckpt_pool + ((size_t)row * H + h) * D * D);
                }
            }
        }
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
    // a loop left early may still have MMAs running: none may be when the
    // TMEM is freed
    cta_sync_tc();
    if (tid == 0) {
        mma_commit(&bar_fin);
        mbar_wait(&bar_fin, 0, nullptr);
    }
    cta_sync_tc();
    if (x.warp == 0) {
        tmem_dealloc(x.tbase, TMEM_COLS);
    }
}

// ====================================================================== split mode
__device__ __forceinline__ int32_t ld_acquire(const int32_t* ptr) {
    int32_t v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int32_t* ptr, int32_t v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// Tells producers that a ring slot may be rewritten.  The slot's bulk copy
// into this CTA's shared memory has completed (its mbarrier phase was
// observed) before this store is issued, so no data needs publishing with it:
// a relaxed store, which does not wait for this CTA's output stores to drain
// as a release would.
__device__ __forceinline__ void st_relaxed(int32_t* ptr, int32_t v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(ptr), "r"(v) : "memory");
}

// Bounded wait (one thread) until *ptr >= target: at most `polls` polls.
// False on timeout or when another thread of the CTA raised the abort flag.
__device__ __forceinline__ bool wait_at_least(const int32_t* ptr, int32_t target,
                                              const volatile int* abort_flag, uint32_t polls) {
    for (uint32_t i = 0; i < polls; ++i) {
        if (ld_acquire(ptr) >= target) {
            return true;
        }
        if (*abort_flag) {
            return false;
        }
        __nanosleep(64);
    }
    return false;
}

// orders this thread's generic-proxy global accesses with its later (or
// earlier) async-proxy ones
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}


// Sequence and batch tables, built by every CTA at start (the chunk bases
// only with chunk records).
template <bool kRec>
struct SplitMetaT {
    int32_t cu[kSplitMaxSeqs + 1];       // token start of each sequence (and total_T)
    float eA[kSplitMaxHeads];            // e^{A_h} log2(e)
    int32_t task0[kSplitMaxBatches + 1]; // first task of each batch
    int32_t g0[kSplitMaxBatches + 1];    // first consumer-stream index of each batch
    int32_t ch0[kRec ? kSplitMaxSeqs + 1 : 1];   // records: first chunk of each sequence
    uint8_t* rec;                        // the chunk records, or null (none, or too few)
};

static_assert(REC_BYTES == kChunkRecordBytes, "chunk record size");

// The chunk record of chunk c of sequence n, head h (none without records).
template <bool kRec>
__device__ __forceinline__ uint8_t* chunk_record(const SplitMetaT<kRec>& m,
                                                 const ChunkedParams& p, int n, int c, int h) {
    if constexpr (kRec) {
        return m.rec + ((size_t)(m.ch0[n] + c) * p.H + h) * REC_BYTES;
    } else {
        return nullptr;
    }
}

// Length of sequence n from the clamped starts (never negative).
template <bool kRec>
__device__ __forceinline__ int32_t split_len(const SplitMetaT<kRec>& m, int n) {
    return max(0, m.cu[n + 1] - m.cu[n]);
}

// One producer task: chunk c of unit `unit` (the i-th unit of its batch).
// Task t of batch b is chunk (t - task0[b]) / nu of unit (t - task0[b]) % nu
// (chunk-major), nu the batch's units; in consumer i's stream of chunks it is
// number g = g0[b] + c, and it goes through ring slot i * ring + g % ring.
struct SplitTask {
    int i, unit, h, c, L;
    int32_t t0, g;
};

// False if the task's chunk lies past the end of its sequence.
template <bool kRec>
__device__ __forceinline__ bool decode_task(const SplitMetaT<kRec>& m, const ChunkedParams& p, int t,
                                            SplitTask& o) {
    int lo = 0, hi = p.n_batches - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (m.task0[mid] <= t) {
            lo = mid;
        } else {
            hi = mid - 1;
        }
    }
    const int U = p.N * p.H;
    const int u0 = lo * p.n_cons;
    const int nu = min(U - u0, p.n_cons);
    const int local = t - m.task0[lo];
    const int c = local / nu;
    o.i = local - c * nu;
    o.unit = u0 + o.i;
    const int n = o.unit / p.H;
    o.h = o.unit - n * p.H;
    o.c = c;
    const int32_t bos = m.cu[n];
    const int32_t len = split_len(m, n);
    o.t0 = bos + c * C;
    o.L = min(C, len - c * C);
    o.g = m.g0[lo] + c;
    return c * C < len;
}

// With the convolutions fused: the conv state after sequence n of head h --
// its last W-1 inputs of q, k and v, oldest first (from its conv state in
// where the sequence is shorter), as kda_short_conv writes it.  Every thread
// of the CTA; no barrier.
__device__ __forceinline__ void conv_state_tail(const ChunkedParams& p, int n, int h,
                                                int64_t bos, int64_t eos) {
    const int R = p.conv_W - 1;
    const __nv_bfloat16* st_in = static_cast<const __nv_bfloat16*>(p.conv_state_in);
    __nv_bfloat16* st_out = static_cast<__nv_bfloat16*>(p.conv_state_out);
    for (int e = threadIdx.x; e < R * 3 * D; e += blockDim.x) {
        const int r = e / (3 * D), ch = e - r * 3 * D;
        const int64_t tau = eos - R + r;
        __nv_bfloat16 val = __float2bfloat16_rn(0.0f);
        if (tau >= bos) {
            const void* x = ch < D ? p.q : ch < 2 * D ? p.k : p.v;
            val = static_cast<const __nv_bfloat16*>(x)[((size_t)tau * p.H + h) * D + (ch & (D - 1))];
        } else if (st_in) {
            val = st_in[(((size_t)n * p.H + h) * R + (tau - bos + R)) * 3 * D + ch];
        }
        st_out[(((size_t)n * p.H + h) * R + r) * 3 * D + ch] = val;
    }
}

// kMode: kSplitPlain, kSplitRecords (chunk records for the training
// backward) or kSplitConv (the short convolutions fused in); one
// instantiation each, so that the plain prefill carries none of the others'
// code.
constexpr int kSplitPlain = 0;
constexpr int kSplitRecords = 1;
constexpr int kSplitConv = 2;

template <int kMode>
__global__ void __launch_bounds__(kThreads, 1)
kda_split_kernel(const __grid_constant__ ChunkedArgs args) {
    constexpr bool kRec = kMode == kSplitRecords;
    constexpr bool kConv = kMode == kSplitConv;
    const ChunkedParams& p = args.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = align1024(smem_raw);
    __shared__ SplitMetaT<kRec> meta;
    __shared__ uint64_t bar_raw;       // producer: raw q, k, z landed
    __shared__ uint64_t bar_mma;       // producer: MMA group done
    __shared__ uint64_t bar_full[2];   // consumer: a buffer's slot landed
    __shared__ uint64_t bar_v[kVRing]; // consumer: a v tile landed
    __shared__ uint64_t bar_u;         // consumer: U^T done
    __shared__ uint64_t bar_os;        // consumer: O and the state update done
    __shared__ uint64_t bar_fin;       // every MMA of this CTA done
    __shared__ uint64_t bar_gram[2];   // producer: Gram products of task j done (buffer j & 1)
    __shared__ uint64_t bar_bdone[2];  // producer: B finished task j (K+, beta buffer j & 1 free)
    __shared__ uint64_t bar_aw[2];     // producer: A's writes of task j into its slot done
    __shared__ uint64_t bar_w;         // producer: W^T of a task done
    __shared__ uint64_t bar_finb;      // producer: every MMA of group B done
    __shared__ uint32_t tmem_base_s;
    __shared__ int s_issued;
    __shared__ int s_vissued;
    __shared__ int s_slot_free;
    __shared__ int s_ck;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int H = p.H;
    const int U = p.N * H;

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar_raw, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        for (int j = 0; j < kVRing; ++j) {
            mbar_init(&bar_v[j], 1);
        }
        mbar_init(&bar_u, 1);
        mbar_init(&bar_os, 1);
        mbar_init(&bar_fin, 1);
        mbar_init(&bar_gram[0], 1);
        mbar_init(&bar_gram[1], 1);
        mbar_init(&bar_bdone[0], 1);
        mbar_init(&bar_bdone[1], 1);
        mbar_init(&bar_aw[0], 1);
        mbar_init(&bar_aw[1], 1);
        mbar_init(&bar_w, 1);
        mbar_init(&bar_finb, 1);
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
    // sequence starts and gate constants
    // each entry clamped to [0, total_T]; a sequence's length is then
    // max(0, cu[n + 1] - cu[n]) (split_len), so it stays inside the tokens
    for (int n = tid; n <= p.N; n += kThreads) {
        meta.cu[n] = p.cu_seqlens ? (int32_t)clamp_token(p.cu_seqlens[n], p.total_T)
                                  : n * (p.total_T / p.N);
    }
    for (int h = tid; h < H; h += kThreads) {
        meta.eA[h] = exp2_approx(p.A[h] * kLog2e) * kLog2e;
    }
    __syncthreads();
    // per batch: tasks (its longest sequence's chunks x its units) and stream length
    for (int b = tid; b < p.n_batches; b += kThreads) {
        const int u0 = b * p.n_cons;
        const int u1 = min(U, u0 + p.n_cons);
        int maxc = 0;
        for (int n = u0 / H; n <= (u1 - 1) / H; ++n) {
            maxc = max(maxc, (split_len(meta, n) + C - 1) / C);
        }
        meta.task0[b + 1] = maxc * (u1 - u0);
        meta.g0[b + 1] = maxc;
    }
    if (tid == 0 && !kRec) {
        meta.rec = nullptr;
    }
    if (kRec && (tid >> 5) == 1) {   // chunk bases of the sequences (one warp)
        const int l = tid & 31;
        const int per = (p.N + 31) >> 5;
        const int n0 = min(l * per, p.N), n1 = min(n0 + per, p.N);
        int32_t a = 0;
        for (int n = n0; n < n1; ++n) {
            a += (split_len(meta, n) + C - 1) / C;
        }
        int32_t incl = a;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, incl, off);
            if (l >= off) {
                incl += t;
            }
        }
        int32_t run = incl - a;
        for (int n = n0; n < n1; ++n) {
            meta.ch0[n] = run;
            run += (split_len(meta, n) + C - 1) / C;
        }
        if (l == 31) {
            meta.ch0[p.N] = incl;
            // more chunks than the records hold (only a cu_seqlens the host has
            // not checked): an error, and the chunks go through the ring
            meta.rec = incl <= p.rec_chunks ? p.records : nullptr;
            if (!meta.rec) {
                atomicCAS(p.status, 0, kStatusRecords);
            }
        }
    }
    __syncthreads();
    if (tid < 32) {  // exclusive prefix sums over the batches (one warp)
        const int nb = p.n_batches;
        const int per = (nb + 31) >> 5;
        const int b0 = tid * per;
        int a = 0, g = 0;
        for (int j = 0; j < per; ++j) {
            if (b0 + j < nb) {
                a += meta.task0[b0 + j + 1];
                g += meta.g0[b0 + j + 1];
            }
        }
        int ai = a, gi = g;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int ta = __shfl_up_sync(0xffffffffu, ai, off);
            const int tg = __shfl_up_sync(0xffffffffu, gi, off);
            if (tid >= off) {
                ai += ta;
                gi += tg;
            }
        }
        int ra = ai - a, rg = gi - g;
        for (int j = 0; j < per; ++j) {
            if (b0 + j < nb) {
                ra += meta.task0[b0 + j + 1];
                meta.task0[b0 + j + 1] = ra;
                rg += meta.g0[b0 + j + 1];
                meta.g0[b0 + j + 1] = rg;
            }
        }
        if (tid == 0) {
            meta.task0[0] = 0;
            meta.g0[0] = 0;
        }
    }
    cta_sync_tc();
    const Ctx x = make_ctx(sm, tmem_base_s);
    const __nv_bfloat16* beta_g = static_cast<const __nv_bfloat16*>(p.beta);

    if ((int)blockIdx.x < p.n_cons) {
        // ------------------------------------------------------------ consumer
        const int i = blockIdx.x;
        __nv_bfloat16* o_g = static_cast<__nv_bfloat16*>(p.o);
        // with the convolutions fused, the convolved v tile comes in the slot
        // (buffers of HO_BYTES_CONV) and the v ring is not used
        constexpr bool conv = kConv;
        constexpr uint32_t cbuf = conv ? HO_BYTES_CONV : CB_BYTES;
        auto tiles = [&](uint32_t b, uint32_t vb) -> StateTiles {
            const uint32_t cb = b * cbuf;
            return StateTiles{cb + HO_WT, cb + HO_QP,  cb + HO_KE, cb + HO_AQK, cb + HO_TM,
                              cb + HO_GAM, conv ? cb + HO_V : CB_VRING + vb * 16384, 0, 0};
        };
        uint32_t cnt = 0;  // buffer fills so far (buffer = count & 1, parity = (count >> 1) & 1)
        uint32_t vcnt = 0; // v tiles loaded so far (ring slot = count % 4, parity = (count / 4) & 1)
        uint32_t ph_u = 0, ph_os = 0;
        {   // O^T starts at zero; every chunk's output epilogue zeroes it again
            uint32_t z[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) z[k] = 0u;
            tmem_st16(x.tbase + x.lane_base + TC_O + 16 * x.sub, z);
            tmem_wait_st();
        }
        for (int bt = 0; bt < p.n_batches && !abort_flag; ++bt) {
            const int unit = bt * p.n_cons + i;
            if (unit >= U) {
                break;
            }
            const int n = unit / H;
            const int h = unit - n * H;
            const int32_t bos = meta.cu[n];
            const int32_t len = split_len(meta, n);
            const int nch = (len + C - 1) / C;
            const int32_t g0 = meta.g0[bt];
            const size_t state_off = (size_t)unit * D * D;

            load_state(x, p.initial_state ? p.initial_state + state_off : nullptr);
            cta_sync_tc();
            const int64_t ck_base =
                p.ckpt_interval > 0
                    ? ckpt_base(n, p.ckpt_interval,
                                [&](int m) { return (int)split_len(meta, m); },
                                &s_ck)
                    : 0;

            // Thread 0 issues the tensor-core products and the v tiles; thread 32
            // polls the ring flags and issues the slot copies, so that their
            // acquire loads and proxy fences do not hold up the next products.
            int fetched = 0;  // thread 32: chunks of this unit whose copies are issued
            int waited = 0;   // chunks of this unit every thread has waited for
            int v_issued = 0, v_waited = 0;   // thread 0: v tiles of this unit
            // thread 0: load chunk c's v tile (an input, independent of the
            // producers) into the v ring, up to kVRing chunks ahead of use
            auto issue_v = [&](int c) {
                if (conv) {
                    return;
                }
                const uint32_t vb = (vcnt + c) % kVRing;
                uint8_t* vbuf = sm + CB_VRING + vb * 16384;
                mbar_arrive_expect_tx(&bar_v[vb], 16384);
                tma_load_3d(vbuf, &args.tm_v, 0, h, bos + c * C, &bar_v[vb]);
                tma_load_3d(vbuf + 8192, &args.tm_v, 64, h, bos + c * C, &bar_v[vb]);
                v_issued = c + 1;
            };
            // thread 0: wait for chunk c's v tile
            auto wait_v = [&](int c) -> bool {
                if (conv) {
                    return true;
                }
                const uint32_t r = vcnt + c;
                const bool ok = mbar_wait(&bar_v[r % kVRing], (r / kVRing) & 1, &abort_flag);
                if (ok) {
                    v_waited = c + 1;
                }
                return ok;
            };
            // thread 32: the ring flag of chunk c
            auto flag_of = [&](int c) -> const int32_t* {
                return p.flags + i * p.ring + (g0 + c) % p.ring;
            };
            // thread 32: copy chunk c's slot into buffer (cnt + c) & 1 (block: wait
            // for its flag; ready: an earlier acquire load of it saw it raised)
            auto fetch = [&](int c, bool block, bool ready = false) -> bool {
                const int32_t g = g0 + c;
                const int32_t slot = i * p.ring + g % p.ring;
                if (ready) {
                } else if (block) {
                    if (!wait_at_least(p.flags + slot, g + 1, &abort_flag, p.peer_wait_polls)) {
                        record_timeout(p.status, &abort_flag, 667);
                        return false;
                    }
                } else if (ld_acquire(p.flags + slot) < g + 1) {
                    return false;
                }
                // the acquire (and this CTA's earlier use of the buffer) before the copies
                fence_proxy_async_global();
                fence_proxy_async();
                const uint32_t b = (cnt + c) & 1;
                uint8_t* buf = sm + b * cbuf;
                const uint32_t bytes = conv ? HO_BYTES_CONV : HO_BYTES;
                mbar_arrive_expect_tx(&bar_full[b], bytes);
                bulk_load(buf,
                          kRec && meta.rec ? chunk_record(meta, p, n, c, h)
                                    : p.handoff + (size_t)slot * bytes,
                          bytes, &bar_full[b]);
                fetched = c + 1;
                return true;
            };
            // every thread: wait for chunk c's buffer; then its slot may be reused
            // (a copy whose wait gave up is drained below, before the buffers
            // are reused or the CTA exits)
            auto wait_full = [&](int c) {
                const uint32_t r = cnt + c;
                if (mbar_wait(&bar_full[r & 1], (r >> 1) & 1, &abort_flag)) {
                    waited = c + 1;
                } else {
                    record_timeout(p.status, &abort_flag, 691);
                }
                if (tid == 32 && !abort_flag) {
                    st_relaxed(p.cons_done + i, g0 + c + 1);
                }
            };

            if (nch > 0) {
                if (tid == 0) {
                    for (int c = 0; c < nch && c < kVRing; ++c) {
                        issue_v(c);
                    }
                }
                if (tid == 32) {
                    if (fetch(0, true) && nch > 1) {
                        fetch(1, false);
                    }
                }
                wait_full(0);
                tc_fence_after();
                if (tid == 0 && !abort_flag) {
                    if (wait_v(0)) {
                        tc_fence_after();
                        issue_u_prime_tc(x, tiles(cnt & 1, vcnt % kVRing));   // U'^T = V^T Tm^T
                    } else {
                        record_timeout(p.status, &abort_flag, 714);
                    }
                }
                // S^T -> bf16 operand (and chunk 0's record); S^T *= Gamma of chunk 0
                phase_state_to_tmem_decay(
                    x, reinterpret_cast<const float*>(sm + tiles(cnt & 1, 0).gam),
                    kRec && meta.rec ? chunk_record(meta, p, n, 0, h) + REC_S0 : nullptr);
                cta_sync_tc();
            }
            uint32_t ob[8];   // the last chunk's O^T as bf16 pairs, stored one chunk later
            // thread 32: flags read during the last chunk's products: of the next
            // chunk (pf1, when it was not copied yet) and of the one after (pf2)
            int32_t pf1 = 0, pf2 = 0;
            for (int c = 0; c < nch && !abort_flag; ++c) {
                const StateTiles st = tiles((cnt + c) & 1, (vcnt + c) % kVRing);
                // [O^T | U^T] += S^T [Q+^T | -W^T]  (U^T holds U', O^T zero)
                if (tid == 0) {
                    issue_ou_tc(x, st);
                    mma_commit(&bar_u);
                }
                // chunk c + 1 into the buffer chunk c - 1 left, if the flag read
                // during the last chunk's products showed it published (before
                // this thread's output stores below, which the copy's proxy
                // fence would otherwise wait for)
                if (tid == 32 && fetched == c + 1 && c + 1 < nch && pf2 >= g0 + c + 2) {
                    fetch(c + 1, false, true);
                }
                // the previous chunk's o while the tensor core works
                if (c > 0 && o_g) {
                    phase_ot_store(x, o_g, bos + (c - 1) * C, C, h, H, ob);
                }
                if (!mbar_wait(&bar_u, ph_u, &abort_flag)) {
                    record_timeout(p.status, &abort_flag, 745);
                }
                ph_u ^= 1;
                tc_fence_after();
                phase_u_to_tmem(x);
                cta_sync_tc();
                if (abort_flag) {
                    break;
                }
                // [S^T | O^T] += U^T [Kend ; Aqk]
                if (tid == 0) {
                    issue_so_tc(x, st);
                    mma_commit(&bar_os);
                }
                if (tid == 32) {
                    // the flag of the chunk after next, read while the tensor core
                    // works (the acquire load's latency overlaps the products); its
                    // copy is issued at the top of the next chunk
                    pf1 = pf2 = 0;
                    if (c + 1 < nch && fetched == c + 1) {
                        pf1 = ld_acquire(flag_of(c + 1));
                    }
                    if (c + 2 < nch && fetched <= c + 2) {
                        pf2 = ld_acquire(flag_of(c + 2));
                    }
                }
                if (!mbar_wait(&bar_os, ph_os, &abort_flag)) {
                    record_timeout(p.status, &abort_flag, 770);
                }
                ph_os ^= 1;
                tc_fence_after();
                // the next chunk's slot, if not copied yet (a chunk the producers
                // have not published yet is waited for)
                if (tid == 32 && !abort_flag) {
                    if (c + 1 < nch && fetched < c + 2) {
                        fetch(c + 1, pf1 < g0 + c + 2, pf1 >= g0 + c + 2);
                    }
                    // chunk c's buffer is free once its products are done: the chunk
                    // after next goes into it now if its flag showed it published
                    if (c + 2 < nch && fetched == c + 2 && pf2 >= g0 + c + 3) {
                        fetch(c + 2, false, true);
                    }
                }
                if (tid == 0 && !abort_flag) {
                    if (c + 1 < nch) {
                        // the next chunk's U' = V Tm^T, once its slot has landed
                        const uint32_t r = cnt + c + 1;
                        if (mbar_wait(&bar_full[r & 1], (r >> 1) & 1, &abort_flag) &&
                            wait_v(c + 1)) {
                            tc_fence_after();
                            issue_u_prime_tc(x, tiles(r & 1, (vcnt + c + 1) % kVRing));
                        } else {
                            record_timeout(p.status, &abort_flag, 785);
                        }
                    }
                    // U'(c) and the products of chunk c are done: its v slot takes
                    // chunk c + kVRing
                    if (c + kVRing < nch) {
                        issue_v(c + kVRing);
                    }
                }
                if (c + 1 < nch) {
                    wait_full(c + 1);
                }
                // state checkpoint after this chunk (S^T in TMEM is the state after it)
                if (p.ckpt_interval > 0) {
                    const int64_t done = (int64_t)(c + 1) * C;
                    const int64_t idx = ck_base + done / p.ckpt_interval - 1;
                    if (done % p.ckpt_interval == 0 && done <= len && idx < p.ckpt_count) {
                        const int64_t row = p.ckpt_slots ? (int64_t)p.ckpt_slots[idx] : idx;
                        if (row >= 0 && row < p.ckpt_pool_size) {
                            store_state(x, p.ckpt_pool + ((size_t)row * H + h) * D * D);
                        }
                    }
                }
                // O^T -> registers (stored during the next chunk's products); the
                // next chunk's S^T -> bf16 operand and S^T *= its Gamma
                phase_ot_take(x, ob);
                if (c + 1 < nch) {
                    phase_state_to_tmem_decay(
                        x, reinterpret_cast<const float*>(
                               sm + tiles((cnt + c + 1) & 1, 0).gam),
                        kRec && meta.rec ? chunk_record(meta, p, n, c + 1, h) + REC_S0
                                         : nullptr);
                }
                cta_sync_tc();
                if (c + 1 == nch && o_g) {   // the last chunk's o
                    phase_ot_store(x, o_g, bos + c * C, len - c * C, h, H, ob);
                }
            }
            // copies still in flight into this CTA's buffers (a loop left early)
            if (tid == 32) {
                s_issued = fetched;
            }
            if (tid == 0) {
                for (int c = v_waited; c < v_issued; ++c) {
                    const uint32_t r = vcnt + c;
                    mbar_wait(&bar_v[r % kVRing], (r / kVRing) & 1, nullptr);
                }
                s_vissued = v_issued;
            }
            __syncthreads();
            const int issued = s_issued;
            for (int c = waited; c < issued; ++c) {
                const uint32_t r = cnt + c;
                mbar_wait(&bar_full[r & 1], (r >> 1) & 1, nullptr);
            }
            cnt += issued;
            vcnt += s_vissued;
            if (!abort_flag && p.final_state) {
                store_state(x, p.final_state + state_off);
            }
            if (conv && p.conv_state_out) {
                conv_state_tail(p, n, h, meta.cu[n], meta.cu[n] + len);
            }
            cta_sync_tc();
            if (tid == 32 && !abort_flag) {  // skip the stream positions this unit leaves unused
                st_release(p.cons_done + i, meta.g0[bt + 1]);
            }
        }
    } else {
        // ------------------------------------------------------------ producer
        // Producer k takes tasks k, k + P, k + 2P, ... (P producers; tasks past
        // the end of their sequence are skipped), the j-th of them through two
        // warp groups (kda_split_phases.cuh): group A (warps 0-7) runs the
        // prologue of task j and issues its Gram products into TMEM buffer
        // j & 1 while group B (warps 8-15) finishes task j - 1 (Gram epilogue,
        // UT solve, W) out of the other buffer.  Hand-overs, all mbarriers with
        // one arrival: bar_gram[j & 1] (task j's Gram done: B reads it, A may
        // overwrite the operand tiles; one barrier per buffer, so that a waiter
        // never faces a phase two tasks ahead), bar_aw[j & 1] (A's writes of
        // task j into its slot done), bar_bdone[j & 1] (B finished task j: its
        // TMEM buffer, K+ and beta buffers are free).  Group B raises each
        // slot's flag (release) once it has finished the task: B waits on
        // nothing outside the CTA, so every flag is raised without depending on
        // a consumer, and the release's wait for the slot writes to drain falls
        // in B's idle time instead of holding up group A's barriers.
        using namespace split;
        const int total = meta.task0[p.n_batches];
        constexpr bool conv = kConv;
        constexpr uint32_t slot_bytes = conv ? HO_BYTES_CONV : HO_BYTES;
        ConvSrc cs;
        cs.w = p.conv_w;
        cs.q = static_cast<const __nv_bfloat16*>(p.q);
        cs.k = static_cast<const __nv_bfloat16*>(p.k);
        cs.v = static_cast<const __nv_bfloat16*>(p.v);
        cs.st = static_cast<const __nv_bfloat16*>(p.conv_state_in);
        cs.R = p.conv_W - 1;
        cs.silu = p.conv_silu != 0;
        cs.H = H;
        const int P = (int)gridDim.x - p.n_cons;
        const bool grpA = x.warp < 8;
        const int lt = grpA ? tid : tid - 256;   // thread within the group
        const int lw = lt >> 5;                  // warp within the group
        auto next_task = [&](int t, SplitTask& tk) -> int {
            while (t < total && !decode_task(meta, p, t, tk)) {
                t += P;
            }
            return t;
        };
        SplitTask cur;
        int t = next_task((int)blockIdx.x - p.n_cons, cur);
        if (grpA) {
            // ---------------------------------------------------- group A
            constexpr int kChecker = 32;     // lane 0 of warp 1: the slot checks
            auto issue_raw = [&](const SplitTask& tk) {
                mbar_arrive_expect_tx(&bar_raw, 3 * 16384);
                tma_load_3d(sm + P_RAWQ, &args.tm_q, 0, tk.h, tk.t0, &bar_raw);
                tma_load_3d(sm + P_RAWK, &args.tm_k, 0, tk.h, tk.t0, &bar_raw);
                tma_load_3d(sm + P_RAWZ, &args.tm_z, 0, tk.h, tk.t0, &bar_raw);
            };
            if (tid == 0 && t < total) {
                issue_raw(cur);
            }
            // beta of the current task, loaded one task ahead (threads < 64)
            float beta_r = 0.0f;
            if (t < total && lt < cur.L) {
                beta_r = __bfloat162float(beta_g[(size_t)(cur.t0 + lt) * H + cur.h]);
            }
            bool raw_pending = t < total;   // a raw load issued and not waited for
            uint32_t raw_par = 0;           // (and the parity it completes)
            // slot checker: consumer cons_i's counter, read earlier (it only grows)
            int32_t cons_seen = 0;
            int cons_i = -1;
            const int c = lt & (D - 1);
            // the thread's two 16-token blocks: {0, 3} or {1, 2}, so that both
            // halves of the group write the same number of key copies (block a
            // is in the copies a..3)
            const int hb = lt >> 7;
            const int blk0 = hb ? 1 : 0, blk1 = hb ? 2 : 3;
            int j = 0;
            while (t < total) {
                SplitTask nt;
                const int tn = next_task(t + P, nt);
                const bool has_next = tn < total;
                const int32_t slot = cur.i * p.ring + cur.g % p.ring;
                uint8_t* rec =
                    kRec && meta.rec ? chunk_record(meta, p, cur.unit / H, cur.c, cur.h)
                                     : nullptr;
                uint8_t* pub = rec ? rec : p.handoff + (size_t)slot * slot_bytes;
                float* s_beta = reinterpret_cast<float*>(sm + P_BETA) + (j & 1) * 64;
                uint8_t* kp = sm + P_KP + (j & 1) * 16384;
                // K+ and beta buffer j & 1 are free once B finished task j - 2
                bool ok = true;
                if (j >= 2) {
                    ok = mbar_wait(&bar_bdone[j & 1], ((j - 2) >> 1) & 1, &abort_flag);
                }
                if (ok && mbar_wait(&bar_raw, j & 1, &abort_flag)) {
                    raw_pending = false;
                } else {
                    record_timeout(p.status, &abort_flag, 932);
                }
                // beta, norms and gate of task j
                if (lt < C) {
                    s_beta[lt] = beta_r;
                    beta_r = (has_next && lt < nt.L)
                                 ? __bfloat162float(beta_g[(size_t)(nt.t0 + lt) * H + nt.h])
                                 : 0.0f;
                }
                if (conv) {   // the short convolutions of q and k, in place
                    float hq[3], hk[3];
                    a_conv_halo(sm, lt, cs, cur.t0, cur.c, cur.unit / H, cur.h, hq, hk);
                    group_sync(kBarA);
                    a_conv_apply(sm, lt, cs, cur.h, hq, hk);
                    group_sync(kBarA);
                }
                a_norms(sm, lw, x.lane, cur.L, p.scale, p.l2norm);
                float al0[16], al1[16];
                a_gate_block(sm, c, blk0, cur.L, meta.eA[cur.h], al0);
                a_gate_block(sm, c, blk1, cur.L, meta.eA[cur.h], al1);
                // is the slot free (its consumer has copied out the chunk that was in it)?
                if (lt == kChecker) {
                    if (cons_i != cur.i || cons_seen < cur.g - p.ring + 1) {
                        cons_seen = ld_acquire(p.cons_done + cur.i);
                        cons_i = cur.i;
                    }
                    s_slot_free = cons_seen >= cur.g - p.ring + 1;
                }
                if (group_sync_or(kBarA, abort_flag != 0)) {
                    break;
                }
                if (!s_slot_free) {
                    if (lt == kChecker &&
                        !wait_at_least(p.cons_done + cur.i, cur.g - p.ring + 1, &abort_flag,
                                       p.peer_wait_polls)) {
                        record_timeout(p.status, &abort_flag, 962);
                    }
                    group_sync(kBarA);
                }
                // X~, K~ are free once the previous task's Gram products are done
                if (j >= 1 &&
                    !mbar_wait(&bar_gram[(j - 1) & 1], ((j - 1) >> 1) & 1, &abort_flag)) {
                    record_timeout(p.status, &abort_flag, 969);
                }
                // the operand tiles
                a_operands_block(sm, c, blk0, al0, kp, pub, rec);
                a_operands_block(sm, c, blk1, al1, kp, pub, rec);
                fence_proxy_async();
                tc_fence_before();
                const bool stop = group_sync_or(kBarA, abort_flag != 0);
                tc_fence_after();
                if (stop) {
                    break;
                }
                if (tid == 0) {
                    // every thread of A has written its part of task j's slot
                    mbar_arrive(&bar_aw[j & 1]);
                    if (has_next) {   // the raw tiles are consumed: fetch the next task's
                        issue_raw(nt);
                    }
                    // task j's Gram products into TMEM buffer j & 1 (free: B
                    // finished task j - 2, waited for at the top of this task)
                    a_issue_gram(x.smem_base, x.tbase + (j & 1) * kGramBufCols);
                    mma_commit(&bar_gram[j & 1]);
                }
                raw_pending = has_next;
                raw_par = (j + 1) & 1;
                // the next slot's consumer counter, read ahead of its use
                if (lt == kChecker && has_next) {
                    cons_seen = ld_acquire(p.cons_done + nt.i);
                    cons_i = nt.i;
                }
                cur = nt;
                t = tn;
                ++j;
            }
            // a loop left early may still have a raw load in flight into this CTA's smem
            if (raw_pending) {
                mbar_wait(&bar_raw, raw_par, nullptr);
            }
        } else {
            // ---------------------------------------------------- group B
            int j = 0;
            while (t < total) {
                SplitTask nt;
                const int tn = next_task(t + P, nt);
                const int32_t slot = cur.i * p.ring + cur.g % p.ring;
                uint8_t* rec =
                    kRec && meta.rec ? chunk_record(meta, p, cur.unit / H, cur.c, cur.h)
                                     : nullptr;
                uint8_t* pub = rec ? rec : p.handoff + (size_t)slot * slot_bytes;
                const float* s_beta = reinterpret_cast<const float*>(sm + P_BETA) + (j & 1) * 64;
                // task j's Gram products, issued by group A once it has written
                // their operands (the slot is then free: A checked it first)
                const uint32_t tg = x.tbase + (j & 1) * kGramBufCols;
                if (!mbar_wait(&bar_gram[j & 1], (j >> 1) & 1, &abort_flag)) {
                    record_timeout(p.status, &abort_flag, 1033);
                }
                if (conv) {   // the convolved v into the slot
                    b_conv_v(pub + HO_V, lt, cs, cur.t0, cur.L, cur.c, cur.unit / H, cur.h);
                }
                tc_fence_after();
                b_gram_epilogue(sm, tg, x.warp, x.lane, lw >> 2, s_beta, pub, rec);
                tc_fence_before();
                const bool stop = group_sync_or(kBarB, abort_flag != 0);
                if (stop) {
                    break;
                }
                b_solve(sm, lt, lw, x.lane, s_beta, pub, rec);
                fence_proxy_async();
                tc_fence_before();
                group_sync(kBarB);
                tc_fence_after();
                if (lt == 0) {
                    b_issue_w(x.smem_base, tg, P_KP + (j & 1) * 16384);
                    mma_commit(&bar_w);
                }
                if (!mbar_wait(&bar_w, j & 1, &abort_flag)) {
                    record_timeout(p.status, &abort_flag, 1052);
                }
                tc_fence_after();
                b_neg_w(tg, x.warp, lw, x.lane, pub + HO_WT);
                tc_fence_before();
                group_sync(kBarB);
                if (lt == 0) {
                    // A's writes of task j (ordered before its arrival, which came
                    // before the Gram products B waited for) and B's (ordered by
                    // the group barrier) are all done: raise the slot's flag.
                    // bar_aw[j & 1] cannot complete again before this wait: A
                    // arrives for task j + 2 only after B finished task j.
                    const bool aw = mbar_wait(&bar_aw[j & 1], (j >> 1) & 1, &abort_flag);
                    mbar_arrive(&bar_bdone[j & 1]);
                    if (aw) {
                        st_release(p.flags + slot, cur.g + 1);
                    } else {
                        record_timeout(p.status, &abort_flag, 1064);
                    }
                }

                cur = nt;
                t = tn;
                ++j;
            }
            // no W^T product of this group may still be running when the TMEM
            // is freed (a wait above may have given up)
            if (lt == 0) {
                mma_commit(&bar_finb);
                mbar_wait(&bar_finb, 0, nullptr);
            }
        }
    }
    // no MMA of this CTA may still be running when its TMEM is freed
    cta_sync_tc();
    if (tid == 0) {
        mma_commit(&bar_fin);
        mbar_wait(&bar_fin, 0, nullptr);
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

bool make_map_impl(CUtensorMap* map, const void* base, int total_T, int H, int box_c,
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

}  // namespace

bool make_token_map(CUtensorMap* map, const void* base, int total_T, int H, bool swizzled) {
    return make_map_impl(map, base, total_T, H, swizzled ? 64 : 128,
                         swizzled ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE);
}

namespace {

bool make_args(ChunkedArgs* args, const ChunkedParams& p) {
    memset(args, 0, sizeof(*args));
    args->p = p;
    return make_token_map(&args->tm_q, p.q, p.total_T, p.H, false) &&
           make_token_map(&args->tm_k, p.k, p.total_T, p.H, false) &&
           make_token_map(&args->tm_z, p.z, p.total_T, p.H, false) &&
           make_token_map(&args->tm_v, p.v, p.total_T, p.H, true);
}

}  // namespace

size_t chunked_workspace_bytes(int32_t N, int32_t H) {
    return 256 + (size_t)N * H * sizeof(int32_t);
}

namespace {
constexpr int32_t kSplitRing = 16;      // slots per consumer
constexpr int32_t kSplitRingWide = 24;  // with a third of the SMs as consumers
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
size_t split_flags_offset() { return 256; }
size_t split_done_offset(const SplitPlan& plan) {
    return split_flags_offset() + round256((size_t)plan.consumers * plan.ring * sizeof(int32_t));
}
}  // namespace

bool split_plan(int32_t N, int32_t H, int num_sms, SplitPlan* plan) {
    if (num_sms < 8 || N < 1 || H < 1 || N > kSplitMaxSeqs || H > kSplitMaxHeads) {
        return false;
    }
    // Producers need most of the GPU: at most a quarter of the SMs are
    // consumers -- or a third where that cuts the units into at most two
    // batches instead of three or more (96 heads: two batches of 48 instead
    // of three of 32), with a deeper ring so that the fewer producers can run
    // further ahead.  (Measured on a GB300: 7.27 -> 6.82 ms for 96 heads x
    // 65,536 tokens; for many batches, as with 1,024 units, a third of the
    // SMs as consumers was slower, 9.7 -> 11.9 ms.)
    const int64_t U = (int64_t)N * H;
    int64_t max_cons = num_sms / 4;
    int32_t ring = kSplitRing;
    const int64_t wide = num_sms / 3;
    if ((U + max_cons - 1) / max_cons > 2 && (U + wide - 1) / wide <= 2) {
        max_cons = wide;
        ring = kSplitRingWide;
    }
    int64_t batches = (U + max_cons - 1) / max_cons;
    if (batches > kSplitMaxBatches) {
        return false;
    }
    const int64_t cons = (U + batches - 1) / batches;  // even batches
    batches = (U + cons - 1) / cons;                    // none left empty
    plan->consumers = (int32_t)cons;
    plan->batches = (int32_t)batches;
    plan->ring = ring;
    return true;
}

size_t split_zeroed_bytes(const SplitPlan& plan) {
    return split_done_offset(plan) + round256((size_t)plan.consumers * sizeof(int32_t));
}

size_t split_workspace_bytes(const SplitPlan& plan, bool conv) {
    return split_zeroed_bytes(plan) +
           (size_t)plan.consumers * plan.ring * (conv ? HO_BYTES_CONV : HO_BYTES);
}

void split_bind(const SplitPlan& plan, void* workspace, ChunkedParams* p) {
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p->flags = reinterpret_cast<int32_t*>(ws + split_flags_offset());
    p->cons_done = reinterpret_cast<int32_t*>(ws + split_done_offset(plan));
    p->handoff = ws + split_zeroed_bytes(plan);
    p->n_cons = plan.consumers;
    p->n_batches = plan.batches;
    p->ring = plan.ring;
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

namespace {
template <int kMode>
cudaError_t launch_split_mode(ChunkedArgs& args, int num_sms, cudaStream_t stream) {
    cudaError_t err = cudaFuncSetAttribute(kda_split_kernel<kMode>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kSplitSmemBytes);
    if (err != cudaSuccess) {
        return err;
    }
    // The CTAs wait on one another (ring flags, consumer counters), so every
    // one of them must be resident at once: a cooperative launch guarantees
    // that, or fails (cudaErrorCooperativeLaunchTooLarge) without running
    // anything when the grid cannot be co-resident -- the caller then runs the
    // single-pass kernel instead.  The ring flags and consumer counters were
    // zeroed by the caller on this stream.
    void* kargs[] = {&args};
    err = cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(&kda_split_kernel<kMode>),
                                      dim3((unsigned)num_sms), dim3(kThreads), kargs,
                                      kSplitSmemBytes, stream);
    if (err != cudaSuccess) {
        cudaGetLastError();  // clear the launch error; it is returned instead
    }
    return err;
}
}  // namespace

cudaError_t launch_split_prefill(const ChunkedParams& p, int num_sms, cudaStream_t stream) {
    ChunkedArgs args;
    if (!make_args(&args, p)) {
        return cudaErrorInvalidValue;
    }
    if (p.records) {
        return launch_split_mode<kSplitRecords>(args, num_sms, stream);
    }
    if (p.conv_w) {
        return launch_split_mode<kSplitConv>(args, num_sms, stream);
    }
    return launch_split_mode<kSplitPlain>(args, num_sms, stream);
}

}  // namespace kda
