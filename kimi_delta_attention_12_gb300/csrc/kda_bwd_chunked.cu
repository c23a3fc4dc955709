// kda_bwd_chunked.cu -- chunked training backward of KDA on tcgen05 tensor
// cores (sm_103a): the gradients of the chunked prefill of "Kimi K3 Open
// Weights: What Is Actually New In Its 2.8 Trillion Parameter Architecture",
// section 1, with respect to q, k, v, z, beta, A and the initial state.
//
// The forward of one 64-token chunk (start state S0; the algebra of
// kda_chunk_phases.cuh, Minv = (I + Akk)^-1, Akk = Diag(beta) Gkk):
//   X = V - K+ S0,  U = Minv Diag(beta) X,
//   O = Q+ S0 + Aqk U,  S_L = Diag(Gamma) S0 + Kend^T U.
// Its adjoint, given dO and dS_L = dL/dS_L:
//   dU = Aqk^T dO + Kend dS_L,  dY = Minv^T dU,  dV = dX = Diag(beta) dY,
//   dS0 = Diag(Gamma) dS_L + Q+^T dO - W^T dU      (W = Minv Diag(beta) K+),
//   dQ+ = dO S0^T,  dK+ = -dX S0^T,  dKend = U dS_L^T,
//   dAqk = dO U^T (i <= r),  dAkk = -dY U^T (i < r),  dGkk = Diag(beta) dAkk,
//   dbeta_r = sum_v dY X + sum_i dAkk Gkk,
// then the decay chains of Q+ = q e^gamma, K+ = k e^gamma, Kend = k
// e^(gamma_L - gamma), Aqk and Gkk (whose entries carry e^(gamma_r -
// gamma_i)) into q_hat, k_hat and gamma, dg = the reverse cumulative sum of
// dgamma over the chunk (plus dgamma_L, from Gamma and Kend), and per token
// the gate and normalisation derivatives.
//
// Two kernels run after the split prefill has kept every chunk's operand
// tiles in a chunk record and the state at every chunk start:
//   kda_bwd_chain_kernel: one CTA per (sequence, head) walks the chunks last
//     to first with dS^T (fp32) in TMEM; per chunk two tensor-core rounds,
//     dU^T = dO^T Aqk + dS^T Kend with dS^T += dO^T Q+, then dS^T += dU^T
//     (-W^T), and the dS_L of every chunk is stored (bf16) for the assembly;
//   kda_bwd_assemble_kernel: one CTA per (chunk, head), all at once: the
//     products above on the tensor core with the value dimension (or the key
//     channel) as M = 128, the decay chains on the CUDA cores in fp32 with
//     one reference point per 16-token block (the bounded gate keeps every
//     factor inside fp32), and every per-token gradient.
// dL/dA is then the sum of the per-token shares (kda_backward.cu).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_chunk_phases.cuh"
#include "kda_chunked.h"
#include "kda_seqlens.cuh"
#include "sm103_ptx.cuh"

namespace kda {
namespace {

using namespace sm103;
using namespace chunk;

struct BwdArgs {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_z;
    CUtensorMap tm_v;
    CUtensorMap tm_do;
    BwdChunkedParams p;
};

__device__ __forceinline__ uint8_t* bw_align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) &
                                      ~static_cast<uintptr_t>(1023));
}

__device__ __forceinline__ Ctx bw_ctx(uint8_t* sm, uint32_t tbase) {
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

// CTA barrier (ordering tcgen05 operations around it) that also tells every
// thread whether any thread passed true: a loop left on it is left by all.
__device__ __forceinline__ bool cta_sync_tc_or(bool pred) {
    tc_fence_before();
    const bool r = __syncthreads_or(pred) != 0;
    tc_fence_after();
    return r;
}

// Sum over the sequences m < n of f(m); every thread of the CTA calls it.
template <typename F>
__device__ __forceinline__ int64_t seq_prefix(int n, F f, int* s_acc) {
    if (threadIdx.x == 0) {
        *s_acc = 0;
    }
    __syncthreads();
    int part = 0;
    for (int m = threadIdx.x; m < n; m += blockDim.x) {
        part += f(m);
    }
    if (part) {
        atomicAdd(s_acc, part);
    }
    __syncthreads();
    const int64_t r = *s_acc;
    __syncthreads();
    return r;
}

__device__ __forceinline__ float bf16_at(const uint8_t* p) {
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(p));
}

// ====================================================================== chain
// Shared memory: two record buffers (the published part of a chunk record,
// HO_BYTES) and a ring of dO tiles, both prefetched ahead of use.
constexpr uint32_t CH_BUF = 66560;
constexpr uint32_t CH_DO = 2 * CH_BUF;
constexpr int kDoRing = 4;
constexpr uint32_t kChainSmem = CH_DO + kDoRing * 16384 + 1024;

// (one thread) dU^T = dO^T Aqk + dS_L^T Kend into TC_U, and dS^T += dO^T Q+
// (dS^T already scaled by Gamma).  rec: the record buffer; dob: the dO tile
// (two v-halves [64 r][64 v]).
__device__ __forceinline__ void chain_issue_du(const Ctx& x, uint32_t rec, uint32_t dob) {
    const uint32_t id_a = idesc_bf16(128, 64, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = smem_desc(x.smem_base + dob + kk * 2048, 8192, 1024);
        const uint64_t b = smem_desc(x.smem_base + rec + HO_AQK + kk * 2048, 8192, 1024);
        mma_bf16(x.tbase + TC_U, a, b, id_a, kk > 0);
    }
    const uint32_t id_k = idesc_bf16(128, 64, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t b = smem_desc(x.smem_base + rec + HO_KE + kk * 2048, 8192, 1024);
        mma_bf16_ta(x.tbase + TC_U, x.tbase + TC_SB + kk * 8, b, id_k, 1);
    }
    const uint32_t id_q = idesc_bf16(128, 128, 1, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t a = smem_desc(x.smem_base + dob + kk * 2048, 8192, 1024);
        const uint64_t b = smem_desc(x.smem_base + rec + HO_QP + kk * 32, 16, 1024);
        mma_bf16(x.tbase + TC_S, a, b, id_q, 1);
    }
}

// (one thread) dS^T += dU^T (-W^T).
__device__ __forceinline__ void chain_issue_ds(const Ctx& x, uint32_t rec) {
    const uint32_t id = idesc_bf16(128, 128, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t b = smem_desc(x.smem_base + rec + HO_WT + kk * 32, 16, 1024);
        mma_bf16_ta(x.tbase + TC_S, x.tbase + TC_UB + kk * 8, b, id, 1);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
kda_bwd_chain_kernel(const __grid_constant__ BwdArgs args) {
    const BwdChunkedParams& p = args.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = bw_align1024(smem_raw);
    __shared__ uint64_t bar_full[2];       // a record buffer landed
    __shared__ uint64_t bar_do[kDoRing];   // a dO tile landed
    __shared__ uint64_t bar_u;             // dU^T and the dO^T Q+ part done
    __shared__ uint64_t bar_s;             // the dU^T (-W^T) part done
    __shared__ uint64_t bar_fin;           // every MMA of this CTA done
    __shared__ uint32_t tmem_base_s;
    __shared__ int s_acc;
    __shared__ int s_fetched;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x;
    const int unit = blockIdx.x;
    const int n = unit / p.H;
    const int h = unit - n * p.H;
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar_full[0], 1);
        mbar_init(&bar_full[1], 1);
        for (int j = 0; j < kDoRing; ++j) {
            mbar_init(&bar_do[j], 1);
        }
        mbar_init(&bar_u, 1);
        mbar_init(&bar_s, 1);
        mbar_init(&bar_fin, 1);
        fence_mbar_init();
        prefetch_tmap(&args.tm_do);
    }
    if ((tid >> 5) == 0) {
        tmem_alloc(&tmem_base_s, TMEM_COLS);
        tmem_relinquish();
    }
    int64_t bos, eos;
    clamped_seq(p.cu_seqlens, n, p.N, p.total_T, bos, eos);
    const int nch = (int)((eos - bos + C - 1) / C);
    auto len_of = [&](int m) { return (int)clamped_len(p.cu_seqlens, m, p.N, p.total_T); };
    // first chunk of this sequence among all chunks
    const int64_t ch_base = seq_prefix(n, [&](int m) { return (len_of(m) + C - 1) / C; }, &s_acc);
    if (h == 0) {
        for (int c = tid; c < nch; c += kThreads) {
            const int64_t g = ch_base + c;
            if (g < p.max_chunks) {
                reinterpret_cast<int4*>(p.chunk_map)[g] = make_int4(n, c, 0, 0);
            }
        }
    }
    cta_sync_tc();
    const Ctx x = bw_ctx(sm, tmem_base_s);
    const size_t state_off = (size_t)unit * D * D;
    load_state(x, p.dS_final ? p.dS_final + state_off : nullptr);
    cta_sync_tc();

    // step s works on chunk nch - 1 - s; its record goes through buffer s & 1
    // and its dO tile through ring slot s % kDoRing
    int fetched = 0, do_issued = 0, do_waited = 0;   // thread 0
    auto usable = [&](int s) { return ch_base + (nch - 1 - s) < p.max_chunks; };
    auto fetch = [&](int s) {
        const uint32_t b = s & 1;
        const uint8_t* rec =
            p.records + ((size_t)(ch_base + nch - 1 - s) * p.H + h) * REC_BYTES;
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar_full[b], HO_BYTES);
        bulk_load(sm + b * CH_BUF, rec, HO_BYTES, &bar_full[b]);
        fetched = s + 1;
    };
    auto issue_do = [&](int s) {
        const int t0 = (int)(bos + (int64_t)(nch - 1 - s) * C);
        const uint32_t r = s % kDoRing;
        uint8_t* d = sm + CH_DO + r * 16384;
        mbar_arrive_expect_tx(&bar_do[r], 16384);
        tma_load_3d(d, &args.tm_do, 0, h, t0, &bar_do[r]);
        tma_load_3d(d + 8192, &args.tm_do, 64, h, t0, &bar_do[r]);
        do_issued = s + 1;
    };
    const int steps = (nch > 0 && usable(0)) ? nch : 0;
    if (tid == 0) {
        for (int s = 0; s < steps && s < kDoRing; ++s) {
            issue_do(s);
        }
        for (int s = 0; s < steps && s < 2; ++s) {
            fetch(s);
        }
    }
    uint32_t ph_u = 0, ph_s = 0;
    int waited = 0;
    for (int s = 0; s < steps; ++s) {
        const int c = nch - 1 - s;
        const uint32_t b = s & 1;
        if (mbar_wait(&bar_full[b], (s >> 1) & 1, &abort_flag)) {
            waited = s + 1;
        } else {
            record_timeout(p.status, &abort_flag, 190);
        }
        if (!abort_flag) {
            uint8_t* dst = p.dsl + ((size_t)(ch_base + c) * p.H + h) * kBwdDslBytes;
            // dS_L -> bf16 operand and the chunk's dS_L tile; dS *= Gamma
            phase_state_to_tmem_decay(
                x, reinterpret_cast<const float*>(sm + b * CH_BUF + HO_GAM), dst);
        }
        if (cta_sync_tc_or(abort_flag != 0)) {
            break;
        }
        if (tid == 0) {
            if (mbar_wait(&bar_do[s % kDoRing], (s / kDoRing) & 1, &abort_flag)) {
                do_waited = s + 1;
                tc_fence_after();
                chain_issue_du(x, b * CH_BUF, CH_DO + (s % kDoRing) * 16384);
                mma_commit(&bar_u);
            } else {
                record_timeout(p.status, &abort_flag, 209);
            }
        }
        if (!mbar_wait(&bar_u, ph_u, &abort_flag)) {
            record_timeout(p.status, &abort_flag, 214);
        }
        ph_u ^= 1;
        tc_fence_after();
        phase_u_to_tmem(x);   // dU^T -> bf16 at TC_UB
        if (cta_sync_tc_or(abort_flag != 0)) {
            break;
        }
        if (tid == 0) {
            chain_issue_ds(x, b * CH_BUF);
            mma_commit(&bar_s);
        }
        if (!mbar_wait(&bar_s, ph_s, &abort_flag)) {
            record_timeout(p.status, &abort_flag, 226);
        }
        ph_s ^= 1;
        tc_fence_after();
        // the buffers of this step are free again
        if (tid == 0 && !abort_flag) {
            if (s + 2 < steps && usable(s + 2)) {
                fetch(s + 2);
            }
            if (s + kDoRing < steps) {
                issue_do(s + kDoRing);
            }
        }
        if (s + 1 < steps && !usable(s + 1)) {
            break;   // (only a chunk count above the bound gets here)
        }
    }
    // copies still in flight into this CTA's buffers (a loop left early)
    if (tid == 0) {
        s_fetched = fetched;
        for (int s = do_waited; s < do_issued; ++s) {
            mbar_wait(&bar_do[s % kDoRing], (s / kDoRing) & 1, nullptr);
        }
    }
    __syncthreads();
    for (int s = waited; s < s_fetched; ++s) {
        mbar_wait(&bar_full[s & 1], (s >> 1) & 1, nullptr);
    }
    if (!abort_flag) {
        store_state(x, p.dS0 + state_off);
    }
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

// =================================================================== assembly
// Shared memory (byte offsets from a 1024-aligned base).  Operand tiles:
constexpr uint32_t AS_DO = 0;          // per v-half (+16384 h): dO [64 r][64 v], then -dY [64 i][64 v]
constexpr uint32_t AS_S0 = 32768;      // S0 bf16, per v-half [128 c][64 v] (from the record)
constexpr uint32_t AS_DSL = 65536;     // dS_L bf16, the same layout
constexpr uint32_t AS_V = 98304;       // V, 2 v-halves [64 r][64 v]
constexpr uint32_t AS_KP = 114688;     // K+ [128 c][64 r]; later U^T [128 v][64 r]
constexpr uint32_t AS_KE = 131072;     // Kend [128 c][64 r]; later -dX^T [128 v][64 i]
constexpr uint32_t AS_AQK = 147456;    // Aqk [64 r][64 i]
constexpr uint32_t AS_MINV = 155648;   // (I + Akk)^-1 [64 r][64 i]
constexpr uint32_t AS_G = 163840;      // Gkk [64 r][64 i]
constexpr uint32_t AS_RAWQ = 172032;   // raw q [64 t][128 c] bf16, row-major
constexpr uint32_t AS_RAWK = 188416;   // raw k
// small arrays
constexpr uint32_t AS_GAM = 204800;    // Gamma = e^{gamma_L}, fp32 [128]
constexpr uint32_t AS_BETA = 205312;   // beta fp32 [64] (0 past the chunk's end)
constexpr uint32_t AS_INVQ = 205568;   // scale / |q_t| (0 past the end)
constexpr uint32_t AS_INVK = 205824;   // 1 / |k_t| (0 past the end)
constexpr uint32_t AS_RQ = 206080;     // 1 / |q_t|
constexpr uint32_t AS_DB1 = 206336;    // [4][64]: sum_v dY X over each lane quadrant
constexpr uint32_t AS_DB2 = 207360;    // [4][64]: sum_i dAkk Gkk over each column quarter
constexpr uint32_t AS_TOT = 208384;    // [4][128]: block totals of g (log2 units)
constexpr uint32_t AS_DGT = 210432;    // [4][128]: block sums of dgamma
constexpr uint32_t AS_DGL = 212480;    // [4][128]: partial sums of sum_v dS_L S0
constexpr uint32_t AS_DKE = 214528;    // [4][128]: partial sums of sum_t dKend Kend
constexpr uint32_t AS_RHO = 216576;    // [4][128]: gamma at each block's middle token (log2)
constexpr uint32_t AS_END = 218624;
constexpr uint32_t kAsmSmem = AS_END + 1024;
// the z tile [64 t][128 c] bf16, over V (dead after the X epilogue)
constexpr uint32_t AS_Z = AS_V;
// the decay chains, over the operand tiles (dead after the last products)
constexpr int kDP = 68;                // row pitch (floats) of the dA arrays
constexpr uint32_t AS_DAQ = 0;         // dAqk fp32 [64 r][kDP]
constexpr uint32_t AS_DGG = 17408;     // dGkk fp32 [64 r][kDP]
constexpr uint32_t AS_DAQT = 34816;    // dAqk^T [64 i][kDP]
constexpr uint32_t AS_DGGT = 52224;    // dGkk^T [64 i][kDP]
constexpr uint32_t AS_WROW = 69632;    // kh_t e^{rho_b - gamma_t}   fp32 [64 t][128 c] (b: t's block)
constexpr uint32_t AS_WCK = 102400;    // kh_t e^{gamma_t - rho_b}
constexpr uint32_t AS_WCQ = 135168;    // qh_t e^{gamma_t - rho_b}
// the four sums of the decay chains, over the decay-chain arrays once they
// are read: RowQ, RowK, ColK, ColQ fp32 [64 t][128 c] each; dq_hat and dk_hat
// then overwrite RowQ and RowK, dx * x (the terms of a token's share of
// dL/dA) ColK
constexpr uint32_t AS_OUT = 0;
constexpr uint32_t AS_DQH = AS_OUT;
constexpr uint32_t AS_DKH = AS_OUT + 32768;
constexpr uint32_t AS_DXX = AS_OUT + 65536;
static_assert(AS_WCQ + 32768 <= AS_RAWQ, "decay-chain arrays overlap the raw tiles");

// TMEM columns (fp32 accumulators, M = 128 lanes)
constexpr uint32_t TX = 0;       // X^T    [v][r]   (lane v)
constexpr uint32_t TU = 64;      // U^T    [v][r]
constexpr uint32_t TDU = 128;    // dU^T   [v][r]
constexpr uint32_t TDY = 192;    // dY^T   [v][i]
constexpr uint32_t TDQ = 256;    // dQ+^T  [c][r]   (lane c)
constexpr uint32_t TDK = 320;    // dK+^T  [c][i]
constexpr uint32_t TDKE = 384;   // dKend^T [c][r]
constexpr uint32_t TDA = 448;    // [dAqk ; dAkk] [r][i] (lanes 0-63, 64-127)
constexpr uint32_t TXB = 384;    // (beta X)^T bf16 A operand (32 columns; before TDKE is written)
constexpr uint32_t TDUB = 448;   // dU^T bf16 A operand (32 columns; before TDA is written)
// after the last products (lane c, column 16 b + j for token 16 b + j)
constexpr uint32_t TG2 = 0;      // gamma (log2 units)
constexpr uint32_t TXZ = 448;    // x = e^A z

// Sum over the 32 lanes of 16 values per lane: lane l returns the sum of
// entry l % 16 (a transposing butterfly, 16 shuffles).
__device__ __forceinline__ float warp_sum16(float (&v)[16], int lane) {
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const bool up = lane & 8;
        const float send = up ? v[k] : v[k + 8];
        const float keep = up ? v[k + 8] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const bool up = lane & 4;
        const float send = up ? v[k] : v[k + 4];
        const float keep = up ? v[k + 4] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        const bool up = lane & 2;
        const float send = up ? v[k] : v[k + 2];
        const float keep = up ? v[k + 2] : v[k];
        v[k] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
    }
    {
        const bool up = lane & 1;
        const float send = up ? v[0] : v[1];
        const float keep = up ? v[1] : v[0];
        v[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
    }
    return v[0] + __shfl_xor_sync(0xffffffffu, v[0], 16);
}

// (one thread) the first round, from the loaded tiles:
//   X^T  (TX)  = S0^T K+^T           (V^T subtracted in the epilogue)
//   dU^T (TDU) = dO^T Aqk + dS_L^T Kend
//   dQ+^T (TDQ) = S0 dO^T
__device__ __forceinline__ void asm_issue_round1(const Ctx& x) {
    const uint32_t sb = x.smem_base;
    const uint32_t id_mm = idesc_bf16(128, 64, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        mma_bf16(x.tbase + TX, smem_desc(sb + AS_S0 + kk * 2048, 16384, 1024),
                 smem_desc(sb + AS_KP + kk * 2048, 8192, 1024), id_mm, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        mma_bf16(x.tbase + TDU, smem_desc(sb + AS_DO + kk * 2048, 16384, 1024),
                 smem_desc(sb + AS_AQK + kk * 2048, 8192, 1024), id_mm, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        mma_bf16(x.tbase + TDU, smem_desc(sb + AS_DSL + kk * 2048, 16384, 1024),
                 smem_desc(sb + AS_KE + kk * 2048, 8192, 1024), id_mm, 1);
    }
    const uint32_t id_kk = idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        mma_bf16(x.tbase + TDQ, smem_desc(sb + AS_S0 + off, 16, 1024),
                 smem_desc(sb + AS_DO + off, 16, 1024), id_kk, kk > 0);
    }
}

// (one thread) the second round: U^T (TU) = (beta X)^T Minv^T, dY^T (TDY) = dU^T Minv.
__device__ __forceinline__ void asm_issue_round2(const Ctx& x) {
    const uint32_t sb = x.smem_base;
    const uint32_t id_u = idesc_bf16(128, 64, 0, 0);
    const uint32_t id_y = idesc_bf16(128, 64, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        mma_bf16_ta(x.tbase + TU, x.tbase + TXB + kk * 8,
                    smem_desc(sb + AS_MINV + kk * 32, 16, 1024), id_u, kk > 0);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        mma_bf16_ta(x.tbase + TDY, x.tbase + TDUB + kk * 8,
                    smem_desc(sb + AS_MINV + kk * 2048, 8192, 1024), id_y, kk > 0);
    }
}

// (one thread) the third round:
//   dK+^T (TDK) = S0 (-dX)^T,  dKend^T (TDKE) = dS_L U^T,
//   [dAqk ; dAkk] (TDA) = [dO ; -dY] U^T
__device__ __forceinline__ void asm_issue_round3(const Ctx& x) {
    const uint32_t sb = x.smem_base;
    const uint32_t id = idesc_bf16(128, 64, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
        const uint64_t bdx = smem_desc(sb + AS_KE + kk * 2048, 8192, 1024);
        const uint64_t bu = smem_desc(sb + AS_KP + kk * 2048, 8192, 1024);
        mma_bf16(x.tbase + TDK, smem_desc(sb + AS_S0 + off, 16, 1024), bdx, id, kk > 0);
        mma_bf16(x.tbase + TDKE, smem_desc(sb + AS_DSL + off, 16, 1024), bu, id, kk > 0);
        mma_bf16(x.tbase + TDA, smem_desc(sb + AS_DO + off, 16, 1024), bu, id, kk > 0);
    }
}

__global__ void __launch_bounds__(kThreads, 1)
kda_bwd_assemble_kernel(const __grid_constant__ BwdArgs args) {
    const BwdChunkedParams& p = args.p;
    const int H = p.H;
    const int gid = blockIdx.x / H;
    const int h = blockIdx.x - gid * H;
    const int4 cm = reinterpret_cast<const int4*>(p.chunk_map)[gid];
    if (cm.x < 0 || cm.x >= p.N) {
        return;   // past the last chunk
    }
    const int n = cm.x, c = cm.y;
    int64_t bos, eos;
    clamped_seq(p.cu_seqlens, n, p.N, p.total_T, bos, eos);
    const int64_t t0 = bos + (int64_t)c * C;
    const int L = (int)min((int64_t)C, eos - t0);
    if (L <= 0) {
        return;
    }
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = bw_align1024(smem_raw);
    __shared__ uint64_t bar_ld, bar_z, bar_m1, bar_m2, bar_m3, bar_fin;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat16* beta_g = static_cast<const __nv_bfloat16*>(p.beta);

    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar_ld, 1);
        mbar_init(&bar_z, 1);
        mbar_init(&bar_m1, 1);
        mbar_init(&bar_m2, 1);
        mbar_init(&bar_m3, 1);
        mbar_init(&bar_fin, 1);
        fence_mbar_init();
        const uint8_t* rec = p.records + ((size_t)gid * H + h) * REC_BYTES;
        const uint8_t* dsl = p.dsl + ((size_t)gid * H + h) * kBwdDslBytes;
        mbar_arrive_expect_tx(&bar_ld, 188928);
        bulk_load(sm + AS_S0, rec + REC_S0, 32768, &bar_ld);
        bulk_load(sm + AS_KP, rec + REC_KP, 16384, &bar_ld);
        bulk_load(sm + AS_KE, rec + HO_KE, 16384, &bar_ld);
        bulk_load(sm + AS_AQK, rec + HO_AQK, 8192, &bar_ld);
        bulk_load(sm + AS_MINV, rec + REC_MINV, 8192, &bar_ld);
        bulk_load(sm + AS_G, rec + REC_G, 8192, &bar_ld);
        bulk_load(sm + AS_GAM, rec + HO_GAM, 512, &bar_ld);
        bulk_load(sm + AS_DSL, dsl, 32768, &bar_ld);
        const int tt = (int)t0;
        tma_load_3d(sm + AS_DO, &args.tm_do, 0, h, tt, &bar_ld);
        tma_load_3d(sm + AS_DO + 16384, &args.tm_do, 64, h, tt, &bar_ld);
        tma_load_3d(sm + AS_V, &args.tm_v, 0, h, tt, &bar_ld);
        tma_load_3d(sm + AS_V + 8192, &args.tm_v, 64, h, tt, &bar_ld);
        tma_load_3d(sm + AS_RAWQ, &args.tm_q, 0, h, tt, &bar_ld);
        tma_load_3d(sm + AS_RAWK, &args.tm_k, 0, h, tt, &bar_ld);
    }
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, TMEM_COLS);
        tmem_relinquish();
    }
    if (tid < C) {
        reinterpret_cast<float*>(sm + AS_BETA)[tid] =
            tid < L ? __bfloat162float(beta_g[(size_t)(t0 + tid) * H + h]) : 0.0f;
    }
    fence_proxy_async();
    cta_sync_tc();
    const Ctx x = bw_ctx(sm, tmem_base_s);
    // the work; returns early (every thread alike) once a wait gave up
    [&]() {
    if (!mbar_wait(&bar_ld, 0, &abort_flag)) {
        record_timeout(p.status, &abort_flag, 520);
    }
    if (tid == 0 && !abort_flag) {
        tc_fence_after();
        asm_issue_round1(x);
        mma_commit(&bar_m1);
    }
    // per-token norms while the tensor core works (4 tokens per warp)
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
        const int t = 4 * warp + tt;
        const uint2 qv = *reinterpret_cast<const uint2*>(sm + AS_RAWQ + t * 256 + lane * 8);
        const uint2 kv = *reinterpret_cast<const uint2*>(sm + AS_RAWK + t * 256 + lane * 8);
        float sq = bf16lo(qv.x) * bf16lo(qv.x) + bf16hi(qv.x) * bf16hi(qv.x) +
                   bf16lo(qv.y) * bf16lo(qv.y) + bf16hi(qv.y) * bf16hi(qv.y);
        float sk = bf16lo(kv.x) * bf16lo(kv.x) + bf16hi(kv.x) * bf16hi(kv.x) +
                   bf16lo(kv.y) * bf16lo(kv.y) + bf16hi(kv.y) * bf16hi(kv.y);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            sq += __shfl_xor_sync(0xffffffffu, sq, off);
            sk += __shfl_xor_sync(0xffffffffu, sk, off);
        }
        if (lane == 0) {
            const bool valid = t < L;
            const float rq = p.l2norm ? rsqrtf(sq + kNormEps) : 1.0f;
            const float rk = p.l2norm ? rsqrtf(sk + kNormEps) : 1.0f;
            reinterpret_cast<float*>(sm + AS_INVQ)[t] = valid ? rq * p.scale : 0.0f;
            reinterpret_cast<float*>(sm + AS_INVK)[t] = valid ? rk : 0.0f;
            reinterpret_cast<float*>(sm + AS_RQ)[t] = rq;
        }
    }
    const int v = 32 * x.qd + x.lane;   // TMEM lane of this thread in the value-side epilogues
    const int r0 = 16 * x.sub;          // its 16 columns
    const float* s_beta = reinterpret_cast<const float*>(sm + AS_BETA);
    // ---- round 1 done: X = V - S0^T K+^T (kept fp32 in TX), (beta X)^T and
    // dU^T as bf16 A operands
    if (!mbar_wait(&bar_m1, 0, &abort_flag)) {
        record_timeout(p.status, &abort_flag, 560);
    }
    tc_fence_after();
    {
        uint32_t ax[16], au[16];
        tmem_ld16(x.tbase + x.lane_base + TX + r0, ax);
        tmem_ld16(x.tbase + x.lane_base + TDU + r0, au);
        tmem_wait_ld();
        const uint8_t* vt = sm + AS_V + (v >> 6) * 8192;
        const uint32_t vb = 2 * (v & 63);
        uint32_t xb[8], ub[8];
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
            const float x0 = bf16_at(vt + sw128(r0 + j, vb)) - __uint_as_float(ax[j]);
            const float x1 = bf16_at(vt + sw128(r0 + j + 1, vb)) - __uint_as_float(ax[j + 1]);
            ax[j] = __float_as_uint(x0);
            ax[j + 1] = __float_as_uint(x1);
            xb[j >> 1] = pack_bf16x2(s_beta[r0 + j] * x0, s_beta[r0 + j + 1] * x1);
            ub[j >> 1] = pack_bf16x2(__uint_as_float(au[j]), __uint_as_float(au[j + 1]));
        }
        tmem_st16(x.tbase + x.lane_base + TX + r0, ax);
        tmem_st8(x.tbase + x.lane_base + TXB + 8 * x.sub, xb);
        tmem_st8(x.tbase + x.lane_base + TDUB + 8 * x.sub, ub);
        tmem_wait_st();
    }
    fence_proxy_async();   // the V tile's reads before the z tile lands over it
    if (cta_sync_tc_or(abort_flag != 0)) {
        return;
    }
    if (tid == 0) {
        asm_issue_round2(x);
        mma_commit(&bar_m2);
        mbar_arrive_expect_tx(&bar_z, 16384);
        tma_load_3d(sm + AS_Z, &args.tm_z, 0, h, (int)t0, &bar_z);
    }
    // ---- round 2 done: U^T -> bf16 B operand, dY: dv, -dX^T and -dY
    // operands, sum_v dY X
    if (!mbar_wait(&bar_m2, 0, &abort_flag)) {
        record_timeout(p.status, &abort_flag, 598);
    }
    tc_fence_after();
    {
        uint32_t au[16], ay[16], ax[16];
        tmem_ld16(x.tbase + x.lane_base + TU + r0, au);
        tmem_ld16(x.tbase + x.lane_base + TDY + r0, ay);
        tmem_ld16(x.tbase + x.lane_base + TX + r0, ax);
        tmem_wait_ld();
        float f[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(au[j]);
        store_row16(sm + AS_KP, v, 2 * r0, f);          // U^T row v (K+ is dead)
#pragma unroll
        for (int j = 0; j < 16; ++j) f[j] = -s_beta[r0 + j] * __uint_as_float(ay[j]);
        store_row16(sm + AS_KE, v, 2 * r0, f);          // -dX^T row v (Kend is dead)
        float* dv_g = p.dv + ((size_t)t0 * H + h) * D + v;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            if (r0 + j < L) {
                dv_g[(size_t)(r0 + j) * H * D] = -f[j];
            }
        }
        uint8_t* yb = sm + AS_DO + (v >> 6) * 16384 + 8192;
        const uint32_t vb = 2 * (v & 63);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            *reinterpret_cast<__nv_bfloat16*>(yb + sw128(r0 + j, vb)) =
                __float2bfloat16_rn(-__uint_as_float(ay[j]));
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) f[j] = __uint_as_float(ay[j]) * __uint_as_float(ax[j]);
        const float s = warp_sum16(f, x.lane);
        if (x.lane < 16) {
            reinterpret_cast<float*>(sm + AS_DB1)[x.qd * 64 + r0 + x.lane] = s;
        }
    }
    fence_proxy_async();
    if (cta_sync_tc_or(abort_flag != 0)) {
        return;
    }
    if (tid == 0) {
        asm_issue_round3(x);
        mma_commit(&bar_m3);
    }
    // ---- while the tensor core works: sum_v dS_L S0 (partials over four
    // 32-value slices) and the gate of this thread's (channel cc, block pb)
    const int cc = tid & (D - 1), pb = tid >> 7;
    {
        const uint8_t* srow = sm + AS_S0 + (pb >> 1) * 16384;
        const uint8_t* drow = sm + AS_DSL + (pb >> 1) * 16384;
        float acc = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t off = sw128(cc, 64 * (pb & 1) + 16 * k);
            const uint4 a = *reinterpret_cast<const uint4*>(srow + off);
            const uint4 b = *reinterpret_cast<const uint4*>(drow + off);
            acc += bf16lo(a.x) * bf16lo(b.x) + bf16hi(a.x) * bf16hi(b.x) +
                   bf16lo(a.y) * bf16lo(b.y) + bf16hi(a.y) * bf16hi(b.y) +
                   bf16lo(a.z) * bf16lo(b.z) + bf16hi(a.z) * bf16hi(b.z) +
                   bf16lo(a.w) * bf16lo(b.w) + bf16hi(a.w) * bf16hi(b.w);
        }
        reinterpret_cast<float*>(sm + AS_DGL)[pb * D + cc] = acc;
    }
    // the gate: g2 = -5 log2(e) sigmoid(x), x = e^A z (log2 units, 0 past
    // the end), cumulated within the block; x kept for the gate derivative
    float g2[16];
    const float eA = expf(p.A[h]);
    if (!mbar_wait(&bar_z, 0, &abort_flag)) {
        record_timeout(p.status, &abort_flag, 694);
    }
    {
        float run = 0.f;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = 16 * pb + j;
            // (the forward's arithmetic: sigmoid(x) = 1 / (1 + 2^{-x log2 e}))
            const float xv = eA * bf16_at(sm + AS_Z + t * 256 + 2 * cc);
            const float sg = rcp_approx(1.0f + exp2_approx(-kLog2e * xv));
            const float g = t < L ? -5.0f * kLog2e * sg : 0.0f;
            run += g;
            g2[j] = run;
        }
        reinterpret_cast<float*>(sm + AS_TOT)[pb * D + cc] = run;
    }
    __syncthreads();   // block totals published; S0 and dS_L reads done
    {
        const float* tot = reinterpret_cast<const float*>(sm + AS_TOT);
        float base = 0.f;
        for (int b = 0; b < pb; ++b) base += tot[b * D + cc];
#pragma unroll
        for (int j = 0; j < 16; ++j) g2[j] += base;
        reinterpret_cast<float*>(sm + AS_RHO)[pb * D + cc] = g2[7];
    }
    if (!mbar_wait(&bar_m3, 0, &abort_flag)) {
        record_timeout(p.status, &abort_flag, 722);
    }
    tc_fence_after();
    // ---- round 3 done: the dA epilogue (masked, fp32, both layouts) and the
    // Gkk part of dbeta; then x into the dA columns (this warp's own)
    {
        float* daq = reinterpret_cast<float*>(sm + AS_DAQ);
        float* dgg = reinterpret_cast<float*>(sm + AS_DGG);
        float* daqt = reinterpret_cast<float*>(sm + AS_DAQT);
        float* dggt = reinterpret_cast<float*>(sm + AS_DGGT);
        uint32_t ad[16];
        tmem_ld16(x.tbase + x.lane_base + TDA + r0, ad);
        tmem_wait_ld();
        if (x.qd < 2) {
            const int r = v;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = r0 + j;
                const float val = (i <= r && r < L) ? __uint_as_float(ad[j]) : 0.0f;
                daq[r * kDP + i] = val;
                daqt[i * kDP + r] = val;
            }
        } else {
            const int r = v - 64;
            const float br = s_beta[r];
            float acc = 0.f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int i = r0 + j;
                const float val = (i < r && r < L) ? __uint_as_float(ad[j]) : 0.0f;
                acc += val * bf16_at(sm + AS_G + sw128(r, 2 * i));
                dgg[r * kDP + i] = br * val;
                dggt[i * kDP + r] = br * val;
            }
            reinterpret_cast<float*>(sm + AS_DB2)[x.sub * 64 + r] = acc;
        }
        // (thread (cc, pb) is lane cc of this warp's quadrant, columns 16 pb;
        // the z tile is still intact)
        uint32_t xr[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            xr[j] = __float_as_uint(eA * bf16_at(sm + AS_Z + (16 * pb + j) * 256 + 2 * cc));
        }
        tmem_st16(x.tbase + x.lane_base + TXZ + 16 * pb, xr);
        tmem_wait_st();
    }
    cta_sync_tc();   // dA arrays written; Gkk and the operand tiles are dead
    // ---- the decayed key / query factors of this thread's tokens, with its
    // block's middle token as reference rho (each factor at most e^{40});
    // gamma of the thread's tokens parked in TMEM meanwhile
    const float rho = g2[7];
    {
        const float* invq = reinterpret_cast<const float*>(sm + AS_INVQ);
        const float* invk = reinterpret_cast<const float*>(sm + AS_INVK);
        float* wrow = reinterpret_cast<float*>(sm + AS_WROW);
        float* wck = reinterpret_cast<float*>(sm + AS_WCK);
        float* wcq = reinterpret_cast<float*>(sm + AS_WCQ);
        uint32_t gr[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = 16 * pb + j;
            const float kh = bf16_at(sm + AS_RAWK + t * 256 + 2 * cc) * invk[t];
            const float qh = bf16_at(sm + AS_RAWQ + t * 256 + 2 * cc) * invq[t];
            const float up = exp2_approx(g2[j] - rho);
            const float dn = exp2_approx(rho - g2[j]);
            wrow[t * D + cc] = kh * dn;
            wck[t * D + cc] = kh * up;
            wcq[t * D + cc] = qh * up;
            gr[j] = __float_as_uint(g2[j]);
        }
        tmem_st16(x.tbase + x.lane_base + TG2 + 16 * pb, gr);
        tmem_wait_st();
    }
    cta_sync_tc();
    // ---- decay chains (CUDA cores, fp32).  For the tokens of block b
    // (rows r or columns i there):
    //   RowQ[r] = sum_{i<=r} dAqk[r,i] e^{gamma_r - gamma_i} kh_i,
    //   RowK[r] = sum_{i<r}  dGkk[r,i] e^{gamma_r - gamma_i} kh_i,
    //   ColK[i] = sum_{r>i}  dGkk[r,i] e^{gamma_r - gamma_i} kh_r,
    //   ColQ[i] = sum_{r>=i} dAqk[r,i] e^{gamma_r - gamma_i} qh_r,
    // each factor split at the middle token of block b (gamma there = rho_b):
    // the tables hold every token's factor against its own block's reference,
    // moved to rho_b by e^{rho_b' - rho_b} (at most 1 for other blocks); the
    // factor of the output token, e^{+-(gamma - rho_b)}, is applied later.
    // Warp w: sum (w % 4: RowQ, RowK, ColK, ColQ) of block w / 4, all 128
    // channels (lane l: channels 4 l .. 4 l + 3), 16 outputs per channel; the
    // 4 sums of a block share one SM sub-partition's worth of loads each way.
    {
        const int kind = warp & 3, b = warp >> 2;
        const int c0 = 4 * lane;
        const float* rhos = reinterpret_cast<const float*>(sm + AS_RHO);
        const float4 rb = *reinterpret_cast<const float4*>(rhos + b * D + c0);
        float acc[16][4];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
        }
        const bool row = kind < 2;
        // row sums: source tokens i of blocks 0..b (table WROW, dA^T rows i);
        // column sums: source tokens r of blocks b..3 (WCK / WCQ, dA rows r)
        const float* wt = reinterpret_cast<const float*>(
            sm + (row ? AS_WROW : kind == 2 ? AS_WCK : AS_WCQ));
        const float* da = reinterpret_cast<const float*>(
            sm + (kind == 0 ? AS_DAQT : kind == 1 ? AS_DGGT : kind == 2 ? AS_DGG : AS_DAQ));
        const int s0 = row ? 0 : b, s1 = row ? b : 3;
        for (int sb = s0; sb <= s1; ++sb) {
            const float4 rs = *reinterpret_cast<const float4*>(rhos + sb * D + c0);
            float4 f;
            if (row) {
                f = make_float4(exp2_approx(rb.x - rs.x), exp2_approx(rb.y - rs.y),
                                exp2_approx(rb.z - rs.z), exp2_approx(rb.w - rs.w));
            } else {
                f = make_float4(exp2_approx(rs.x - rb.x), exp2_approx(rs.y - rb.y),
                                exp2_approx(rs.z - rb.z), exp2_approx(rs.w - rb.w));
            }
#pragma unroll 1
            for (int u = 0; u < 16; ++u) {
                const int s = 16 * sb + u;
                float4 w = *reinterpret_cast<const float4*>(wt + s * D + c0);
                w.x *= f.x; w.y *= f.y; w.z *= f.z; w.w *= f.w;
                const float4* a4 = reinterpret_cast<const float4*>(da + s * kDP + 16 * b);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 a = a4[k];
                    const float av[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        acc[4 * k + e][0] += av[e] * w.x;
                        acc[4 * k + e][1] += av[e] * w.y;
                        acc[4 * k + e][2] += av[e] * w.z;
                        acc[4 * k + e][3] += av[e] * w.w;
                    }
                }
            }
        }
        __syncthreads();   // every read of the dA arrays and the tables is done
        float* out = reinterpret_cast<float*>(sm + AS_OUT + kind * 32768);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            *reinterpret_cast<float4*>(out + (16 * b + j) * D + c0) =
                make_float4(acc[j][0], acc[j][1], acc[j][2], acc[j][3]);
        }
    }
    __syncthreads();
    // ---- per (token, channel): the output tokens' factors; dq_hat, dk_hat
    // (over RowQ and RowK in shared memory) and dgamma
    float dgam[16];
    {
        const float* invq = reinterpret_cast<const float*>(sm + AS_INVQ);
        const float* invk = reinterpret_cast<const float*>(sm + AS_INVK);
        const float* tot = reinterpret_cast<const float*>(sm + AS_TOT);
        float* o_rq = reinterpret_cast<float*>(sm + AS_OUT);
        float* o_rk = reinterpret_cast<float*>(sm + AS_OUT + 32768);
        const float* o_ck = reinterpret_cast<const float*>(sm + AS_OUT + 65536);
        const float* o_cq = reinterpret_cast<const float*>(sm + AS_OUT + 98304);
        const float gL = tot[cc] + tot[D + cc] + tot[2 * D + cc] + tot[3 * D + cc];
        const uint32_t tl = x.tbase + x.lane_base;
        uint32_t ta[16], tb[16], tg[16];
        tmem_ld16(tl + TG2 + 16 * pb, tg);
        tmem_ld16(tl + TDQ + 16 * pb, ta);
        tmem_wait_ld();
        // Q side: dq_hat = dQ+ e^gamma + RowQ;  dgamma = qh dq_hat
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = 16 * pb + j;
            const float gj = __uint_as_float(tg[j]);
            const float qh = bf16_at(sm + AS_RAWQ + t * 256 + 2 * cc) * invq[t];
            const float dqh = __uint_as_float(ta[j]) * exp2_approx(gj) +
                              o_rq[t * D + cc] * exp2_approx(gj - rho);
            const bool valid = t < L;
            o_rq[t * D + cc] = valid ? dqh : 0.0f;   // becomes dq_hat
            dgam[j] = valid ? qh * dqh : 0.0f;
        }
        // K side: dk_hat = dK+ e^gamma + dKend e^{gamma_L - gamma} + RowK + ColK + ColQ;
        // dgamma += kh (dK+ e^gamma - dKend e^{gamma_L - gamma} + RowK - ColK - ColQ)
        float dke_sum = 0.f, dg_sum = 0.f;
        tmem_ld16(tl + TDK + 16 * pb, ta);
        tmem_ld16(tl + TDKE + 16 * pb, tb);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int t = 16 * pb + j;
            const float gj = __uint_as_float(tg[j]);
            const float kh = bf16_at(sm + AS_RAWK + t * 256 + 2 * cc) * invk[t];
            const float a = __uint_as_float(ta[j]) * exp2_approx(gj);
            const float e = __uint_as_float(tb[j]) * exp2_approx(gL - gj);
            const float up = exp2_approx(gj - rho), dn = exp2_approx(rho - gj);
            const float rk = o_rk[t * D + cc] * up;
            const float cs = (o_ck[t * D + cc] + o_cq[t * D + cc]) * dn;
            const bool valid = t < L;
            o_rk[t * D + cc] = valid ? a + e + rk + cs : 0.0f;   // becomes dk_hat
            dgam[j] += valid ? kh * (a - e + rk - cs) : 0.0f;
            dke_sum += valid ? kh * e : 0.0f;
            dg_sum += dgam[j];
        }
        reinterpret_cast<float*>(sm + AS_DGT)[pb * D + cc] = dg_sum;
        reinterpret_cast<float*>(sm + AS_DKE)[pb * D + cc] = dke_sum;
    }
    __syncthreads();   // block sums published; ColK, ColQ read
    // ---- dg = reverse cumulative sum of dgamma (+ dgamma_L), gate
    // derivative, dz; dx * x to shared memory
    {
        const float* dgt = reinterpret_cast<const float*>(sm + AS_DGT);
        const float* dgl = reinterpret_cast<const float*>(sm + AS_DGL);
        const float* dke = reinterpret_cast<const float*>(sm + AS_DKE);
        const float gamL = reinterpret_cast<const float*>(sm + AS_GAM)[cc];
        float run = gamL * (dgl[cc] + dgl[D + cc] + dgl[2 * D + cc] + dgl[3 * D + cc]) +
                    (dke[cc] + dke[D + cc] + dke[2 * D + cc] + dke[3 * D + cc]);
        for (int b = pb + 1; b < 4; ++b) run += dgt[b * D + cc];
        float* dxx_s = reinterpret_cast<float*>(sm + AS_DXX);
        uint32_t xr[16];
        tmem_ld16(x.tbase + x.lane_base + TXZ + 16 * pb, xr);
        tmem_wait_ld();
#pragma unroll
        for (int j = 15; j >= 0; --j) {
            const int t = 16 * pb + j;
            run += dgam[j];
            float dxx = 0.f;
            if (t < L) {
                const float zx = __uint_as_float(xr[j]);
                const float sg = rcp_approx(1.0f + exp2_approx(-kLog2e * zx));
                const float dx = run * (-5.0f) * sg * (1.0f - sg);
                p.dz[((size_t)(t0 + t) * H + h) * D + cc] = dx * eA;
                dxx = dx * zx;
            }
            dxx_s[t * D + cc] = dxx;
        }
    }
    __syncthreads();
    // ---- per token: normalisation derivatives, dq, dk, dbeta and the token's
    // share of dL/dA (warp w: tokens w, w + 16, ...; lane: 4 channels)
    {
        const float* dqh_s = reinterpret_cast<const float*>(sm + AS_DQH);
        const float* dkh_s = reinterpret_cast<const float*>(sm + AS_DKH);
        const float* dxx_s = reinterpret_cast<const float*>(sm + AS_DXX);
        const float* rqv = reinterpret_cast<const float*>(sm + AS_RQ);
        const float* rkv = reinterpret_cast<const float*>(sm + AS_INVK);
        const float* db1 = reinterpret_cast<const float*>(sm + AS_DB1);
        const float* db2 = reinterpret_cast<const float*>(sm + AS_DB2);
        for (int t = warp; t < L; t += kThreads / 32) {
            const float4 dq4 = *reinterpret_cast<const float4*>(dqh_s + t * D + 4 * lane);
            const float4 dk4 = *reinterpret_cast<const float4*>(dkh_s + t * D + 4 * lane);
            const float4 dx4 = *reinterpret_cast<const float4*>(dxx_s + t * D + 4 * lane);
            const uint2 qv = *reinterpret_cast<const uint2*>(sm + AS_RAWQ + t * 256 + lane * 8);
            const uint2 kv = *reinterpret_cast<const uint2*>(sm + AS_RAWK + t * 256 + lane * 8);
            const float q0 = bf16lo(qv.x), q1 = bf16hi(qv.x), q2 = bf16lo(qv.y), q3 = bf16hi(qv.y);
            const float k0 = bf16lo(kv.x), k1 = bf16hi(kv.x), k2 = bf16lo(kv.y), k3 = bf16hi(kv.y);
            float s1 = q0 * dq4.x + q1 * dq4.y + q2 * dq4.z + q3 * dq4.w;
            float s2 = k0 * dk4.x + k1 * dk4.y + k2 * dk4.z + k3 * dk4.w;
            float s3 = dx4.x + dx4.y + dx4.z + dx4.w;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                s1 += __shfl_xor_sync(0xffffffffu, s1, off);
                s2 += __shfl_xor_sync(0xffffffffu, s2, off);
                s3 += __shfl_xor_sync(0xffffffffu, s3, off);
            }
            const size_t o = ((size_t)(t0 + t) * H + h) * D + 4 * lane;
            float4 oq, ok;
            if (p.l2norm) {
                const float rq = rqv[t], rk = rkv[t];
                const float cq = rq * rq * rq * s1, ck = rk * rk * rk * s2;
                oq = make_float4(p.scale * (rq * dq4.x - cq * q0), p.scale * (rq * dq4.y - cq * q1),
                                 p.scale * (rq * dq4.z - cq * q2), p.scale * (rq * dq4.w - cq * q3));
                ok = make_float4(rk * dk4.x - ck * k0, rk * dk4.y - ck * k1, rk * dk4.z - ck * k2,
                                 rk * dk4.w - ck * k3);
            } else {
                oq = make_float4(p.scale * dq4.x, p.scale * dq4.y, p.scale * dq4.z,
                                 p.scale * dq4.w);
                ok = dk4;
            }
            *reinterpret_cast<float4*>(p.dq + o) = oq;
            *reinterpret_cast<float4*>(p.dk + o) = ok;
            if (lane == 0) {
                const size_t th = (size_t)(t0 + t) * H + h;
                p.dbeta[th] = db1[t] + db1[64 + t] + db1[128 + t] + db1[192 + t] + db2[t] +
                              db2[64 + t] + db2[128 + t] + db2[192 + t];
                p.dA_tok[th] = s3;
            }
        }
    }
    }();
    // a wait that gave up may leave copies or products in flight
    if (abort_flag) {
        mbar_wait(&bar_ld, 0, nullptr);
        mbar_wait(&bar_z, 0, nullptr);
    }
    cta_sync_tc();
    if (tid == 0) {
        mma_commit(&bar_fin);
        mbar_wait(&bar_fin, 0, nullptr);
    }
    cta_sync_tc();
    if (warp == 0) {
        tmem_dealloc(x.tbase, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_bwd_chunked(const BwdChunkedParams& p, cudaStream_t stream) {
    if (p.N < 1 || p.H < 1 || p.total_T < 1) {
        return cudaErrorInvalidValue;
    }
    BwdArgs args;
    memset(&args, 0, sizeof(args));
    args.p = p;
    if (!make_token_map(&args.tm_q, p.q, p.total_T, p.H, false) ||
        !make_token_map(&args.tm_k, p.k, p.total_T, p.H, false) ||
        !make_token_map(&args.tm_z, p.z, p.total_T, p.H, false) ||
        !make_token_map(&args.tm_v, p.v, p.total_T, p.H, true) ||
        !make_token_map(&args.tm_do, p.dO, p.total_T, p.H, true)) {
        return cudaErrorInvalidValue;
    }
    cudaError_t err = cudaFuncSetAttribute(kda_bwd_chain_kernel,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)kChainSmem);
    if (err != cudaSuccess) {
        return err;
    }
    err = cudaFuncSetAttribute(kda_bwd_assemble_kernel,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAsmSmem);
    if (err != cudaSuccess) {
        return err;
    }
    kda_bwd_chain_kernel<<<(unsigned)((int64_t)p.N * p.H), kThreads, kChainSmem, stream>>>(args);
    err = cudaGetLastError();
    if (err != cudaSuccess) {
        return err;
    }
    kda_bwd_assemble_kernel<<<(unsigned)((int64_t)p.max_chunks * p.H), kThreads, kAsmSmem,
                              stream>>>(args);
    return cudaGetLastError();
}

}  // namespace kda
