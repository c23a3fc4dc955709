// kda_prefill_sm103.cu -- chunked KDA prefill on tcgen05 tensor cores (sm_103a).
//
// The pages' prefill ("Kimi K3 Open Weights: What Is Actually New In Its 2.8
// Trillion Parameter Architecture", section 1) processes tokens "parallel
// within chunks, recurrent between", with decay products, triangular
// intra-chunk interactions and dense matrix tiles; the bounded gate
// (g >= -5) keeps the reciprocal decay factors of a 16-token tile inside the
// bf16 range (e^80 < 3.4e38), so the diagonal tiles use dense matmuls too.
//
// Algebra used per chunk of C = 64 tokens (start state S0, d_k = d_v = 128),
// derived by unrolling the recurrence; gamma_r = inclusive cumulative g:
//   Akk[r,i] = beta_r <k_r e^{gamma_r - gamma_i}, k_i>   (i < r)
//   Aqk[r,i] =        <q_r e^{gamma_r - gamma_i}, k_i>   (i <= r)
//   Tm       = (I + Akk)^-1 Diag(beta)                    (UT solve, fp32)
//   U        = Tm V - (Tm K+) S0,    K+ = k * e^{gamma}
//   O        = Q+ S0 + Aqk U,        Q+ = q * e^{gamma}
//   S_next   = Diag(e^{gamma_C}) S0 + Kend^T U,   Kend = k * e^{gamma_C - gamma}
// The Gram products use one reference point per 16-token block a
// (rho_a = gamma at the end of the previous block): the query/key side is
// scaled by e^{gamma_r - rho_a} <= 1 and the key side of the products with
// block a by e^{rho_a - gamma_i} (<= e^80 inside the block, <= 1 before it).
//
// Execution (one CTA of 8 warps per (sequence, head); one TMEM allocation of
// 512 columns; fp32 state S^T kept in TMEM for the whole sequence):
//   P0  TMA: raw q, k, z tiles [64 tok][128 ch]; v as a 128B-swizzled operand
//   P1  prologue on the CUDA cores: L2 norms, gate, per-block cumulative
//       decay, and the bf16 operand tiles (X~, K~^(a), K+, Q+, Kend)
//   P2  tcgen05: Gram Aqk/Akk (two M=128 x N=64 x K=128 products)
//   P3  Gram -> smem (masking, beta);  S^T -> bf16 operand; S^T *= Gamma
//   P4  UT solve in shared memory (fp32): Tm
//   P5  tcgen05: W^T = K+^T Tm^T, U^T = V^T Tm^T
//   P6  W^T -> bf16 operand
//   P7  tcgen05: U^T += S^T (-W^T), O^T = S^T Q+^T
//   P8  U^T -> bf16 operand
//   P9  tcgen05: O^T += U^T Aqk^T, S^T += U^T Kend
//   P10 O^T -> o (bf16)
// Every MMA is M=128 with the head dimension on M (the transposed form), so
// the TMEM accumulator layout is row m -> lane m.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "kda_internal.h"
#include "sm103_ptx.cuh"

namespace kda {
namespace {

using namespace sm103;

constexpr int C = 64;          // chunk length
constexpr int D = 128;         // head dim (d_k = d_v)
constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNormEps = 1e-6f;
constexpr int kStatusTimeout = 1;

// ---- shared memory map (byte offsets from a 1024-aligned base) ----
// Region 1 (48 KB): raw q, k, z tiles, dedicated so that the next chunk's
// loads can be issued as soon as the prologue has consumed them.
constexpr uint32_t OFF_RAWQ = 0;
constexpr uint32_t OFF_RAWK = 16384;
constexpr uint32_t OFF_RAWZ = 32768;
// Region 2 (96 KB): X~ and K~ (Gram operands, P1-P2); then S^T bf16, Aqk, Tm
// and the solve scratch (P3-P4); then W^T and U^T (P6-P9).
constexpr uint32_t OFF_XT = 49152;          // 2 N-blocks x [128 c][64 e]  (MN-major B)
constexpr uint32_t OFF_KT = 49152 + 32768;  // 4 M-blocks x [128 c][64 i] (MN-major A)
constexpr uint32_t OFF_ST = 49152;          // [2 atoms][128 j][64 c]     (K-major A)
constexpr uint32_t OFF_AQK = 81920;         // [64 r][64 i]               (K-major B)
constexpr uint32_t OFF_TM = 90112;          // [64 r][64 i]               (K-major B)
constexpr uint32_t OFF_AKK = 98304;         // fp32 [64][65]
constexpr uint32_t OFF_NMAT = 114944;       // fp32 [64][65]
constexpr uint32_t OFF_MSCR = 131584;       // fp32 [3 x 16][65]
constexpr uint32_t OFF_WT = 98304;          // bf16 [128 c][64 r]  (MN-major B)
constexpr uint32_t OFF_UT = 114688;         // bf16 [128 j][64 i]  (K-major A)
// dedicated operand tiles
constexpr uint32_t OFF_V = 147456;          // [2 blocks][64 i][64 j]     (MN-major A)
constexpr uint32_t OFF_KP = 163840;         // [128 c][64 i]              (K-major A)
constexpr uint32_t OFF_QP = 180224;         // [128 c][64 r]              (MN-major B)
constexpr uint32_t OFF_KE = 196608;         // [128 c][64 i]              (K-major B)
// small fp32 arrays
constexpr uint32_t OFF_INVQ = 212992;       // [64]
constexpr uint32_t OFF_INVK = OFF_INVQ + 256;
constexpr uint32_t OFF_BETA = OFF_INVK + 256;
constexpr uint32_t OFF_TOT = OFF_BETA + 256;  // [4][128]
constexpr uint32_t OFF_GAM = OFF_TOT + 2048;  // [128]
constexpr uint32_t SMEM_USED = OFF_GAM + 512;
constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // slack for 1024-byte alignment

// TMEM columns
constexpr uint32_t TM_S = 0;      // S^T  [128 j lanes][128 c]
constexpr uint32_t TM_G1 = 128;   // Gram blocks 3, 2
constexpr uint32_t TM_G2 = 192;   // Gram blocks 1, 0
constexpr uint32_t TM_W = 256;    // W^T  [128 c][64 r]
constexpr uint32_t TM_U = 320;    // U^T  [128 j][64 r]
constexpr uint32_t TM_O = 384;    // O    [64 r][128 j]  (M = 64 layout)
constexpr uint32_t TMEM_COLS = 512;

struct ChunkedArgs {
    CUtensorMap tm_q;
    CUtensorMap tm_k;
    CUtensorMap tm_z;
    CUtensorMap tm_v;
    ChunkedParams p;
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ float bf16lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

// Store 16 consecutive fp32 values (tokens) of one operand row as bf16 into a
// 128B-swizzled tile: row `row`, starting byte `byte0` (multiple of 32).
__device__ __forceinline__ void store_row16(uint8_t* tile, uint32_t row, uint32_t byte0,
                                            const float (&v)[16]) {
    uint4 a, b;
    a.x = pack_bf16x2(v[0], v[1]);   a.y = pack_bf16x2(v[2], v[3]);
    a.z = pack_bf16x2(v[4], v[5]);   a.w = pack_bf16x2(v[6], v[7]);
    b.x = pack_bf16x2(v[8], v[9]);   b.y = pack_bf16x2(v[10], v[11]);
    b.z = pack_bf16x2(v[12], v[13]); b.w = pack_bf16x2(v[14], v[15]);
    *reinterpret_cast<uint4*>(tile + sw128(row, byte0)) = a;
    *reinterpret_cast<uint4*>(tile + sw128(row, byte0 + 16)) = b;
}

// 2^x and 1/x with the hardware approximations (ex2.approx handles subnormal
// results, so decay factors down to 2^-149 are kept).
__device__ __forceinline__ float exp2_approx(float x) {
    float y;
    asm("ex2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ---- UT-solve helpers: warp-level 16x16x16 products on fp32 [..][65] tiles ----
__device__ __forceinline__ uint32_t to_tf32(float x) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ void mma_tf32_16x8x8(float (&d)[4], const uint32_t (&a)[4],
                                                const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// acc (+)= X[xr0.., xc0..] * Y[yr0.., yc0..], all 16x16, row stride 65 floats.
// acc holds the two 16x8 column halves in the m16n8 accumulator layout.
__device__ __forceinline__ void warp_gemm16(float (&acc)[2][4], const float* X, int xr0, int xc0,
                                            const float* Y, int yr0, int yc0, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int kb = 0; kb < 16; kb += 8) {
        uint32_t a[4];
        a[0] = to_tf32(X[(xr0 + g) * 65 + xc0 + kb + t]);
        a[1] = to_tf32(X[(xr0 + g + 8) * 65 + xc0 + kb + t]);
        a[2] = to_tf32(X[(xr0 + g) * 65 + xc0 + kb + t + 4]);
        a[3] = to_tf32(X[(xr0 + g + 8) * 65 + xc0 + kb + t + 4]);
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            uint32_t b[2];
            b[0] = to_tf32(Y[(yr0 + kb + t) * 65 + yc0 + nt * 8 + g]);
            b[1] = to_tf32(Y[(yr0 + kb + t + 4) * 65 + yc0 + nt * 8 + g]);
            mma_tf32_16x8x8(acc[nt], a, b);
        }
    }
}

__device__ __forceinline__ void warp_store16(const float (&acc)[2][4], float* Z, int zr0, int zc0,
                                             float sign, int lane) {
    const int g = lane >> 2, t = lane & 3;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        Z[(zr0 + g) * 65 + zc0 + nt * 8 + 2 * t] = sign * acc[nt][0];
        Z[(zr0 + g) * 65 + zc0 + nt * 8 + 2 * t + 1] = sign * acc[nt][1];
        Z[(zr0 + g + 8) * 65 + zc0 + nt * 8 + 2 * t] = sign * acc[nt][2];
        Z[(zr0 + g + 8) * 65 + zc0 + nt * 8 + 2 * t + 1] = sign * acc[nt][3];
    }
}

// CTA-wide barrier that also orders tcgen05 operations around it.
__device__ __forceinline__ void cta_sync_tc() {
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

__device__ void record_timeout(int32_t* status, volatile int* abort_flag) {
    atomicExch(status, kStatusTimeout);
    *abort_flag = 1;
}

__global__ void __launch_bounds__(kThreads, 1)
kda_chunked_kernel(const __grid_constant__ ChunkedArgs args) {
    const ChunkedParams& p = args.p;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
    __shared__ uint64_t bar_raw;   // raw q, k, z of a chunk landed
    __shared__ uint64_t bar_v;     // v of a chunk landed
    __shared__ uint64_t bar_mma;
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    float* s_invq = reinterpret_cast<float*>(sm + OFF_INVQ);
    float* s_invk = reinterpret_cast<float*>(sm + OFF_INVK);
    float* s_beta = reinterpret_cast<float*>(sm + OFF_BETA);
    float* s_tot = reinterpret_cast<float*>(sm + OFF_TOT);
    float* s_gam = reinterpret_cast<float*>(sm + OFF_GAM);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    const int qd = warp & 3;           // TMEM lane quadrant this warp may access
    const int sub = warp >> 2;         // 0..3: which of the four warps of that quadrant
    const uint32_t lane_base = (uint32_t)(32 * qd) << 16;
    const int H = p.H;
    const int unit = blockIdx.x;
    const int n = unit / H;
    const int h = unit % H;

    int64_t bos, eos;
    if (p.cu_seqlens) {
        bos = p.cu_seqlens[n];
        eos = p.cu_seqlens[n + 1];
    } else {
        const int64_t len = p.total_T / p.N;
        bos = (int64_t)n * len;
        eos = bos + len;
    }
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
    if (warp == 0) {
        tmem_alloc(&tmem_base_s, TMEM_COLS);
        tmem_relinquish();
    }
    cta_sync_tc();
    const uint32_t tbase = tmem_base_s;
    const uint32_t smem_base = smem_u32(sm);

    // ---- initial state -> TMEM: lane j holds column j of S (S^T row j) ----
    {
        const int j = 32 * qd + lane;
        const uint32_t taddr = tbase + lane_base + TM_S;
#pragma unroll 1
        for (int cb = 32 * sub; cb < 32 * sub + 32; cb += 16) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float x = p.initial_state
                                    ? __ldg(p.initial_state + state_off + (size_t)(cb + i) * D + j)
                                    : 0.0f;
                r[i] = __float_as_uint(x);
            }
            tmem_st16(taddr + cb, r);
        }
        tmem_wait_st();
    }
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

        // ---------------- P1a: per-token L2 norms (4 tokens per warp) ----------------
        {
            const uint8_t* rq = sm + OFF_RAWQ;
            const uint8_t* rk = sm + OFF_RAWK;
            float sq[4], sk[4];
#pragma unroll
            for (int tt = 0; tt < 4; ++tt) {
                const int r = warp * 4 + tt;
                const uint2 qv = *reinterpret_cast<const uint2*>(rq + r * 256 + lane * 8);
                const uint2 kv = *reinterpret_cast<const uint2*>(rk + r * 256 + lane * 8);
                const float q0 = bf16lo(qv.x), q1 = bf16hi(qv.x), q2 = bf16lo(qv.y), q3 = bf16hi(qv.y);
                const float k0 = bf16lo(kv.x), k1 = bf16hi(kv.x), k2 = bf16lo(kv.y), k3 = bf16hi(kv.y);
                sq[tt] = q0 * q0 + q1 * q1 + q2 * q2 + q3 * q3;
                sk[tt] = k0 * k0 + k1 * k1 + k2 * k2 + k3 * k3;
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
                for (int tt = 0; tt < 4; ++tt) {
                    sq[tt] += __shfl_xor_sync(0xffffffffu, sq[tt], off);
                    sk[tt] += __shfl_xor_sync(0xffffffffu, sk[tt], off);
                }
            }
            if (lane < 4) {
                const int r = warp * 4 + lane;
                const float a = lane == 0 ? sq[0] : lane == 1 ? sq[1] : lane == 2 ? sq[2] : sq[3];
                const float b = lane == 0 ? sk[0] : lane == 1 ? sk[1] : lane == 2 ? sk[2] : sk[3];
                const bool valid = r < L;
                s_invq[r] = valid ? (p.l2norm ? rsqrtf(a + kNormEps) : 1.0f) * p.scale : 0.0f;
                s_invk[r] = valid ? (p.l2norm ? rsqrtf(b + kNormEps) : 1.0f) : 0.0f;
            }
        }
        __syncthreads();

        // ---------------- P1b: gate and per-token decay (one channel, 16 tokens per thread) ----------------
        const int c = tid & (D - 1);   // channel
        const int ab = tid >> 7;       // token block: tokens 16ab .. 16ab+15
        float qh[16], kh[16], al[16];
        {
            float tot = 0.f;           // block total of g, log2 units
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = 16 * ab + rr;
                const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                    sm + OFF_RAWQ + r * 256 + 2 * c));
                const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                    sm + OFF_RAWK + r * 256 + 2 * c));
                const float zv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                    sm + OFF_RAWZ + r * 256 + 2 * c));
                // g = -5 sigmoid(e^A z) in log2 units; invalid tokens: g = 0
                const float sg = rcp_approx(1.0f + exp2_approx(-eA_log2 * zv));
                const float g = r < L ? -5.0f * kLog2e * sg : 0.0f;
                tot += g;
                al[rr] = exp2_approx(g);
                qh[rr] = qv * s_invq[r];
                kh[rr] = kv * s_invk[r];
            }
            s_tot[ab * D + c] = tot;
        }
        __syncthreads();

        // ---------------- P1c: operand tiles ----------------
        {
            float t[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) t[b] = s_tot[b * D + c];
            float rho[5];  // rho[b] = log2 decay before block b; rho[4] = chunk total
            rho[0] = 0.f;
#pragma unroll
            for (int b = 0; b < 4; ++b) rho[b + 1] = rho[b] + t[b];
            if (ab == 0) {
                s_gam[c] = exp2_approx(rho[4]);
            }
            const float rho_a = ab == 0 ? rho[0] : ab == 1 ? rho[1] : ab == 2 ? rho[2] : rho[3];
            const float rho_a1 = ab == 0 ? rho[1] : ab == 1 ? rho[2] : ab == 2 ? rho[3] : rho[4];
            const float eRa = exp2_approx(rho_a);               // e^{rho_a}          <= 1
            const float cF = exp2_approx(rho_a - rho_a1);       // e^{-block total}   <= e^80
            const float eEnd = exp2_approx(rho[4] - rho_a1);    // e^{gamma_C - rho_{a+1}} <= 1

            // In-block decay factors as running products of alpha:
            //   E_r = e^{gamma_r - rho_a}      = prod_{t<=r} alpha_t        in [e^-80, 1]
            //   G_r = e^{rho_{a+1} - gamma_r}  = prod_{t>r, t in block}     in [e^-80, 1]
            //   F_r = e^{rho_a - gamma_r}      = G_r e^{-block total}       in [1, e^80]
            float E[16], G[16];
            E[0] = al[0];
#pragma unroll
            for (int rr = 1; rr < 16; ++rr) E[rr] = E[rr - 1] * al[rr];
            G[15] = 1.0f;
#pragma unroll
            for (int rr = 14; rr >= 0; --rr) G[rr] = G[rr + 1] * al[rr + 1];

            float v[16];
            // X~ : Gram B operand; N-block 0 = [Q3 K3 Q2 K2], N-block 1 = [Q1 K1 Q0 K0]
            const uint32_t nb = ab >= 2 ? 0u : 1u;
            const uint32_t e0 = (ab >= 2 ? (3 - ab) : (1 - ab)) * 32;
            uint8_t* xt = sm + OFF_XT + nb * 16384;
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) v[rr] = qh[rr] * E[rr];
            store_row16(xt, c, 2 * e0, v);
            // Q+ = q e^{gamma} = (q e^{gamma - rho_a}) e^{rho_a}
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) v[rr] *= eRa;
            store_row16(sm + OFF_QP, c, 32 * ab, v);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) v[rr] = kh[rr] * E[rr];
            store_row16(xt, c, 2 * (e0 + 16), v);
            // K+ = k e^{gamma}
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) v[rr] *= eRa;
            store_row16(sm + OFF_KP, c, 32 * ab, v);
            // key side with the end-of-block reference: k e^{rho_{a+1} - gamma_r} <= 1
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) G[rr] *= kh[rr];
            // Kend = k e^{gamma_C - gamma}
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) v[rr] = G[rr] * eEnd;
            store_row16(sm + OFF_KE, c, 32 * ab, v);
            // K~^(ab) = k e^{rho_a - gamma}: M-block (3 - ab) of the Gram A operand
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) v[rr] = G[rr] * cF;
            store_row16(sm + OFF_KT + (3 - ab) * 16384, c, 32 * ab, v);
            // K~^(a') for a' > ab: k e^{rho_{a'} - gamma} = (k e^{rho_{a+1} - gamma}) e^{rho_{a'} - rho_{a+1}}
#pragma unroll
            for (int ap = 1; ap < 4; ++ap) {
                if (ap > ab) {
                    const float f = exp2_approx((ap == 1 ? rho[1] : ap == 2 ? rho[2] : rho[3]) - rho_a1);
#pragma unroll
                    for (int rr = 0; rr < 16; ++rr) v[rr] = G[rr] * f;
                    store_row16(sm + OFF_KT + (3 - ap) * 16384, c, 32 * ab, v);
                }
            }
        }
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
            const uint32_t idg = idesc_bf16(128, 64, 1, 1);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t a1 = smem_desc(smem_base + OFF_KT + kk * 2048, 16384, 1024);
                const uint64_t b1 = smem_desc(smem_base + OFF_XT + kk * 2048, 16384, 1024);
                mma_bf16(tbase + TM_G1, a1, b1, idg, kk > 0);
                const uint64_t a2 = smem_desc(smem_base + OFF_KT + 32768 + kk * 2048, 16384, 1024);
                const uint64_t b2 = smem_desc(smem_base + OFF_XT + 16384 + kk * 2048, 16384, 1024);
                mma_bf16(tbase + TM_G2, a2, b2, idg, kk > 0);
            }
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

        // ---------------- P3: Gram -> Akk (fp32), Aqk (bf16);  S^T -> bf16, S^T *= Gamma ----------------
        if (warp < 8) {
            // warps 0-3: Gram blocks 3 (lanes 0-63) and 2 (lanes 64-127) in TM_G1;
            // warps 4-7: Gram blocks 1 and 0 in TM_G2
            const int g = warp >> 2;
            float* akk = reinterpret_cast<float*>(sm + OFF_AKK);
            const int blk = g == 0 ? (qd < 2 ? 3 : 2) : (qd < 2 ? 1 : 0);
            const uint32_t col = (g == 0 ? TM_G1 : TM_G2) + (qd < 2 ? 0 : 32);
            const int i = (qd < 2 ? 32 * qd : 32 * (qd - 2)) + lane;
            uint32_t vq[16], vk[16];
            tmem_ld16(tbase + lane_base + col, vq);
            tmem_ld16(tbase + lane_base + col + 16, vk);
            tmem_wait_ld();
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) {
                const int r = 16 * blk + rr;
                const float aq = i <= r ? __uint_as_float(vq[rr]) : 0.0f;
                const float ak = i < r ? s_beta[r] * __uint_as_float(vk[rr]) : 0.0f;
                akk[r * 65 + i] = ak;
                *reinterpret_cast<__nv_bfloat16*>(sm + OFF_AQK + sw128(r, 2 * i)) =
                    __float2bfloat16_rn(aq);
            }
        } else {
            // warps 8-15: S^T row j = lane, columns [64 half, 64 half + 64)
            const int j = 32 * qd + lane;
            const int half = sub - 2;
            const uint32_t taddr = tbase + lane_base + TM_S;
#pragma unroll 1
            for (int cb = 64 * half; cb < 64 * half + 64; cb += 32) {
                uint32_t r0[16], r1[16];
                tmem_ld16(taddr + cb, r0);
                tmem_ld16(taddr + cb + 16, r1);
                tmem_wait_ld();
                float v0[16], v1[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    v0[i] = __uint_as_float(r0[i]);
                    v1[i] = __uint_as_float(r1[i]);
                }
                store_row16(sm + OFF_ST + half * 16384, j, 2 * (cb % 64), v0);
                store_row16(sm + OFF_ST + half * 16384, j, 2 * (cb % 64) + 32, v1);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    r0[i] = __float_as_uint(v0[i] * s_gam[cb + i]);
                    r1[i] = __float_as_uint(v1[i] * s_gam[cb + 16 + i]);
                }
                tmem_st16(taddr + cb, r0);
                tmem_st16(taddr + cb + 16, r1);
            }
            tmem_wait_st();
        }
        cta_sync_tc();

        // ---------------- P4: UT solve  Tm = (I + Akk)^-1 Diag(beta) ----------------
        // N = (I + L)^-1, L = Akk strictly lower, in 16x16 blocks: the diagonal
        // blocks by forward substitution (one column per thread), then the
        // off-diagonal blocks by block rows, N_ab = -N_aa sum_{c=b}^{a-1} L_ac N_cb,
        // in three waves of warp-level tf32 products.
        {
            const float* Lm = reinterpret_cast<const float*>(sm + OFF_AKK);
            float* Nm = reinterpret_cast<float*>(sm + OFF_NMAT);
            float* Ms = reinterpret_cast<float*>(sm + OFF_MSCR);
            if (tid < 64) {
                const int a = tid >> 4, jj = tid & 15;
                const float* Lb = Lm + (16 * a) * 65 + 16 * a;
                float acc[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) acc[r] = (r == jj) ? 1.0f : 0.0f;
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float xi = (i < jj) ? 0.0f : acc[i];
                    acc[i] = xi;
#pragma unroll
                    for (int r = i + 1; r < 16; ++r) acc[r] -= Lb[r * 65 + i] * xi;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Nm[(16 * a + r) * 65 + 16 * a + jj] = acc[r];
            }
            __syncthreads();
#pragma unroll 1
            for (int wave = 1; wave < 4; ++wave) {
                // wave w computes the blocks N_{a, a-w}, one warp per block
                if (warp < 4 - wave) {
                    const int a = warp + wave, b = a - wave;
                    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    for (int cc = b; cc < a; ++cc) {
                        warp_gemm16(acc, Lm, 16 * a, 16 * cc, Nm, 16 * cc, 16 * b, lane);
                    }
                    warp_store16(acc, Ms, 16 * warp, 0, 1.0f, lane);
                    __syncwarp();
                    float acc2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
                    warp_gemm16(acc2, Nm, 16 * a, 16 * a, Ms, 16 * warp, 0, lane);
                    warp_store16(acc2, Nm, 16 * a, 16 * b, -1.0f, lane);
                }
                __syncthreads();
            }
            // Tm[r][i] = N[r][i] beta_i (lower triangle), bf16, rows of 64 -> K-major B tile
            {
                const int r = tid >> 3, i0 = (tid & 7) * 8;  // 512 chunks of 8 values
                uint4 w;
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int i = i0 + u;
                    v[u] = i <= r ? Nm[r * 65 + i] * s_beta[i] : 0.0f;
                }
                w.x = pack_bf16x2(v[0], v[1]); w.y = pack_bf16x2(v[2], v[3]);
                w.z = pack_bf16x2(v[4], v[5]); w.w = pack_bf16x2(v[6], v[7]);
                *reinterpret_cast<uint4*>(sm + OFF_TM + sw128(r, 2 * i0)) = w;
            }
        }
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
            const uint32_t idw = idesc_bf16(128, 64, 0, 0);
            const uint32_t idu = idesc_bf16(128, 64, 1, 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t bT = smem_desc(smem_base + OFF_TM + kk * 32, 16, 1024);
                const uint64_t aK = smem_desc(smem_base + OFF_KP + kk * 32, 16, 1024);
                mma_bf16(tbase + TM_W, aK, bT, idw, kk > 0);
                const uint64_t aV = smem_desc(smem_base + OFF_V + kk * 2048, 8192, 1024);
                mma_bf16(tbase + TM_U, aV, bT, idu, kk > 0);
            }
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

        // ---------------- P6: W^T -> bf16 operand (row c = lane, 16 tokens per warp) ----------------
        {
            uint32_t r[16];
            tmem_ld16(tbase + lane_base + TM_W + 16 * sub, r);
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
            store_row16(sm + OFF_WT, 32 * qd + lane, 32 * sub, v);
        }
        fence_proxy_async();
        cta_sync_tc();

        // ---------------- P7: U^T += S^T (-W^T),  O = Q+ S ----------------
        if (tid == 0) {
            const uint32_t idu = idesc_bf16(128, 64, 0, 1, /*neg_b=*/1);
            const uint32_t ido = idesc_bf16(64, 128, 1, 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t aS =
                    smem_desc(smem_base + OFF_ST + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                const uint64_t bW = smem_desc(smem_base + OFF_WT + kk * 2048, 16384, 1024);
                mma_bf16(tbase + TM_U, aS, bW, idu, 1);
            }
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t aQ = smem_desc(smem_base + OFF_QP + kk * 2048, 16384, 1024);
                const uint64_t bS =
                    smem_desc(smem_base + OFF_ST + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
                mma_bf16(tbase + TM_O, aQ, bS, ido, kk > 0);
            }
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

        // ---------------- P8: U^T -> bf16 operand (row j = lane, 16 tokens per warp) ----------------
        {
            uint32_t r[16];
            tmem_ld16(tbase + lane_base + TM_U + 16 * sub, r);
            tmem_wait_ld();
            float v[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
            store_row16(sm + OFF_UT, 32 * qd + lane, 32 * sub, v);
        }
        fence_proxy_async();
        cta_sync_tc();

        // ---------------- P9: O += Aqk U,  S^T += U^T Kend ----------------
        if (tid == 0) {
            const uint32_t ido = idesc_bf16(64, 128, 0, 0);
            const uint32_t ids = idesc_bf16(128, 128, 0, 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t aA = smem_desc(smem_base + OFF_AQK + kk * 32, 16, 1024);
                const uint64_t bU = smem_desc(smem_base + OFF_UT + kk * 32, 16, 1024);
                mma_bf16(tbase + TM_O, aA, bU, ido, 1);
                const uint64_t aU = smem_desc(smem_base + OFF_UT + kk * 32, 16, 1024);
                const uint64_t bK = smem_desc(smem_base + OFF_KE + kk * 32, 16, 1024);
                mma_bf16(tbase + TM_S, aU, bK, ids, 1);
            }
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
        // O (M = 64 tokens) sits in TMEM lanes 32q .. 32q+15 for tokens
        // 16q .. 16q+15; each warp stores 32 value columns of its 16 tokens.
        {
            uint32_t r0[16], r1[16];
            tmem_ld16(tbase + lane_base + TM_O + 32 * sub, r0);
            tmem_ld16(tbase + lane_base + TM_O + 32 * sub + 16, r1);
            tmem_wait_ld();
            const int rtok = 16 * qd + lane;
            if (lane < 16 && rtok < L) {
                uint4 w[4];
                uint32_t* wp = reinterpret_cast<uint32_t*>(w);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    wp[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
                    wp[8 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
                }
                uint4* dst = reinterpret_cast<uint4*>(o_g + ((size_t)(t0 + rtok) * H + h) * D + 32 * sub);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = w[i];
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

    // ---- final state: TMEM S^T -> final_state (coalesced along j) ----
    if (!abort_flag && p.final_state) {
        const int j = 32 * qd + lane;
        const uint32_t taddr = tbase + lane_base + TM_S;
#pragma unroll 1
        for (int cb = 32 * sub; cb < 32 * sub + 32; cb += 16) {
            uint32_t r[16];
            tmem_ld16(taddr + cb, r);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                p.final_state[state_off + (size_t)(cb + i) * D + j] = __uint_as_float(r[i]);
            }
        }
    }
    cta_sync_tc();
    if (warp == 0) {
        tmem_dealloc(tbase, TMEM_COLS);
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

}  // namespace

size_t chunked_workspace_bytes(int32_t N, int32_t H) {
    return 256 + (size_t)N * H * sizeof(int32_t);
}

cudaError_t launch_chunked_prefill(const ChunkedParams& p, cudaStream_t stream) {
    ChunkedArgs args;
    memset(&args, 0, sizeof(args));
    args.p = p;
    if (!make_map(&args.tm_q, p.q, p.total_T, p.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&args.tm_k, p.k, p.total_T, p.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&args.tm_z, p.z, p.total_T, p.H, 128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&args.tm_v, p.v, p.total_T, p.H, 64, CU_TENSOR_MAP_SWIZZLE_128B)) {
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

}  // namespace kda
