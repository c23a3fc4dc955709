// kda_chunk_phases.cuh -- the phases of one 64-token chunk of the chunked KDA
// prefill, shared by the single-pass kernel and the split (producer /
// consumer) kernel in kda_prefill_sm103.cu.
//
// Algebra per chunk (start state S0, d_k = d_v = 128, gamma_r = inclusive
// cumulative g), derived by unrolling the recurrence of "Kimi K3 Open Weights:
// What Is Actually New In Its 2.8 Trillion Parameter Architecture", section 1:
//   Akk[r,i] = beta_r <k_r e^{gamma_r - gamma_i}, k_i>   (i < r)
//   Aqk[r,i] =        <q_r e^{gamma_r - gamma_i}, k_i>   (i <= r)
//   Tm       = (I + Akk)^-1 Diag(beta)                    (UT solve, fp32)
//   U        = Tm V - (Tm K+) S0,    K+ = k * e^{gamma}
//   O        = Q+ S0 + Aqk U,        Q+ = q * e^{gamma}  (computed as O^T)
//   S_next   = Diag(e^{gamma_C}) S0 + Kend^T U,   Kend = k * e^{gamma_C - gamma}
// The Gram products use one reference point per 16-token block a (rho_a =
// gamma at the end of the previous block): the query/key side is scaled by
// e^{gamma_r - rho_a} <= 1, the key side of the products with block a by
// e^{rho_a - gamma_i} (<= e^80 inside the block, <= 1 before it) -- the
// section's bounded-gate / 16-token-tile argument.
//
// Every function here is executed by all threads of the CTA (512 threads,
// 16 warps) unless its comment says otherwise; functions that contain a
// CTA barrier say so.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_chunked.h"
#include "sm103_ptx.cuh"

namespace kda {
namespace chunk {

using namespace sm103;

constexpr int C = 64;          // chunk length
constexpr int D = 128;         // head dim (d_k = d_v)
constexpr int kThreads = 512;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNormEps = 1e-6f;
constexpr int kStatusTimeout = 1;
constexpr int kStatusRecords = 2;   // more chunks than the chunk records hold

// ---- shared memory map of a chunk's intra work (byte offsets from a 1024-aligned base) ----
// Region 1 (48 KB): raw q, k, z tiles.
constexpr uint32_t OFF_RAWQ = 0;
constexpr uint32_t OFF_RAWK = 16384;
constexpr uint32_t OFF_RAWZ = 32768;
// Region 2 (96 KB): X~ and K~ (Gram operands); then S^T bf16, Aqk, Tm and the
// solve scratch; then W^T and U^T.
constexpr uint32_t OFF_XT = 49152;          // 2 N-blocks x [128 c][64 e]  (MN-major B)
constexpr uint32_t OFF_KT = 49152 + 32768;  // 4 M-blocks x [128 c][64 i] (MN-major A)
constexpr uint32_t OFF_ST = 49152;          // [2 atoms][128 j][64 c]     (K-major A)
constexpr uint32_t OFF_AQK = 81920;         // [64 r][64 i]               (K-major B)
constexpr uint32_t OFF_TM = 90112;          // [64 r][64 i]               (K-major B)
constexpr uint32_t OFF_AKK = 98304;         // fp32 [64][65]
constexpr uint32_t OFF_NMAT = 114944;       // fp32 [64][65]
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

// A published chunk (split mode): the operand tiles the state chain needs,
// laid out as the shared-memory tiles are, so one bulk copy loads it.
// Q+ and -W^T are adjacent MN-major N-blocks (one N = 128 B operand), and so
// are the K-major rows of Kend and Aqk (one N = 192 B operand).
constexpr uint32_t HO_QP = 0;        // Q+    bf16 [128 c][64 r]
constexpr uint32_t HO_WT = 16384;    // -W^T  bf16 [128 c][64 r]
constexpr uint32_t HO_KE = 32768;    // Kend  bf16 [128 c][64 i]
constexpr uint32_t HO_AQK = 49152;   // Aqk   bf16 [64 r][64 i]
constexpr uint32_t HO_TM = 57344;    // Tm    bf16 [64 r][64 i]
constexpr uint32_t HO_GAM = 65536;   // Gamma_C fp32 [128]
constexpr uint32_t HO_BYTES = 66048; // multiple of 256
// With the short convolutions fused (split kernel), a slot also carries the
// chunk's convolved v tile, as the consumer's V operand (two halves
// [64 i][64 j], 128-byte swizzle: the layout TMA gives the plain kernel).
constexpr uint32_t HO_V = 66560;
constexpr uint32_t HO_BYTES_CONV = HO_V + 16384;

// A chunk record (the training backward keeps one per (chunk, head)): the
// published tiles above, then K+ and the two matrices of the UT transform
// that the gradient assembly needs.  Every tile starts on a 1024-byte
// boundary, so a byte copy of it into 1024-aligned shared memory is a valid
// 128B-swizzled operand.
constexpr uint32_t REC_KP = 66560;    // K+    bf16 [128 c][64 i]
constexpr uint32_t REC_G = 82944;     // Gkk   bf16 [64 r][64 i]: <k_r e^{gamma_r - gamma_i}, k_i>, i < r
constexpr uint32_t REC_MINV = 91136;  // (I + Akk)^-1 bf16 [64 r][64 i] (lower, unit diagonal)
constexpr uint32_t REC_S0 = 99328;    // the chunk's start state S, bf16, per v-half [128 c][64 v]
constexpr uint32_t REC_BYTES = 132096; // multiple of 1024

// TMEM columns
constexpr uint32_t TM_S = 0;      // S^T  [128 j lanes][128 c]
constexpr uint32_t TM_G1 = 128;   // Gram blocks 3, 2
constexpr uint32_t TM_G2 = 192;   // Gram blocks 1, 0
constexpr uint32_t TM_W = 256;    // W^T  [128 c][64 r]
constexpr uint32_t TM_U = 320;    // U^T  [128 j][64 r]
constexpr uint32_t TM_O = 384;    // O^T  [128 j][64 r]
constexpr uint32_t TMEM_COLS = 512;

// Where the state-side phases find a chunk's operand tiles.
struct StateTiles {
    uint32_t wt;   // W^T  bf16 [128 c][64 r]  MN-major B
    uint32_t qp;   // Q+   bf16 [128 c][64 r]  MN-major B
    uint32_t ke;   // Kend bf16 [128 c][64 i]  K-major B
    uint32_t aqk;  // Aqk  bf16 [64 r][64 i]   K-major A
    uint32_t tm;   // Tm   bf16 [64 r][64 i]   K-major B
    uint32_t gam;  // Gamma_C fp32 [128]
    uint32_t v;    // V    bf16 2 x [64 i][64 j] MN-major A
    uint32_t st;   // S^T  bf16 [2 atoms][128 j][64 c] K-major (written by phase_state_epilogue)
    uint32_t ut;   // U^T  bf16 [128 j][64 i] K-major (written from TMEM TM_U)
};

__device__ __forceinline__ StateTiles local_tiles() {
    return StateTiles{OFF_WT, OFF_QP, OFF_KE, OFF_AQK, OFF_TM, OFF_GAM, OFF_V, OFF_ST, OFF_UT};
}

// Per-thread view of the CTA.
struct Ctx {
    uint8_t* sm;           // 1024-aligned dynamic shared memory
    uint32_t smem_base;    // its shared-window address
    uint32_t tbase;        // TMEM base address
    int tid, warp, lane;
    int qd;                // TMEM lane quadrant this warp may access (warp % 4)
    int sub;               // which of the four warps of that quadrant (warp / 4)
    uint32_t lane_base;    // (32 * qd) << 16
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

// A bounded wait gave up: the first one to do so records where (a nonzero
// code, the source line of the wait) in the status word, and the CTA leaves
// its loops.  Any nonzero status is reported as a timeout.
__device__ __forceinline__ void record_timeout(int32_t* status, volatile int* abort_flag,
                                               int site = kStatusTimeout) {
    atomicCAS(status, 0, site);
    *abort_flag = 1;
}

// ---------------------------------------------------------------- P1a
// Per-token L2 norms of the raw q, k tiles (4 tokens per warp).  Writes
// inv_q (times scale) and inv_k; tokens r >= L get 0.  No barrier.
__device__ __forceinline__ void phase_norms(const Ctx& x, int L, float scale, int l2norm) {
    const uint8_t* rq = x.sm + OFF_RAWQ;
    const uint8_t* rk = x.sm + OFF_RAWK;
    float* s_invq = reinterpret_cast<float*>(x.sm + OFF_INVQ);
    float* s_invk = reinterpret_cast<float*>(x.sm + OFF_INVK);
    float sq[4], sk[4];
#pragma unroll
    for (int tt = 0; tt < 4; ++tt) {
        const int r = x.warp * 4 + tt;
        const uint2 qv = *reinterpret_cast<const uint2*>(rq + r * 256 + x.lane * 8);
        const uint2 kv = *reinterpret_cast<const uint2*>(rk + r * 256 + x.lane * 8);
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
    if (x.lane < 4) {
        const int r = x.warp * 4 + x.lane;
        const float a = x.lane == 0 ? sq[0] : x.lane == 1 ? sq[1] : x.lane == 2 ? sq[2] : sq[3];
        const float b = x.lane == 0 ? sk[0] : x.lane == 1 ? sk[1] : x.lane == 2 ? sk[2] : sk[3];
        const bool valid = r < L;
        s_invq[r] = valid ? (l2norm ? rsqrtf(a + kNormEps) : 1.0f) * scale : 0.0f;
        s_invk[r] = valid ? (l2norm ? rsqrtf(b + kNormEps) : 1.0f) : 0.0f;
    }
}

// ---------------------------------------------------------------- P1b + P1c
// Gate, in-block decay products and the bf16 operand tiles X~, K~^(a), K+,
// Q+, Kend, plus Gamma_C = e^{gamma_C} (fp32, OFF_GAM).  Each thread owns one
// (channel c = tid % 128, 16-token block ab = tid / 128) unit.  Two halves:
// phase_prologue_gate (gate, alpha, block totals; raw q, k kept in the
// thread's registers) and, after a CTA barrier that also publishes the norms
// phase_norms wrote, phase_prologue_operands (the tiles).  The same thread
// must run both halves of its unit.
// kPub (split producer): Q+, Kend and Gamma_C go straight to the published
// chunk at `pub` (global memory) instead of shared memory, after the
// thread's shared-memory tiles and their proxy fence.
struct GateRegs {
    float qh[16], kh[16], al[16];
};

__device__ __forceinline__ void phase_prologue_gate(const Ctx& x, int L, float eA_log2,
                                                    GateRegs& gr) {
    uint8_t* sm = x.sm;
    float* s_tot = reinterpret_cast<float*>(sm + OFF_TOT);
    const int c = x.tid & (D - 1);   // channel
    const int ab = (x.tid >> 7) & 3; // token block: tokens 16ab .. 16ab+15
    float tot = 0.f;                 // block total of g, log2 units
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * ab + rr;
        const float qv = __bfloat162float(
            *reinterpret_cast<const __nv_bfloat16*>(sm + OFF_RAWQ + r * 256 + 2 * c));
        const float kv = __bfloat162float(
            *reinterpret_cast<const __nv_bfloat16*>(sm + OFF_RAWK + r * 256 + 2 * c));
        const float zv = __bfloat162float(
            *reinterpret_cast<const __nv_bfloat16*>(sm + OFF_RAWZ + r * 256 + 2 * c));
        // g = -5 sigmoid(e^A z) in log2 units; invalid tokens: g = 0
        const float sg = rcp_approx(1.0f + exp2_approx(-eA_log2 * zv));
        const float g = r < L ? -5.0f * kLog2e * sg : 0.0f;
        tot += g;
        gr.al[rr] = exp2_approx(g);
        gr.qh[rr] = qv;
        gr.kh[rr] = kv;
    }
    s_tot[ab * D + c] = tot;
}

template <bool kPub = false>
__device__ __forceinline__ void phase_prologue_operands(const Ctx& x, int L, GateRegs& gr,
                                                        uint8_t* pub = nullptr) {
    uint8_t* sm = x.sm;
    const float* s_invq = reinterpret_cast<const float*>(sm + OFF_INVQ);
    const float* s_invk = reinterpret_cast<const float*>(sm + OFF_INVK);
    const float* s_tot = reinterpret_cast<const float*>(sm + OFF_TOT);
    float* s_gam = kPub ? reinterpret_cast<float*>(pub + HO_GAM)
                        : reinterpret_cast<float*>(sm + OFF_GAM);
    uint8_t* qp_tile = kPub ? pub + HO_QP : sm + OFF_QP;
    uint8_t* ke_tile = kPub ? pub + HO_KE : sm + OFF_KE;
    const int c = x.tid & (D - 1);
    const int ab = (x.tid >> 7) & 3;
    float* qh = gr.qh;
    float* kh = gr.kh;
    const float* al = gr.al;
    // the norms (written before the barrier) are applied now
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        qh[rr] *= s_invq[16 * ab + rr];
        kh[rr] *= s_invk[16 * ab + rr];
    }
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
    uint32_t qp_w[8];
    if (kPub) {
#pragma unroll
        for (int i = 0; i < 8; ++i) qp_w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    } else {
        store_row16(qp_tile, c, 32 * ab, v);
    }
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
    uint32_t ke_w[8];
    if (kPub) {
#pragma unroll
        for (int i = 0; i < 8; ++i) ke_w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    } else {
        store_row16(ke_tile, c, 32 * ab, v);
    }
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
    if (kPub) {
        // shared-memory tiles before the tensor core reads them; then the
        // published tiles (global stores the fence need not wait for)
        fence_proxy_async();
        uint4* q4 = reinterpret_cast<uint4*>(qp_tile + sw128(c, 32 * ab));
        uint4* q5 = reinterpret_cast<uint4*>(qp_tile + sw128(c, 32 * ab + 16));
        uint4* k4 = reinterpret_cast<uint4*>(ke_tile + sw128(c, 32 * ab));
        uint4* k5 = reinterpret_cast<uint4*>(ke_tile + sw128(c, 32 * ab + 16));
        *q4 = make_uint4(qp_w[0], qp_w[1], qp_w[2], qp_w[3]);
        *q5 = make_uint4(qp_w[4], qp_w[5], qp_w[6], qp_w[7]);
        *k4 = make_uint4(ke_w[0], ke_w[1], ke_w[2], ke_w[3]);
        *k5 = make_uint4(ke_w[4], ke_w[5], ke_w[6], ke_w[7]);
    }
}


// Both halves with the barrier between them; after_gate() runs right after
// the barrier (every thread).
struct NoHook {
    __device__ void operator()() const {}
};
template <bool kPub = false, typename Hook = NoHook>
__device__ __forceinline__ void phase_prologue(const Ctx& x, int L, float eA_log2,
                                               uint8_t* pub = nullptr,
                                               Hook after_gate = Hook()) {
    GateRegs gr;
    phase_prologue_gate(x, L, eA_log2, gr);
    __syncthreads();
    after_gate();
    phase_prologue_operands<kPub>(x, L, gr, pub);
}

// ---------------------------------------------------------------- P2 (one thread)
__device__ __forceinline__ void issue_gram(const Ctx& x) {
    const uint32_t idg = idesc_bf16(128, 64, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t a1 = smem_desc(x.smem_base + OFF_KT + kk * 2048, 16384, 1024);
        const uint64_t b1 = smem_desc(x.smem_base + OFF_XT + kk * 2048, 16384, 1024);
        mma_bf16(x.tbase + TM_G1, a1, b1, idg, kk > 0);
        const uint64_t a2 = smem_desc(x.smem_base + OFF_KT + 32768 + kk * 2048, 16384, 1024);
        const uint64_t b2 = smem_desc(x.smem_base + OFF_XT + 16384 + kk * 2048, 16384, 1024);
        mma_bf16(x.tbase + TM_G2, a2, b2, idg, kk > 0);
    }
}

// ---------------------------------------------------------------- P3a (warps 0-7)
// Gram -> Akk (fp32, beta-scaled, strictly lower) and Aqk (bf16 tile, lower).
// Warps 0-3: blocks 3 (lanes 0-63) and 2 (lanes 64-127) of TM_G1; warps 4-7:
// blocks 1 and 0 of TM_G2.
// kPub: Aqk goes straight to the published chunk at `pub`.
template <bool kPub = false>
__device__ __forceinline__ void phase_gram_epilogue(const Ctx& x, uint8_t* pub = nullptr) {
    uint8_t* aqk_tile = kPub ? pub + HO_AQK : x.sm + OFF_AQK;
    const float* s_beta = reinterpret_cast<const float*>(x.sm + OFF_BETA);
    float* akk = reinterpret_cast<float*>(x.sm + OFF_AKK);
    const int g = x.warp >> 2;
    const int qd = x.qd;
    const int blk = g == 0 ? (qd < 2 ? 3 : 2) : (qd < 2 ? 1 : 0);
    const uint32_t col = (g == 0 ? TM_G1 : TM_G2) + (qd < 2 ? 0 : 32);
    const int i = (qd < 2 ? 32 * qd : 32 * (qd - 2)) + x.lane;
    uint32_t vq[16], vk[16];
    tmem_ld16(x.tbase + x.lane_base + col, vq);
    tmem_ld16(x.tbase + x.lane_base + col + 16, vk);
    tmem_wait_ld();
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * blk + rr;
        const float aq = i <= r ? __uint_as_float(vq[rr]) : 0.0f;
        const float ak = i < r ? s_beta[r] * __uint_as_float(vk[rr]) : 0.0f;
        akk[r * 65 + i] = ak;
        *reinterpret_cast<__nv_bfloat16*>(aqk_tile + sw128(r, 2 * i)) =
            __float2bfloat16_rn(aq);
    }
}

// ---------------------------------------------------------------- P3b
// S^T (TMEM, fp32) -> bf16 A-operand tile at st_tile, then S^T *= Gamma_C in
// TMEM.  Warps with sub in [sub0, sub0 + nsub) take part; each covers
// 128 / nsub columns of its lane quadrant.
__device__ __forceinline__ void phase_state_epilogue(const Ctx& x, const float* gam,
                                                     uint32_t st_tile, int sub0, int nsub) {
    const int part = x.sub - sub0;
    if (part < 0 || part >= nsub) {
        return;
    }
    const int ncol = D / nsub;
    const int j = 32 * x.qd + x.lane;
    const uint32_t taddr = x.tbase + x.lane_base + TM_S;
#pragma unroll 1
    for (int cb = part * ncol; cb < (part + 1) * ncol; cb += 32) {
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
        store_row16(x.sm + st_tile + (cb / 64) * 16384, j, 2 * (cb % 64), v0);
        store_row16(x.sm + st_tile + (cb / 64) * 16384, j, 2 * (cb % 64) + 32, v1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            r0[i] = __float_as_uint(v0[i] * gam[cb + i]);
            r1[i] = __float_as_uint(v1[i] * gam[cb + 16 + i]);
        }
        tmem_st16(taddr + cb, r0);
        tmem_st16(taddr + cb + 16, r1);
    }
    tmem_wait_st();
}

// ---------------------------------------------------------------- split consumer
// The split kernel's consumer keeps the bf16 copies of S^T and U^T that feed
// the tensor core in TMEM (A operands read from TMEM: lane = row, two K
// elements per column) and places its accumulators so that one instruction
// computes two products: [O^T | U^T] += S^T [Q+^T | -W^T] (N = 128) and
// [S^T | O^T] += U^T [Kend ; Aqk] (N = 192).
constexpr uint32_t TC_S = 0;      // S^T  fp32 [128 j][128 c]
constexpr uint32_t TC_O = 128;    // O^T  fp32 [128 j][64 r]
constexpr uint32_t TC_U = 192;    // U^T  fp32 [128 j][64 r]
constexpr uint32_t TC_SB = 256;   // S^T  bf16, 64 columns
constexpr uint32_t TC_UB = 320;   // U^T  bf16, 32 columns

// S^T (TMEM, fp32) -> bf16 at TC_SB, and S^T *= Gamma in the same pass (the
// next chunk's products read the bf16 copy of the undecayed state and
// accumulate onto the decayed one); all 16 warps, 32 c each.  No barrier.
// With `dump` (global memory) the bf16 state also goes there as an operand
// tile S [c][v]: v-half v / 64 at 16384 (v / 64), row c, 128-byte swizzle.
__device__ __forceinline__ void phase_state_to_tmem_decay(const Ctx& x, const float* gam,
                                                          uint8_t* dump = nullptr) {
    const int cb = 32 * x.sub;
    const uint32_t taddr = x.tbase + x.lane_base + TC_S + cb;
    uint32_t r0[16], r1[16];
    tmem_ld16(taddr, r0);
    tmem_ld16(taddr + 16, r1);
    tmem_wait_ld();
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w[i] = pack_bf16x2(__uint_as_float(r0[2 * i]), __uint_as_float(r0[2 * i + 1]));
        w[8 + i] = pack_bf16x2(__uint_as_float(r1[2 * i]), __uint_as_float(r1[2 * i + 1]));
    }
    tmem_st16(x.tbase + x.lane_base + TC_SB + cb / 2, w);
    if (dump) {
        const int v = 32 * x.qd + x.lane;
        uint8_t* half = dump + (v >> 6) * 16384;
        const uint32_t vb = 2 * (v & 63);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const uint32_t pr = w[i >> 1];
            *reinterpret_cast<uint16_t*>(half + sw128(cb + i, vb)) =
                (i & 1) ? (uint16_t)(pr >> 16) : (uint16_t)(pr & 0xffffu);
        }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        r0[i] = __float_as_uint(__uint_as_float(r0[i]) * gam[cb + i]);
        r1[i] = __float_as_uint(__uint_as_float(r1[i]) * gam[cb + 16 + i]);
    }
    tmem_st16(taddr, r0);
    tmem_st16(taddr + 16, r1);
    tmem_wait_st();
}

// O^T (TMEM lane j, columns r0 .. r0 + 15 of this warp) -> 8 registers of
// bf16 pairs, then O^T = 0 for the next chunk's accumulation.  The global
// stores follow later (phase_ot_store), off the chunk's critical path.  No
// barrier.
__device__ __forceinline__ void phase_ot_take(const Ctx& x, uint32_t (&ob)[8]) {
    const uint32_t taddr = x.tbase + x.lane_base + TC_O + 16 * x.sub;
    uint32_t r[16];
    tmem_ld16(taddr, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        ob[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = 0u;
    tmem_st16(taddr, r);
    tmem_wait_st();
}

// The values phase_ot_take kept -> o (bf16): this warp's 16 tokens of its 32
// value columns; for a token the warp's lanes cover 64 contiguous bytes of o.
__device__ __forceinline__ void phase_ot_store(const Ctx& x, __nv_bfloat16* o_g, int64_t t0,
                                               int L, int h, int H, const uint32_t (&ob)[8]) {
    const int j = 32 * x.qd + x.lane;
    const int r0 = 16 * x.sub;
    uint16_t* dst = reinterpret_cast<uint16_t*>(o_g + ((size_t)(t0 + r0) * H + h) * D + j);
    const size_t row = (size_t)H * D;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (r0 + i < L) {
            dst[i * row] = (uint16_t)((i & 1) ? (ob[i >> 1] >> 16) : (ob[i >> 1] & 0xffffu));
        }
    }
}

// U^T (TMEM, fp32) -> bf16 at TC_UB; all 16 warps, 16 r each.  No barrier.
__device__ __forceinline__ void phase_u_to_tmem(const Ctx& x) {
    uint32_t r[16];
    tmem_ld16(x.tbase + x.lane_base + TC_U + 16 * x.sub, r);
    tmem_wait_ld();
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        w[i] = pack_bf16x2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1]));
    }
    tmem_st8(x.tbase + x.lane_base + TC_UB + 8 * x.sub, w);
    tmem_wait_st();
}

// (one thread) O^T = 0 in TMEM is the caller's; U'^T = V^T Tm^T into TC_U.
__device__ __forceinline__ void issue_u_prime_tc(const Ctx& x, const StateTiles& st) {
    const uint32_t idu = idesc_bf16(128, 64, 1, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bT = smem_desc(x.smem_base + st.tm + kk * 32, 16, 1024);
        const uint64_t aV = smem_desc(x.smem_base + st.v + kk * 2048, 8192, 1024);
        mma_bf16(x.tbase + TC_U, aV, bT, idu, kk > 0);
    }
}

// (one thread) [O^T | U^T] += S^T [Q+^T | -W^T]: st.qp holds Q+ then -W^T.
__device__ __forceinline__ void issue_ou_tc(const Ctx& x, const StateTiles& st) {
    const uint32_t id = idesc_bf16(128, 128, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t b = smem_desc(x.smem_base + st.qp + kk * 2048, 16384, 1024);
        mma_bf16_ta(x.tbase + TC_O, x.tbase + TC_SB + kk * 8, b, id, 1);
    }
}

// (one thread) [S^T | O^T] += U^T [Kend ; Aqk]: st.ke holds Kend then Aqk rows.
__device__ __forceinline__ void issue_so_tc(const Ctx& x, const StateTiles& st) {
    const uint32_t id = idesc_bf16(128, 192, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t b = smem_desc(x.smem_base + st.ke + kk * 32, 16, 1024);
        mma_bf16_ta(x.tbase + TC_S, x.tbase + TC_UB + kk * 8, b, id, 1);
    }
}

// ---------------------------------------------------------------- P4
// UT solve  Tm = (I + Akk)^-1 Diag(beta) -> bf16 tile at OFF_TM.
// N = (I + L)^-1, L = Akk strictly lower, in 16x16 blocks:
//   diagonal blocks N_aa by right-looking forward substitution (one column
//   per thread);
//   wave 0: B_ac = N_aa L_ac for the six blocks below the diagonal (one warp
//   each, written over L_ac, which only that warp reads);
//   waves 1..3: N_ab = -sum_{c=b}^{a-1} B_ac N_cb for a - b = wave.
// All products are warp-level tf32 MMAs.  Contains CTA barriers; the caller
// must have synchronised after phase_gram_epilogue.
// kPub: Tm is also copied to the published chunk at `pub`.
template <bool kPub = false>
__device__ __forceinline__ void phase_solve(const Ctx& x, uint8_t* pub = nullptr) {
    const float* s_beta = reinterpret_cast<const float*>(x.sm + OFF_BETA);
    float* Lm = reinterpret_cast<float*>(x.sm + OFF_AKK);
    float* Nm = reinterpret_cast<float*>(x.sm + OFF_NMAT);
    if (x.tid < 64) {
        const int a = x.tid >> 4, jj = x.tid & 15;
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
    if (x.warp < 6) {
        // (a, c) = (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
        const int a = x.warp < 1 ? 1 : x.warp < 3 ? 2 : 3;
        const int c = x.warp < 1 ? 0 : x.warp < 3 ? x.warp - 1 : x.warp - 3;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        warp_gemm16(acc, Nm, 16 * a, 16 * a, Lm, 16 * a, 16 * c, x.lane);
        warp_store16(acc, Lm, 16 * a, 16 * c, 1.0f, x.lane);
    }
    __syncthreads();
#pragma unroll 1
    for (int wave = 1; wave < 4; ++wave) {
        // wave w computes the blocks N_{a, a-w}, one warp per block
        if (x.warp < 4 - wave) {
            const int a = x.warp + wave, b = x.warp;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int cc = b; cc < a; ++cc) {
                warp_gemm16(acc, Lm, 16 * a, 16 * cc, Nm, 16 * cc, 16 * b, x.lane);
            }
            warp_store16(acc, Nm, 16 * a, 16 * b, -1.0f, x.lane);
        }
        __syncthreads();
    }
    // Tm[r][i] = N[r][i] beta_i (lower triangle), bf16, rows of 64 -> K-major B tile
    {
        const int r = x.tid >> 3, i0 = (x.tid & 7) * 8;  // 512 chunks of 8 values
        uint4 w;
        float v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u;
            v[u] = i <= r ? Nm[r * 65 + i] * s_beta[i] : 0.0f;
        }
        w.x = pack_bf16x2(v[0], v[1]); w.y = pack_bf16x2(v[2], v[3]);
        w.z = pack_bf16x2(v[4], v[5]); w.w = pack_bf16x2(v[6], v[7]);
        *reinterpret_cast<uint4*>(x.sm + OFF_TM + sw128(r, 2 * i0)) = w;
        if (kPub) {
            *reinterpret_cast<uint4*>(pub + HO_TM + sw128(r, 2 * i0)) = w;
        }
    }
}

// ---------------------------------------------------------------- P5 (one thread)
// W^T = K+^T Tm^T  (TMEM TM_W).
__device__ __forceinline__ void issue_w(const Ctx& x) {
    const uint32_t idw = idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bT = smem_desc(x.smem_base + OFF_TM + kk * 32, 16, 1024);
        const uint64_t aK = smem_desc(x.smem_base + OFF_KP + kk * 32, 16, 1024);
        mma_bf16(x.tbase + TM_W, aK, bT, idw, kk > 0);
    }
}

// U'^T = V^T Tm^T  (TMEM TM_U), operands at the given tiles.
__device__ __forceinline__ void issue_u_prime(const Ctx& x, const StateTiles& st) {
    const uint32_t idu = idesc_bf16(128, 64, 1, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bT = smem_desc(x.smem_base + st.tm + kk * 32, 16, 1024);
        const uint64_t aV = smem_desc(x.smem_base + st.v + kk * 2048, 8192, 1024);
        mma_bf16(x.tbase + TM_U, aV, bT, idu, kk > 0);
    }
}

// ---------------------------------------------------------------- P6 / P8
// A 128-lane x 64-token fp32 TMEM block -> bf16 tile rows (lane = row), 16
// tokens per warp (all 16 warps).  No barrier.
__device__ __forceinline__ void phase_tile_from_tmem(const Ctx& x, uint32_t tm_col, uint32_t tile) {
    uint32_t r[16];
    tmem_ld16(x.tbase + x.lane_base + tm_col + 16 * x.sub, r);
    tmem_wait_ld();
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
    store_row16(x.sm + tile, 32 * x.qd + x.lane, 32 * x.sub, v);
}

// ---------------------------------------------------------------- P7 (one thread)
// U^T += S^T (-W^T)   (S^T bf16 tile at st.st).
__device__ __forceinline__ void issue_u(const Ctx& x, const StateTiles& st) {
    const uint32_t idu = idesc_bf16(128, 64, 0, 1, /*neg_b=*/1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t aS =
            smem_desc(x.smem_base + st.st + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        const uint64_t bW = smem_desc(x.smem_base + st.wt + kk * 2048, 16384, 1024);
        mma_bf16(x.tbase + TM_U, aS, bW, idu, 1);
    }
}

// O^T = S^T Q+^T   (S^T bf16 tile at st.st; Q+ [128 c][64 r] is the MN-major B).
__device__ __forceinline__ void issue_o(const Ctx& x, const StateTiles& st) {
    const uint32_t ido = idesc_bf16(128, 64, 0, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t aS =
            smem_desc(x.smem_base + st.st + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024);
        const uint64_t bQ = smem_desc(x.smem_base + st.qp + kk * 2048, 16384, 1024);
        mma_bf16(x.tbase + TM_O, aS, bQ, ido, kk > 0);
    }
}

__device__ __forceinline__ void issue_uo(const Ctx& x, const StateTiles& st) {
    issue_u(x, st);
    issue_o(x, st);
}

// ---------------------------------------------------------------- P9 (one thread)
// S^T += U^T Kend (first: the next chunk waits for it);  O^T += U^T Aqk^T
// (U^T bf16 tile at st.ut; Kend [128 c][64 i] and Aqk [64 r][64 i] K-major B).
__device__ __forceinline__ void issue_os(const Ctx& x, const StateTiles& st) {
    const uint32_t ids = idesc_bf16(128, 128, 0, 0);
    const uint32_t ido = idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t aU = smem_desc(x.smem_base + st.ut + kk * 32, 16, 1024);
        const uint64_t bK = smem_desc(x.smem_base + st.ke + kk * 32, 16, 1024);
        mma_bf16(x.tbase + TM_S, aU, bK, ids, 1);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t aU = smem_desc(x.smem_base + st.ut + kk * 32, 16, 1024);
        const uint64_t bA = smem_desc(x.smem_base + st.aqk + kk * 32, 16, 1024);
        mma_bf16(x.tbase + TM_O, aU, bA, ido, 1);
    }
}

// ---------------------------------------------------------------- P10
// O^T (TMEM lane j = value column, column r = token) -> o (bf16).  Each warp
// stores 16 tokens of its 32 value columns; for a token the warp's lanes
// cover 64 contiguous bytes of o.  No barrier.
__device__ __forceinline__ void phase_o_epilogue(const Ctx& x, __nv_bfloat16* o_g, int64_t t0,
                                                 int L, int h, int H) {
    const int j = 32 * x.qd + x.lane;
    const int r0 = 16 * x.sub;
    uint32_t r[16];
    tmem_ld16(x.tbase + x.lane_base + TM_O + r0, r);
    tmem_wait_ld();
    __nv_bfloat16* dst = o_g + ((size_t)(t0 + r0) * H + h) * D + j;
    const size_t row = (size_t)H * D;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        if (r0 + i < L) {
            dst[i * row] = __float2bfloat16_rn(__uint_as_float(r[i]));
        }
    }
}

// ---------------------------------------------------------------- state checkpoints
// Index of sequence n's first checkpoint: the sum over earlier sequences of
// floor(length / interval).  `len_of(m)` gives sequence m's length; every
// thread of the CTA calls this (one CTA barrier inside, two with the reset).
template <typename LenOf>
__device__ __forceinline__ int64_t ckpt_base(int n, int interval, LenOf len_of, int* s_acc) {
    if (threadIdx.x == 0) {
        *s_acc = 0;
    }
    __syncthreads();
    int part = 0;
    for (int m = threadIdx.x; m < n; m += blockDim.x) {
        part += len_of(m) / interval;
    }
    if (part) {
        atomicAdd(s_acc, part);
    }
    __syncthreads();
    const int64_t r = *s_acc;
    __syncthreads();
    return r;
}

// ---------------------------------------------------------------- state load / store
// initial state -> TMEM: lane j holds column j of S (S^T row j).
__device__ __forceinline__ void load_state(const Ctx& x, const float* src) {
    const int j = 32 * x.qd + x.lane;
    const uint32_t taddr = x.tbase + x.lane_base + TM_S;
#pragma unroll 1
    for (int cb = 32 * x.sub; cb < 32 * x.sub + 32; cb += 16) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float v = src ? __ldg(src + (size_t)(cb + i) * D + j) : 0.0f;
            r[i] = __float_as_uint(v);
        }
        tmem_st16(taddr + cb, r);
    }
    tmem_wait_st();
}

// TMEM S^T -> dst (coalesced along j).
__device__ __forceinline__ void store_state(const Ctx& x, float* dst) {
    const int j = 32 * x.qd + x.lane;
    const uint32_t taddr = x.tbase + x.lane_base + TM_S;
#pragma unroll 1
    for (int cb = 32 * x.sub; cb < 32 * x.sub + 32; cb += 16) {
        uint32_t r[16];
        tmem_ld16(taddr + cb, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) dst[(size_t)(cb + i) * D + j] = __uint_as_float(r[i]);
    }
}

}  // namespace chunk
}  // namespace kda
