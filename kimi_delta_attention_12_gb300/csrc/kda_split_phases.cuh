// kda_split_phases.cuh -- the producer side of the split chunked prefill
// (kda_split_kernel in kda_prefill_sm103.cu), run by two warp groups that
// work on consecutive tasks at once.
//
// A producer task is the state-independent part of one 64-token chunk of one
// (sequence, head) unit -- the algebra of kda_chunk_phases.cuh:
//   group A (warps 0-7): L2 norms, gate and per-block cumulative decay, the
//     bf16 operand tiles (X~, K~^(a), K+, and Q+, Kend, Gamma_C straight into
//     the chunk's ring slot), then one thread issues the Gram products;
//   group B (warps 8-15): the Gram epilogue (Akk fp32 in shared memory, Aqk
//     into the slot), the UT solve Tm = (I + Akk)^-1 Diag(beta) (Tm into the
//     slot), W^T = K+^T Tm^T on the tensor core and -W^T into the slot.
// Group A runs task j + 1 (and issues its Gram products into the other TMEM
// buffer) while group B finishes task j.  The two groups share no barrier:
// they hand the Gram accumulator, K+ and beta over through mbarriers (see
// the kernel), so each group synchronises with a named barrier of its own
// 256 threads.
//
// The Gram products are one M = 128 x N = 256 x K = 128 product: A = X~ (the
// q and k rows of the four 16-token blocks, [Q3 K3 Q2 K2 Q1 K1 Q0 K0], stored
// MN-major), B = the four key copies K~^(3), K~^(2), K~^(1), K~^(0) (MN-major
// 64-token blocks).  TMEM lane m is row m of X~, column 64 q + i is token i
// of copy 3 - q, so warp quadrant q reads the 64 columns that belong to its
// own rows (block a = 3 - q) and writes whole rows of Aqk and Akk.  Eight
// instructions instead of sixteen of N = 64: a tcgen05.mma at M = 128 costs
// about the same time for any N up to 192.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_chunk_phases.cuh"
#include "kda_conv_math.cuh"
#include "sm103_ptx.cuh"

namespace kda {
namespace split {

using namespace sm103;
using chunk::C;
using chunk::D;
using chunk::kLog2e;
using chunk::kNormEps;

// ---- producer shared memory (byte offsets from a 1024-aligned base) ----
constexpr uint32_t P_RAWQ = 0;          // raw q, k, z tiles [64 tok][128 ch] bf16 (TMA)
constexpr uint32_t P_RAWK = 16384;
constexpr uint32_t P_RAWZ = 32768;
constexpr uint32_t P_XT = 49152;        // X~ : 2 M-blocks [128 c][64 rows] MN-major A
constexpr uint32_t P_KT = 81920;        // K~ : 4 N-blocks [128 c][64 i] MN-major B
constexpr uint32_t P_KP = 147456;       // K+ : 2 buffers [128 c][64 i] K-major A (W)
constexpr uint32_t P_AKK = 180224;      // Akk fp32 [64][65]; after the solve Tm bf16 [64][64]
constexpr uint32_t P_TM = P_AKK;        //   (K-major B of W; Akk is dead by then)
constexpr uint32_t P_NMAT = 196864;     // (I + Akk)^-1 fp32 [64][65]
constexpr uint32_t P_INVQ = 213504;     // [64] scale / |q|
constexpr uint32_t P_INVK = 213760;     // [64] 1 / |k|
constexpr uint32_t P_BETA = 214016;     // 2 buffers [64] beta (0 past the chunk's end)
constexpr uint32_t P_TOT = 214528;      // [4][128] block totals of g (log2 units)
constexpr uint32_t P_END = 216576;

// TMEM columns of a producer: two buffers of 256 columns, task j in buffer
// j & 1 -- its Gram products, then (once the epilogue has read them) W^T in
// its first 64 columns -- so that group A can issue the next task's Gram
// products while group B still works on this one.  Offsets within a buffer:
constexpr uint32_t TG_G = 0;            // Gram: 256 columns
constexpr uint32_t TG_W = 0;            // W^T [128 c][64 r]
constexpr uint32_t kGramBufCols = 256;

constexpr int kGroupThreads = 256;
constexpr int kBarA = 1;                // named barrier of group A
constexpr int kBarB = 2;                // named barrier of group B

__device__ __forceinline__ void group_sync(int id) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(kGroupThreads) : "memory");
}

// group_sync that also returns whether any thread of the group passed true:
// a decision every thread of the group takes alike (a loop left on one
// thread's view of the abort flag would leave the others at the next barrier).
__device__ __forceinline__ bool group_sync_or(int id, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(kGroupThreads)
        : "memory");
    return r != 0;
}

// ---------------------------------------------------------- fused convolutions
// The short convolutions of kda_short_conv.cu (conv_step, the same arithmetic
// and rounding), fused into the producers: q and k in place in the raw tiles
// (group A, before the norms), v into the published chunk (group B).  The
// inputs before a chunk's first token are the previous chunk's last ones, or
// for a sequence's first chunk the rows of its conv state (zeros without one).

// Where a convolution finds a chunk's inputs.
struct ConvSrc {
    const float* w;            // taps [H][384][W] fp32
    const __nv_bfloat16* q;    // raw inputs [total_T][H][128]
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const __nv_bfloat16* st;   // conv states in [N][H][W-1][384], or null
    int R;                     // W - 1 (0 .. 3)
    bool silu;
    int H;
};

// Taps of channel ch (of the 384) of head h: w[0 .. R] (the rest 0).
__device__ __forceinline__ void conv_taps(const ConvSrc& cs, int h, int ch, float (&w)[4]) {
    const float* src = cs.w + ((size_t)h * 384 + ch) * (cs.R + 1);
#pragma unroll
    for (int j = 0; j < 4; ++j) w[j] = j <= cs.R ? __ldg(src + j) : 0.0f;
}

// Group A, step 1 (before a barrier of the group): thread lt takes channel
// c = lt % 128 of tokens 32 hb .. 32 hb + 31 (hb = lt / 128) of q and k; its
// window gets the R inputs before its first token (win[3 - R + r]: the r-th of
// them, oldest first), read before the thread ahead of it overwrites them.
__device__ __forceinline__ void a_conv_halo(const uint8_t* sm, int lt, const ConvSrc& cs,
                                            int64_t t0, int chunk, int n, int h,
                                            float (&wq)[3], float (&wk)[3]) {
    const int c = lt & (D - 1), hb = lt >> 7;
#pragma unroll
    for (int r = 0; r < 3; ++r) {
        wq[r] = 0.0f;
        wk[r] = 0.0f;
    }
    for (int r = 0; r < cs.R; ++r) {
        const int rel = 32 * hb - cs.R + r;   // token within the chunk (< 0: before it)
        float a = 0.0f, b = 0.0f;
        if (rel >= 0) {
            a = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16*>(sm + P_RAWQ + rel * 256 + 2 * c));
            b = __bfloat162float(
                *reinterpret_cast<const __nv_bfloat16*>(sm + P_RAWK + rel * 256 + 2 * c));
        } else if (chunk > 0) {
            const size_t o = ((size_t)(t0 + rel) * cs.H + h) * D + c;
            a = __bfloat162float(cs.q[o]);
            b = __bfloat162float(cs.k[o]);
        } else if (cs.st) {
            const size_t o = (((size_t)n * cs.H + h) * cs.R + (rel + cs.R)) * 384 + c;
            a = __bfloat162float(cs.st[o]);
            b = __bfloat162float(cs.st[o + D]);
        }
        wq[3 - cs.R + r] = a;
        wk[3 - cs.R + r] = b;
    }
}

template <int R>
__device__ __forceinline__ void a_conv_rows(uint8_t* sm, int c, int hb, const float (&tq)[4],
                                            const float (&tk)[4], float (&wq)[3],
                                            float (&wk)[3], bool silu) {
    __nv_bfloat16* rq = reinterpret_cast<__nv_bfloat16*>(sm + P_RAWQ);
    __nv_bfloat16* rk = reinterpret_cast<__nv_bfloat16*>(sm + P_RAWK);
#pragma unroll 4
    for (int j = 0; j < 32; ++j) {
        const int e = (32 * hb + j) * D + c;
        const float xq = __bfloat162float(rq[e]), xk = __bfloat162float(rk[e]);
        rq[e] = __float2bfloat16_rn(conv_step<R>(tq, wq, xq, silu));
        rk[e] = __float2bfloat16_rn(conv_step<R>(tk, wk, xk, silu));
        wq[0] = wq[1]; wq[1] = wq[2]; wq[2] = xq;
        wk[0] = wk[1]; wk[1] = wk[2]; wk[2] = xk;
    }
}

// Group A, step 2 (after that barrier): the thread's 32 outputs of q and k,
// rounded to bf16, over its inputs in the raw tiles.  No barrier.
__device__ __forceinline__ void a_conv_apply(uint8_t* sm, int lt, const ConvSrc& cs, int h,
                                             float (&wq)[3], float (&wk)[3]) {
    const int c = lt & (D - 1), hb = lt >> 7;
    float tq[4], tk[4];
    conv_taps(cs, h, c, tq);
    conv_taps(cs, h, D + c, tk);
    switch (cs.R) {
        case 0: a_conv_rows<0>(sm, c, hb, tq, tk, wq, wk, cs.silu); break;
        case 1: a_conv_rows<1>(sm, c, hb, tq, tk, wq, wk, cs.silu); break;
        case 2: a_conv_rows<2>(sm, c, hb, tq, tk, wq, wk, cs.silu); break;
        default: a_conv_rows<3>(sm, c, hb, tq, tk, wq, wk, cs.silu); break;
    }
}

template <int R>
__device__ __forceinline__ void b_conv_rows(uint8_t* tile, int c0, int tq, const float (&t0w)[4],
                                            const float (&t1w)[4], const uint32_t (&raw)[19],
                                            bool silu) {
    float w0[3], w1[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) {   // raw[r]: the input 3 - r tokens before the first
        w0[r] = chunk::bf16lo(raw[r]);
        w1[r] = chunk::bf16hi(raw[r]);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const float x0 = chunk::bf16lo(raw[3 + j]), x1 = chunk::bf16hi(raw[3 + j]);
        const uint32_t y = chunk::pack_bf16x2(conv_step<R>(t0w, w0, x0, silu),
                                              conv_step<R>(t1w, w1, x1, silu));
        *reinterpret_cast<uint32_t*>(tile + (c0 >> 6) * 8192 + sw128(16 * tq + j, 2 * (c0 & 63))) =
            y;
        w0[0] = w0[1]; w0[1] = w0[2]; w0[2] = x0;
        w1[0] = w1[1]; w1[1] = w1[2]; w1[2] = x1;
    }
}

// Group B: the chunk's convolved v into the published chunk's V tile (the
// consumer's operand layout).  Thread lt: channels c0 = 2 (lt % 64), c0 + 1
// of tokens 16 tq .. 16 tq + 15 (tq = lt / 64); its 16 + 3 input pairs are
// loaded first, all in flight at once.  Tokens at or past the chunk's end L
// read as 0.  No barrier.
__device__ __forceinline__ void b_conv_v(uint8_t* tile, int lt, const ConvSrc& cs, int64_t t0,
                                         int L, int chunk, int n, int h) {
    const int c0 = 2 * (lt & 63), tq = lt >> 6;
    uint32_t raw[19];
#pragma unroll
    for (int i = 0; i < 19; ++i) {
        const int rel = 16 * tq - 3 + i;   // token within the chunk
        uint32_t val = 0u;
        if (rel >= 0) {
            if (rel < L) {
                val = __ldg(reinterpret_cast<const uint32_t*>(
                    cs.v + ((size_t)(t0 + rel) * cs.H + h) * D + c0));
            }
        } else if (rel >= -cs.R) {
            if (chunk > 0) {
                val = __ldg(reinterpret_cast<const uint32_t*>(
                    cs.v + ((size_t)(t0 + rel) * cs.H + h) * D + c0));
            } else if (cs.st) {
                val = __ldg(reinterpret_cast<const uint32_t*>(
                    cs.st + (((size_t)n * cs.H + h) * cs.R + (rel + cs.R)) * 384 + 2 * D + c0));
            }
        }
        raw[i] = val;
    }
    float t0w[4], t1w[4];
    conv_taps(cs, h, 2 * D + c0, t0w);
    conv_taps(cs, h, 2 * D + c0 + 1, t1w);
    switch (cs.R) {
        case 0: b_conv_rows<0>(tile, c0, tq, t0w, t1w, raw, cs.silu); break;
        case 1: b_conv_rows<1>(tile, c0, tq, t0w, t1w, raw, cs.silu); break;
        case 2: b_conv_rows<2>(tile, c0, tq, t0w, t1w, raw, cs.silu); break;
        default: b_conv_rows<3>(tile, c0, tq, t0w, t1w, raw, cs.silu); break;
    }
}

// ---------------------------------------------------------------- group A
// Per-token L2 norms, 8 tokens per warp (lw = warp in the group).  Tokens
// r >= L get 0.  No barrier.
__device__ __forceinline__ void a_norms(uint8_t* sm, int lw, int lane, int L, float scale,
                                        int l2norm) {
    const uint8_t* rq = sm + P_RAWQ;
    const uint8_t* rk = sm + P_RAWK;
    float* s_invq = reinterpret_cast<float*>(sm + P_INVQ);
    float* s_invk = reinterpret_cast<float*>(sm + P_INVK);
    float sq[8], sk[8];
#pragma unroll
    for (int tt = 0; tt < 8; ++tt) {
        const int r = lw * 8 + tt;
        const uint2 qv = *reinterpret_cast<const uint2*>(rq + r * 256 + lane * 8);
        const uint2 kv = *reinterpret_cast<const uint2*>(rk + r * 256 + lane * 8);
        const float q0 = chunk::bf16lo(qv.x), q1 = chunk::bf16hi(qv.x);
        const float q2 = chunk::bf16lo(qv.y), q3 = chunk::bf16hi(qv.y);
        const float k0 = chunk::bf16lo(kv.x), k1 = chunk::bf16hi(kv.x);
        const float k2 = chunk::bf16lo(kv.y), k3 = chunk::bf16hi(kv.y);
        sq[tt] = q0 * q0 + q1 * q1 + q2 * q2 + q3 * q3;
        sk[tt] = k0 * k0 + k1 * k1 + k2 * k2 + k3 * k3;
    }
    // The 16 sums (8 tokens of q, then of k) over the 32 lanes, halving the
    // values at each step: at offset o a lane keeps the half of its values
    // that its lane bit o selects and adds the partner's copy of that half.
    // Afterwards lanes 2m and 2m + 1 hold sum number ((m >> 3) & 1) * 8 +
    // (m & 7) -- tensor bit 4 of the lane, token bits 3..1.
    float v16[16];
#pragma unroll
    for (int tt = 0; tt < 8; ++tt) {
        v16[tt] = sq[tt];
        v16[8 + tt] = sk[tt];
    }
#pragma unroll
    for (int off = 16, n = 16; off >= 2; off >>= 1, n >>= 1) {
        const bool hi = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = hi ? v16[n / 2 + i] : v16[i];
            const float send = hi ? v16[i] : v16[n / 2 + i];
            v16[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
    }
    const float tot = v16[0] + __shfl_xor_sync(0xffffffffu, v16[0], 1);
    if ((lane & 1) == 0) {
        const int r = lw * 8 + ((lane >> 1) & 7);
        const bool valid = r < L;
        if (lane & 16) {
            s_invk[r] = valid ? (l2norm ? rsqrtf(tot + kNormEps) : 1.0f) : 0.0f;
        } else {
            s_invq[r] = valid ? (l2norm ? rsqrtf(tot + kNormEps) : 1.0f) * scale : 0.0f;
        }
    }
}

// Gate of token block ab for channel c: alpha = 2^g, g = -5 log2(e)
// sigmoid(e^A z) (0 past the chunk's end); the block total of g -> P_TOT.
__device__ __forceinline__ void a_gate_block(uint8_t* sm, int c, int ab, int L, float eA_log2,
                                             float (&al)[16]) {
    float tot = 0.f;
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * ab + rr;
        const float zv = __bfloat162float(
            *reinterpret_cast<const __nv_bfloat16*>(sm + P_RAWZ + r * 256 + 2 * c));
        const float sg = chunk::rcp_approx(1.0f + chunk::exp2_approx(-eA_log2 * zv));
        const float g = r < L ? -5.0f * kLog2e * sg : 0.0f;
        tot += g;
        al[rr] = chunk::exp2_approx(g);
    }
    reinterpret_cast<float*>(sm + P_TOT)[ab * D + c] = tot;
}

// The operand tiles of token block ab for channel c, from its alpha (al, 16
// tokens) and the raw q, k in shared memory: X~ and K~^(a) (all a >= ab) for
// the Gram, K+ into kp, and Q+, Kend (and, for block 0, Gamma_C) straight
// into the published chunk at pub; with `rec` (a chunk record, which pub
// then points into) K+ goes to its REC_KP tile as well.  The arithmetic is
// that of chunk::phase_prologue_operands.
__device__ __forceinline__ void a_operands_block(uint8_t* sm, int c, int ab,
                                                 const float (&al)[16], uint8_t* kp,
                                                 uint8_t* pub, uint8_t* rec) {
    const float* s_invq = reinterpret_cast<const float*>(sm + P_INVQ);
    const float* s_invk = reinterpret_cast<const float*>(sm + P_INVK);
    const float* s_tot = reinterpret_cast<const float*>(sm + P_TOT);
    float t[4];
#pragma unroll
    for (int b = 0; b < 4; ++b) t[b] = s_tot[b * D + c];
    float rho[5];  // rho[b] = log2 decay before block b; rho[4] = chunk total
    rho[0] = 0.f;
#pragma unroll
    for (int b = 0; b < 4; ++b) rho[b + 1] = rho[b] + t[b];
    if (ab == 0) {
        reinterpret_cast<float*>(pub + chunk::HO_GAM)[c] = chunk::exp2_approx(rho[4]);
    }
    const float rho_a = ab == 0 ? rho[0] : ab == 1 ? rho[1] : ab == 2 ? rho[2] : rho[3];
    const float rho_a1 = ab == 0 ? rho[1] : ab == 1 ? rho[2] : ab == 2 ? rho[3] : rho[4];
    const float eRa = chunk::exp2_approx(rho_a);             // e^{rho_a}               <= 1
    const float cF = chunk::exp2_approx(rho_a - rho_a1);     // e^{-block total}        <= e^80
    const float eEnd = chunk::exp2_approx(rho[4] - rho_a1);  // e^{gamma_C - rho_{a+1}} <= 1

    // E_r = e^{gamma_r - rho_a} (running product of alpha), G_r = e^{rho_{a+1} - gamma_r}
    float G[16];
    G[15] = 1.0f;
#pragma unroll
    for (int rr = 14; rr >= 0; --rr) G[rr] = G[rr + 1] * al[rr + 1];
    float E[16];
    E[0] = al[0];
#pragma unroll
    for (int rr = 1; rr < 16; ++rr) E[rr] = E[rr - 1] * al[rr];

    // X~ M-blocks: 0 = [Q3 K3 Q2 K2], 1 = [Q1 K1 Q0 K0]
    const uint32_t mb = ab >= 2 ? 0u : 1u;
    const uint32_t e0 = (ab >= 2 ? (3 - ab) : (1 - ab)) * 32;
    uint8_t* xt = sm + P_XT + mb * 16384;
    float v[16];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const float qv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
            sm + P_RAWQ + (16 * ab + rr) * 256 + 2 * c));
        v[rr] = qv * s_invq[16 * ab + rr] * E[rr];
    }
    chunk::store_row16(xt, c, 2 * e0, v);
    // Q+ = q e^{gamma} -> slot
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = chunk::pack_bf16x2(v[2 * i] * eRa, v[2 * i + 1] * eRa);
    *reinterpret_cast<uint4*>(pub + chunk::HO_QP + sw128(c, 32 * ab)) =
        make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(pub + chunk::HO_QP + sw128(c, 32 * ab + 16)) =
        make_uint4(w[4], w[5], w[6], w[7]);
    float kh[16];
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) {
        const float kv = __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
            sm + P_RAWK + (16 * ab + rr) * 256 + 2 * c));
        kh[rr] = kv * s_invk[16 * ab + rr];
        v[rr] = kh[rr] * E[rr];
    }
    chunk::store_row16(xt, c, 2 * (e0 + 16), v);
    // K+ = k e^{gamma}
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) v[rr] *= eRa;
    chunk::store_row16(kp, c, 32 * ab, v);
    if (rec) {
        chunk::store_row16(rec + chunk::REC_KP, c, 32 * ab, v);
    }
    // key side with the end-of-block reference: k e^{rho_{a+1} - gamma_r} <= 1
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) G[rr] *= kh[rr];
    // Kend = k e^{gamma_C - gamma} -> slot
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = chunk::pack_bf16x2(G[2 * i] * eEnd, G[2 * i + 1] * eEnd);
    *reinterpret_cast<uint4*>(pub + chunk::HO_KE + sw128(c, 32 * ab)) =
        make_uint4(w[0], w[1], w[2], w[3]);
    *reinterpret_cast<uint4*>(pub + chunk::HO_KE + sw128(c, 32 * ab + 16)) =
        make_uint4(w[4], w[5], w[6], w[7]);
    // K~^(ab) = k e^{rho_a - gamma}: N-block (3 - ab) of the Gram B operand
#pragma unroll
    for (int rr = 0; rr < 16; ++rr) v[rr] = G[rr] * cF;
    chunk::store_row16(sm + P_KT + (3 - ab) * 16384, c, 32 * ab, v);
    // K~^(a') for a' > ab: (k e^{rho_{a+1} - gamma}) e^{rho_{a'} - rho_{a+1}}
#pragma unroll
    for (int ap = 1; ap < 4; ++ap) {
        if (ap > ab) {
            const float f = chunk::exp2_approx((ap == 1 ? rho[1] : ap == 2 ? rho[2] : rho[3]) -
                                               rho_a1);
#pragma unroll
            for (int rr = 0; rr < 16; ++rr) v[rr] = G[rr] * f;
            chunk::store_row16(sm + P_KT + (3 - ap) * 16384, c, 32 * ab, v);
        }
    }
}

// (one thread) the Gram products into TG_G of the buffer at tbase: [X~ rows]
// x [4 key copies].
__device__ __forceinline__ void a_issue_gram(uint32_t smem_base, uint32_t tbase) {
    const uint32_t id = idesc_bf16(128, 256, 1, 1);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
        const uint64_t a = smem_desc(smem_base + P_XT + kk * 2048, 16384, 1024);
        const uint64_t b = smem_desc(smem_base + P_KT + kk * 2048, 16384, 1024);
        mma_bf16(tbase + TG_G, a, b, id, kk > 0);
    }
}

// ---------------------------------------------------------------- group B
// Gram epilogue: warp quadrant q holds the rows of block a = 3 - q (lanes
// 0-15 the q rows, 16-31 the k rows); part (0, 1) selects 32 of the block's
// 64 key tokens.  Aqk (bf16, i <= r) goes to the published chunk, Akk (fp32,
// beta_r-scaled, i < r) to P_AKK and, with a chunk record `rec`, the key
// Gram without beta (bf16, i < r) to its REC_G tile.  No barrier.
__device__ __forceinline__ void b_gram_epilogue(uint8_t* sm, uint32_t tbase, int warp, int lane,
                                                int part, const float* s_beta, uint8_t* pub,
                                                uint8_t* rec) {
    const int q = warp & 3;
    const int a = 3 - q;
    const int row = 16 * a + (lane & 15);
    const bool is_k = lane >= 16;
    const int i0 = 32 * part;
    const uint32_t taddr = tbase + ((uint32_t)(32 * q) << 16) + TG_G + 64 * q + i0;
    uint32_t r0[16], r1[16];
    tmem_ld16(taddr, r0);
    tmem_ld16(taddr + 16, r1);
    tmem_wait_ld();
    if (!is_k) {
        uint32_t w[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = i0 + 2 * k;
            w[k] = chunk::pack_bf16x2(i <= row ? __uint_as_float(r0[2 * k]) : 0.0f,
                                      i + 1 <= row ? __uint_as_float(r0[2 * k + 1]) : 0.0f);
            w[8 + k] = chunk::pack_bf16x2(i + 16 <= row ? __uint_as_float(r1[2 * k]) : 0.0f,
                                          i + 17 <= row ? __uint_as_float(r1[2 * k + 1]) : 0.0f);
        }
        uint8_t* t = pub + chunk::HO_AQK;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            *reinterpret_cast<uint4*>(t + sw128(row, 2 * i0 + 16 * k)) =
                make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
        }
    } else {
        const float br = s_beta[row];
        float* akk = reinterpret_cast<float*>(sm + P_AKK) + row * 65 + i0;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            akk[k] = i0 + k < row ? br * __uint_as_float(r0[k]) : 0.0f;
            akk[16 + k] = i0 + 16 + k < row ? br * __uint_as_float(r1[k]) : 0.0f;
        }
        if (rec) {
            uint32_t w[16];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = i0 + 2 * k;
                w[k] = chunk::pack_bf16x2(i < row ? __uint_as_float(r0[2 * k]) : 0.0f,
                                          i + 1 < row ? __uint_as_float(r0[2 * k + 1]) : 0.0f);
                w[8 + k] = chunk::pack_bf16x2(i + 16 < row ? __uint_as_float(r1[2 * k]) : 0.0f,
                                              i + 17 < row ? __uint_as_float(r1[2 * k + 1]) : 0.0f);
            }
            uint8_t* t = rec + chunk::REC_G;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                *reinterpret_cast<uint4*>(t + sw128(row, 2 * i0 + 16 * k)) =
                    make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            }
        }
    }
}

// UT solve Tm = (I + Akk)^-1 Diag(beta) on group B (lt = thread, lw = warp in
// the group; named barrier kBarB), Tm -> P_TM (over Akk) and the published
// chunk; with a chunk record `rec`, (I + Akk)^-1 itself to its REC_MINV
// tile.  The blocked forward substitution of chunk::phase_solve.  The group
// must have synchronised after the Gram epilogue; ends with Tm written (no
// barrier after it).
__device__ __forceinline__ void b_solve(uint8_t* sm, int lt, int lw, int lane,
                                        const float* s_beta, uint8_t* pub, uint8_t* rec) {
    float* Lm = reinterpret_cast<float*>(sm + P_AKK);
    float* Nm = reinterpret_cast<float*>(sm + P_NMAT);
    if (lt < 64) {
        const int a = lt >> 4, jj = lt & 15;
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
    group_sync(kBarB);
    if (lw < 6) {
        // (a, c) = (1,0) (2,0) (2,1) (3,0) (3,1) (3,2)
        const int a = lw < 1 ? 1 : lw < 3 ? 2 : 3;
        const int c = lw < 1 ? 0 : lw < 3 ? lw - 1 : lw - 3;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        chunk::warp_gemm16(acc, Nm, 16 * a, 16 * a, Lm, 16 * a, 16 * c, lane);
        chunk::warp_store16(acc, Lm, 16 * a, 16 * c, 1.0f, lane);
    }
    group_sync(kBarB);
#pragma unroll 1
    for (int wave = 1; wave < 4; ++wave) {
        if (lw < 4 - wave) {
            const int a = lw + wave, b = lw;
            float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            for (int cc = b; cc < a; ++cc) {
                chunk::warp_gemm16(acc, Lm, 16 * a, 16 * cc, Nm, 16 * cc, 16 * b, lane);
            }
            chunk::warp_store16(acc, Nm, 16 * a, 16 * b, -1.0f, lane);
        }
        group_sync(kBarB);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int r = (lt >> 3) + 32 * h, i0 = (lt & 7) * 8;
        float v[8], nv[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int i = i0 + u;
            nv[u] = i <= r ? Nm[r * 65 + i] : 0.0f;
            v[u] = nv[u] * s_beta[i];
        }
        const uint4 w = make_uint4(chunk::pack_bf16x2(v[0], v[1]), chunk::pack_bf16x2(v[2], v[3]),
                                   chunk::pack_bf16x2(v[4], v[5]), chunk::pack_bf16x2(v[6], v[7]));
        *reinterpret_cast<uint4*>(sm + P_TM + sw128(r, 2 * i0)) = w;
        *reinterpret_cast<uint4*>(pub + chunk::HO_TM + sw128(r, 2 * i0)) = w;
        if (rec) {
            *reinterpret_cast<uint4*>(rec + chunk::REC_MINV + sw128(r, 2 * i0)) =
                make_uint4(chunk::pack_bf16x2(nv[0], nv[1]), chunk::pack_bf16x2(nv[2], nv[3]),
                           chunk::pack_bf16x2(nv[4], nv[5]), chunk::pack_bf16x2(nv[6], nv[7]));
        }
    }
}

// (one thread) W^T = K+^T Tm^T into TG_W of the buffer at tbase (K+ at kp_off).
__device__ __forceinline__ void b_issue_w(uint32_t smem_base, uint32_t tbase, uint32_t kp_off) {
    const uint32_t idw = idesc_bf16(128, 64, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bT = smem_desc(smem_base + P_TM + kk * 32, 16, 1024);
        const uint64_t aK = smem_desc(smem_base + kp_off + kk * 32, 16, 1024);
        mma_bf16(tbase + TG_W, aK, bT, idw, kk > 0);
    }
}

// -W^T (TMEM) -> the published chunk; each warp of group B covers 32 of the
// 64 token columns of its lane quadrant.  No barrier.
__device__ __forceinline__ void b_neg_w(uint32_t tbase, int warp, int lw, int lane,
                                        uint8_t* tile) {
    const int q = warp & 3;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int sub = 2 * (lw >> 2) + h;
        uint32_t r[16];
        tmem_ld16(tbase + ((uint32_t)(32 * q) << 16) + TG_W + 16 * sub, r);
        tmem_wait_ld();
        float v[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = -__uint_as_float(r[i]);
        chunk::store_row16(tile, 32 * q + lane, 32 * sub, v);
    }
}

}  // namespace split
}  // namespace kda
