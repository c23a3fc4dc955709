// kda_recurrent.cu -- fused recurrent KDA kernel for sm_103a.
//
// One CTA owns one (row, head) state S (d_k x d_v, fp32) in registers and
// walks that row's tokens in order.  Per token it fuses everything the
// recurrence of "Kimi K3 Open Weights: What Is Actually New In Its 2.8
// Trillion Parameter Architecture", section 1, asks for:
//   gate     alpha = exp(-5 * sigmoid(e^A z))           (gate equation; or
//            sigmoid(-e^A z) = exp(-softplus(e^A z)), the unbounded gate the
//            section says K3 replaced)
//   decay    S'    = Diag(alpha) S
//   erase    u     = beta (v - S'^T k_hat)
//   write    S     = S' + k_hat u^T                     (delta-rule update)
//   read     o     = S^T q_hat = S'^T q_hat + (k_hat . q_hat) u
// q_hat/k_hat are the L2-normalised q/k (the section's "Q/K normalization").
//
// Decode (the section's "fused recurrent kernel" with the state kept
// persistent) is the case of one token per row: the state streams from HBM
// once, is updated in registers and streams back once, with 128-bit loads and
// stores that are coalesced across each warp (a warp covers whole state rows).
// The same kernel serves as the exact fp32 prefill path (any head dim, fp32
// inputs).
//
// Thread layout: the value columns of a head are split over NSPLIT CTAs (the
// columns of S are independent).  Decode: a CTA's slice of DVS = d_v/NSPLIT
// columns is covered by LPR = DVS/4 lanes holding one float4 each; a warp
// covers RPW = 32/LPR rows per pass; the CTA covers RSTEP = 8*RPW rows per
// pass and each thread keeps RPT = d_k/RSTEP float4 of the state.  Column
// sums over the d_k rows (S'^T k, S'^T q) are reduced with warp shuffles
// inside a warp and through shared memory across the 8 warps.  Prefill
// (32-column CTAs): warp w owns the 4 whole columns 4w .. 4w+3 and lane l the
// rows l + 32 r, so the column sums, u and o of a token stay inside the warp
// and the token loop has no CTA barrier.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kda_internal.h"
#include "kda_lanes.cuh"
#include "kda_seqlens.cuh"

namespace kda {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kGmin = -5.0f;
constexpr float kNormEps = 1e-6f;

__device__ __forceinline__ float load_elem(const float* p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float load_elem(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}
__device__ __forceinline__ void store_elem(float* p, size_t i, float x) { p[i] = x; }
// a value of the input dtype as float, from any memory space (shared included)
__device__ __forceinline__ float as_float(float x) { return x; }
__device__ __forceinline__ float as_float(__nv_bfloat16 x) { return __bfloat162float(x); }

// Prefill prepares the next kStage tokens at once, in dynamic shared memory
// (fp32): the normalised and scaled q_hat, k_hat, the decay alpha, the CTA's
// v columns, beta and q_hat . k_hat.  These depend on the inputs only, so the
// whole CTA computes them in parallel (one warp per token); the token-serial
// loop is then left with the state update, warp by warp.
// The stretch's raw inputs are first copied into shared memory with 16-byte
// loads, all in flight at once; for fp32 inputs they land in the prepared
// arrays themselves (each warp reads its token's row before overwriting it),
// for bf16 in a raw area after them.
constexpr int kStage = 64;
template <int DK, int DVS, typename T>
constexpr size_t stage_raw_bytes() {
    return sizeof(T) == 4 ? 0 : (size_t)kStage * (3 * DK + DVS + 1) * sizeof(T);
}
template <int DK, int DVS, typename T>
constexpr size_t stage_bytes() {
    return (size_t)kStage * (3 * DK + DVS + 2) * sizeof(float) + stage_raw_bytes<DK, DVS, T>();
}
__device__ __forceinline__ void store_elem(__nv_bfloat16* p, size_t i, float x) {
    p[i] = __float2bfloat16_rn(x);
}

// sigmoid on the branch that cannot overflow
__device__ __forceinline__ float sigmoid_f(float x) {
    if (x >= 0.0f) {
        return 1.0f / (1.0f + expf(-x));
    }
    const float e = expf(x);
    return e / (1.0f + e);
}

// Launch modes.  Each is its own instantiation so that the decode kernel,
// whose occupancy (and so its HBM bandwidth) depends on its register count,
// carries none of the prefill bookkeeping.
constexpr int kModeDecode = 0;    // one token per row, state pool with slots
constexpr int kModePrefill = 1;   // a sequence per row
constexpr int kModeCkpt = 2;      // prefill that also stores state checkpoints

template <int DK, int DV, int NSPLIT, typename T, int kMode>
__global__ void __launch_bounds__(kThreads)
kda_recurrent_kernel(const RecurrentParams p) {
    constexpr bool kDecode = kMode == kModeDecode;
    constexpr bool kCkpt = kMode == kModeCkpt;
    constexpr int DVS = DV / NSPLIT;
    constexpr int LPR = DVS / 4;
    constexpr int RPW = 32 / LPR;
    constexpr int RSTEP = kWarps * RPW;
    constexpr int RPT = DK / RSTEP;
    static_assert(RPT >= 1 && RPT * RSTEP == DK, "bad state tiling");
    static_assert(DK + DVS <= kThreads, "stage-1 loaders need DK + DVS threads");
    static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "bad column split");

    __shared__ float s_q[DK];
    __shared__ float s_k[DK];
    __shared__ float s_a[DK];
    __shared__ float s_v[DVS];
    __shared__ float s_u[DVS];
    __shared__ float s_red[kWarps][2][DVS];
    __shared__ float s_nrm[DK / 32][3];
    __shared__ float s_beta;

    const int tid = threadIdx.x;
    const int w = tid >> 5;
    const int lane = tid & 31;
    const int cg = lane % LPR;
    const int rs = lane / LPR;
    const int split = blockIdx.x % NSPLIT;
    const int h = (blockIdx.x / NSPLIT) % p.H;
    const int row = blockIdx.x / (NSPLIT * p.H);
    const int col0 = split * DVS;
    const int H = p.H;

    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    const T* z = static_cast<const T*>(p.z);
    const T* beta = static_cast<const T*>(p.beta);
    T* o = static_cast<T*>(p.o);

    int64_t bos, eos;
    int64_t sidx = row;  // index of this row's state in state_in / state_out
    bool valid = true;
    if constexpr (kDecode) {
        bos = row;
        eos = row + 1;
        if (p.slots) {
            sidx = p.slots[row];
        }
        valid = sidx >= 0 && sidx < p.pool_size;
    } else {
        clamped_seq(p.cu_seqlens, row, p.rows, p.total_T, bos, eos);
    }
    if (!valid) {
        // Decode row with an out-of-range slot: state untouched, o = NaN.
        for (int j = tid; j < DVS; j += kThreads) {
            store_elem(o, ((size_t)bos * H + h) * DV + col0 + j, __int_as_float(0x7fc00000));
        }
        return;
    }

    // float4 index, in a d_k x d_v state, of the thread's part of its r-th
    // state row.  Decode: rows r * RSTEP + w * RPW + rs, the CTA's columns
    // spread over the lanes (each warp pass reads whole rows).  Prefill: rows
    // lane + 32 r, warp w owning the 4 columns 4w .. 4w+3 of the CTA's 32, so
    // that a token's column sums never leave the warp.
    auto st4 = [=](int r) -> size_t {
        if constexpr (kDecode) {
            return ((size_t)(r * RSTEP + w * RPW + rs) * DV + col0) / 4 + cg;
        } else {
            return ((size_t)(lane + 32 * r) * DV + col0 + 4 * w) / 4;
        }
    };

    // ---- state load (128-bit) ----
    float4 S[RPT];
    const size_t soff = ((size_t)sidx * H + h) * DK * DV;
    if (p.state_in) {
        const float4* sp = reinterpret_cast<const float4*>(p.state_in + soff);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            S[r] = __ldcs(sp + st4(r));
        }
    } else {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            S[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }

    const float eA = expf(p.A[h]);
    const float scale = p.scale;

    // prefill state checkpoints: index of this row's first one (the sum over
    // earlier sequences of floor(length / interval))
    int64_t ck_idx = 0;               // pool index of the row's next checkpoint
    int64_t ck_next = INT64_MAX;      // token after which it is taken
    if constexpr (kCkpt) {
        __shared__ int s_ck;
        if (tid == 0) {
            s_ck = 0;
        }
        __syncthreads();
        int part = 0;
        for (int m = tid; m < row; m += kThreads) {
            part += (int)(clamped_len(p.cu_seqlens, m, p.rows, p.total_T) / p.ckpt_interval);
        }
        if (part) {
            atomicAdd(&s_ck, part);
        }
        __syncthreads();
        ck_idx = s_ck;
        ck_next = bos + p.ckpt_interval - 1;
    }

    extern __shared__ __align__(16) unsigned char rc_stage[];
    float* sq_h = reinterpret_cast<float*>(rc_stage);   // [kStage][DK] scale q / |q|
    float* sk_h = sq_h + kStage * DK;                   // [kStage][DK] k / |k|
    float* sa_h = sk_h + kStage * DK;                   // [kStage][DK] alpha
    float* sv_h = sa_h + kStage * DK;                   // [kStage][DVS]
    float* sb_h = sv_h + kStage * DVS;                  // [kStage] beta
    float* sd_h = sb_h + kStage;                        // [kStage] q_hat . k_hat
    // raw inputs of the stretch: in place (fp32) or in the raw area (bf16)
    unsigned char* raw_area = rc_stage + (size_t)kStage * (3 * DK + DVS + 2) * sizeof(float);
    T* rq = sizeof(T) == 4 ? reinterpret_cast<T*>(sq_h) : reinterpret_cast<T*>(raw_area);
    T* rk_ = sizeof(T) == 4 ? reinterpret_cast<T*>(sk_h) : rq + kStage * DK;
    T* rz = sizeof(T) == 4 ? reinterpret_cast<T*>(sa_h) : rk_ + kStage * DK;
    T* rv = sizeof(T) == 4 ? reinterpret_cast<T*>(sv_h) : rz + kStage * DK;
    T* rb = sizeof(T) == 4 ? reinterpret_cast<T*>(sb_h) : rv + kStage * DVS;
    auto stage_raw = [&](int64_t t0, int n) {
        constexpr int VE = 16 / sizeof(T);
        constexpr int RK = DK / VE, RV = DVS / VE;
        for (int e = tid; e < n * RK; e += kThreads) {
            const int j = e / RK, c4 = e - j * RK;
            const size_t g = ((size_t)(t0 + j) * H + h) * DK + (size_t)c4 * VE;
            const int l = j * DK + c4 * VE;
            *reinterpret_cast<uint4*>(rq + l) = __ldg(reinterpret_cast<const uint4*>(q + g));
            *reinterpret_cast<uint4*>(rk_ + l) = __ldg(reinterpret_cast<const uint4*>(k + g));
            *reinterpret_cast<uint4*>(rz + l) = __ldg(reinterpret_cast<const uint4*>(z + g));
        }
        for (int e = tid; e < n * RV; e += kThreads) {
            const int j = e / RV, c4 = e - j * RV;
            const size_t g = ((size_t)(t0 + j) * H + h) * DV + col0 + (size_t)c4 * VE;
            *reinterpret_cast<uint4*>(rv + j * DVS + c4 * VE) =
                __ldg(reinterpret_cast<const uint4*>(v + g));
        }
        if (tid < n) {
            rb[tid] = beta[(size_t)(t0 + tid) * H + h];
        }
        __syncthreads();
    };
    // tokens t0 .. t0+n-1 from the raw copy: warp w prepares tokens w, w + 8,
    // ...; lane l holds channels l, l + 32, ... (and column l of v, l < DVS)
    auto prepare = [&](int64_t t0, int n) {
        constexpr int CPL = DK / 32;
        stage_raw(t0, n);
        for (int j = w; j < n; j += kWarps) {
            float qv[CPL], kv[CPL], zv[CPL];
            float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
            for (int m = 0; m < CPL; ++m) {
                const int c = j * DK + lane + 32 * m;
                qv[m] = as_float(rq[c]);
                kv[m] = as_float(rk_[c]);
                zv[m] = as_float(rz[c]);
                sq += qv[m] * qv[m];
                sk += kv[m] * kv[m];
                sqk += qv[m] * kv[m];
            }
            const float vv = lane < DVS ? as_float(rv[j * DVS + lane]) : 0.0f;
            const float bv = as_float(rb[j]);
            __syncwarp();   // (fp32: the row is read before it is overwritten)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
            }
            const float iq = p.l2norm ? rsqrtf(sq + kNormEps) : 1.0f;
            const float ik = p.l2norm ? rsqrtf(sk + kNormEps) : 1.0f;
#pragma unroll
            for (int m = 0; m < CPL; ++m) {
                const int c = lane + 32 * m;
                sq_h[j * DK + c] = qv[m] * iq * scale;
                sk_h[j * DK + c] = kv[m] * ik;
                // alpha = e^g: K3's g = -5 sigmoid(e^A z), or Kimi Linear's
                // g = -softplus(e^A z), for which e^g = sigmoid(-e^A z)
                const float sg = sigmoid_f(p.softplus_gate ? -eA * zv[m] : eA * zv[m]);
                sa_h[j * DK + c] = p.softplus_gate ? sg : expf(kGmin * sg);
            }
            if (lane < DVS) {
                sv_h[j * DVS + lane] = vv;
            }
            if (lane == 0) {
                sb_h[j] = bv;
                sd_h[j] = sqk * iq * ik * scale;
            }
        }
        __syncthreads();
    };

    if constexpr (!kDecode) {
        static_assert(DVS == 32, "prefill CTAs hold 32 value columns");
        for (int64_t t0 = bos; t0 < eos; t0 += kStage) {
            const int n = (int)min((int64_t)kStage, eos - t0);
            __syncthreads();   // the previous stretch's last token has been read
            prepare(t0, n);
            for (int jt = 0; jt < n; ++jt) {
                const int64_t t = t0 + jt;
                // ---- decay, and the two column sums of S' over the d_k rows
                // (warp w holds whole columns 4w .. 4w+3: no other warp and no
                // barrier takes part) ----
                float4 ak = make_float4(0.f, 0.f, 0.f, 0.f);
                float4 aq = make_float4(0.f, 0.f, 0.f, 0.f);
                float kreg[RPT];
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const int i = lane + 32 * r;
                    const float a = sa_h[jt * DK + i];
                    const float kk = sk_h[jt * DK + i];
                    const float qq = sq_h[jt * DK + i];
                    kreg[r] = kk;
                    S[r].x *= a; S[r].y *= a; S[r].z *= a; S[r].w *= a;
                    ak.x += kk * S[r].x; ak.y += kk * S[r].y;
                    ak.z += kk * S[r].z; ak.w += kk * S[r].w;
                    aq.x += qq * S[r].x; aq.y += qq * S[r].y;
                    aq.z += qq * S[r].z; aq.w += qq * S[r].w;
                }
                // Transposed sums over the 32 lanes: lane bit 4 picks ak or aq,
                // bits 3 and 2 the column c = 2 b3 + b2 that the lane finishes;
                // bits 1 and 0 are then summed by two butterflies (9 shuffles
                // for the 8 sums).
                constexpr unsigned F = 0xffffffffu;
                const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4;
                const float x0 = (b4 ? aq.x : ak.x) + __shfl_xor_sync(F, b4 ? ak.x : aq.x, 16);
                const float x1 = (b4 ? aq.y : ak.y) + __shfl_xor_sync(F, b4 ? ak.y : aq.y, 16);
                const float x2 = (b4 ? aq.z : ak.z) + __shfl_xor_sync(F, b4 ? ak.z : aq.z, 16);
                const float x3 = (b4 ? aq.w : ak.w) + __shfl_xor_sync(F, b4 ? ak.w : aq.w, 16);
                const float y0 = (b3 ? x2 : x0) + __shfl_xor_sync(F, b3 ? x0 : x2, 8);
                const float y1 = (b3 ? x3 : x1) + __shfl_xor_sync(F, b3 ? x1 : x3, 8);
                float zc = (b2 ? y1 : y0) + __shfl_xor_sync(F, b2 ? y0 : y1, 4);
                zc += __shfl_xor_sync(F, zc, 2);
                zc += __shfl_xor_sync(F, zc, 1);
                const int c = (b3 ? 2 : 0) + (b2 ? 1 : 0);
                // u_c = beta (v_c - (S'^T k)_c) on the lanes that hold
                // (S'^T k)_c; o_c = (S'^T q)_c + (q . k) u_c on those that
                // hold (S'^T q)_c, which take u_c from lane ^ 16
                const float uc = sb_h[jt] * (sv_h[jt * DVS + 4 * w + c] - zc);
                const float u_other = __shfl_xor_sync(F, uc, 16);
                if (b4 && (lane & 3) == 0) {
                    store_elem(o, ((size_t)t * H + h) * DV + col0 + 4 * w + c,
                               zc + sd_h[jt] * u_other);
                }
                // ---- rank-1 write (u of the warp's 4 columns from lanes 0, 4, 8, 12) ----
                float4 u4;
                u4.x = __shfl_sync(F, uc, 0);
                u4.y = __shfl_sync(F, uc, 4);
                u4.z = __shfl_sync(F, uc, 8);
                u4.w = __shfl_sync(F, uc, 12);
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    const float kk = kreg[r];
                    S[r].x += kk * u4.x; S[r].y += kk * u4.y;
                    S[r].z += kk * u4.z; S[r].w += kk * u4.w;
                }
                // ---- state checkpoint after every ckpt_interval tokens of the row ----
                if constexpr (kCkpt) {
                    if (t == ck_next && ck_idx < p.ckpt_count) {
                        const int64_t idx = ck_idx++;
                        ck_next += p.ckpt_interval;
                        const int64_t prow = p.ckpt_slots ? (int64_t)p.ckpt_slots[idx] : idx;
                        if (prow >= 0 && prow < p.ckpt_pool_size) {
                            float4* cp = reinterpret_cast<float4*>(
                                p.ckpt_pool + ((size_t)prow * H + h) * DK * DV);
#pragma unroll
                            for (int r = 0; r < RPT; ++r) {
                                __stcs(cp + st4(r), S[r]);
                            }
                        }
                    }
                }
            }
        }
    }

    // decode: one token per row, straight from global memory
    for (int64_t t = bos; kDecode && t < eos; ++t) {
        // ---- stage 1: token inputs, gate, norm partial sums ----
        const size_t rk = ((size_t)t * H + h) * DK;
        if (tid < DK) {
            const float qv = load_elem(q, rk + tid);
            const float kv = load_elem(k, rk + tid);
            const float zv = load_elem(z, rk + tid);
            s_q[tid] = qv;
            s_k[tid] = kv;
            // alpha = e^g: K3's g = -5 sigmoid(e^A z), or Kimi Linear's
            // g = -softplus(e^A z), for which e^g = sigmoid(-e^A z)
            const float sg = sigmoid_f(p.softplus_gate ? -eA * zv : eA * zv);
            s_a[tid] = p.softplus_gate ? sg : expf(kGmin * sg);
            float sq = qv * qv, sk = kv * kv, sqk = qv * kv;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
            }
            if (lane == 0) {
                s_nrm[w][0] = sq;
                s_nrm[w][1] = sk;
                s_nrm[w][2] = sqk;
            }
        } else if (tid < DK + DVS) {
            const int j = tid - DK;
            s_v[j] = load_elem(v, ((size_t)t * H + h) * DV + col0 + j);
            if (j == 0) {
                s_beta = load_elem(beta, (size_t)t * H + h);
            }
        }
        __syncthreads();

        float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
        for (int i = 0; i < DK / 32; ++i) {
            sq += s_nrm[i][0];
            sk += s_nrm[i][1];
            sqk += s_nrm[i][2];
        }
        const float inv_q = p.l2norm ? rsqrtf(sq + kNormEps) : 1.0f;
        const float inv_k = p.l2norm ? rsqrtf(sk + kNormEps) : 1.0f;
        const float qscale = inv_q * scale;

        // ---- stage 2: decay, and the two column sums of S' ----
        float4 ak = make_float4(0.f, 0.f, 0.f, 0.f);
        float4 aq = make_float4(0.f, 0.f, 0.f, 0.f);
        float kreg[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int i = r * RSTEP + w * RPW + rs;
            const float a = s_a[i];
            const float kk = s_k[i];
            const float qq = s_q[i];
            kreg[r] = kk * inv_k;
            S[r].x *= a; S[r].y *= a; S[r].z *= a; S[r].w *= a;
            ak.x += kk * S[r].x; ak.y += kk * S[r].y; ak.z += kk * S[r].z; ak.w += kk * S[r].w;
            aq.x += qq * S[r].x; aq.y += qq * S[r].y; aq.z += qq * S[r].z; aq.w += qq * S[r].w;
        }
#pragma unroll
        for (int off = LPR; off < 32; off <<= 1) {
            ak.x += __shfl_xor_sync(0xffffffffu, ak.x, off);
            ak.y += __shfl_xor_sync(0xffffffffu, ak.y, off);
            ak.z += __shfl_xor_sync(0xffffffffu, ak.z, off);
            ak.w += __shfl_xor_sync(0xffffffffu, ak.w, off);
            aq.x += __shfl_xor_sync(0xffffffffu, aq.x, off);
            aq.y += __shfl_xor_sync(0xffffffffu, aq.y, off);
            aq.z += __shfl_xor_sync(0xffffffffu, aq.z, off);
            aq.w += __shfl_xor_sync(0xffffffffu, aq.w, off);
        }
        if (rs == 0) {
            *reinterpret_cast<float4*>(&s_red[w][0][4 * cg]) = ak;
            *reinterpret_cast<float4*>(&s_red[w][1][4 * cg]) = aq;
        }
        __syncthreads();

        // ---- stage 3: u and o per value column ----
        if (tid < DVS) {
            float rkj = 0.f, rqj = 0.f;
#pragma unroll
            for (int ww = 0; ww < kWarps; ++ww) {
                rkj += s_red[ww][0][tid];
                rqj += s_red[ww][1][tid];
            }
            rkj *= inv_k;
            rqj *= qscale;
            const float u = s_beta * (s_v[tid] - rkj);
            s_u[tid] = u;
            const float dot = sqk * inv_k * qscale;  // k_hat . q_hat
            store_elem(o, ((size_t)t * H + h) * DV + col0 + tid, rqj + dot * u);
        }
        __syncthreads();

        // ---- stage 4: rank-1 write ----
        const float4 u4 = *reinterpret_cast<const float4*>(&s_u[4 * cg]);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const float kk = kreg[r];
            S[r].x += kk * u4.x; S[r].y += kk * u4.y; S[r].z += kk * u4.z; S[r].w += kk * u4.w;
        }

    }

    if (p.state_out) {
        float4* sp = reinterpret_cast<float4*>(p.state_out + soff);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            __stcs(sp + st4(r), S[r]);
        }
    }
}

// Value-column split per head.  Decode of d_v = 128 uses two CTAs per head
// (half the registers per CTA, twice the state bytes in flight per SM; more
// CTAs per head would shrink the 128-bit rows each warp streams).  Prefill,
// token-serial and latency-bound, uses 32-column CTAs: a quarter of the
// per-token work of each CTA at d_v = 128, on four times the SMs.
template <int DV>
constexpr int decode_split() { return DV == 128 ? 2 : 1; }
template <int DV>
constexpr int prefill_split() { return DV / 32; }

template <int DK, int DV, int NS, typename T, int kMode>
cudaError_t launch_one(const RecurrentParams& p, cudaStream_t stream) {
    const dim3 grid((unsigned)((int64_t)p.rows * p.H * NS));
    if (grid.x == 0) {
        return cudaSuccess;
    }
    // decode has one token per row: no staging, no dynamic shared memory.
    // The attribute belongs to the current device, so it is set on every launch.
    constexpr size_t smem = kMode == kModeDecode ? 0 : stage_bytes<DK, DV / NS, T>();
    if (smem > 0) {
        const cudaError_t e = cudaFuncSetAttribute(kda_recurrent_kernel<DK, DV, NS, T, kMode>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem);
        if (e != cudaSuccess) {
            return e;
        }
    }
    kda_recurrent_kernel<DK, DV, NS, T, kMode><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int DK, int DV, typename T>
cudaError_t launch_mode(int mode, const RecurrentParams& p, cudaStream_t stream) {
    constexpr int NSD = decode_split<DV>();
    constexpr int NSP = prefill_split<DV>();
    switch (mode) {
        case kModeDecode: return launch_one<DK, DV, NSD, T, kModeDecode>(p, stream);
        case kModeCkpt: return launch_one<DK, DV, NSP, T, kModeCkpt>(p, stream);
        default: return launch_one<DK, DV, NSP, T, kModePrefill>(p, stream);
    }
}

template <int DK, int DV>
cudaError_t launch_dims(const RecurrentParams& p, int dtype, cudaStream_t stream) {
    const int mode = p.decode ? kModeDecode : p.ckpt_interval > 0 ? kModeCkpt : kModePrefill;
    return dtype == 0 ? launch_mode<DK, DV, float>(mode, p, stream)
                      : launch_mode<DK, DV, __nv_bfloat16>(mode, p, stream);
}

template <int DK>
cudaError_t launch_dk(const RecurrentParams& p, int d_v, int dtype, cudaStream_t stream) {
    switch (d_v) {
        case 32: return launch_dims<DK, 32>(p, dtype, stream);
        case 64: return launch_dims<DK, 64>(p, dtype, stream);
        case 128: return launch_dims<DK, 128>(p, dtype, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_recurrent(const RecurrentParams& p, int d_k, int d_v, int dtype,
                             cudaStream_t stream) {
    switch (d_k) {
        case 32: return launch_dk<32>(p, d_v, dtype, stream);
        case 64: return launch_dk<64>(p, d_v, dtype, stream);
        case 128: return launch_dk<128>(p, d_v, dtype, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace kda
