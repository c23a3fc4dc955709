// kda_backward.cu -- gradients of the KDA recurrence (training backward),
// recurrent form, fp32, for sm_103a.
//
// The forward step of "Kimi K3 Open Weights: What Is Actually New In Its 2.8
// Trillion Parameter Architecture", section 1 (per head, per token):
//   qh = scale q / |q|, kh = k / |k|,  a = e^g (g = -5 sigmoid(e^A z), or
//   -softplus(e^A z)),  S' = Diag(a) S_{t-1},  u = b (v - S'^T kh),
//   S_t = S' + kh u^T,  o_t = S_t^T qh.
// With G = dL/dS_t carried backwards from dL/dS_T, each token in reverse:
//   G += qh do^T;  dqh = S_t do;  du = G^T kh;  dkh = G u - b S' du;
//   dv = b du;  db = du . (v - S'^T kh);  G' = G - b kh du^T;
//   da[c] = sum_j G'[c][j] S_{t-1}[c][j];  G = Diag(a) G'
// followed by the gate and normalisation derivatives, written out per token.
//
// The value columns of a head are independent in the recurrence (column j of
// S, G, u, du only meets column j), so each (sequence, head) runs as NS =
// d_v / 32 CTAs of 32 columns, each holding its d_k x 32 slices of the state
// and of G in registers.  What sums over the columns (dqh, dkh, da, db) is
// written per token as one partial per CTA; kda_backward_finalize_kernel adds
// the partials and applies the gate and normalisation derivatives.  The
// reverse pass needs S_{t-1} for every token.  The states at the 64-token
// chunk starts come from the library's checkpointed prefill (run by the host
// before this kernel: checkpoint m of sequence n, the state after its first
// 64 m tokens, at pool row (checkpoints of earlier sequences) + m - 1); the
// kernel walks the chunks last to first, recomputes each chunk's states
// forward into a scratch buffer (S_{t-1} of its 64 tokens), then walks its
// tokens backwards.  The scratch keeps memory at 64 states per (sequence,
// head).  Both walks over a chunk read its tokens' q_hat, k_hat, alpha, v and
// dO columns and beta from shared memory, computed once for the chunk by the
// whole CTA, so the token chain has no global loads and no reductions over
// the key channels.  Each warp owns 4 whole value columns, so the
// recurrence's column sums never leave the warp and neither walk takes a CTA
// barrier per token; the outputs are summed over the warps every kBwRed
// tokens.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "kda_internal.h"
#include "kda_lanes.cuh"
#include "kda_seqlens.cuh"

namespace kda {
namespace {

constexpr int kBwThreads = 256;
constexpr int kBwWarps = kBwThreads / 32;
constexpr float kBwGmin = -5.0f;
constexpr float kBwEps = 1e-6f;

__device__ __forceinline__ float ldf(const float* p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p, size_t i) {
    return __bfloat162float(p[i]);
}


__device__ __forceinline__ float as_f32(float x) { return x; }
__device__ __forceinline__ float as_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

__device__ __forceinline__ float bw_sigmoid(float x) {
    if (x >= 0.0f) {
        return 1.0f / (1.0f + expf(-x));
    }
    const float e = expf(x);
    return e / (1.0f + e);
}

constexpr int kBwCols = 32;   // value columns per CTA (8 lanes x float4 per state row)

// Tokens whose per-warp output partials are staged in shared memory before
// the CTA sums them over its warps.
constexpr int kBwRed = 8;

// Dynamic shared memory: the chunk's prepared token quantities and the
// forward walk's v - S'^T k_hat per token (fp32), then one area used first
// for the chunk's raw 16-bit inputs (fp32 inputs are copied in place into the
// prepared arrays) and then, in the reverse walk, for the warps' staged
// output partials.
template <int DK, typename T>
constexpr size_t chunk_raw_bytes() {
    return sizeof(T) == 4 ? 0 : (size_t)kBwChunk * (3 * DK + 2 * kBwCols + 1) * sizeof(T);
}
template <int DK>
constexpr size_t chunk_red_bytes() {
    return (size_t)kBwRed * kBwWarps * (3 * DK + 1) * sizeof(float);
}
template <int DK, typename T>
constexpr size_t chunk_stage_bytes() {
    return (size_t)kBwChunk * (3 * DK + 3 * kBwCols + 2) * sizeof(float) +
           (chunk_raw_bytes<DK, T>() > chunk_red_bytes<DK>() ? chunk_raw_bytes<DK, T>()
                                                             : chunk_red_bytes<DK>());
}

// Thread layout: warp w owns the 4 whole value columns 4w .. 4w+3 of the
// CTA's 32 and lane l the state rows l + 32 r, so that every column sum of
// the recurrence (S'^T k_hat forward, G^T k_hat in reverse) and the values
// formed from it (u, du) stay inside the warp: neither walk needs a CTA
// barrier for the recurrence.  Only the per-row outputs (dq_hat, dk_hat,
// dalpha) and dbeta are summed over the 8 warps, kBwRed tokens at a time.
template <int DK, int DV, typename T>
__global__ void __launch_bounds__(kBwThreads, 2)
kda_backward_kernel(const BackwardParams p) {
    constexpr int NS = DV / kBwCols;       // CTAs per (sequence, head)
    constexpr int DVS = kBwCols;
    constexpr int RPT = DK / 32;           // rows per thread
    constexpr int C = kBwChunk;
    constexpr int PW = 3 * DK + 1;         // partials per (split, token, head)
    static_assert(RPT >= 1 && RPT * 32 == DK, "bad state tiling");
    static_assert(DVS == 4 * kBwWarps, "a warp owns 4 value columns");

    const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
    const int split = blockIdx.x % NS;
    const int h = (blockIdx.x / NS) % p.H;
    const int n = blockIdx.x / (NS * p.H);
    const int col0 = split * DVS;
    const int wc0 = 4 * w;                 // the warp's first column within the CTA's
    const int H = p.H;
    const T* q = static_cast<const T*>(p.q);
    const T* k = static_cast<const T*>(p.k);
    const T* v = static_cast<const T*>(p.v);
    const T* z = static_cast<const T*>(p.z);
    const T* beta = static_cast<const T*>(p.beta);
    const T* dO = static_cast<const T*>(p.dO);

    int64_t bos, eos;
    clamped_seq(p.cu_seqlens, n, p.N, p.total_T, bos, eos);
    const int64_t len = eos - bos;
    const int64_t nchunks = (len + C - 1) / C;
    const size_t SS = (size_t)DK * DV;
    // this CTA's part of its pair's chunk scratch, thread-major: the float4 of
    // token j, row pass r, thread tid at (j * RPT + r) * kBwThreads + tid
    float4* scratch = reinterpret_cast<float4*>(p.scratch + ((size_t)n * H + h) * C * SS +
                                                (size_t)split * C * DK * DVS);
    const float eA = expf(p.A[h]);
    const float scale = p.scale;

    // float4 index of the thread's part of its r-th row in a full d_k x d_v state
    auto st_idx = [=](int r) { return ((size_t)(lane + 32 * r) * DV + col0 + wc0) / 4; };
    auto sc_idx = [=](int j, int r) { return ((size_t)j * RPT + r) * kBwThreads + tid; };

    // ---- the chunk's token quantities, prepared in shared memory (fp32) ----
    // q_hat (normalised, scaled), k_hat, alpha, the CTA's v and dO columns,
    // beta and q_hat . k_hat depend on the inputs only: the whole CTA first
    // copies the chunk's raw inputs in with 16-byte loads, all in flight at
    // once, then computes them (one warp per token) before the two token walks.
    extern __shared__ __align__(16) unsigned char bw_stage[];
    float* pq = reinterpret_cast<float*>(bw_stage);   // [C][DK]
    float* pk = pq + C * DK;
    float* pa = pk + C * DK;
    float* pv = pa + C * DK;                          // [C][DVS]
    float* pdo = pv + C * DVS;
    float* pw = pdo + C * DVS;                        // [C][DVS]: v - S'^T k_hat
    float* pb = pw + C * DVS;                         // [C]
    float* pqk = pb + C;                              // [C]
    // the raw copy: in place for fp32 inputs, in the shared area else; the
    // staged output partials [kBwRed][kBwWarps][PW] in the same area
    float* red = pqk + C;
    T* rq;
    T* rk_;
    T* rz;
    T* rv;
    T* rdo;
    T* rb;
    if constexpr (sizeof(T) == 4) {
        rq = reinterpret_cast<T*>(pq);
        rk_ = reinterpret_cast<T*>(pk);
        rz = reinterpret_cast<T*>(pa);
        rv = reinterpret_cast<T*>(pv);
        rdo = reinterpret_cast<T*>(pdo);
        rb = reinterpret_cast<T*>(pb);
    } else {
        rq = reinterpret_cast<T*>(red);
        rk_ = rq + C * DK;
        rz = rk_ + C * DK;
        rv = rz + C * DK;
        rdo = rv + C * DVS;
        rb = rdo + C * DVS;
    }
    auto stage_raw = [&](int64_t t0, int cl) {
        constexpr int VE = 16 / sizeof(T);
        constexpr int RK = DK / VE, RV = DVS / VE;
        for (int e = tid; e < cl * RK; e += kBwThreads) {
            const int j = e / RK, c4 = e - j * RK;
            const size_t g = ((size_t)(t0 + j) * H + h) * DK + (size_t)c4 * VE;
            const int l = j * DK + c4 * VE;
            *reinterpret_cast<uint4*>(rq + l) = __ldg(reinterpret_cast<const uint4*>(q + g));
            *reinterpret_cast<uint4*>(rk_ + l) = __ldg(reinterpret_cast<const uint4*>(k + g));
            *reinterpret_cast<uint4*>(rz + l) = __ldg(reinterpret_cast<const uint4*>(z + g));
        }
        for (int e = tid; e < cl * RV; e += kBwThreads) {
            const int j = e / RV, c4 = e - j * RV;
            const size_t g = ((size_t)(t0 + j) * H + h) * DV + col0 + (size_t)c4 * VE;
            const int l = j * DVS + c4 * VE;
            *reinterpret_cast<uint4*>(rv + l) = __ldg(reinterpret_cast<const uint4*>(v + g));
            *reinterpret_cast<uint4*>(rdo + l) = __ldg(reinterpret_cast<const uint4*>(dO + g));
        }
        if (tid < cl) {
            rb[tid] = beta[(size_t)(t0 + tid) * H + h];
        }
        __syncthreads();
    };
    auto prepare = [&](int64_t t0, int cl) {
        constexpr int CPL = DK / 32;
        stage_raw(t0, cl);
        for (int j = w; j < cl; j += kBwWarps) {
            float qv[CPL], kv[CPL], zv[CPL];
            float sq = 0.f, sk = 0.f, sqk = 0.f;
#pragma unroll
            for (int m = 0; m < CPL; ++m) {
                const int c = j * DK + lane + 32 * m;
                qv[m] = as_f32(rq[c]);
                kv[m] = as_f32(rk_[c]);
                zv[m] = as_f32(rz[c]);
                sq += qv[m] * qv[m];
                sk += kv[m] * kv[m];
                sqk += qv[m] * kv[m];
            }
            const float vv = as_f32(rv[j * DVS + lane]);   // lane < 32 = DVS
            const float dov = as_f32(rdo[j * DVS + lane]);
            const float bv = as_f32(rb[j]);
            __syncwarp();   // (fp32: the row is read before it is overwritten)
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sqk += __shfl_xor_sync(0xffffffffu, sqk, off);
            }
            const float iq = p.l2norm ? rsqrtf(sq + kBwEps) : 1.0f;
            const float ik = p.l2norm ? rsqrtf(sk + kBwEps) : 1.0f;
#pragma unroll
            for (int m = 0; m < CPL; ++m) {
                const int c = lane + 32 * m;
                pq[j * DK + c] = qv[m] * iq * scale;
                pk[j * DK + c] = kv[m] * ik;
                const float sg = bw_sigmoid(p.softplus_gate ? -eA * zv[m] : eA * zv[m]);
                pa[j * DK + c] = p.softplus_gate ? sg : expf(kBwGmin * sg);
            }
            pv[j * DVS + lane] = vv;
            pdo[j * DVS + lane] = dov;
            if (lane == 0) {
                pb[j] = bv;
                pqk[j] = sqk * iq * ik * scale;
            }
        }
        __syncthreads();
    };

    // ---- one forward step on S (registers) for token jt of the chunk; it
    // also keeps w = v - S'^T k_hat of the token (S' = Diag(alpha) S_{t-1})
    // for the reverse walk.  Warp-local: lanes 8c .. 8c+7 finish column c. ----
    float4 S[RPT];
    const int cw = lane >> 3;   // the warp column whose sums this lane finishes
    auto forward_step = [&](int jt) {
        float4 ak = make_float4(0.f, 0.f, 0.f, 0.f);
        float kreg[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const int i = lane + 32 * r;
            const float a = pa[jt * DK + i], kk = pk[jt * DK + i];
            kreg[r] = kk;
            S[r].x *= a; S[r].y *= a; S[r].z *= a; S[r].w *= a;
            ak.x += kk * S[r].x; ak.y += kk * S[r].y; ak.z += kk * S[r].z; ak.w += kk * S[r].w;
        }
        const float wv = pv[jt * DVS + wc0 + cw] - warp_colsum4(ak, lane);
        if ((lane & 7) == 0) {
            pw[jt * DVS + wc0 + cw] = wv;
        }
        const float4 u4 = gather4(pb[jt] * wv);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            const float kk = kreg[r];
            S[r].x += kk * u4.x; S[r].y += kk * u4.y; S[r].z += kk * u4.z; S[r].w += kk * u4.w;
        }
    };
    auto load_state = [&](const float* src) {
        const float4* sp = reinterpret_cast<const float4*>(src);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            S[r] = sp[st_idx(r)];
        }
    };

    // index of this sequence's first checkpoint in the pool: the sum over
    // earlier sequences of floor(length / 64)
    __shared__ int s_base;
    if (tid == 0) {
        s_base = 0;
    }
    __syncthreads();
    {
        int part = 0;
        for (int m = tid; m < n; m += kBwThreads) {
            part += (int)(clamped_len(p.cu_seqlens, m, p.N, p.total_T) / C);
        }
        if (part) {
            atomicAdd(&s_base, part);
        }
    }
    __syncthreads();
    const int64_t ck_base = s_base;

    // ---- phase 2: chunks last to first ----
    float4 G[RPT];
    if (p.dS_final) {
        const float4* gp = reinterpret_cast<const float4*>(p.dS_final + ((size_t)n * H + h) * SS);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            G[r] = gp[st_idx(r)];
        }
    } else {
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            G[r] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    for (int64_t c = nchunks - 1; c >= 0; --c) {
        const int64_t i0 = c * C;
        const int64_t cl = min((int64_t)C, len - i0);
        // 2a: the chunk's states S_{t-1} into the scratch, from the state at
        // the chunk start (the initial state for chunk 0, else checkpoint c)
        __syncthreads();   // the previous chunk's partials and last token have been read
        prepare(bos + i0, (int)cl);
        if (c > 0 && ck_base + c - 1 < p.pool_rows) {
            load_state(p.pool + ((size_t)(ck_base + c - 1) * H + h) * SS);
        } else if (c > 0) {
            // only a malformed cu_seqlens gets here (more checkpoints than the pool holds)
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                S[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        } else if (p.initial_state) {
            load_state(p.initial_state + ((size_t)n * H + h) * SS);
        } else {
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                S[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        for (int j = 0; j < (int)cl; ++j) {
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                scratch[sc_idx(j, r)] = S[r];
            }
            forward_step(j);   // (after the last token only its w is used)
        }
        __syncwarp();   // the warp's w entries are visible to all its lanes
        // 2b: the chunk's tokens in reverse (each thread reads back the
        // scratch elements it wrote).  The next reverse token's S_{t-1} is
        // loaded while this token is worked on.
        float4 Snext[RPT];
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            Snext[r] = scratch[sc_idx((int)cl - 1, r)];
        }
        int slot = 0;   // staged tokens j + slot - 1 .. j + 1 (one per slot, in walk order)
        for (int j = (int)cl - 1; j >= 0; --j) {
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                S[r] = Snext[r];                           // S = S_{t-1}
            }
            if (j > 0) {
#pragma unroll
                for (int r = 0; r < RPT; ++r) {
                    Snext[r] = scratch[sc_idx(j - 1, r)];
                }
            }
            // u = beta w (from the forward walk); dq_hat = S_t dO needs no G:
            // S_t = S' + k_hat u^T, S' = Diag(alpha) S_{t-1}
            const float b = pb[j];
            const float4 w4 = *reinterpret_cast<const float4*>(&pw[j * DVS + wc0]);
            const float4 u4 = make_float4(b * w4.x, b * w4.y, b * w4.z, b * w4.w);
            const float4 do4 = *reinterpret_cast<const float4*>(&pdo[j * DVS + wc0]);
            float dqv[RPT], dkv[RPT], dav[RPT];
            // column sums gk = G^T k_hat (G = dL/dS_t from the future)
            float4 ag = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int i = lane + 32 * r;
                const float a = pa[j * DK + i], kk = pk[j * DK + i];
                ag.x += kk * G[r].x; ag.y += kk * G[r].y; ag.z += kk * G[r].z; ag.w += kk * G[r].w;
                dqv[r] = (a * S[r].x + kk * u4.x) * do4.x + (a * S[r].y + kk * u4.y) * do4.y +
                         (a * S[r].z + kk * u4.z) * do4.z + (a * S[r].w + kk * u4.w) * do4.w;
            }
            // du = G^T kh + (qh . kh) dO, finished for column cw on lanes 8cw ..
            const float duc = warp_colsum4(ag, lane) + pqk[j] * pdo[j * DVS + wc0 + cw];
            const int64_t t = bos + i0 + j;
            if ((lane & 7) == 0) {
                p.dv[((size_t)t * H + h) * DV + col0 + wc0 + cw] = b * duc;
            }
            const float4 du4 = gather4(duc);
            // per state row: dkh, da and the new G
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int i = lane + 32 * r;
                const float a = pa[j * DK + i], kk = pk[j * DK + i], qq = pq[j * DK + i];
                const float4 sp = make_float4(a * S[r].x, a * S[r].y, a * S[r].z, a * S[r].w);
                float4 g = make_float4(G[r].x + qq * do4.x, G[r].y + qq * do4.y,
                                       G[r].z + qq * do4.z, G[r].w + qq * do4.w);
                dkv[r] = g.x * u4.x + g.y * u4.y + g.z * u4.z + g.w * u4.w -
                         b * (sp.x * du4.x + sp.y * du4.y + sp.z * du4.z + sp.w * du4.w);
                g.x -= b * kk * du4.x; g.y -= b * kk * du4.y;
                g.z -= b * kk * du4.z; g.w -= b * kk * du4.w;
                dav[r] = g.x * S[r].x + g.y * S[r].y + g.z * S[r].z + g.w * S[r].w;
                G[r] = make_float4(a * g.x, a * g.y, a * g.z, a * g.w);
            }
            // stage the warp's partials (its 4 columns) of dq_hat, dk_hat,
            // dalpha and dbeta for this token
            float* rw = red + ((size_t)slot * kBwWarps + w) * PW;
#pragma unroll
            for (int r = 0; r < RPT; ++r) {
                const int i = lane + 32 * r;
                rw[i] = dqv[r];
                rw[DK + i] = dkv[r];
                rw[2 * DK + i] = dav[r];
            }
            if (lane == 0) {
                rw[3 * DK] = du4.x * w4.x + du4.y * w4.y + du4.z * w4.z + du4.w * w4.w;
            }
            ++slot;
            if (slot == kBwRed || j == 0) {
                // the CTA's partials of the staged tokens: slot s holds token
                // j + slot - 1 - s; summed over the warps in a fixed order
                __syncthreads();
                for (int e = tid; e < slot * PW; e += kBwThreads) {
                    const int sl = e / PW, x = e - sl * PW;
                    float acc = 0.f;
#pragma unroll
                    for (int ww = 0; ww < kBwWarps; ++ww) {
                        acc += red[((size_t)sl * kBwWarps + ww) * PW + x];
                    }
                    const int64_t ts = bos + i0 + j + slot - 1 - sl;
                    p.part[(((size_t)split * p.total_T + ts) * H + h) * PW + x] = acc;
                }
                __syncthreads();   // the staging area is free again
                slot = 0;
            }
        }
    }
    // dL/dS_0 (this CTA's columns)
    {
        float4* dp = reinterpret_cast<float4*>(p.dS0 + ((size_t)n * H + h) * SS);
#pragma unroll
        for (int r = 0; r < RPT; ++r) {
            dp[st_idx(r)] = G[r];
        }
    }
}

// Per (token, head): the column partials of dqh, dkh, da and db added up,
// then the gate derivative (a = e^g, x = e^A z; g = -5 sigmoid(x): dx = da a
// (-5) sigmoid(x) (1 - sigmoid(x)); g = -softplus(x), a = sigmoid(-x): dx = -da
// a (1 - a)), dz = dx e^A, the token's share dx . x of dL/dA, and the
// normalisation derivative (xh = m x / sqrt(sum x^2 + eps): dx = m (rho dxh -
// rho^3 (x . dxh) x)).  One thread per key channel.
template <int DK, int NS, typename T>
__global__ void __launch_bounds__(DK)
kda_backward_finalize_kernel(const BackwardParams p) {
    constexpr int PW = 3 * DK + 1;
    constexpr int NW = DK / 32;
    __shared__ float red[NW][5];
    const int c = threadIdx.x, lane = c & 31, w = c >> 5;
    const int64_t th = blockIdx.x;               // t * H + h
    const int h = (int)(th % p.H);
    float dqh = 0.f, dkh = 0.f, da = 0.f, db = 0.f;
#pragma unroll
    for (int s = 0; s < NS; ++s) {
        const float* part = p.part + ((size_t)s * p.total_T * p.H + th) * PW;
        dqh += part[c];
        dkh += part[DK + c];
        da += part[2 * DK + c];
        if (c == 0) {
            db += part[3 * DK];
        }
    }
    const size_t o = (size_t)th * DK + c;
    const float qv = ldf(static_cast<const T*>(p.q), o);
    const float kv = ldf(static_cast<const T*>(p.k), o);
    const float eA = expf(p.A[h]);
    const float x = eA * ldf(static_cast<const T*>(p.z), o);
    float dx;
    if (p.softplus_gate) {
        const float a = bw_sigmoid(-x);
        dx = -da * a * (1.0f - a);
    } else {
        const float sg = bw_sigmoid(x);
        const float a = expf(kBwGmin * sg);
        dx = da * a * kBwGmin * sg * (1.0f - sg);
    }
    float v5[5] = {qv * qv, kv * kv, qv * dqh, kv * dkh, dx * x};
#pragma unroll
    for (int i = 0; i < 5; ++i) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            v5[i] += __shfl_xor_sync(0xffffffffu, v5[i], off);
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            red[w][i] = v5[i];
        }
    }
    __syncthreads();
    float t5[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int ww = 0; ww < NW; ++ww) {
#pragma unroll
        for (int i = 0; i < 5; ++i) {
            t5[i] += red[ww][i];
        }
    }
    p.dz[o] = dx * eA;
    if (p.l2norm) {
        const float rq = rsqrtf(t5[0] + kBwEps), rk = rsqrtf(t5[1] + kBwEps);
        p.dq[o] = p.scale * (rq * dqh - rq * rq * rq * t5[2] * qv);
        p.dk[o] = rk * dkh - rk * rk * rk * t5[3] * kv;
    } else {
        p.dq[o] = p.scale * dqh;
        p.dk[o] = dkh;
    }
    if (c == 0) {
        p.dbeta[th] = db;
        p.dA_tok[th] = t5[4];
    }
}

// dA[h] = the sum over all tokens of their shares, as a fixed tree (the same
// order on every call).  One CTA of 256 threads per head.
__global__ void __launch_bounds__(256)
kda_backward_dA_kernel(const float* dA_tok, float* dA, int64_t total_T, int H) {
    __shared__ float red[256];
    const int h = blockIdx.x;
    float s = 0.0f;
    for (int64_t t = threadIdx.x; t < total_T; t += 256) {
        s += dA_tok[(size_t)t * H + h];
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int width = 128; width > 0; width >>= 1) {
        if ((int)threadIdx.x < width) {
            red[threadIdx.x] += red[threadIdx.x + width];
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        dA[h] = red[0];
    }
}

template <int DK, int DV, typename T>
cudaError_t launch_main(const BackwardParams& p, dim3 grid, cudaStream_t stream) {
    constexpr size_t smem = chunk_stage_bytes<DK, T>();
    // the attribute belongs to the current device: set on every launch
    const cudaError_t e = cudaFuncSetAttribute(kda_backward_kernel<DK, DV, T>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
    if (e != cudaSuccess) {
        return e;
    }
    kda_backward_kernel<DK, DV, T><<<grid, kBwThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t launch_dims(const BackwardParams& p, int dtype, cudaStream_t stream) {
    constexpr int NS = DV / kBwCols;
    const dim3 grid((unsigned)((int64_t)p.N * p.H * NS));
    const int64_t tokens = (int64_t)p.total_T * p.H;
    if (dtype == 0) {
        const cudaError_t e = launch_main<DK, DV, float>(p, grid, stream);
        if (e != cudaSuccess) {
            return e;
        }
        if (tokens > 0) {
            kda_backward_finalize_kernel<DK, NS, float><<<(unsigned)tokens, DK, 0, stream>>>(p);
        }
    } else {
        const cudaError_t e = launch_main<DK, DV, __nv_bfloat16>(p, grid, stream);
        if (e != cudaSuccess) {
            return e;
        }
        if (tokens > 0) {
            kda_backward_finalize_kernel<DK, NS, __nv_bfloat16>
                <<<(unsigned)tokens, DK, 0, stream>>>(p);
        }
    }
    return cudaGetLastError();
}

template <int DK>
cudaError_t launch_dk(const BackwardParams& p, int d_v, int dtype, cudaStream_t stream) {
    switch (d_v) {
        case 32: return launch_dims<DK, 32>(p, dtype, stream);
        case 64: return launch_dims<DK, 64>(p, dtype, stream);
        case 128: return launch_dims<DK, 128>(p, dtype, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_backward_dA(const float* dA_tok, float* dA, int64_t total_T, int H,
                               cudaStream_t stream) {
    kda_backward_dA_kernel<<<H, 256, 0, stream>>>(dA_tok, dA, total_T, H);
    return cudaGetLastError();
}

cudaError_t launch_backward(const BackwardParams& p, int d_k, int d_v, int dtype,
                            cudaStream_t stream) {
    if (p.N > 0) {
        cudaError_t err;
        switch (d_k) {
            case 32: err = launch_dk<32>(p, d_v, dtype, stream); break;
            case 64: err = launch_dk<64>(p, d_v, dtype, stream); break;
            case 128: err = launch_dk<128>(p, d_v, dtype, stream); break;
            default: return cudaErrorInvalidValue;
        }
        if (err != cudaSuccess) {
            return err;
        }
    }
    kda_backward_dA_kernel<<<p.H, 256, 0, stream>>>(p.dA_tok, p.dA, p.total_T, p.H);
    return cudaGetLastError();
}

}  // namespace kda
