/*
 * kda_oracle.c -- fp64 CPU oracle for Kimi Delta Attention (KDA).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path links,
 * loads or calls this file: only the tests, the smoke check and the timed
 * CPU baseline of the benchmark do.  It shares no code, header, table or
 * constant with the CUDA library.
 *
 * What it computes (sources are the pages' titles and sections):
 *
 *  - "Kimi K3 Open Weights: What Is Actually New In Its 2.8 Trillion
 *    Parameter Architecture", section 1 "Kimi Delta Attention is a real new
 *    kernel family", displayed recurrence:
 *        S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *        o_t = S_t^T q_t                       (read after the write)
 *  - same section, gate equation:
 *        g_t = g_min * sigmoid(e^A z_t),  alpha_t = e^{g_t},  g_min = -5
 *  - same section, prefill bullet: Q/K normalization is part of the KDA op.
 *
 * Readings where the pages are silent (each one is applied identically by
 * the CUDA library, which implements it independently):
 *  - q and k are L2-normalised per token and head inside the op when
 *    `l2norm` is set:  x_hat = x / sqrt(sum x^2 + eps), eps = 1e-6; q is
 *    then multiplied by `scale` (default 1.0).
 *  - A is one scalar per head; e^A multiplies every channel of z.
 *  - z, g and alpha have d_k channels (Diag(alpha) left-multiplies the
 *    d_k x d_v state).
 *  - beta is given already in [0, 1].
 *  - the state is stored [N, H, d_k, d_v] row-major (d_v contiguous).
 *
 * Two forms are provided:
 *  kda_oracle_recurrent  -- the token loop, written straight from the
 *                           recurrence.  This is THE oracle.
 *  kda_oracle_chunked    -- the chunkwise form ("parallel within chunks,
 *                           recurrent between"), derived by unrolling the
 *                           recurrence inside a chunk; it exists only so
 *                           that tests can pin the chunk algebra against
 *                           the recurrent form.  It uses the pairwise decay
 *                           factors exp(gamma_r - gamma_i) directly, with no
 *                           reciprocal rescaling.
 * Both are fp64 throughout; every input arrives already converted exactly
 * from its stored bf16/fp32 value.
 *
 * kda_oracle_backward is reverse mode of the token loop (the gradients of a
 * loss through every step, in reverse), kda_oracle_short_conv the short
 * convolutions that precede the step.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define KDA_ORACLE_GMIN (-5.0)

/* sigmoid, evaluated on the branch that cannot overflow. */
static double oracle_sigmoid(double x)
{
    if (x >= 0.0) {
        return 1.0 / (1.0 + exp(-x));
    }
    double e = exp(x);
    return e / (1.0 + e);
}

/* Kimi Linear's unbounded negative-softplus decay, which the same section
 * says K3 replaced: g = -softplus(e^A * z) = -log(1 + e^{e^A z}) (the pages
 * give its name, not its argument; the argument e^A z of the K3 gate is the
 * reading).  Evaluated without overflow: softplus(x) = max(x, 0) + log1p(e^-|x|). */
static double oracle_neg_softplus(double x)
{
    return -((x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x))));
}

double kda_oracle_gate_softplus(double z, double A)
{
    return oracle_neg_softplus(exp(A) * z);
}

/* Gate equation of section 1: g = g_min * sigmoid(e^A * z). */
double kda_oracle_gate(double z, double A)
{
    return KDA_ORACLE_GMIN * oracle_sigmoid(exp(A) * z);
}

void kda_oracle_gate_vec(const double* z, int64_t n, double A, double* g)
{
    for (int64_t i = 0; i < n; ++i) {
        g[i] = kda_oracle_gate(z[i], A);
    }
}

/* x_hat = mult * x / sqrt(sum x^2 + eps)  (or mult * x when l2norm == 0). */
static void oracle_normalise(const double* x, int d, int l2norm, double eps,
                             double mult, double* out)
{
    double inv = 1.0;
    if (l2norm) {
        double ss = 0.0;
        for (int c = 0; c < d; ++c) {
            ss += x[c] * x[c];
        }
        inv = 1.0 / sqrt(ss + eps);
    }
    for (int c = 0; c < d; ++c) {
        out[c] = mult * x[c] * inv;
    }
}

typedef struct {
    const double* q;      /* [total_T, H, dk] */
    const double* k;      /* [total_T, H, dk] */
    const double* v;      /* [total_T, H, dv] */
    const double* z;      /* [total_T, H, dk] */
    const double* beta;   /* [total_T, H]     */
    const double* A;      /* [H]              */
    const double* S0;     /* [N, H, dk, dv] or NULL */
    const int64_t* cu;    /* [N + 1]          */
    int N, H, dk, dv;
    double scale, eps;
    int l2norm;
    int softplus;         /* 1: Kimi Linear's negative-softplus gate instead of the K3 one */
    int chunk;            /* 0 = recurrent form, >0 = chunked form with this C */
    double* o;            /* [total_T, H, dv] */
    double* S_out;        /* [N, H, dk, dv] or NULL */
    const int32_t* units; /* optional list of (n, h) pairs; NULL = all */
    int64_t ckpt_interval;       /* > 0: record S after every this many tokens of a sequence */
    const int64_t* ckpt_base;    /* [N]: index of each sequence's first checkpoint */
    double* ckpt;                /* [n_checkpoints, H, dk, dv] */
    int64_t n_units;
    /* reverse mode (kda_oracle_backward): upstream gradients in, gradients out */
    int backward;
    const double* dO;     /* [total_T, H, dv] */
    const double* dSf;    /* [N, H, dk, dv] or NULL */
    double* gq;           /* [total_T, H, dk] */
    double* gk;
    double* gv;           /* [total_T, H, dv] */
    double* gz;           /* [total_T, H, dk] */
    double* gbeta;        /* [total_T, H] */
    double* gA_part;      /* [N, H]: this pair's share of dL/dA_h */
    double* gS0;          /* [N, H, dk, dv] */
    int64_t next;         /* work counter, guarded by mu */
    pthread_mutex_t mu;
    int failed;
} oracle_job;

/* ---- recurrent form: one (sequence, head) pair ------------------------- */
static int oracle_unit_recurrent(oracle_job* J, int n, int h)
{
    const int dk = J->dk, dv = J->dv, H = J->H;
    double* S = (double*)malloc(sizeof(double) * (size_t)dk * dv);
    double* qh = (double*)malloc(sizeof(double) * dk);
    double* kh = (double*)malloc(sizeof(double) * dk);
    double* alpha = (double*)malloc(sizeof(double) * dk);
    double* u = (double*)malloc(sizeof(double) * dv);
    if (!S || !qh || !kh || !alpha || !u) {
        free(S); free(qh); free(kh); free(alpha); free(u);
        return -1;
    }
    if (J->S0) {
        memcpy(S, J->S0 + ((size_t)n * H + h) * dk * dv, sizeof(double) * dk * dv);
    } else {
        memset(S, 0, sizeof(double) * dk * dv);
    }
    const double eA = exp(J->A[h]);
    for (int64_t t = J->cu[n]; t < J->cu[n + 1]; ++t) {
        const size_t rowk = ((size_t)t * H + h) * dk;
        const size_t rowv = ((size_t)t * H + h) * dv;
        oracle_normalise(J->q + rowk, dk, J->l2norm, J->eps, J->scale, qh);
        oracle_normalise(J->k + rowk, dk, J->l2norm, J->eps, 1.0, kh);
        for (int c = 0; c < dk; ++c) {
            /* gate equation (same as kda_oracle_gate, with e^A hoisted) */
            const double x = eA * J->z[rowk + c];
            alpha[c] = exp(J->softplus ? oracle_neg_softplus(x)
                                       : KDA_ORACLE_GMIN * oracle_sigmoid(x));
        }
        const double b = J->beta[(size_t)t * H + h];
        /* S' = Diag(alpha) S */
        for (int c = 0; c < dk; ++c) {
            for (int j = 0; j < dv; ++j) {
                S[(size_t)c * dv + j] *= alpha[c];
            }
        }
        /* u = beta (v - S'^T k);  S = S' + k u^T  ==  (I - beta k k^T) S' + beta k v^T */
        for (int j = 0; j < dv; ++j) {
            double r = 0.0;
            for (int c = 0; c < dk; ++c) {
                r += S[(size_t)c * dv + j] * kh[c];
            }
            u[j] = b * (J->v[rowv + j] - r);
        }
        for (int c = 0; c < dk; ++c) {
            for (int j = 0; j < dv; ++j) {
                S[(size_t)c * dv + j] += kh[c] * u[j];
            }
        }
        /* o_t = S_t^T q_t */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c) {
                acc += S[(size_t)c * dv + j] * qh[c];
            }
            J->o[rowv + j] = acc;
        }
        /* checkpoint: the state after the first m * ckpt_interval tokens */
        const int64_t done = t - J->cu[n] + 1;
        if (J->ckpt && J->ckpt_interval > 0 && done % J->ckpt_interval == 0) {
            const int64_t idx = J->ckpt_base[n] + done / J->ckpt_interval - 1;
            memcpy(J->ckpt + ((size_t)idx * H + h) * dk * dv, S, sizeof(double) * dk * dv);
        }
    }
    if (J->S_out) {
        memcpy(J->S_out + ((size_t)n * H + h) * dk * dv, S, sizeof(double) * dk * dv);
    }
    free(S); free(qh); free(kh); free(alpha); free(u);
    return 0;
}

/* ---- chunked form: one (sequence, head) pair ----------------------------
 * Inside a chunk of C tokens with start state S0 and inclusive cumulative
 * log-decay gamma_r = sum_{t<=r} g_t (per channel), unrolling the recurrence
 * gives, with u_r = beta_r (v_r - (Diag(alpha_r) S_{r-1})^T k_r):
 *   S_r = Diag(e^{gamma_r}) S0 + sum_{i<=r} Diag(e^{gamma_r - gamma_i}) k_i u_i^T
 *   u_r + beta_r sum_{i<r} Akk[r,i] u_i = beta_r (v_r - S0^T (k_r * e^{gamma_r}))
 *   o_r = S0^T (q_r * e^{gamma_r}) + sum_{i<=r} Aqk[r,i] u_i
 *   S_C = Diag(e^{gamma_C}) S0 + sum_i (k_i * e^{gamma_C - gamma_i}) u_i^T
 * with Akk[r,i] = <k_r * e^{gamma_r - gamma_i}, k_i>, Aqk[r,i] = <q_r * e^{gamma_r - gamma_i}, k_i>.
 * The triangular system is solved by forward substitution, row by row. */
static int oracle_unit_chunked(oracle_job* J, int n, int h)
{
    const int dk = J->dk, dv = J->dv, H = J->H, C = J->chunk;
    const size_t SZ = (size_t)dk * dv;
    double* S = (double*)malloc(sizeof(double) * SZ);
    double* Snew = (double*)malloc(sizeof(double) * SZ);
    double* Q = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* K = (double*)malloc(sizeof(double) * (size_t)C * dk);
    double* G = (double*)malloc(sizeof(double) * (size_t)C * dk); /* gamma */
    double* U = (double*)malloc(sizeof(double) * (size_t)C * dv);
    double* Akk = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* Aqk = (double*)malloc(sizeof(double) * (size_t)C * C);
    double* bet = (double*)malloc(sizeof(double) * C);
    if (!S || !Snew || !Q || !K || !G || !U || !Akk || !Aqk || !bet) {
        free(S); free(Snew); free(Q); free(K); free(G); free(U); free(Akk); free(Aqk); free(bet);
        return -1;
    }
    if (J->S0) {
        memcpy(S, J->S0 + ((size_t)n * H + h) * SZ, sizeof(double) * SZ);
    } else {
        memset(S, 0, sizeof(double) * SZ);
    }
    const int64_t bos = J->cu[n], eos = J->cu[n + 1];
    for (int64_t t0 = bos; t0 < eos; t0 += C) {
        const int L = (int)((eos - t0) < C ? (eos - t0) : C);
        /* normalised q, k; cumulative gate; beta */
        for (int r = 0; r < L; ++r) {
            const size_t rowk = ((size_t)(t0 + r) * H + h) * dk;
            oracle_normalise(J->q + rowk, dk, J->l2norm, J->eps, J->scale, Q + (size_t)r * dk);
            oracle_normalise(J->k + rowk, dk, J->l2norm, J->eps, 1.0, K + (size_t)r * dk);
            for (int c = 0; c < dk; ++c) {
                const double g = J->softplus ? kda_oracle_gate_softplus(J->z[rowk + c], J->A[h])
                                             : kda_oracle_gate(J->z[rowk + c], J->A[h]);
                G[(size_t)r * dk + c] = (r == 0 ? 0.0 : G[(size_t)(r - 1) * dk + c]) + g;
            }
            bet[r] = J->beta[(size_t)(t0 + r) * H + h];
        }
        /* pairwise intra-chunk interactions */
        for (int r = 0; r < L; ++r) {
            for (int i = 0; i < L; ++i) {
                double skk = 0.0, sqk = 0.0;
                if (i <= r) {
                    for (int c = 0; c < dk; ++c) {
                        const double dec = exp(G[(size_t)r * dk + c] - G[(size_t)i * dk + c]);
                        skk += K[(size_t)r * dk + c] * dec * K[(size_t)i * dk + c];
                        sqk += Q[(size_t)r * dk + c] * dec * K[(size_t)i * dk + c];
                    }
                }
                Akk[(size_t)r * C + i] = (i < r) ? skk : 0.0;
                Aqk[(size_t)r * C + i] = (i <= r) ? sqk : 0.0;
            }
        }
        /* forward substitution: u_r = beta_r (v_r - S0^T k_r^+) - beta_r sum_{i<r} Akk[r,i] u_i */
        for (int r = 0; r < L; ++r) {
            const size_t rowv = ((size_t)(t0 + r) * H + h) * dv;
            for (int j = 0; j < dv; ++j) {
                double sk = 0.0;
                for (int c = 0; c < dk; ++c) {
                    sk += S[(size_t)c * dv + j] * K[(size_t)r * dk + c] * exp(G[(size_t)r * dk + c]);
                }
                double acc = J->v[rowv + j] - sk;
                double corr = 0.0;
                for (int i = 0; i < r; ++i) {
                    corr += Akk[(size_t)r * C + i] * U[(size_t)i * dv + j];
                }
                U[(size_t)r * dv + j] = bet[r] * (acc - corr);
            }
        }
        /* outputs */
        for (int r = 0; r < L; ++r) {
            const size_t rowv = ((size_t)(t0 + r) * H + h) * dv;
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int c = 0; c < dk; ++c) {
                    acc += S[(size_t)c * dv + j] * Q[(size_t)r * dk + c] * exp(G[(size_t)r * dk + c]);
                }
                for (int i = 0; i <= r; ++i) {
                    acc += Aqk[(size_t)r * C + i] * U[(size_t)i * dv + j];
                }
                J->o[rowv + j] = acc;
            }
        }
        /* state carried to the next chunk */
        for (int c = 0; c < dk; ++c) {
            const double gC = G[(size_t)(L - 1) * dk + c];
            for (int j = 0; j < dv; ++j) {
                double acc = exp(gC) * S[(size_t)c * dv + j];
                for (int i = 0; i < L; ++i) {
                    acc += K[(size_t)i * dk + c] * exp(gC - G[(size_t)i * dk + c]) * U[(size_t)i * dv + j];
                }
                Snew[(size_t)c * dv + j] = acc;
            }
        }
        memcpy(S, Snew, sizeof(double) * SZ);
    }
    if (J->S_out) {
        memcpy(J->S_out + ((size_t)n * H + h) * SZ, S, sizeof(double) * SZ);
    }
    free(S); free(Snew); free(Q); free(K); free(G); free(U); free(Akk); free(Aqk); free(bet);
    return 0;
}

/* ---- reverse mode of the recurrent form: one (sequence, head) pair ------
 * Given dL/do_t for every token and dL/dS_T, the gradients of L with respect
 * to q, k, v, z, beta, A (this pair's share) and S_0, by the chain rule taken
 * through the forward steps in reverse order.  With G = dL/dS_t:
 *   o_t = S_t^T qh          G += qh do^T;          dqh = S_t do
 *   S_t = S' + kh u^T       du = G^T kh;           dkh = G u;      dS' = G
 *   u = b (v - S'^T kh)     dv = b du;  db = du . (v - S'^T kh);
 *                           dS' -= b kh du^T;      dkh -= b S' du
 *   S' = Diag(a) S_{t-1}    da[c] = sum_j dS'[c][j] S_{t-1}[c][j];  G = Diag(a) dS'
 * then through the gate (a = e^g, x = e^A z; g = -5 sigma(x): dx = da a (-5)
 * sigma(x) (1 - sigma(x)); g = -softplus(x), a = sigma(-x): dx = -da a (1 - a);
 * dz = dx e^A, dA += dx x) and the normalisation (xh = m rho x with rho =
 * (sum x^2 + eps)^(-1/2): dx = m (rho dxh - rho^3 (x . dxh) x)).  The forward
 * pass keeps every state S_0 .. S_T of the pair. */
static void oracle_normalise_backward(const double* x, const double* dxh, int d, int l2norm,
                                      double eps, double mult, double* dx)
{
    if (!l2norm) {
        for (int c = 0; c < d; ++c) {
            dx[c] = mult * dxh[c];
        }
        return;
    }
    double ss = 0.0, xd = 0.0;
    for (int c = 0; c < d; ++c) {
        ss += x[c] * x[c];
        xd += x[c] * dxh[c];
    }
    const double rho = 1.0 / sqrt(ss + eps);
    for (int c = 0; c < d; ++c) {
        dx[c] = mult * (rho * dxh[c] - rho * rho * rho * xd * x[c]);
    }
}

static int oracle_unit_backward(oracle_job* J, int n, int h)
{
    const int dk = J->dk, dv = J->dv, H = J->H;
    const int64_t bos = J->cu[n], T = J->cu[n + 1] - bos;
    const size_t SS = (size_t)dk * dv;
    double* Sall = (double*)malloc(sizeof(double) * SS * (size_t)(T + 1));
    double* qh = (double*)malloc(sizeof(double) * dk * (size_t)(T > 0 ? T : 1));
    double* kh = (double*)malloc(sizeof(double) * dk * (size_t)(T > 0 ? T : 1));
    double* al = (double*)malloc(sizeof(double) * dk * (size_t)(T > 0 ? T : 1));
    double* uu = (double*)malloc(sizeof(double) * dv * (size_t)(T > 0 ? T : 1));
    double* G = (double*)malloc(sizeof(double) * SS);
    double* Sp = (double*)malloc(sizeof(double) * SS);
    double* du = (double*)malloc(sizeof(double) * dv);
    double* dqh = (double*)malloc(sizeof(double) * dk);
    double* dkh = (double*)malloc(sizeof(double) * dk);
    double* da = (double*)malloc(sizeof(double) * dk);
    if (!Sall || !qh || !kh || !al || !uu || !G || !Sp || !du || !dqh || !dkh || !da) {
        free(Sall); free(qh); free(kh); free(al); free(uu); free(G); free(Sp);
        free(du); free(dqh); free(dkh); free(da);
        return -1;
    }
    const double eA = exp(J->A[h]);
    /* forward, keeping S_0 .. S_T */
    if (J->S0) {
        memcpy(Sall, J->S0 + ((size_t)n * H + h) * SS, sizeof(double) * SS);
    } else {
        memset(Sall, 0, sizeof(double) * SS);
    }
    for (int64_t i = 0; i < T; ++i) {
        const int64_t t = bos + i;
        const size_t rowk = ((size_t)t * H + h) * dk, rowv = ((size_t)t * H + h) * dv;
        oracle_normalise(J->q + rowk, dk, J->l2norm, J->eps, J->scale, qh + i * dk);
        oracle_normalise(J->k + rowk, dk, J->l2norm, J->eps, 1.0, kh + i * dk);
        for (int c = 0; c < dk; ++c) {
            const double x = eA * J->z[rowk + c];
            al[i * dk + c] = exp(J->softplus ? oracle_neg_softplus(x)
                                             : KDA_ORACLE_GMIN * oracle_sigmoid(x));
        }
        const double b = J->beta[(size_t)t * H + h];
        const double* Sprev = Sall + (size_t)i * SS;
        double* Snext = Sall + (size_t)(i + 1) * SS;
        for (int c = 0; c < dk; ++c) {
            for (int j = 0; j < dv; ++j) {
                Snext[(size_t)c * dv + j] = al[i * dk + c] * Sprev[(size_t)c * dv + j];
            }
        }
        for (int j = 0; j < dv; ++j) {
            double r = 0.0;
            for (int c = 0; c < dk; ++c) {
                r += Snext[(size_t)c * dv + j] * kh[i * dk + c];
            }
            uu[i * dv + j] = b * (J->v[rowv + j] - r);
        }
        for (int c = 0; c < dk; ++c) {
            for (int j = 0; j < dv; ++j) {
                Snext[(size_t)c * dv + j] += kh[i * dk + c] * uu[i * dv + j];
            }
        }
    }
    /* reverse */
    if (J->dSf) {
        memcpy(G, J->dSf + ((size_t)n * H + h) * SS, sizeof(double) * SS);
    } else {
        memset(G, 0, sizeof(double) * SS);
    }
    double gA = 0.0;
    for (int64_t i = T - 1; i >= 0; --i) {
        const int64_t t = bos + i;
        const size_t rowk = ((size_t)t * H + h) * dk, rowv = ((size_t)t * H + h) * dv;
        const double* dO = J->dO + rowv;
        const double* Sprev = Sall + (size_t)i * SS;
        const double* St = Sall + (size_t)(i + 1) * SS;
        const double* q_ = qh + i * dk;
        const double* k_ = kh + i * dk;
        const double* a_ = al + i * dk;
        const double* u_ = uu + i * dv;
        const double b = J->beta[(size_t)t * H + h];
        /* o_t = S_t^T qh */
        for (int c = 0; c < dk; ++c) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                G[(size_t)c * dv + j] += q_[c] * dO[j];
                acc += St[(size_t)c * dv + j] * dO[j];
            }
            dqh[c] = acc;
        }
        /* S_t = S' + kh u^T */
        for (int j = 0; j < dv; ++j) {
            double acc = 0.0;
            for (int c = 0; c < dk; ++c) {
                acc += G[(size_t)c * dv + j] * k_[c];
            }
            du[j] = acc;
        }
        for (int c = 0; c < dk; ++c) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                acc += G[(size_t)c * dv + j] * u_[j];
            }
            dkh[c] = acc;
        }
        /* u = b (v - S'^T kh) */
        for (int c = 0; c < dk; ++c) {
            for (int j = 0; j < dv; ++j) {
                Sp[(size_t)c * dv + j] = a_[c] * Sprev[(size_t)c * dv + j];
            }
        }
        double db = 0.0;
        for (int j = 0; j < dv; ++j) {
            double r = 0.0;
            for (int c = 0; c < dk; ++c) {
                r += Sp[(size_t)c * dv + j] * k_[c];
            }
            J->gv[rowv + j] = b * du[j];
            db += du[j] * (J->v[rowv + j] - r);
        }
        J->gbeta[(size_t)t * H + h] = db;
        for (int c = 0; c < dk; ++c) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                G[(size_t)c * dv + j] -= b * k_[c] * du[j];
                acc += Sp[(size_t)c * dv + j] * du[j];
            }
            dkh[c] -= b * acc;
        }
        /* S' = Diag(a) S_{t-1} */
        for (int c = 0; c < dk; ++c) {
            double acc = 0.0;
            for (int j = 0; j < dv; ++j) {
                acc += G[(size_t)c * dv + j] * Sprev[(size_t)c * dv + j];
                G[(size_t)c * dv + j] *= a_[c];
            }
            da[c] = acc;
        }
        /* gate and normalisation */
        for (int c = 0; c < dk; ++c) {
            const double x = eA * J->z[rowk + c];
            double dx;
            if (J->softplus) {
                dx = -da[c] * a_[c] * (1.0 - a_[c]);
            } else {
                const double sg = oracle_sigmoid(x);
                dx = da[c] * a_[c] * KDA_ORACLE_GMIN * sg * (1.0 - sg);
            }
            J->gz[rowk + c] = dx * eA;
            gA += dx * x;
        }
        oracle_normalise_backward(J->q + rowk, dqh, dk, J->l2norm, J->eps, J->scale,
                                  J->gq + rowk);
        oracle_normalise_backward(J->k + rowk, dkh, dk, J->l2norm, J->eps, 1.0, J->gk + rowk);
    }
    memcpy(J->gS0 + ((size_t)n * H + h) * SS, G, sizeof(double) * SS);
    J->gA_part[(size_t)n * H + h] = gA;
    free(Sall); free(qh); free(kh); free(al); free(uu); free(G); free(Sp);
    free(du); free(dqh); free(dkh); free(da);
    return 0;
}

static void* oracle_worker(void* arg)
{
    oracle_job* J = (oracle_job*)arg;
    const int64_t total = J->units ? J->n_units : (int64_t)J->N * J->H;
    for (;;) {
        pthread_mutex_lock(&J->mu);
        const int64_t w = J->next++;
        pthread_mutex_unlock(&J->mu);
        if (w >= total) {
            break;
        }
        int n, h;
        if (J->units) {
            n = J->units[2 * w];
            h = J->units[2 * w + 1];
        } else {
            n = (int)(w / J->H);
            h = (int)(w % J->H);
        }
        const int rc = J->backward ? oracle_unit_backward(J, n, h)
                       : J->chunk > 0 ? oracle_unit_chunked(J, n, h)
                                      : oracle_unit_recurrent(J, n, h);
        if (rc != 0) {
            pthread_mutex_lock(&J->mu);
            J->failed = 1;
            pthread_mutex_unlock(&J->mu);
        }
    }
    return NULL;
}

static int oracle_run(oracle_job* J, int nthreads)
{
    if (J->N < 0 || J->H <= 0 || J->dk <= 0 || J->dv <= 0 || !J->cu) {
        return -1;
    }
    for (int n = 0; n < J->N; ++n) {
        if (J->cu[n + 1] < J->cu[n]) {
            return -1;
        }
    }
    if (nthreads <= 0) {
        long np = sysconf(_SC_NPROCESSORS_ONLN);
        nthreads = np > 0 ? (int)np : 1;
    }
    const int64_t total = J->units ? J->n_units : (int64_t)J->N * J->H;
    if (nthreads > total) {
        nthreads = total > 0 ? (int)total : 1;
    }
    pthread_mutex_init(&J->mu, NULL);
    J->next = 0;
    J->failed = 0;
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * nthreads);
    if (!th) {
        pthread_mutex_destroy(&J->mu);
        return -1;
    }
    int started = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (pthread_create(&th[i], NULL, oracle_worker, J) == 0) {
            ++started;
        }
    }
    if (started == 0) {
        oracle_worker(J);
    }
    for (int i = 0; i < started; ++i) {
        pthread_join(th[i], NULL);
    }
    free(th);
    pthread_mutex_destroy(&J->mu);
    return J->failed ? -2 : started > 0 ? started : 1;
}

/* Returns the number of threads used (> 0), or a negative value on error.
 * `l2norm`: bit 0 = L2-normalise q and k, bit 1 = the negative-softplus gate.
 * `units`: NULL for every (sequence, head) pair, else n_units (n, h) pairs;
 * outputs are written only for the listed pairs. */
int kda_oracle_run(const double* q, const double* k, const double* v, const double* z,
                   const double* beta, const double* A, const double* S0,
                   const int64_t* cu_seqlens, int N, int H, int dk, int dv,
                   double scale, int l2norm, double eps, int chunk,
                   const int32_t* units, int64_t n_units,
                   double* o, double* S_out, int nthreads)
{
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.z = z; J.beta = beta; J.A = A; J.S0 = S0;
    J.cu = cu_seqlens; J.N = N; J.H = H; J.dk = dk; J.dv = dv;
    J.scale = scale; J.eps = eps; J.l2norm = l2norm & 1; J.softplus = (l2norm >> 1) & 1;
    J.chunk = chunk;
    J.o = o; J.S_out = S_out; J.units = units; J.n_units = n_units;
    return oracle_run(&J, nthreads);
}

/* kda_oracle_run plus state checkpoints (recurrent form only): for every
 * sequence n and m >= 1 with m * ckpt_interval <= its length, the state after
 * its first m * ckpt_interval tokens goes to ckpt[(ckpt_base[n] + m - 1), h]. */
int kda_oracle_run_ckpt(const double* q, const double* k, const double* v, const double* z,
                        const double* beta, const double* A, const double* S0,
                        const int64_t* cu_seqlens, int N, int H, int dk, int dv,
                        double scale, int l2norm, double eps,
                        const int32_t* units, int64_t n_units,
                        double* o, double* S_out, int64_t ckpt_interval,
                        const int64_t* ckpt_base, double* ckpt, int nthreads)
{
    if (ckpt_interval <= 0 || !ckpt_base || !ckpt) {
        return -1;
    }
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.z = z; J.beta = beta; J.A = A; J.S0 = S0;
    J.cu = cu_seqlens; J.N = N; J.H = H; J.dk = dk; J.dv = dv;
    J.scale = scale; J.eps = eps; J.l2norm = l2norm & 1; J.softplus = (l2norm >> 1) & 1;
    J.chunk = 0;
    J.o = o; J.S_out = S_out; J.units = units; J.n_units = n_units;
    J.ckpt_interval = ckpt_interval; J.ckpt_base = ckpt_base; J.ckpt = ckpt;
    return oracle_run(&J, nthreads);
}

/* ---- short convolution ---------------------------------------------------
 * Section 1 lists "short convolutions" first among the prefill steps and
 * keeps a "convolution state" persistent through decode; the section "Why
 * 104B active still understates the systems problem" counts a fixed-size
 * short-convolution state per request and layer.  The pages give no formula.  Reading: a causal,
 * depthwise convolution along time of width W on every channel,
 *     y_t[c] = sum_{j=0}^{W-1} w[c][j] * x_{t-(W-1)+j}[c]
 * (w[c][W-1] weights the current token), optionally followed by SiLU,
 * y * sigmoid(y).  Inputs before a sequence's first token come from that
 * sequence's conv state, whose row r (0 <= r < W-1) holds the input at
 * position bos - (W-1) + r (oldest first); with no state they are zero.  The
 * final conv state is the last W-1 inputs of the sequence, taking rows of
 * the initial state where the sequence is shorter than W-1.
 *
 * Layouts: x, y [total_T, C]; w [C, W]; state_in, state_out [N, W-1, C]
 * (state_in may be NULL = zeros; state_out may be NULL).  Returns 0, or -1
 * on a bad argument. */
int kda_oracle_short_conv(const double* x, int64_t total_T, int64_t C,
                          const int64_t* cu_seqlens, int N, const double* w, int W,
                          const double* state_in, int silu, double* y, double* state_out)
{
    if (W < 1 || C < 0 || N < 0 || !cu_seqlens || cu_seqlens[0] != 0 ||
        cu_seqlens[N] != total_T) {
        return -1;
    }
    const int R = W - 1;  /* rows of conv state */
    for (int n = 0; n < N; ++n) {
        const int64_t bos = cu_seqlens[n], eos = cu_seqlens[n + 1];
        if (eos < bos) {
            return -1;
        }
        for (int64_t c = 0; c < C; ++c) {
            /* input at absolute position tau of this sequence (tau < eos) */
#define ORACLE_CONV_IN(tau)                                                        \
    ((tau) >= bos ? x[(tau) * C + c]                                               \
                  : (state_in ? state_in[((int64_t)n * R + ((tau) - bos + R)) * C + c] \
                              : 0.0))
            for (int64_t t = bos; t < eos; ++t) {
                double acc = 0.0;
                for (int j = 0; j < W; ++j) {
                    acc += w[c * W + j] * ORACLE_CONV_IN(t - R + j);
                }
                y[t * C + c] = silu ? acc * oracle_sigmoid(acc) : acc;
            }
            if (state_out) {
                for (int r = 0; r < R; ++r) {
                    state_out[((int64_t)n * R + r) * C + c] = ORACLE_CONV_IN(eos - R + r);
                }
            }
#undef ORACLE_CONV_IN
        }
    }
    return 0;
}

/* Gradients of L = sum_t do_t . o_t + dSf . S_T (reverse mode of the
 * recurrent form, oracle_unit_backward) for every (sequence, head) pair:
 * gq, gk, gz [total_T, H, dk]; gv [total_T, H, dv]; gbeta [total_T, H];
 * gA_part [N, H] (dL/dA_h is the sum over n); gS0 [N, H, dk, dv].
 * `flags` as kda_oracle_run's `l2norm` (bit 0 normalise, bit 1 softplus
 * gate); dSf may be NULL (zero).  Returns the threads used or a negative
 * value on error. */
int kda_oracle_backward(const double* q, const double* k, const double* v, const double* z,
                        const double* beta, const double* A, const double* S0,
                        const int64_t* cu_seqlens, int N, int H, int dk, int dv,
                        double scale, int flags, double eps, const double* dO,
                        const double* dSf, double* gq, double* gk, double* gv, double* gz,
                        double* gbeta, double* gA_part, double* gS0, int nthreads)
{
    if (!dO || !gq || !gk || !gv || !gz || !gbeta || !gA_part || !gS0) {
        return -1;
    }
    oracle_job J;
    memset(&J, 0, sizeof(J));
    J.q = q; J.k = k; J.v = v; J.z = z; J.beta = beta; J.A = A; J.S0 = S0;
    J.cu = cu_seqlens; J.N = N; J.H = H; J.dk = dk; J.dv = dv;
    J.scale = scale; J.eps = eps; J.l2norm = flags & 1; J.softplus = (flags >> 1) & 1;
    J.backward = 1; J.dO = dO; J.dSf = dSf;
    J.gq = gq; J.gk = gk; J.gv = gv; J.gz = gz; J.gbeta = gbeta; J.gA_part = gA_part;
    J.gS0 = gS0;
    return oracle_run(&J, nthreads);
}
