"""fp64 CPU oracle for Kimi Delta Attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it, and
the two share no code: this side is a plain C token loop in fp64
(``kda_oracle.c``) plus this ctypes wrapper.

Sources (page titles and sections):
  * "Kimi K3 Open Weights: What Is Actually New In Its 2.8 Trillion Parameter
    Architecture", section 1 "Kimi Delta Attention is a real new kernel
    family": the delta-rule recurrence with o_t = S_t^T q_t, the bounded gate
    g = -5 sigmoid(e^A z), alpha = e^g, and Q/K normalisation inside the op;
    the short convolutions before it and their persistent conv state (the
    prefill and decode bullets of the same section); and the gradients of a
    loss through the recurrence (reverse mode, for the training form), also
    in the chunked form a chunk-parallel backward computes.

Every function here is pinned by ``tests/test_oracle_pins.py`` against closed
forms, brute force and invariants that do not reuse this code.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

EPS = 1e-6
G_MIN = -5.0


def build(force: bool = False) -> str:
    """Compile kda_oracle.c with gcc into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)) or (
        os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC))
    if force or stale:
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            lib = ctypes.CDLL(path)
            dp = ctypes.POINTER(ctypes.c_double)
            lib.kda_oracle_run.restype = ctypes.c_int
            lib.kda_oracle_run.argtypes = [
                dp, dp, dp, dp, dp, dp, dp,
                ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                ctypes.c_double, ctypes.c_int, ctypes.POINTER(ctypes.c_int32),
                ctypes.c_int64, dp, dp, ctypes.c_int]
            lib.kda_oracle_run_ckpt.restype = ctypes.c_int
            lib.kda_oracle_run_ckpt.argtypes = [
                dp, dp, dp, dp, dp, dp, dp,
                ctypes.POINTER(ctypes.c_int64), ctypes.c_int, ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                ctypes.c_double, ctypes.POINTER(ctypes.c_int32), ctypes.c_int64, dp, dp,
                ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), dp, ctypes.c_int]
            lib.kda_oracle_gate_softplus.restype = ctypes.c_double
            lib.kda_oracle_gate_softplus.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.kda_oracle_gate.restype = ctypes.c_double
            lib.kda_oracle_gate.argtypes = [ctypes.c_double, ctypes.c_double]
            lib.kda_oracle_short_conv.restype = ctypes.c_int
            lib.kda_oracle_short_conv.argtypes = [
                dp, ctypes.c_int64, ctypes.c_int64, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                dp, ctypes.c_int, dp, ctypes.c_int, dp, dp]
            lib.kda_oracle_backward.restype = ctypes.c_int
            lib.kda_oracle_backward.argtypes = [
                dp, dp, dp, dp, dp, dp, dp, ctypes.POINTER(ctypes.c_int64), ctypes.c_int,
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                ctypes.c_double, dp, dp, dp, dp, dp, dp, dp, dp, dp, ctypes.c_int]
            lib.kda_oracle_gate_vec.restype = None
            lib.kda_oracle_gate_vec.argtypes = [dp, ctypes.c_int64, ctypes.c_double, dp]
            _lib = lib
    return _lib


def _f64(x):
    """Exact conversion of a bf16/fp32/fp64 array (numpy or torch) to fp64."""
    if x is None:
        return None
    if hasattr(x, "detach"):  # torch tensor
        x = x.detach().to("cpu")
        import torch
        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def gate_softplus(z, A: float):
    """Kimi Linear's negative-softplus gate g = -softplus(e^A z), elementwise (fp64)."""
    lib = _load()
    zz = np.asarray(z, dtype=np.float64)
    return np.vectorize(lambda v: lib.kda_oracle_gate_softplus(float(v), float(A)))(zz)


def gate(z, A: float):
    """g = -5 * sigmoid(e^A z), elementwise, in fp64."""
    lib = _load()
    zz = _f64(z)
    out = np.empty_like(zz)
    lib.kda_oracle_gate_vec(_ptr(zz), zz.size, float(A), _ptr(out))
    return out


def kda_reference(q, k, v, z, beta, A, initial_state=None, cu_seqlens=None,
                  scale: float = 1.0, l2norm: bool = True, eps: float = EPS,
                  chunk: int = 0, units=None, nthreads: int = 0, softplus_gate: bool = False):
    """Run the oracle.

    Layouts (token-major, packed):
      q, k, z: [total_T, H, d_k];  v: [total_T, H, d_v];  beta: [total_T, H]
      A: [H];  initial_state: [N, H, d_k, d_v] or None (zeros)
      cu_seqlens: [N + 1] int, or None for one sequence of length total_T.
    chunk: 0 = recurrent form (the oracle), C > 0 = the chunked form.
    units: optional iterable of (n, h) pairs; only those are computed and the
      other outputs are left as NaN.
    softplus_gate: Kimi Linear's unbounded gate g = -softplus(e^A z) instead of
      K3's g = -5 sigmoid(e^A z).
    Returns (o [total_T, H, d_v] fp64, final_state [N, H, d_k, d_v] fp64,
    threads_used).
    """
    lib = _load()
    q, k, v, z, beta, A = (_f64(t) for t in (q, k, v, z, beta, A))
    if q.ndim == 4:  # [B, T, H, d] -> packed
        B, T = q.shape[0], q.shape[1]
        q, k, v, z = (t.reshape(B * T, *t.shape[2:]) for t in (q, k, v, z))
        beta = beta.reshape(B * T, -1)
        if cu_seqlens is None:
            cu_seqlens = np.arange(B + 1, dtype=np.int64) * T
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        cu_seqlens = np.array([0, total_T], dtype=np.int64)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    N = cu.size - 1
    if cu[0] != 0 or cu[-1] != total_T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must be non-decreasing from 0 to total_T")
    S0 = _f64(initial_state)
    if S0 is not None and S0.shape != (N, H, dk, dv):
        raise ValueError(f"initial_state shape {S0.shape} != {(N, H, dk, dv)}")
    o = np.full((total_T, H, dv), np.nan)
    S_out = np.full((N, H, dk, dv), np.nan)
    if units is not None:
        u = np.ascontiguousarray(np.asarray(list(units), dtype=np.int32).reshape(-1, 2))
        n_units = u.shape[0]
        uptr = _ptr(u, ctypes.c_int32)
    else:
        u, n_units, uptr = None, 0, None
    rc = lib.kda_oracle_run(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(S0),
        _ptr(cu, ctypes.c_int64), N, H, dk, dv, float(scale),
        int(bool(l2norm)) | (2 if softplus_gate else 0),
        float(eps), int(chunk), uptr, n_units, _ptr(o), _ptr(S_out), int(nthreads))
    if rc <= 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    return o, S_out, rc


def checkpoint_counts(cu_seqlens, interval: int):
    """Checkpoints per sequence (floor(length / interval)) and the index of
    each sequence's first one (exclusive prefix sum), for the state
    checkpoints of kda_reference_checkpoints."""
    cu = np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens,
                    dtype=np.int64)
    counts = np.diff(cu) // int(interval)
    base = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int64)
    return counts, base


def kda_reference_checkpoints(q, k, v, z, beta, A, initial_state=None, cu_seqlens=None,
                              interval: int = 64, scale: float = 1.0, l2norm: bool = True,
                              eps: float = EPS, units=None, nthreads: int = 0):
    """The oracle (recurrent form) plus state checkpoints: for every sequence n
    and m = 1, 2, ... with m * interval <= its length, the state after its
    first m * interval tokens, at index base[n] + m - 1 (checkpoint_counts).

    Layouts as kda_reference (packed only).  Returns (o, final_state,
    checkpoints [n_checkpoints, H, d_k, d_v] fp64, threads_used); entries of
    pairs not listed in `units` stay NaN.
    """
    lib = _load()
    q, k, v, z, beta, A = (_f64(t) for t in (q, k, v, z, beta, A))
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    if cu_seqlens is None:
        cu_seqlens = np.array([0, total_T], dtype=np.int64)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    N = cu.size - 1
    if cu[0] != 0 or cu[-1] != total_T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must be non-decreasing from 0 to total_T")
    if int(interval) <= 0:
        raise ValueError("interval must be positive")
    counts, base = checkpoint_counts(cu, interval)
    base = np.ascontiguousarray(base)
    S0 = _f64(initial_state)
    o = np.full((total_T, H, dv), np.nan)
    S_out = np.full((N, H, dk, dv), np.nan)
    ck = np.full((max(int(counts.sum()), 1), H, dk, dv), np.nan)
    if units is not None:
        u = np.ascontiguousarray(np.asarray(list(units), dtype=np.int32).reshape(-1, 2))
        n_units, uptr = u.shape[0], _ptr(u, ctypes.c_int32)
    else:
        u, n_units, uptr = None, 0, None
    rc = lib.kda_oracle_run_ckpt(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(S0),
        _ptr(cu, ctypes.c_int64), N, H, dk, dv, float(scale), int(bool(l2norm)),
        float(eps), uptr, n_units, _ptr(o), _ptr(S_out), int(interval),
        _ptr(base, ctypes.c_int64), _ptr(ck), int(nthreads))
    if rc <= 0:
        raise RuntimeError(f"oracle failed with status {rc}")
    return o, S_out, ck[:int(counts.sum())], rc


def _cu(cu_seqlens, total_T):
    if cu_seqlens is None:
        cu_seqlens = np.array([0, total_T], dtype=np.int64)
    cu = np.ascontiguousarray(np.asarray(
        cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu") else cu_seqlens, dtype=np.int64))
    if cu[0] != 0 or cu[-1] != total_T or np.any(np.diff(cu) < 0):
        raise ValueError("cu_seqlens must be non-decreasing from 0 to total_T")
    return cu


def short_conv(x, w, cu_seqlens=None, state_in=None, silu: bool = False):
    """Causal depthwise convolution along time (the short convolution).

    x: [total_T, C]; w: [C, W] (w[:, W-1] weights the current token);
    state_in: [N, W-1, C] or None (zeros), row r = the input W-1-r tokens
    before the sequence's first one.  Returns (y [total_T, C],
    state_out [N, W-1, C]): y_t = sum_j w[:, j] x_{t-W+1+j} (then y*sigmoid(y)
    if silu) and the last W-1 inputs of every sequence, all fp64."""
    lib = _load()
    x, w = _f64(x), _f64(w)
    total_T, C = x.shape
    W = w.shape[1]
    if w.shape[0] != C:
        raise ValueError("w must be [C, W]")
    cu = _cu(cu_seqlens, total_T)
    N = cu.size - 1
    s_in = _f64(state_in)
    if s_in is not None and s_in.shape != (N, W - 1, C):
        raise ValueError(f"state_in shape {s_in.shape} != {(N, W - 1, C)}")
    y = np.empty((total_T, C))
    s_out = np.empty((N, W - 1, C))
    rc = lib.kda_oracle_short_conv(_ptr(x), total_T, C, _ptr(cu, ctypes.c_int64), N,
                                   _ptr(w), W, _ptr(s_in), int(bool(silu)), _ptr(y),
                                   _ptr(s_out))
    if rc != 0:
        raise RuntimeError(f"oracle short_conv failed with status {rc}")
    return y, s_out


def short_conv_qkv(q, k, v, conv_w, cu_seqlens=None, conv_state=None, silu: bool = False):
    """The short convolutions of q, k and v with the per-head packed layouts
    of the library: conv_w [H, 2 d_k + d_v, W] fp32 and conv_state
    [N, H, W-1, 2 d_k + d_v], channels of a head ordered q | k | v.

    Returns (q_c, k_c, v_c, conv_state_out), fp64."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    Cc = 2 * dk + dv
    w = _f64(conv_w)
    W = w.shape[-1]
    x = np.concatenate([q, k, v], axis=-1).reshape(total_T, H * Cc)
    st = _f64(conv_state)
    if st is not None:
        st = np.ascontiguousarray(st.transpose(0, 2, 1, 3).reshape(st.shape[0], W - 1, H * Cc))
    y, s_out = short_conv(x, w.reshape(H * Cc, W), cu_seqlens, st, silu)
    y = y.reshape(total_T, H, Cc)
    s_out = s_out.reshape(s_out.shape[0], W - 1, H, Cc).transpose(0, 2, 1, 3)
    return (np.ascontiguousarray(y[..., :dk]), np.ascontiguousarray(y[..., dk:2 * dk]),
            np.ascontiguousarray(y[..., 2 * dk:]), np.ascontiguousarray(s_out))


def kda_reference_conv(q, k, v, z, beta, A, conv_w, conv_state=None, initial_state=None,
                       cu_seqlens=None, silu: bool = False, scale: float = 1.0,
                       l2norm: bool = True, eps: float = EPS, softplus_gate: bool = False,
                       nthreads: int = 0):
    """Short convolutions of q, k, v (short_conv_qkv) followed by the KDA
    recurrence (kda_reference) on the convolved q, k, v.

    Returns (o, final_state, conv_state_out), fp64."""
    qc, kc, vc, cs = short_conv_qkv(q, k, v, conv_w, cu_seqlens, conv_state, silu)
    o, S, _ = kda_reference(qc, kc, vc, z, beta, A, initial_state, cu_seqlens, scale=scale,
                            l2norm=l2norm, eps=eps, softplus_gate=softplus_gate,
                            nthreads=nthreads)
    return o, S, cs


def kda_reference_backward(q, k, v, z, beta, A, initial_state=None, cu_seqlens=None, dO=None,
                           dS_final=None, scale: float = 1.0, l2norm: bool = True,
                           eps: float = EPS, softplus_gate: bool = False, nthreads: int = 0):
    """Gradients of L = sum(dO * o) + sum(dS_final * S_T) with respect to every
    input of kda_reference (reverse mode of the recurrent form, fp64).

    Layouts as kda_reference (packed); dO [total_T, H, d_v]; dS_final
    [N, H, d_k, d_v] or None.  Returns a dict with dq, dk, dz [total_T, H, d_k],
    dv [total_T, H, d_v], dbeta [total_T, H], dA [H], dS0 [N, H, d_k, d_v]
    and the number of threads used ("threads")."""
    lib = _load()
    q, k, v, z, beta, A = (_f64(t) for t in (q, k, v, z, beta, A))
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    cu = _cu(cu_seqlens, total_T)
    N = cu.size - 1
    S0 = _f64(initial_state)
    dO = _f64(dO)
    dSf = _f64(dS_final)
    if dO is None or dO.shape != (total_T, H, dv):
        raise ValueError("dO must be [total_T, H, d_v]")
    out = dict(dq=np.empty((total_T, H, dk)), dk=np.empty((total_T, H, dk)),
               dv=np.empty((total_T, H, dv)), dz=np.empty((total_T, H, dk)),
               dbeta=np.empty((total_T, H)), dS0=np.empty((N, H, dk, dv)))
    gA = np.empty((N, H))
    rc = lib.kda_oracle_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(S0),
        _ptr(cu, ctypes.c_int64), N, H, dk, dv, float(scale),
        int(bool(l2norm)) | (2 if softplus_gate else 0), float(eps), _ptr(dO), _ptr(dSf),
        _ptr(out["dq"]), _ptr(out["dk"]), _ptr(out["dv"]), _ptr(out["dz"]),
        _ptr(out["dbeta"]), _ptr(gA), _ptr(out["dS0"]), int(nthreads))
    if rc <= 0:
        raise RuntimeError(f"oracle backward failed with status {rc}")
    out["dA"] = gA.sum(axis=0)
    out["threads"] = int(rc)
    return out


def _sigmoid(x):
    """Logistic function in fp64, without overflow for any x."""
    return 0.5 * (1.0 + np.tanh(0.5 * x))


def kda_reference_backward_chunked(q, k, v, z, beta, A, initial_state=None, cu_seqlens=None,
                                   dO=None, dS_final=None, chunk: int = 64, scale: float = 1.0,
                                   l2norm: bool = True, eps: float = EPS,
                                   softplus_gate: bool = False):
    """The gradients of kda_reference_backward by the chunked form of the
    recurrence (fp64 numpy): the algebra a chunk-parallel backward computes.

    Forward inside a chunk of the sequence (tokens r = 1..L, start state S0),
    from the recurrence of the section by unrolling it with the in-chunk
    cumulative gate gamma_r = sum_{j<=r} g_j (per key channel):
      E[r, i]   = e^(gamma_r - gamma_i)  for i <= r (0 above the diagonal)
      A_kk[r,i] = beta_r sum_c kh_r kh_i E[r,i]    (i < r)
      A_qk[r,i] = sum_c qh_r kh_i E[r,i]           (i <= r)
      K+ = kh e^gamma,  Q+ = qh e^gamma,  K_end = kh e^(gamma_L - gamma)
      X = V - K+ S0;  (I + A_kk) U = Diag(beta) X
      O = Q+ S0 + A_qk U;  S_L = Diag(e^gamma_L) S0 + K_end^T U
    Backward of that chunk, given dO and dS_L (the next chunk's dS0):
      dU = A_qk^T dO + K_end dS_L;  dY = (I + A_kk)^-T dU;  dA_kk = -dY U^T
      (strictly lower);  dX = Diag(beta) dY;  dbeta += rowsum(dY * X);
      dV = dX;  dS0 = Q+^T dO + Diag(e^gamma_L) dS_L - K+^T dX
    then the elementwise chains of K+, Q+, K_end, A_kk, A_qk into qh, kh,
    beta and gamma, dg = the reverse cumulative sum of dgamma over the chunk,
    and, per token, the gate and normalisation derivatives (as
    kda_reference_backward).  Chunks are walked last to first, the state at
    each chunk start taken from a forward pass over the chunks.

    Same layouts and return dict as kda_reference_backward (without
    "threads")."""
    q, k, v, z, beta, A = (_f64(t) for t in (q, k, v, z, beta, A))
    total_T, H, dk = q.shape
    dv = v.shape[-1]
    cu = _cu(cu_seqlens, total_T)
    N = cu.size - 1
    S0all = _f64(initial_state)
    dO = _f64(dO)
    dSf = _f64(dS_final)
    if dO is None or dO.shape != (total_T, H, dv):
        raise ValueError("dO must be [total_T, H, d_v]")
    if chunk < 1:
        raise ValueError("chunk must be >= 1")
    out = dict(dq=np.zeros((total_T, H, dk)), dk=np.zeros((total_T, H, dk)),
               dv=np.zeros((total_T, H, dv)), dz=np.zeros((total_T, H, dk)),
               dbeta=np.zeros((total_T, H)), dA=np.zeros(H), dS0=np.zeros((N, H, dk, dv)))
    for n in range(N):
        bos, eos = int(cu[n]), int(cu[n + 1])
        L = eos - bos
        for h in range(H):
            S = np.zeros((dk, dv)) if S0all is None else S0all[n, h].copy()
            dS = np.zeros((dk, dv)) if dSf is None else dSf[n, h].copy()
            if L == 0:
                out["dS0"][n, h] = dS
                continue
            qq, kk, vv = q[bos:eos, h], k[bos:eos, h], v[bos:eos, h]
            zz, bb = z[bos:eos, h], beta[bos:eos, h]
            if l2norm:
                rq = 1.0 / np.sqrt((qq * qq).sum(axis=1) + eps)
                rk = 1.0 / np.sqrt((kk * kk).sum(axis=1) + eps)
            else:
                rq = np.ones(L)
                rk = np.ones(L)
            qh = scale * qq * rq[:, None]
            kh = kk * rk[:, None]
            g = gate_softplus(zz, A[h]) if softplus_gate else gate(zz, A[h])

            def chunk_terms(c0, c1, S0):
                Qh, Kh, V, B = qh[c0:c1], kh[c0:c1], vv[c0:c1], bb[c0:c1]
                gam = np.cumsum(g[c0:c1], axis=0)
                Lc = c1 - c0
                le = np.tril(np.ones((Lc, Lc), dtype=bool))
                lt = np.tril(np.ones((Lc, Lc), dtype=bool), -1)
                D = np.where(le[:, :, None], gam[:, None, :] - gam[None, :, :], -np.inf)
                E = np.exp(D)
                Akk = B[:, None] * np.einsum("rc,ic,ric->ri", Kh, Kh, E) * lt
                Aqk = np.einsum("rc,ic,ric->ri", Qh, Kh, E)
                eg = np.exp(gam)
                Kp, Qp = Kh * eg, Qh * eg
                Kend = Kh * np.exp(gam[-1][None, :] - gam)
                X = V - Kp @ S0
                Mt = np.eye(Lc) + Akk
                U = np.linalg.solve(Mt, B[:, None] * X)
                return dict(Qh=Qh, Kh=Kh, B=B, gam=gam, le=le, lt=lt, E=E, Akk=Akk, Aqk=Aqk,
                            eg=eg, Kp=Kp, Qp=Qp, Kend=Kend, X=X, Mt=Mt, U=U)

            starts = list(range(0, L, chunk))
            S_start = []
            for c0 in starts:
                c1 = min(c0 + chunk, L)
                S_start.append(S.copy())
                t_ = chunk_terms(c0, c1, S)
                S = np.exp(t_["gam"][-1])[:, None] * S + t_["Kend"].T @ t_["U"]

            dqh = np.zeros((L, dk))
            dkh = np.zeros((L, dk))
            dg = np.zeros((L, dk))
            for ci in range(len(starts) - 1, -1, -1):
                c0 = starts[ci]
                c1 = min(c0 + chunk, L)
                S0 = S_start[ci]
                t_ = chunk_terms(c0, c1, S0)
                Qh, Kh, B, E, U, X = t_["Qh"], t_["Kh"], t_["B"], t_["E"], t_["U"], t_["X"]
                gam, Kp, Qp, Kend, eg = t_["gam"], t_["Kp"], t_["Qp"], t_["Kend"], t_["eg"]
                egL = np.exp(gam[-1])
                dOc = dO[bos + c0:bos + c1, h]
                dU = t_["Aqk"].T @ dOc + Kend @ dS
                dAqk = (dOc @ U.T) * t_["le"]
                dQp = dOc @ S0.T
                dS0 = Qp.T @ dOc + egL[:, None] * dS
                dKend = U @ dS.T
                dgamL = egL * (dS * S0).sum(axis=1)
                dY = np.linalg.solve(t_["Mt"].T, dU)
                dAkk = -(dY @ U.T) * t_["lt"]
                dX = B[:, None] * dY
                dbc = (dY * X).sum(axis=1)
                dKp = -dX @ S0.T
                dS0 = dS0 - Kp.T @ dX
                dKh = dKp * eg
                dgam = dKp * Kp
                dQh = dQp * eg
                dgam += dQp * Qp
                dKh += dKend * np.exp(gam[-1][None, :] - gam)
                dgam -= dKend * Kend
                dgamL += (dKend * Kend).sum(axis=0)
                T1 = dAkk[:, :, None] * B[:, None, None] * E
                dbc += np.einsum("ri,rc,ic,ric->r", dAkk, Kh, Kh, E)
                dKh += np.einsum("ric,ic->rc", T1, Kh) + np.einsum("ric,rc->ic", T1, Kh)
                P1 = T1 * Kh[:, None, :] * Kh[None, :, :]
                dgam += P1.sum(axis=1) - P1.sum(axis=0)
                T2 = dAqk[:, :, None] * E
                dQh += np.einsum("ric,ic->rc", T2, Kh)
                dKh += np.einsum("ric,rc->ic", T2, Qh)
                P2 = T2 * Qh[:, None, :] * Kh[None, :, :]
                dgam += P2.sum(axis=1) - P2.sum(axis=0)
                dgam[-1] += dgamL
                dg[c0:c1] = np.cumsum(dgam[::-1], axis=0)[::-1]
                dqh[c0:c1] = dQh
                dkh[c0:c1] = dKh
                out["dv"][bos + c0:bos + c1, h] = dX
                out["dbeta"][bos + c0:bos + c1, h] = dbc
                dS = dS0
            out["dS0"][n, h] = dS
            # gate: g = -5 sigmoid(x) or -softplus(x), x = e^A z
            eA = np.exp(A[h])
            x = eA * zz
            if softplus_gate:
                dx = -dg * _sigmoid(x)
            else:
                s = _sigmoid(x)
                dx = dg * (G_MIN * s * (1.0 - s))
            out["dz"][bos:eos, h] = dx * eA
            out["dA"][h] += float((dx * x).sum())
            # normalisation: xh = m x rho, rho = (sum x^2 + eps)^-1/2
            if l2norm:
                out["dq"][bos:eos, h] = scale * (rq[:, None] * dqh - (rq ** 3 * (qq * dqh).sum(
                    axis=1))[:, None] * qq)
                out["dk"][bos:eos, h] = rk[:, None] * dkh - (rk ** 3 * (kk * dkh).sum(
                    axis=1))[:, None] * kk
            else:
                out["dq"][bos:eos, h] = scale * dqh
                out["dk"][bos:eos, h] = dkh
    return out
