"""Kimi Delta Attention (KDA) for one GB300 -- Python binding of libkda.so.

This module only marshals arguments: torch supplies device memory and the
current CUDA stream, and every step of the computation runs in the library's
CUDA kernels behind the C ABI of ``include/kda.h``.  There is no CPU path:
if the library is not built, or no CUDA device is present, calls raise.

Entry points (same names as the C ABI):
  kda_prefill(q, k, v, z, beta, A, ...)      chunked prefill over packed sequences
  kda_decode_step(q, k, v, z, beta, A, state, ...)  one token per sequence, state in place
  kda_state_io(op, dst, src, ...)            zero / copy / gather / scatter of states
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libkda.so")

KDA_OK = 0
KDA_ERR_INVALID_ARG = -1
KDA_ERR_UNSUPPORTED = -2
KDA_ERR_ALIGNMENT = -3
KDA_ERR_WORKSPACE = -4
KDA_ERR_CUDA = -5
KDA_ERR_TIMEOUT = -6

KDA_F32 = 0
KDA_BF16 = 1

KDA_FLAG_L2NORM_QK = 1
KDA_FLAG_RECURRENT = 2
KDA_FLAG_SOFTPLUS_GATE = 4
KDA_FLAG_CONV_SILU = 8
KDA_FLAG_SHORT_PEER_WAITS = 16

KDA_STATE_ZERO = 0
KDA_STATE_COPY = 1
KDA_STATE_GATHER = 2
KDA_STATE_SCATTER = 3

# Every symbol include/kda.h declares.
EXPORTED_SYMBOLS = (
    "kda_prefill_workspace_bytes", "kda_prefill", "kda_workspace_status",
    "kda_decode_step", "kda_state_io", "kda_status_string", "kda_version",
    "kda_prefill_noalloc", "kda_prefill_checkpointed", "kda_checkpoint_count",
    "kda_short_conv", "kda_decode_step_conv", "kda_decode_conv_workspace_bytes",
    "kda_backward", "kda_backward_workspace_bytes", "kda_prefill_noalloc_status",
    "kda_prefill_conv", "kda_prefill_conv_workspace_bytes",
)

_lock = threading.Lock()
_lib = None


class KDAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what} failed: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libkda.so (built by ``__graft_entry__.build()``); raise if absent."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"KDA CUDA library not found at {LIB_PATH}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, u32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
            f32 = ctypes.c_float
            L.kda_prefill_workspace_bytes.restype = sz
            L.kda_prefill_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, ctypes.c_int]
            L.kda_prefill.restype = ctypes.c_int
            L.kda_prefill.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      i32, i32, i32, i32, i32, ctypes.c_int, f32, u32,
                                      vp, vp, vp, sz, vp]
            L.kda_workspace_status.restype = ctypes.c_int
            L.kda_workspace_status.argtypes = [vp, vp]
            L.kda_decode_step.restype = ctypes.c_int
            L.kda_decode_step.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32,
                                          i32, i32, i32, i32, ctypes.c_int, f32, u32, vp, vp]
            L.kda_state_io.restype = ctypes.c_int
            L.kda_state_io.argtypes = [ctypes.c_int, vp, vp, vp, i32, i32, i32, i32, i32, vp]
            L.kda_status_string.restype = ctypes.c_char_p
            L.kda_status_string.argtypes = [ctypes.c_int]
            L.kda_version.restype = ctypes.c_int
            L.kda_version.argtypes = []
            L.kda_prefill_noalloc.restype = ctypes.c_int
            L.kda_prefill_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                              i32, i32, i32, i32, i32, ctypes.c_int, f32, u32,
                                              vp, vp, vp]
            L.kda_prefill_noalloc_status.restype = ctypes.c_int
            L.kda_prefill_noalloc_status.argtypes = [vp]
            L.kda_prefill_checkpointed.restype = ctypes.c_int
            L.kda_prefill_checkpointed.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                                   i32, i32, i32, i32, i32, ctypes.c_int, f32,
                                                   u32, vp, vp, i32, vp, vp, i32, vp, sz, vp]
            L.kda_short_conv.restype = ctypes.c_int
            L.kda_short_conv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                         i32, i32, ctypes.c_int, ctypes.c_uint32, vp, vp, vp,
                                         vp]
            L.kda_decode_step_conv.restype = ctypes.c_int
            L.kda_decode_step_conv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, vp, vp, i32,
                                               i32, i32, i32, i32, ctypes.c_int,
                                               ctypes.c_float, ctypes.c_uint32, vp, vp, sz, vp]
            L.kda_decode_conv_workspace_bytes.restype = sz
            L.kda_decode_conv_workspace_bytes.argtypes = [i32, i32, i32, i32, ctypes.c_int]
            L.kda_backward.restype = ctypes.c_int
            L.kda_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32,
                                       i32, ctypes.c_int, ctypes.c_float, ctypes.c_uint32, vp,
                                       vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.kda_backward_workspace_bytes.restype = sz
            L.kda_backward_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, ctypes.c_int]
            L.kda_prefill_conv.restype = ctypes.c_int
            L.kda_prefill_conv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                           i32, i32, i32, i32, i32, ctypes.c_int, f32, u32,
                                           vp, vp, vp, i32, vp, vp, vp, sz, vp]
            L.kda_prefill_conv_workspace_bytes.restype = sz
            L.kda_prefill_conv_workspace_bytes.argtypes = [i32, i32, i32, i32, i32,
                                                           ctypes.c_int]
            L.kda_checkpoint_count.restype = ctypes.c_int64
            L.kda_checkpoint_count.argtypes = [vp, i32, i32, i32]
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().kda_status_string(int(status)).decode()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.float32:
        return KDA_F32
    if dt == torch.bfloat16:
        return KDA_BF16
    raise TypeError(f"unsupported dtype {dt}; KDA takes float32 or bfloat16")


def _check_cuda(*ts):
    for t in ts:
        if t is not None:
            if not t.is_cuda:
                raise ValueError("KDA tensors must live on a CUDA device")
            if not t.is_contiguous():
                raise ValueError("KDA tensors must be contiguous")


def _expect(t: Optional[torch.Tensor], shape, name: str, dtype: Optional[torch.dtype] = None):
    """The kernels index raw pointers with the sizes they are given: a tensor
    of another shape (or dtype) would be read or written out of bounds, so it
    is refused here."""
    if t is None:
        return
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def _nbytes(t: torch.Tensor) -> int:
    _check_cuda(t)
    return t.numel() * t.element_size()


def prefill_workspace_bytes(N: int, total_T: int, H: int, d_k: int, d_v: int,
                            dtype: torch.dtype) -> int:
    return int(lib().kda_prefill_workspace_bytes(N, total_T, H, d_k, d_v, _dtype_code(dtype)))


def alloc_workspace(N: int, total_T: int, H: int, d_k: int, d_v: int, dtype: torch.dtype,
                    device=None) -> torch.Tensor:
    nbytes = prefill_workspace_bytes(N, total_T, H, d_k, d_v, dtype)
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def kda_prefill(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, z: torch.Tensor,
                beta: torch.Tensor, A: torch.Tensor,
                initial_state: Optional[torch.Tensor] = None,
                cu_seqlens: Optional[torch.Tensor] = None,
                cu_seqlens_host: Optional[torch.Tensor] = None,
                scale: float = 1.0, l2norm: bool = True, recurrent: bool = False,
                softplus_gate: bool = False, output_final_state: bool = True,
                o: Optional[torch.Tensor] = None, final_state: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None,
                ckpt_interval: int = 0, ckpt_pool: Optional[torch.Tensor] = None,
                ckpt_slots: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None, extra_flags: int = 0
                ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """Chunked KDA prefill.  Packed layout: q, k, z [total_T, H, d_k], v
    [total_T, H, d_v], beta [total_T, H]; a 4-D [B, T, H, d] batch is accepted
    and treated as B sequences of length T.  Returns (o, final_state).

    With ckpt_interval > 0 (a multiple of 64) the state after every
    ckpt_interval tokens of each sequence is also written into ckpt_pool
    [pool, H, d_k, d_v] fp32, at row ckpt_slots[i] (int32, default i) for
    checkpoint i (kda_prefill_checkpointed in include/kda.h).

    softplus_gate=True selects Kimi Linear's unbounded gate -softplus(e^A z)
    (KDA_FLAG_SOFTPLUS_GATE; runs the fused recurrent kernel).  extra_flags
    are OR-ed into the call's flags (e.g. KDA_FLAG_SHORT_PEER_WAITS)."""
    batched = q.dim() == 4
    if batched:
        B, T = q.shape[:2]
        q, k, v, z = (t.reshape(B * T, *t.shape[2:]) for t in (q, k, v, z))
        beta = beta.reshape(B * T, -1)
        N = B
    else:
        N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    total_T, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = q.dtype
    for t in (k, v, z, beta):
        if t.dtype != dt:
            raise TypeError("q, k, v, z and beta must share one dtype")
    _check_cuda(q, k, v, z, beta, A, initial_state, cu_seqlens, o, final_state)
    for name, t in (("k", k), ("z", z)):
        _expect(t, (total_T, H, d_k), name)
    _expect(v, (total_T, H, d_v), "v")
    _expect(beta, (total_T, H), "beta")
    _expect(A, (H,), "A", torch.float32)
    _expect(cu_seqlens, (N + 1,), "cu_seqlens", torch.int32)
    _expect(initial_state, (N, H, d_k, d_v), "initial_state", torch.float32)
    _expect(o, (total_T, H, d_v), "o", dt)
    _expect(final_state, (N, H, d_k, d_v), "final_state", torch.float32)
    if o is None:
        o = torch.empty(total_T, H, d_v, dtype=dt, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, d_k, d_v, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(N, total_T, H, d_k, d_v, dt, q.device)
    host_cu = None
    if cu_seqlens_host is not None:
        host_cu = cu_seqlens_host.to(torch.int32).contiguous()
    flags = ((KDA_FLAG_L2NORM_QK if l2norm else 0) | (KDA_FLAG_RECURRENT if recurrent else 0)
             | (KDA_FLAG_SOFTPLUS_GATE if softplus_gate else 0) | int(extra_flags))
    host_ptr = None if host_cu is None else ctypes.c_void_p(host_cu.data_ptr())
    if ckpt_interval:
        _check_cuda(ckpt_pool, ckpt_slots)
        if ckpt_pool is None or ckpt_pool.dtype != torch.float32:
            raise TypeError("ckpt_pool must be a float32 tensor")
        _expect(ckpt_pool, (ckpt_pool.shape[0], H, d_k, d_v), "ckpt_pool", torch.float32)
        if ckpt_slots is not None:
            if ckpt_slots.dtype != torch.int32 or ckpt_slots.dim() != 1:
                raise TypeError("ckpt_slots must be a 1-D int32 tensor")
            cu_h = host_cu if host_cu is not None else (
                None if cu_seqlens is None else cu_seqlens.to("cpu", torch.int32))
            try:
                need = checkpoint_count(cu_h, N, total_T, int(ckpt_interval))
            except KDAError:   # a malformed cu_seqlens: the library bounds the reads itself
                need = -1
            if need >= 0 and ckpt_slots.numel() < need:
                raise ValueError(f"ckpt_slots has {ckpt_slots.numel()} entries for {need} "
                                 "checkpoints")
        st = lib().kda_prefill_checkpointed(
            _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(initial_state),
            _ptr(cu_seqlens), host_ptr, N, total_T, H, d_k, d_v, _dtype_code(dt),
            float(scale), flags, _ptr(o), _ptr(final_state), int(ckpt_interval),
            _ptr(ckpt_pool), _ptr(ckpt_slots), ckpt_pool.shape[0], _ptr(workspace),
            _nbytes(workspace), _stream_ptr(stream))
        name = "kda_prefill_checkpointed"
    else:
        st = lib().kda_prefill(
            _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(initial_state),
            _ptr(cu_seqlens), host_ptr, N, total_T, H, d_k, d_v, _dtype_code(dt),
            float(scale), flags, _ptr(o), _ptr(final_state), _ptr(workspace), _nbytes(workspace),
            _stream_ptr(stream))
        name = "kda_prefill"
    if st != KDA_OK:
        raise KDAError(st, name)
    if batched:
        o = o.reshape(B, T, H, d_v)
    return o, final_state


def checkpoint_count(cu_seqlens_host: Optional[torch.Tensor], N: int, total_T: int,
                     ckpt_interval: int) -> int:
    """Checkpoints kda_prefill writes with this interval (sum of floor(len / interval))."""
    host = None if cu_seqlens_host is None else cu_seqlens_host.to(torch.int32).contiguous()
    n = int(lib().kda_checkpoint_count(None if host is None else ctypes.c_void_p(host.data_ptr()),
                                       N, total_T, ckpt_interval))
    if n < 0:
        raise KDAError(n, "kda_checkpoint_count")
    return n


def workspace_status(workspace: torch.Tensor, stream: Optional[torch.cuda.Stream] = None) -> int:
    return int(lib().kda_workspace_status(_ptr(workspace), _stream_ptr(stream)))


def noalloc_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Status word of the last kda_prefill_noalloc call on the current device."""
    return int(lib().kda_prefill_noalloc_status(_stream_ptr(stream)))


def _expect_decode(q, k, v, z, beta, A, state, slots, o):
    B, H, d_k = q.shape
    d_v = v.shape[-1]
    for name, t in (("k", k), ("z", z)):
        _expect(t, (B, H, d_k), name, q.dtype)
    _expect(v, (B, H, d_v), "v", q.dtype)
    _expect(beta, (B, H), "beta", q.dtype)
    _expect(A, (H,), "A", torch.float32)
    _expect(state, (state.shape[0], H, d_k, d_v), "state", torch.float32)
    _expect(slots, (B,), "slots", torch.int32)
    _expect(o, (B, H, d_v), "o", q.dtype)


def kda_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, z: torch.Tensor,
                    beta: torch.Tensor, A: torch.Tensor, state: torch.Tensor,
                    slots: Optional[torch.Tensor] = None, scale: float = 1.0,
                    l2norm: bool = True, o: Optional[torch.Tensor] = None,
                    stream: Optional[torch.cuda.Stream] = None, softplus_gate: bool = False) -> torch.Tensor:
    """One decode token per sequence: q, k, z [B, H, d_k], v [B, H, d_v],
    beta [B, H]; `state` [pool, H, d_k, d_v] fp32 is updated in place at
    rows `slots` (default 0..B-1).  Returns o [B, H, d_v]."""
    B, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = q.dtype
    _check_cuda(q, k, v, z, beta, A, state, slots, o)
    _expect_decode(q, k, v, z, beta, A, state, slots, o)
    if o is None:
        o = torch.empty(B, H, d_v, dtype=dt, device=q.device)
    flags = (KDA_FLAG_L2NORM_QK if l2norm else 0) | (KDA_FLAG_SOFTPLUS_GATE if softplus_gate else 0)
    st = lib().kda_decode_step(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(state), _ptr(slots),
        state.shape[0], B, H, d_k, d_v, _dtype_code(dt), float(scale), flags, _ptr(o),
        _stream_ptr(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_step")
    return o


def kda_short_conv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, conv_w: torch.Tensor,
                   conv_state_in: Optional[torch.Tensor] = None,
                   conv_state_out: Optional[torch.Tensor] = None,
                   cu_seqlens: Optional[torch.Tensor] = None,
                   cu_seqlens_host: Optional[torch.Tensor] = None, silu: bool = False,
                   outputs: Optional[Tuple[torch.Tensor, torch.Tensor, torch.Tensor]] = None,
                   stream: Optional[torch.cuda.Stream] = None
                   ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Short convolutions of q, k [total_T, H, d_k] and v [total_T, H, d_v]
    (a 4-D [B, T, H, d] batch is taken as B sequences of length T).
    conv_w [H, 2 d_k + d_v, W] fp32; conv states [N, H, W-1, 2 d_k + d_v] in
    the dtype of q.  Returns the convolved (q, k, v); the final conv states go
    to conv_state_out when given (kda_short_conv in include/kda.h)."""
    batched = q.dim() == 4
    if batched:
        B, T = q.shape[:2]
        q, k, v = (t.reshape(B * T, *t.shape[2:]) for t in (q, k, v))
        N = B
    else:
        N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    total_T, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = q.dtype
    if k.dtype != dt or v.dtype != dt:
        raise TypeError("q, k and v must share one dtype")
    _check_cuda(q, k, v, conv_w, conv_state_in, conv_state_out, cu_seqlens)
    if conv_w.dtype != torch.float32 or conv_w.dim() != 3:
        raise TypeError("conv_w must be a float32 [H, 2 d_k + d_v, W] tensor")
    W = conv_w.shape[-1]
    Cc = 2 * d_k + d_v
    _expect(k, (total_T, H, d_k), "k")
    _expect(v, (total_T, H, d_v), "v")
    _expect(conv_w, (H, Cc, W), "conv_w", torch.float32)
    _expect(conv_state_in, (N, H, W - 1, Cc), "conv_state_in", dt)
    _expect(conv_state_out, (N, H, W - 1, Cc), "conv_state_out", dt)
    _expect(cu_seqlens, (N + 1,), "cu_seqlens", torch.int32)
    if outputs is None:
        outputs = (torch.empty_like(q), torch.empty_like(k), torch.empty_like(v))
    qo, ko, vo = outputs
    _check_cuda(qo, ko, vo)
    for name, t, ref in (("q_out", qo, q), ("k_out", ko, k), ("v_out", vo, v)):
        _expect(t, tuple(ref.shape), name, dt)
    host_cu = None if cu_seqlens_host is None else cu_seqlens_host.to(torch.int32).contiguous()
    host_ptr = None if host_cu is None else ctypes.c_void_p(host_cu.data_ptr())
    st = lib().kda_short_conv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(conv_w), _ptr(conv_state_in), _ptr(conv_state_out),
        _ptr(cu_seqlens), host_ptr, N, total_T, H, d_k, d_v, conv_w.shape[-1], _dtype_code(dt),
        KDA_FLAG_CONV_SILU if silu else 0, _ptr(qo), _ptr(ko), _ptr(vo), _stream_ptr(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_short_conv")
    if batched:
        qo, ko, vo = (t.reshape(B, T, *t.shape[1:]) for t in (qo, ko, vo))
    return qo, ko, vo


def decode_conv_workspace_bytes(B: int, H: int, d_k: int, d_v: int, dtype: torch.dtype) -> int:
    return int(lib().kda_decode_conv_workspace_bytes(B, H, d_k, d_v, _dtype_code(dtype)))


def kda_decode_step_conv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, z: torch.Tensor,
                         beta: torch.Tensor, A: torch.Tensor, state: torch.Tensor,
                         conv_w: torch.Tensor, conv_state: Optional[torch.Tensor],
                         slots: Optional[torch.Tensor] = None, scale: float = 1.0,
                         l2norm: bool = True, silu: bool = False, softplus_gate: bool = False,
                         o: Optional[torch.Tensor] = None,
                         workspace: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """kda_decode_step preceded by the token's short convolutions of q, k, v:
    conv_state [pool, H, W-1, 2 d_k + d_v] (dtype of q) is read and shifted in
    place at rows `slots`, like `state`.  `workspace` (uint8, at least
    decode_conv_workspace_bytes) is allocated when not given.
    Returns o [B, H, d_v]."""
    B, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = q.dtype
    _check_cuda(q, k, v, z, beta, A, state, conv_w, conv_state, slots, o)
    _expect_decode(q, k, v, z, beta, A, state, slots, o)
    if conv_w.dtype != torch.float32 or conv_w.dim() != 3:
        raise TypeError("conv_w must be a float32 [H, 2 d_k + d_v, W] tensor")
    W = conv_w.shape[-1]
    _expect(conv_w, (H, 2 * d_k + d_v, W), "conv_w", torch.float32)
    _expect(conv_state, (state.shape[0], H, W - 1, 2 * d_k + d_v), "conv_state", dt)
    if o is None:
        o = torch.empty(B, H, d_v, dtype=dt, device=q.device)
    if workspace is None:
        workspace = torch.empty(decode_conv_workspace_bytes(B, H, d_k, d_v, dt),
                                dtype=torch.uint8, device=q.device)
    flags = ((KDA_FLAG_L2NORM_QK if l2norm else 0) | (KDA_FLAG_SOFTPLUS_GATE if softplus_gate else 0)
             | (KDA_FLAG_CONV_SILU if silu else 0))
    st = lib().kda_decode_step_conv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(state), _ptr(slots),
        state.shape[0], _ptr(conv_w), _ptr(conv_state), conv_w.shape[-1], B, H, d_k, d_v,
        _dtype_code(dt), float(scale), flags, _ptr(o), _ptr(workspace), _nbytes(workspace),
        _stream_ptr(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_decode_step_conv")
    return o


def backward_workspace_bytes(N: int, total_T: int, H: int, d_k: int, d_v: int,
                             dtype: torch.dtype) -> int:
    return int(lib().kda_backward_workspace_bytes(N, total_T, H, d_k, d_v, _dtype_code(dtype)))


def kda_backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, z: torch.Tensor,
                 beta: torch.Tensor, A: torch.Tensor, dO: torch.Tensor,
                 initial_state: Optional[torch.Tensor] = None,
                 cu_seqlens: Optional[torch.Tensor] = None,
                 cu_seqlens_host: Optional[torch.Tensor] = None,
                 dS_final: Optional[torch.Tensor] = None, scale: float = 1.0,
                 l2norm: bool = True, softplus_gate: bool = False,
                 workspace: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> dict:
    """Gradients of the recurrence (kda_backward in include/kda.h) for packed
    inputs as kda_prefill takes them; dO [total_T, H, d_v] in the inputs'
    dtype, dS_final [N, H, d_k, d_v] fp32 or None.  Returns a dict of fp32
    tensors dq, dk, dz [total_T, H, d_k], dv [total_T, H, d_v],
    dbeta [total_T, H], dA [H], dS0 [N, H, d_k, d_v]."""
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    total_T, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = q.dtype
    for t in (k, v, z, beta, dO):
        if t.dtype != dt:
            raise TypeError("q, k, v, z, beta and dO must share one dtype")
    _check_cuda(q, k, v, z, beta, A, dO, initial_state, cu_seqlens, dS_final)
    for name, t in (("k", k), ("z", z)):
        _expect(t, (total_T, H, d_k), name)
    _expect(v, (total_T, H, d_v), "v")
    _expect(beta, (total_T, H), "beta")
    _expect(dO, (total_T, H, d_v), "dO")
    _expect(A, (H,), "A", torch.float32)
    _expect(cu_seqlens, (N + 1,), "cu_seqlens", torch.int32)
    _expect(initial_state, (N, H, d_k, d_v), "initial_state", torch.float32)
    _expect(dS_final, (N, H, d_k, d_v), "dS_final", torch.float32)
    dev = q.device
    f32 = dict(dtype=torch.float32, device=dev)
    g = dict(dq=torch.empty(total_T, H, d_k, **f32), dk=torch.empty(total_T, H, d_k, **f32),
             dv=torch.empty(total_T, H, d_v, **f32), dz=torch.empty(total_T, H, d_k, **f32),
             dbeta=torch.empty(total_T, H, **f32), dA=torch.empty(H, **f32),
             dS0=torch.empty(N, H, d_k, d_v, **f32))
    if workspace is None:
        workspace = torch.empty(backward_workspace_bytes(N, total_T, H, d_k, d_v, dt),
                                dtype=torch.uint8, device=dev)
    host_cu = None if cu_seqlens_host is None else cu_seqlens_host.to(torch.int32).contiguous()
    host_ptr = None if host_cu is None else ctypes.c_void_p(host_cu.data_ptr())
    flags = (KDA_FLAG_L2NORM_QK if l2norm else 0) | (KDA_FLAG_SOFTPLUS_GATE if softplus_gate else 0)
    st = lib().kda_backward(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(initial_state),
        _ptr(cu_seqlens), host_ptr, N, total_T, H, d_k, d_v, _dtype_code(dt), float(scale),
        flags, _ptr(dO), _ptr(dS_final), _ptr(g["dq"]), _ptr(g["dk"]), _ptr(g["dv"]),
        _ptr(g["dz"]), _ptr(g["dbeta"]), _ptr(g["dA"]), _ptr(g["dS0"]), _ptr(workspace),
        _nbytes(workspace), _stream_ptr(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_backward")
    return g


def prefill_conv_workspace_bytes(N: int, total_T: int, H: int, d_k: int, d_v: int,
                                 dtype: torch.dtype) -> int:
    return int(lib().kda_prefill_conv_workspace_bytes(N, total_T, H, d_k, d_v,
                                                      _dtype_code(dtype)))


def kda_prefill_conv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, z: torch.Tensor,
                     beta: torch.Tensor, A: torch.Tensor, conv_w: torch.Tensor,
                     conv_state_in: Optional[torch.Tensor] = None,
                     conv_state_out: Optional[torch.Tensor] = None,
                     initial_state: Optional[torch.Tensor] = None,
                     cu_seqlens: Optional[torch.Tensor] = None,
                     cu_seqlens_host: Optional[torch.Tensor] = None,
                     scale: float = 1.0, l2norm: bool = True, silu: bool = False,
                     softplus_gate: bool = False, output_final_state: bool = True,
                     o: Optional[torch.Tensor] = None,
                     final_state: Optional[torch.Tensor] = None,
                     workspace: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None, extra_flags: int = 0
                     ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """kda_short_conv followed by kda_prefill on its outputs, in one call
    (kda_prefill_conv in include/kda.h: the convolutions fused into the split
    kernel where it runs).  Packed layouts as kda_prefill; conv_w
    [H, 2 d_k + d_v, W] fp32; conv states [N, H, W-1, 2 d_k + d_v] in the
    dtype of q (the final ones go to conv_state_out when given).  Returns
    (o, final_state)."""
    N = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    total_T, H, d_k = q.shape
    d_v = v.shape[-1]
    dt = q.dtype
    for t in (k, v, z, beta):
        if t.dtype != dt:
            raise TypeError("q, k, v, z and beta must share one dtype")
    _check_cuda(q, k, v, z, beta, A, conv_w, conv_state_in, conv_state_out, initial_state,
                cu_seqlens, o, final_state)
    if conv_w.dtype != torch.float32 or conv_w.dim() != 3:
        raise TypeError("conv_w must be a float32 [H, 2 d_k + d_v, W] tensor")
    W = conv_w.shape[-1]
    Cc = 2 * d_k + d_v
    for name, t in (("k", k), ("z", z)):
        _expect(t, (total_T, H, d_k), name)
    _expect(v, (total_T, H, d_v), "v")
    _expect(beta, (total_T, H), "beta")
    _expect(A, (H,), "A", torch.float32)
    _expect(conv_w, (H, Cc, W), "conv_w", torch.float32)
    _expect(conv_state_in, (N, H, W - 1, Cc), "conv_state_in", dt)
    _expect(conv_state_out, (N, H, W - 1, Cc), "conv_state_out", dt)
    _expect(cu_seqlens, (N + 1,), "cu_seqlens", torch.int32)
    _expect(initial_state, (N, H, d_k, d_v), "initial_state", torch.float32)
    _expect(o, (total_T, H, d_v), "o", dt)
    _expect(final_state, (N, H, d_k, d_v), "final_state", torch.float32)
    if o is None:
        o = torch.empty(total_T, H, d_v, dtype=dt, device=q.device)
    if final_state is None and output_final_state:
        final_state = torch.empty(N, H, d_k, d_v, dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = torch.empty(prefill_conv_workspace_bytes(N, total_T, H, d_k, d_v, dt),
                                dtype=torch.uint8, device=q.device)
    host_cu = None if cu_seqlens_host is None else cu_seqlens_host.to(torch.int32).contiguous()
    host_ptr = None if host_cu is None else ctypes.c_void_p(host_cu.data_ptr())
    flags = ((KDA_FLAG_L2NORM_QK if l2norm else 0) | (KDA_FLAG_CONV_SILU if silu else 0)
             | (KDA_FLAG_SOFTPLUS_GATE if softplus_gate else 0) | int(extra_flags))
    st = lib().kda_prefill_conv(
        _ptr(q), _ptr(k), _ptr(v), _ptr(z), _ptr(beta), _ptr(A), _ptr(initial_state),
        _ptr(cu_seqlens), host_ptr, N, total_T, H, d_k, d_v, _dtype_code(dt), float(scale),
        flags, _ptr(conv_w), _ptr(conv_state_in), _ptr(conv_state_out), W, _ptr(o),
        _ptr(final_state), _ptr(workspace), _nbytes(workspace), _stream_ptr(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_prefill_conv")
    return o, final_state


def kda_state_io(op: int, dst: torch.Tensor, src: Optional[torch.Tensor] = None,
                 slots: Optional[torch.Tensor] = None, n: Optional[int] = None,
                 stream: Optional[torch.cuda.Stream] = None) -> None:
    """State movement; shapes [*, H, d_k, d_v] fp32.  n defaults to the
    number of slots, or to the leading size of src (COPY) / dst (ZERO)."""
    H, d_k, d_v = dst.shape[-3:]
    if n is None:
        if slots is not None:
            n = slots.numel()
        elif src is not None:
            n = src.shape[0]
        else:
            n = dst.shape[0]
    pool = dst.shape[0] if op in (KDA_STATE_ZERO, KDA_STATE_SCATTER) else (
        src.shape[0] if op == KDA_STATE_GATHER else 0)
    if op != KDA_STATE_COPY:
        _check_cuda(dst, src, slots)
    elif not dst.is_contiguous() or (src is not None and not src.is_contiguous()):
        raise ValueError("KDA tensors must be contiguous")
    # the kernels and copies move n whole states: every operand must hold them
    for name, t in (("dst", dst), ("src", src)):
        if t is not None:
            if t.dtype != torch.float32 or t.dim() != 4 or tuple(t.shape[1:]) != (H, d_k, d_v):
                raise ValueError(f"{name} must be a float32 [*, {H}, {d_k}, {d_v}] tensor")
    _expect(slots, (int(n),), "slots", torch.int32)
    if slots is None and dst.shape[0] < n:
        raise ValueError(f"dst holds {dst.shape[0]} states, {n} are written")
    if op in (KDA_STATE_COPY, KDA_STATE_SCATTER) and src is not None and src.shape[0] < n:
        raise ValueError(f"src holds {src.shape[0]} states, {n} are read")
    if op == KDA_STATE_GATHER and dst.shape[0] < n:
        raise ValueError(f"dst holds {dst.shape[0]} states, {n} are written")
    st = lib().kda_state_io(int(op), _ptr(dst), _ptr(src), _ptr(slots), int(n), int(pool),
                            H, d_k, d_v, _stream_ptr(stream))
    if st != KDA_OK:
        raise KDAError(st, "kda_state_io")
