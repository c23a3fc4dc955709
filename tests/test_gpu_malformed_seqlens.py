"""A malformed device cu_seqlens (no host mirror to catch it) must not send any
kernel outside the caller's buffers.

The C ABI receives cu_seqlens as a device array and can only validate it when
the caller also passes a host mirror.  Every kernel clamps the entries to
[0, total_T] and ends each sequence no earlier than it starts, so such an
array gives meaningless values but every read and write stays inside the
packed token range.  These tests pass an array that decreases, goes negative
and ends past total_T, to every entry point that takes one, with each output
a view at the start of a larger buffer whose tail holds a sentinel: the call
must finish with a clean status and leave every tail untouched.  (Even a
kernel that ignored the clamp would stay inside these padded buffers, so the
test cannot fault the GPU; it detects the stray writes.)
"""
import ctypes

import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"
T = 256          # total_T of the calls
PAD = 192        # tokens of sentinel tail behind every per-token buffer
SENT = 1234.5


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


def _bad_cu():
    # decreasing (100 -> -5), negative, and ending past total_T
    return torch.tensor([0, 100, -5, 50, T + 70], dtype=torch.int32, device=DEV)


def _padded_inputs(H, d, dtype, seed):
    """q, k, v, z, beta of T tokens, each a view at the start of a buffer of
    T + PAD tokens (the tail holds ordinary random values)."""
    x = inputs.make_prefill_inputs([T + PAD], H, d, d, dtype, seed=seed)
    xd = x.to(DEV)
    views = {n: getattr(xd, n)[:T] for n in ("q", "k", "v", "z", "beta")}
    return xd, views


def _sentinel(shape, dtype):
    return torch.full(shape, SENT, dtype=dtype, device=DEV)


@pytest.mark.parametrize("path", ["split", "single_pass", "recurrent_f32", "checkpointed"])
def test_prefill_stays_in_bounds(path):
    dtype = torch.float32 if path == "recurrent_f32" else torch.bfloat16
    d = 64 if path == "recurrent_f32" else 128
    H, N = 3, 4
    xd, v = _padded_inputs(H, d, dtype, seed=31)
    cu = _bad_cu()
    o_big = _sentinel((T + PAD, H, d), dtype)
    S = torch.empty(N, H, d, d, dtype=torch.float32, device=DEV)
    ws = kda.alloc_workspace(N, T, H, d, d, dtype)
    if path == "single_pass":
        ws = torch.empty(256 + 256, dtype=torch.uint8, device=DEV)
    kw = {}
    if path == "checkpointed":
        pool_big = _sentinel((T // 64 + 8, H, d, d), torch.float32)
        kw = dict(ckpt_interval=64, ckpt_pool=pool_big[:T // 64],
                  ckpt_slots=torch.arange(T // 64, dtype=torch.int32, device=DEV))
    kda.kda_prefill(v["q"], v["k"], v["v"], v["z"], v["beta"], xd.A, None, cu,
                    o=o_big[:T], final_state=S, workspace=ws, **kw)
    assert kda.workspace_status(ws) == kda.KDA_OK
    assert torch.isfinite(o_big[:T].float()).all()
    assert torch.isfinite(S).all()
    assert (o_big[T:] == SENT).all(), "o written past total_T"
    if path == "checkpointed":
        assert (pool_big[T // 64:] == SENT).all(), "checkpoint written past the pool"


def test_short_conv_stays_in_bounds():
    H, d, N, W = 2, 128, 4, 4
    xd, v = _padded_inputs(H, d, torch.bfloat16, seed=32)
    w, cs = inputs.make_conv_params(N, H, d, d, W, torch.bfloat16, seed=33)
    cs_in = cs.to(DEV)
    cs_out_big = _sentinel((N + 2, H, W - 1, 3 * d), torch.bfloat16)
    outs_big = [_sentinel((T + PAD, H, d), torch.bfloat16) for _ in range(3)]
    kda.kda_short_conv(v["q"], v["k"], v["v"], w.to(DEV), cs_in, cs_out_big[:N], _bad_cu(),
                       silu=True, outputs=tuple(b[:T] for b in outs_big))
    torch.cuda.synchronize()
    for b in outs_big:
        assert torch.isfinite(b[:T].float()).all()
        assert (b[T:] == SENT).all(), "convolved output written past total_T"
    assert (cs_out_big[N:] == SENT).all(), "conv state written past N"


def test_backward_stays_in_bounds():
    H, d, N = 2, 128, 4
    dt = torch.bfloat16
    xd, v = _padded_inputs(H, d, dt, seed=34)
    dO, _ = inputs.make_upstream_grads(T, N, H, d, d, dt, seed=35, with_state=False)
    dO = dO.to(DEV)
    big = lambda *shape: _sentinel(shape, torch.float32)
    dq, dk, dz, dv = (big(T + PAD, H, d) for _ in range(4))
    dbeta = big(T + PAD, H)
    dA = big(H + 4)
    dS0 = big(N + 2, H, d, d)
    ws = torch.empty(kda.backward_workspace_bytes(N, T, H, d, d, dt), dtype=torch.uint8,
                     device=DEV)
    L = kda.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = L.kda_backward(p(v["q"]), p(v["k"]), p(v["v"]), p(v["z"]), p(v["beta"]), p(xd.A),
                        None, p(_bad_cu()), None, N, T, H, d, d, kda.KDA_BF16, 1.0,
                        kda.KDA_FLAG_L2NORM_QK, p(dO), None, p(dq), p(dk), p(dv), p(dz),
                        p(dbeta), p(dA), p(dS0), p(ws), ws.numel(),
                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == kda.KDA_OK, kda.status_string(st)
    assert kda.workspace_status(ws) == kda.KDA_OK
    for name, t in (("dq", dq), ("dk", dk), ("dz", dz), ("dv", dv), ("dbeta", dbeta)):
        assert (t[T:] == SENT).all(), f"{name} written past total_T"
    assert (dA[H:] == SENT).all() and (dS0[N:] == SENT).all()
