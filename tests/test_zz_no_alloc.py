"""kda_prefill_noalloc: prefill for callers that cannot allocate device memory.

Some callers of this library (a plugin inside a host framework that owns all
device memory, a latency-critical loop that must not call into the CUDA
allocator after start-up) cannot provide the device workspace kda_prefill
asks for.  kda_prefill_noalloc takes the same arguments minus the workspace
and uses a fixed array in the library's own device memory instead.  This
test calls it through the C ABI and checks that two calls in a row give the
same o and final state as kda_prefill with a caller workspace, that both
agree with the fp64 oracle, and that kda_prefill_noalloc_status (the only
way such a caller can see a device-side timeout) reads KDA_OK after each.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs
from metrics import BF16_TOL, F32_TOL, max_rel, rel_fro

pytestmark = pytest.mark.gpu


def _call_noalloc(L, xd, N, d, dt_code, o, S):
    vp = ctypes.c_void_p
    p = lambda t: vp(t.data_ptr()) if t is not None else None
    return L.kda_prefill_noalloc(p(xd.q), p(xd.k), p(xd.v), p(xd.z), p(xd.beta), p(xd.A),
                                 p(xd.initial_state), p(xd.cu_seqlens), None,
                                 N, xd.q.shape[0], xd.q.shape[1], d, d, dt_code, 1.0,
                                 kda.KDA_FLAG_L2NORM_QK, p(o), p(S),
                                 vp(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("dtype,d,tol", [(torch.bfloat16, 128, BF16_TOL),
                                         (torch.float32, 64, F32_TOL)])
def test_noalloc_matches_prefill_twice(dtype, d, tol):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = kda.lib()
    x = inputs.make_prefill_inputs([300, 0, 77, 129], 4, d, d, dtype, seed=21,
                                   nonzero_state=True)
    xd = x.to("cuda")
    N = len(x.cu_seqlens) - 1
    o_ref, S_ref = kda.kda_prefill(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, xd.initial_state,
                                   xd.cu_seqlens)
    torch.cuda.synchronize()
    import oracle
    o_or, S_or, _ = oracle.kda_reference(x.q, x.k, x.v, x.z, x.beta, x.A, x.initial_state,
                                         x.cu_seqlens)
    err = rel_fro if dtype == torch.bfloat16 else max_rel
    for _ in range(2):
        o = torch.full_like(o_ref, float("nan"))
        S = torch.full_like(S_ref, float("nan"))
        st = _call_noalloc(L, xd, N, d, kda.KDA_BF16 if dtype == torch.bfloat16 else kda.KDA_F32,
                           o, S)
        assert st == kda.KDA_OK, kda.status_string(st)
        assert kda.noalloc_status() == kda.KDA_OK
        assert err(o.float(), o_ref.float()) <= tol
        assert err(S, S_ref) <= tol
        # and against the fp64 oracle
        assert err(o.float(), o_or) <= tol
        assert err(S, S_or) <= tol


def test_noalloc_rejects_sizes_beyond_its_array():
    """More (sequence, head) pairs than the fixed array holds: a clear error
    status, and nothing is launched."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    L = kda.lib()
    vp = ctypes.c_void_p
    fake = vp(0x7F0000000000)
    N, H = 20000, 4      # 80000 pairs > 16384
    st = L.kda_prefill_noalloc(fake, fake, fake, fake, fake, fake, None, fake, None,
                               N, N, H, 128, 128, kda.KDA_BF16, 1.0, 1, fake, None, None)
    assert st == kda.KDA_ERR_WORKSPACE
