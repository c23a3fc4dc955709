"""GPU parity, at the benchmark's own sizes and launch configurations, of the
short convolutions, the softplus-decay gate and the backward, against the
fp64 oracle: every output where the oracle finishes in seconds (the 4K
backward on all 32 heads), sampled heads (heads are independent problems)
where it does not.

Bars as in the other parity tests: relative Frobenius <= 2e-2 for bf16
inputs; the convolved tensors within their bf16 storage rounding; conv states
bit-exact."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs
from metrics import BF16_TOL, check_dA, max_rel_stored, rel_fro

pytestmark = pytest.mark.gpu

DEV = "cuda"
W = 4   # the benchmark's convolution width


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


def _head(x, h):
    """The inputs of head h alone (a one-head problem with the same tokens)."""
    sl = slice(h, h + 1)
    S0 = None if x.initial_state is None else x.initial_state[:, sl]
    return inputs.PrefillInputs(x.q[:, sl], x.k[:, sl], x.v[:, sl], x.z[:, sl], x.beta[:, sl],
                                x.A[sl], S0, x.cu_seqlens)


def test_short_conv_4k_workload_every_output(oracle_mod):
    """kda_short_conv on B=1 H=32 T=4096 d=128 bf16, width 4, SiLU, conv state
    in and out (the benchmark's call): all 50 M convolved values."""
    x = inputs.make_workload_inputs(inputs.PREFILL_4K, seed=0)
    w, s0 = inputs.make_conv_params(1, 32, 128, 128, W, torch.bfloat16, seed=11)
    s_out = torch.empty_like(s0, device=DEV)
    qc, kc, vc = kda.kda_short_conv(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), w.to(DEV),
                                    s0.to(DEV), s_out, x.cu_seqlens.to(DEV), x.cu_seqlens,
                                    silu=True)
    torch.cuda.synchronize()
    rq, rk, rv, rs = oracle_mod.short_conv_qkv(x.q, x.k, x.v, w, x.cu_seqlens, s0, True)
    for got, ref in ((qc, rq), (kc, rk), (vc, rv)):
        assert max_rel_stored(got, ref) <= 1e-5
    assert np.array_equal(s_out.cpu().double().numpy(), rs)


def test_conv_then_prefill_4k_sampled_heads(oracle_mod):
    """The convolutions followed by the split-kernel prefill at the 4K size,
    checked on three heads against the oracle's convolution + recurrence."""
    x = inputs.make_workload_inputs(inputs.PREFILL_4K, seed=0)
    w, s0 = inputs.make_conv_params(1, 32, 128, 128, W, torch.bfloat16, seed=11)
    xd = x.to(DEV)
    qc, kc, vc = kda.kda_short_conv(xd.q, xd.k, xd.v, w.to(DEV), s0.to(DEV), None,
                                    xd.cu_seqlens, x.cu_seqlens, silu=True)
    o, S = kda.kda_prefill(qc, kc, vc, xd.z, xd.beta, xd.A, None, xd.cu_seqlens,
                           cu_seqlens_host=x.cu_seqlens)
    torch.cuda.synchronize()
    for h in (0, 17, 31):
        xh = _head(x, h)
        o_ref, S_ref, _ = oracle_mod.kda_reference_conv(
            xh.q, xh.k, xh.v, xh.z, xh.beta, xh.A, w[h:h + 1], s0[:, h:h + 1], None,
            x.cu_seqlens, silu=True)
        assert rel_fro(o[:, h:h + 1], o_ref) <= BF16_TOL, h
        assert rel_fro(S[:, h:h + 1], S_ref) <= BF16_TOL, h


def test_decode_conv_256_workload_every_row(oracle_mod):
    """kda_decode_step_conv on the decode workload (B=256 H=96 d=128, bf16
    inputs, fp32 state, width 4, SiLU): one step, every row and head."""
    w_ = inputs.DECODE_256
    A, S0 = inputs.make_decode_state(w_.B, w_.H, 128, 128, seed=5)
    cw, cs0 = inputs.make_conv_params(w_.B, w_.H, 128, 128, W, torch.bfloat16, seed=5)
    st = inputs.make_decode_step(w_.B, w_.H, 128, 128, torch.bfloat16, seed=5, step=0)
    sd = st.to(DEV)
    state, cstate = S0.to(DEV), cs0.to(DEV)
    o = kda.kda_decode_step_conv(sd.q, sd.k, sd.v, sd.z, sd.beta, A.to(DEV), state, cw.to(DEV),
                                 cstate, silu=True)
    torch.cuda.synchronize()
    cu = np.arange(w_.B + 1, dtype=np.int64)
    o_ref, S_ref, cs_ref = oracle_mod.kda_reference_conv(st.q, st.k, st.v, st.z, st.beta, A, cw,
                                                         cs0, S0, cu, silu=True)
    assert rel_fro(o, o_ref) <= BF16_TOL
    assert rel_fro(state, S_ref) <= BF16_TOL
    assert np.array_equal(cstate.cpu().double().numpy(), cs_ref)


def test_softplus_prefill_4k_sampled_heads(oracle_mod):
    """The softplus-gate prefill at the 4K size (the recurrent kernel, as the
    benchmark runs it), checked on three heads."""
    x = inputs.make_workload_inputs(inputs.PREFILL_4K, seed=0)
    xd = x.to(DEV)
    o, S = kda.kda_prefill(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, None, xd.cu_seqlens,
                           cu_seqlens_host=x.cu_seqlens, softplus_gate=True)
    torch.cuda.synchronize()
    for h in (0, 13, 31):
        xh = _head(x, h)
        o_ref, S_ref, _ = oracle_mod.kda_reference(xh.q, xh.k, xh.v, xh.z, xh.beta, xh.A, None,
                                                   x.cu_seqlens, softplus_gate=True)
        assert rel_fro(o[:, h:h + 1], o_ref) <= BF16_TOL, h
        assert rel_fro(S[:, h:h + 1], S_ref) <= BF16_TOL, h


def test_backward_4k_workload_all_heads(oracle_mod):
    """kda_backward on the 4K workload with the benchmark's upstream gradients
    (the chunked tensor-core backward: lengths vouched for by the host),
    every gradient of all 32 heads against the oracle's reverse mode."""
    x = inputs.make_workload_inputs(inputs.PREFILL_4K, seed=0)
    dO, dSf = inputs.make_upstream_grads(4096, 1, 32, 128, 128, torch.bfloat16, seed=21)
    xd = x.to(DEV)
    ws = torch.empty(kda.backward_workspace_bytes(1, 4096, 32, 128, 128, torch.bfloat16),
                     dtype=torch.uint8, device=DEV)
    g = kda.kda_backward(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, dO.to(DEV), None,
                         xd.cu_seqlens, x.cu_seqlens, dS_final=dSf.to(DEV), workspace=ws)
    torch.cuda.synchronize()
    assert kda.workspace_status(ws) == kda.KDA_OK
    ref = oracle_mod.kda_reference_backward(x.q, x.k, x.v, x.z, x.beta, x.A, None,
                                            x.cu_seqlens, dO, dSf)
    for key in ("dq", "dk", "dv", "dz", "dbeta", "dS0"):
        for h in range(32):
            got, want = g[key][:, h], ref[key][:, h]
            assert rel_fro(got, want) <= BF16_TOL, (h, key, rel_fro(got, want))
    # dA: its per-token shares at the bar, the sum of its shares, and the
    # relative bar where the sum does not cancel too far
    check_dA(g["dA"], g["dz"], ref["dA"], ref["dz"], x.z)
