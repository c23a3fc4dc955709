"""GPU parity of the short convolutions and their persistent conv state
against the fp64 oracle, through the C ABI: kda_short_conv alone, short conv
followed by kda_prefill, kda_decode_step_conv (the token's convolutions, then
the decode step), and prefill handing both states to decode.

Bars: the convolved tensors within their storage rounding (bf16: 2^-8 of
each value, plus 1e-5 of the tensor's largest value for fp32 accumulation;
fp32: 1e-5 max relative); conv states bit-exact (they are copies of inputs);
KDA outputs and states 1e-4 max relative for fp32 and 2e-2 relative Frobenius
for bf16, as for every other parity test."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs
from metrics import BF16_TOL, F32_TOL, max_rel, max_rel_stored, rel_fro

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


def _check_conv_out(got, ref, dtype):
    if dtype == torch.bfloat16:
        assert max_rel_stored(got, ref) <= 1e-5
    else:
        assert max_rel(got, ref) <= 1e-5


def _exact(got, ref):
    g = got.detach().cpu().double().numpy()
    assert g.shape == ref.shape and np.array_equal(g, ref)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("W", [1, 2, 3, 4])
@pytest.mark.parametrize("silu", [False, True])
@pytest.mark.parametrize("with_state", [False, True])
def test_short_conv_matches_oracle(oracle_mod, dtype, W, silu, with_state):
    """Varlen batch with an empty sequence, sequences shorter than W-1, token
    blocks that straddle sequence boundaries and a ragged tail; d_k != d_v."""
    lens = [70, 0, 2, 1, 33, 64, 7]
    H, dk, dv = 2, 64, 32
    x = inputs.make_prefill_inputs(lens, H, dk, dv, dtype, seed=300 + W)
    w, s0 = inputs.make_conv_params(len(lens), H, dk, dv, W, dtype, seed=300 + W,
                                    with_state=with_state)
    s_out = torch.empty(len(lens), H, W - 1, 2 * dk + dv, dtype=dtype, device=DEV)
    qc, kc, vc = kda.kda_short_conv(x.q.to(DEV), x.k.to(DEV), x.v.to(DEV), w.to(DEV),
                                    None if s0 is None else s0.to(DEV), s_out,
                                    x.cu_seqlens.to(DEV), x.cu_seqlens, silu=silu)
    torch.cuda.synchronize()
    rq, rk, rv, rs = oracle_mod.short_conv_qkv(x.q, x.k, x.v, w, x.cu_seqlens, s0, silu)
    for got, ref in ((qc, rq), (kc, rk), (vc, rv)):
        _check_conv_out(got, ref, dtype)
    _exact(s_out, rs)


def test_short_conv_d128_equal_lengths(oracle_mod):
    """A 4-D batch (equal lengths, no cu_seqlens) at d = 128."""
    B, T, H, d, W = 3, 100, 4, 128, 4
    x = inputs.make_prefill_inputs([T] * B, H, d, d, torch.bfloat16, seed=310)
    w, s0 = inputs.make_conv_params(B, H, d, d, W, torch.bfloat16, seed=310)
    s_out = torch.empty(B, H, W - 1, 3 * d, dtype=torch.bfloat16, device=DEV)
    q4, k4, v4 = (t.reshape(B, T, H, d).to(DEV) for t in (x.q, x.k, x.v))
    qc, kc, vc = kda.kda_short_conv(q4, k4, v4, w.to(DEV), s0.to(DEV), s_out, silu=True)
    torch.cuda.synchronize()
    rq, rk, rv, rs = oracle_mod.short_conv_qkv(x.q, x.k, x.v, w, x.cu_seqlens, s0, True)
    for got, ref in ((qc, rq), (kc, rk), (vc, rv)):
        _check_conv_out(got.reshape(B * T, H, d), ref, torch.bfloat16)
    _exact(s_out, rs)


@pytest.mark.parametrize("dtype,d", [(torch.bfloat16, 128), (torch.float32, 64)])
def test_short_conv_then_prefill(oracle_mod, dtype, d):
    """The prefill pipeline: kda_short_conv, then kda_prefill on its outputs
    (the chunked tensor-core kernel for bf16 d = 128, the recurrent one for
    fp32), against the oracle's convolution followed by the recurrence."""
    lens = [300, 5, 129]
    H, W = 4, 4
    x = inputs.make_prefill_inputs(lens, H, d, d, dtype, seed=320, nonzero_state=True)
    w, s0 = inputs.make_conv_params(len(lens), H, d, d, W, dtype, seed=320)
    xd = x.to(DEV)
    s_out = torch.empty_like(s0, device=DEV)
    qc, kc, vc = kda.kda_short_conv(xd.q, xd.k, xd.v, w.to(DEV), s0.to(DEV), s_out,
                                    xd.cu_seqlens, x.cu_seqlens, silu=True)
    o, S = kda.kda_prefill(qc, kc, vc, xd.z, xd.beta, xd.A, xd.initial_state, xd.cu_seqlens,
                           cu_seqlens_host=x.cu_seqlens)
    torch.cuda.synchronize()
    o_ref, S_ref, cs_ref = oracle_mod.kda_reference_conv(
        x.q, x.k, x.v, x.z, x.beta, x.A, w, s0, x.initial_state, x.cu_seqlens, silu=True)
    if dtype == torch.float32:
        assert max_rel(o, o_ref) <= F32_TOL and max_rel(S, S_ref) <= F32_TOL
    else:
        assert rel_fro(o, o_ref) <= BF16_TOL and rel_fro(S, S_ref) <= BF16_TOL
    _exact(s_out, cs_ref)


def _decode_case(oracle_mod, dtype, d, W, silu, softplus, seed):
    """B rows decoded from a pool through a slot permutation with one
    out-of-range slot; compared with the oracle on B one-token sequences."""
    B, H, pool = 5, 3, 8
    slots = torch.tensor([6, 0, -1, 3, 5], dtype=torch.int32)
    A, S_pool = inputs.make_decode_state(pool, H, d, d, seed=seed)
    w, cs_pool = inputs.make_conv_params(pool, H, d, d, W, dtype, seed=seed,
                                         with_state=W > 1)
    st = inputs.make_decode_step(B, H, d, d, dtype, seed=seed, step=0)
    sd = st.to(DEV)
    state = S_pool.to(DEV)
    cstate = None if cs_pool is None else cs_pool.to(DEV)
    o = kda.kda_decode_step_conv(sd.q, sd.k, sd.v, sd.z, sd.beta, A.to(DEV), state, w.to(DEV),
                                 cstate, slots=slots.to(DEV), silu=silu,
                                 softplus_gate=softplus)
    torch.cuda.synchronize()
    valid = [b for b in range(B) if 0 <= int(slots[b]) < pool]
    rows = [int(slots[b]) for b in valid]
    cu = np.arange(len(valid) + 1, dtype=np.int64)
    sel = lambda t: t[valid]
    o_ref, S_ref, cs_ref = oracle_mod.kda_reference_conv(
        sel(st.q), sel(st.k), sel(st.v), sel(st.z), sel(st.beta), A, w,
        None if cs_pool is None else cs_pool[rows], S_pool[rows], cu, silu=silu,
        softplus_gate=softplus)
    o_got = o[valid]
    if dtype == torch.float32:
        assert max_rel(o_got, o_ref) <= F32_TOL
        assert max_rel(state[rows], S_ref) <= F32_TOL
    else:
        assert rel_fro(o_got, o_ref) <= BF16_TOL
        assert rel_fro(state[rows], S_ref) <= BF16_TOL
    if cs_pool is not None:
        _exact(cstate[rows], cs_ref)
        untouched = [r for r in range(pool) if r not in rows]
        assert torch.equal(cstate[untouched].cpu(), cs_pool[untouched])
    untouched = [r for r in range(pool) if r not in rows]
    assert torch.equal(state[untouched].cpu(), S_pool[untouched])
    assert torch.isnan(o[2].float()).all()


@pytest.mark.parametrize("W,silu", [(4, True), (2, False), (1, True)])
def test_decode_conv_bf16_d128(oracle_mod, W, silu):
    """d_v = 128 (the decode step's two column-split CTAs per head)."""
    _decode_case(oracle_mod, torch.bfloat16, 128, W, silu, False, seed=330 + W)


@pytest.mark.parametrize("W,softplus", [(3, True), (4, False)])
def test_decode_conv_fp32_d64(oracle_mod, W, softplus):
    _decode_case(oracle_mod, torch.float32, 64, W, True, softplus, seed=340 + W)


def test_prefill_hands_both_states_to_decode(oracle_mod):
    """Prompt of 100 tokens through kda_short_conv + kda_prefill, then three
    tokens through kda_decode_step_conv with the recurrent and conv states
    handed over; the oracle runs the 103 tokens as one sequence."""
    T0, steps, H, d, W = 100, 3, 2, 128, 4
    dtype = torch.bfloat16
    x = inputs.make_prefill_inputs([T0 + steps], H, d, d, dtype, seed=350,
                                   nonzero_state=True)
    w, cs0 = inputs.make_conv_params(1, H, d, d, W, dtype, seed=350)
    xd = x.to(DEV)
    wd = w.to(DEV)
    cs = torch.empty_like(cs0, device=DEV)
    cu0 = torch.tensor([0, T0], dtype=torch.int32)
    pre = slice(0, T0)
    qc, kc, vc = kda.kda_short_conv(xd.q[pre], xd.k[pre], xd.v[pre], wd, cs0.to(DEV), cs,
                                    cu0.to(DEV), cu0, silu=True)
    _, S = kda.kda_prefill(qc, kc, vc, xd.z[pre], xd.beta[pre], xd.A, xd.initial_state,
                           cu0.to(DEV), cu_seqlens_host=cu0)
    outs = []
    for t in range(T0, T0 + steps):
        sl = slice(t, t + 1)
        outs.append(kda.kda_decode_step_conv(xd.q[sl], xd.k[sl], xd.v[sl], xd.z[sl],
                                             xd.beta[sl], xd.A, S, wd, cs, silu=True))
    torch.cuda.synchronize()
    o_ref, S_ref, cs_ref = oracle_mod.kda_reference_conv(
        x.q, x.k, x.v, x.z, x.beta, x.A, w, cs0, x.initial_state, x.cu_seqlens, silu=True)
    assert rel_fro(torch.cat(outs), o_ref[T0:]) <= BF16_TOL
    assert rel_fro(S, S_ref) <= BF16_TOL
    _exact(cs, cs_ref)
