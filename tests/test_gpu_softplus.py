"""GPU parity of the Kimi Linear gate variant (KDA_FLAG_SOFTPLUS_GATE:
g = -softplus(e^A z), unbounded below) against the fp64 oracle with the same
gate, through the C ABI.  Prefill runs the fused recurrent kernel for every
dtype and size; decode takes the flag directly.  Bars: max relative <= 1e-4
for fp32 (outputs stored in bf16 get their storage rounding), relative
Frobenius <= 2e-2 for bf16 inputs."""
import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs
from metrics import BF16_TOL, F32_TOL, max_rel, rel_fro

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


def _prefill(x, **kw):
    xd = x.to(DEV)
    o, S = kda.kda_prefill(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, xd.initial_state,
                           xd.cu_seqlens, softplus_gate=True, **kw)
    torch.cuda.synchronize()
    return o, S


def test_softplus_prefill_fp32(oracle_mod):
    x = inputs.make_prefill_inputs([70, 1, 130], 3, 64, 64, torch.float32, seed=51,
                                   nonzero_state=True)
    o, S = _prefill(x)
    o_ref, S_ref, _ = oracle_mod.kda_reference(x.q, x.k, x.v, x.z, x.beta, x.A,
                                               x.initial_state, x.cu_seqlens,
                                               softplus_gate=True)
    assert max_rel(o, o_ref) <= F32_TOL
    assert max_rel(S, S_ref) <= F32_TOL
    # the K3 gate gives a different answer on the same inputs
    o_k3, _ = kda.kda_prefill(*(t.to(DEV) for t in (x.q, x.k, x.v, x.z, x.beta, x.A)),
                              x.initial_state.to(DEV), x.cu_seqlens.to(DEV))
    assert max_rel(o_k3, o_ref) > 1e-3


def test_softplus_prefill_bf16_d128(oracle_mod):
    """bf16, d = 128: the chunked kernels do not apply to the unbounded gate;
    the call runs the recurrent kernel and still meets the bf16 bar."""
    x = inputs.make_prefill_inputs([200, 64, 3], 2, 128, 128, torch.bfloat16, seed=52,
                                   nonzero_state=True)
    o, S = _prefill(x)
    o_ref, S_ref, _ = oracle_mod.kda_reference(x.q, x.k, x.v, x.z, x.beta, x.A,
                                               x.initial_state, x.cu_seqlens,
                                               softplus_gate=True)
    assert rel_fro(o, o_ref) <= BF16_TOL
    assert rel_fro(S, S_ref) <= BF16_TOL


def test_softplus_decode_fp32(oracle_mod):
    A, S0 = inputs.make_decode_state(6, 4, 64, 64, seed=53)
    st = inputs.make_decode_step(6, 4, 64, 64, torch.float32, seed=53, step=0)
    state = S0.to(DEV)
    sd = st.to(DEV)
    o = kda.kda_decode_step(sd.q, sd.k, sd.v, sd.z, sd.beta, A.to(DEV), state,
                            softplus_gate=True)
    torch.cuda.synchronize()
    o_ref, S_ref, _ = oracle_mod.kda_reference(st.q.unsqueeze(1), st.k.unsqueeze(1),
                                               st.v.unsqueeze(1), st.z.unsqueeze(1),
                                               st.beta.unsqueeze(1), A, S0,
                                               softplus_gate=True)
    assert max_rel(o, o_ref.reshape(6, 4, 64)) <= F32_TOL
    assert max_rel(state, S_ref) <= F32_TOL
