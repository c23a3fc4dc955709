"""The Python binding refuses tensors whose shape, dtype or layout the
kernels would index out of bounds (the C ABI only sees raw pointers), before
anything is launched."""
import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


@pytest.fixture(scope="module")
def x():
    return inputs.make_prefill_inputs([70, 30], 2, 64, 64, torch.bfloat16, seed=1).to(DEV)


def test_prefill_rejects_bad_shapes(x):
    bad = dict(o=torch.empty(99, 2, 64, dtype=torch.bfloat16, device=DEV),
               final_state=torch.empty(1, 2, 64, 64, device=DEV))
    for key, val in bad.items():
        with pytest.raises(ValueError):
            kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens, **{key: val})
    with pytest.raises(ValueError):
        kda.kda_prefill(x.q, x.k, x.v[:50], x.z, x.beta, x.A, None, x.cu_seqlens)
    with pytest.raises(ValueError):      # a head slice is not contiguous
        kda.kda_prefill(x.q[:, :1], x.k[:, :1], x.v[:, :1], x.z[:, :1], x.beta[:, :1],
                        x.A[:1], None, x.cu_seqlens)
    with pytest.raises(ValueError):      # too few slots for the checkpoints
        pool = torch.empty(4, 2, 64, 64, device=DEV)
        kda.kda_prefill(x.q, x.k, x.v, x.z, x.beta, x.A, None, x.cu_seqlens,
                        ckpt_interval=64, ckpt_pool=pool,
                        ckpt_slots=torch.zeros(0, dtype=torch.int32, device=DEV))


def test_decode_and_state_io_reject_bad_shapes():
    A, S = inputs.make_decode_state(4, 2, 64, 64, seed=1)
    st = inputs.make_decode_step(4, 2, 64, 64, torch.bfloat16, seed=1).to(DEV)
    A, S = A.to(DEV), S.to(DEV)
    with pytest.raises(ValueError):
        kda.kda_decode_step(st.q, st.k, st.v, st.z, st.beta, A, S,
                            slots=torch.zeros(3, dtype=torch.int32, device=DEV))
    with pytest.raises(ValueError):
        kda.kda_decode_step(st.q, st.k, st.v, st.z, st.beta, A, S[:, :1])
    with pytest.raises(ValueError):
        kda.kda_state_io(kda.KDA_STATE_COPY, torch.empty(2, 2, 64, 64, device=DEV), S, n=4)


def test_conv_and_backward_reject_bad_shapes(x):
    w, s0 = inputs.make_conv_params(2, 2, 64, 64, 4, torch.bfloat16, seed=1)
    w = w.to(DEV)
    with pytest.raises(ValueError):
        kda.kda_short_conv(x.q, x.k, x.v, w[:1], None, None, x.cu_seqlens)
    with pytest.raises(ValueError):
        kda.kda_short_conv(x.q, x.k, x.v, w, s0[:1].to(DEV), None, x.cu_seqlens)
    dO = torch.empty(99, 2, 64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ValueError):
        kda.kda_backward(x.q, x.k, x.v, x.z, x.beta, x.A, dO, None, x.cu_seqlens)
