"""GPU parity of the training backward (kda_backward: gradients of the
recurrence) against the fp64 reverse-mode oracle, through the C ABI.

Every gradient is compared: dq, dk, dv, dz, dbeta, dA and dS0.  Bars as for
the forward: max relative error <= 1e-4 for fp32 inputs, relative Frobenius
<= 2e-2 for bf16 inputs (the gradients themselves are fp32)."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs
from metrics import BF16_TOL, F32_TOL, max_rel, rel_fro

pytestmark = pytest.mark.gpu

DEV = "cuda"
KEYS = ("dq", "dk", "dv", "dz", "dbeta", "dA", "dS0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


def _run(oracle_mod, lens, H, dk, dv, dtype, seed, with_state=True, **flags):
    x = inputs.make_prefill_inputs(lens, H, dk, dv, dtype, seed=seed, nonzero_state=with_state)
    dO, dSf = inputs.make_upstream_grads(sum(lens), len(lens), H, dk, dv, dtype, seed=seed,
                                         with_state=with_state)
    xd = x.to(DEV)
    g = kda.kda_backward(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, dO.to(DEV), xd.initial_state,
                         xd.cu_seqlens, x.cu_seqlens,
                         None if dSf is None else dSf.to(DEV), **flags)
    torch.cuda.synchronize()
    ref = oracle_mod.kda_reference_backward(x.q, x.k, x.v, x.z, x.beta, x.A, x.initial_state,
                                            x.cu_seqlens, dO, dSf, **flags)
    return g, ref


@pytest.mark.parametrize("dk,dv", [(32, 32), (64, 32)])
def test_backward_fp32_varlen(oracle_mod, dk, dv):
    """Varlen with an empty sequence and one spanning three 64-token chunks
    with a ragged tail; nonzero initial state and dL/dS_T; scale != 1."""
    g, ref = _run(oracle_mod, [70, 0, 3, 130], 2, dk, dv, torch.float32, seed=400 + dk,
                  scale=0.8)
    for key in KEYS:
        assert max_rel(g[key], ref[key]) <= F32_TOL, key


def test_backward_fp32_softplus_no_norm_d128(oracle_mod):
    """Kimi Linear's gate and no in-op normalisation, d = 128."""
    g, ref = _run(oracle_mod, [64, 65], 2, 128, 128, torch.float32, seed=410,
                  softplus_gate=True, l2norm=False)
    for key in KEYS:
        assert max_rel(g[key], ref[key]) <= F32_TOL, key


def test_backward_bf16_d128(oracle_mod):
    g, ref = _run(oracle_mod, [200, 64], 2, 128, 128, torch.bfloat16, seed=420)
    for key in KEYS:
        assert rel_fro(g[key], ref[key]) <= BF16_TOL, key


def test_backward_zero_state_and_empty_sequences(oracle_mod):
    """No initial state and no dL/dS_T; two of three sequences empty."""
    g, ref = _run(oracle_mod, [0, 90, 0], 3, 64, 64, torch.float32, seed=430,
                  with_state=False)
    for key in KEYS:
        if key == "dS0":
            # only the sequence with tokens has a nonzero dL/dS0
            assert torch.count_nonzero(g[key][[0, 2]]) == 0
        assert max_rel(g[key], ref[key]) <= F32_TOL, key
