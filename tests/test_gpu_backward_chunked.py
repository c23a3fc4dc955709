"""GPU parity of the chunked training backward (bf16, d_k = d_v = 128, the
bounded gate: the split prefill's chunk records, the reverse state chain and
the chunk-parallel gradient assembly) against the fp64 reverse-mode oracle,
through the C ABI.

Every gradient is compared by relative Frobenius error (the bf16 bar,
2e-2): dq, dk, dv, dz, dbeta, dS0, and per head dA through its per-token
shares (metrics.check_dA).
The cases cover ragged last chunks, empty and one-token sequences, several
full chunks, a nonzero initial state and dL/dS_T, scale != 1, no in-op
normalisation, and the equal split without cu_seqlens; every call's status
word is checked."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs
from metrics import BF16_TOL, check_dA, rel_fro

pytestmark = pytest.mark.gpu

DEV = "cuda"
KEYS = ("dq", "dk", "dv", "dz", "dbeta", "dS0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


def _run(oracle_mod, lens, H, seed, with_state=True, equal_split=False, **flags):
    x = inputs.make_prefill_inputs(lens, H, 128, 128, torch.bfloat16, seed=seed,
                                   nonzero_state=with_state)
    dO, dSf = inputs.make_upstream_grads(sum(lens), len(lens), H, 128, 128, torch.bfloat16,
                                         seed=seed, with_state=with_state)
    xd = x.to(DEV)
    ws = torch.empty(kda.backward_workspace_bytes(len(lens), sum(lens), H, 128, 128,
                                                  torch.bfloat16),
                     dtype=torch.uint8, device=DEV)
    g = kda.kda_backward(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, dO.to(DEV), xd.initial_state,
                         None if equal_split else xd.cu_seqlens,
                         None if equal_split else x.cu_seqlens,
                         None if dSf is None else dSf.to(DEV), workspace=ws, **flags)
    torch.cuda.synchronize()
    assert kda.workspace_status(ws) == kda.KDA_OK
    ref = oracle_mod.kda_reference_backward(x.q, x.k, x.v, x.z, x.beta, x.A, x.initial_state,
                                            x.cu_seqlens, dO, dSf, **flags)
    return g, ref, x


def _check(g, ref, x):
    for key in KEYS:
        assert torch.isfinite(g[key]).all(), key
        assert rel_fro(g[key], ref[key]) <= BF16_TOL, (key, rel_fro(g[key], ref[key]))
    check_dA(g["dA"], g["dz"], ref["dA"], ref["dz"], x.z)


def test_chunked_backward_varlen_ragged(oracle_mod):
    """Five sequences: ragged (200 = 3 x 64 + 8), empty, exactly one chunk,
    two chunks and a tail of 2, and a single token; three heads, scale 0.9."""
    lens = [200, 0, 64, 130, 1]
    g, ref, x = _run(oracle_mod, lens, 3, seed=500, scale=0.9)
    _check(g, ref, x)
    # the empty sequence's dL/dS0 is its dL/dS_T
    _, dSf = inputs.make_upstream_grads(sum(lens), len(lens), 3, 128, 128, torch.bfloat16,
                                        seed=500)
    assert torch.equal(g["dS0"][1].cpu(), dSf[1])


def test_chunked_backward_no_norm_no_state(oracle_mod):
    """No in-op normalisation, no initial state, no dL/dS_T."""
    g, ref, x = _run(oracle_mod, [96, 33], 2, seed=510, with_state=False, l2norm=False)
    _check(g, ref, x)


def test_chunked_backward_equal_split_long(oracle_mod):
    """One sequence of 1,000 tokens (16 chunks, ragged tail) without
    cu_seqlens: the chain carries dL/dS through every chunk."""
    g, ref, x = _run(oracle_mod, [1000], 2, seed=520, equal_split=True)
    _check(g, ref, x)


def test_chunked_backward_short_single_chunk(oracle_mod):
    """A sequence shorter than one chunk, a single head."""
    g, ref, x = _run(oracle_mod, [37], 1, seed=530)
    _check(g, ref, x)


def test_chunked_backward_deterministic(oracle_mod):
    """Two calls on the same inputs give identical gradients (no atomics in
    any sum)."""
    lens = [150, 70]
    x = inputs.make_prefill_inputs(lens, 2, 128, 128, torch.bfloat16, seed=540,
                                   nonzero_state=True)
    dO, dSf = inputs.make_upstream_grads(sum(lens), 2, 2, 128, 128, torch.bfloat16, seed=540)
    xd = x.to(DEV)
    runs = [kda.kda_backward(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, dO.to(DEV),
                             xd.initial_state, xd.cu_seqlens, x.cu_seqlens, dSf.to(DEV))
            for _ in range(2)]
    torch.cuda.synchronize()
    for key in KEYS + ("dA",):
        assert torch.equal(runs[0][key], runs[1][key]), key
