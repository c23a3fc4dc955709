"""GPU parity of kda_prefill_conv -- the short convolutions fused into the
split prefill (bf16, d = 128, all pairs in one batch; two passes otherwise)
-- through the C ABI.

Two bars:
- bit-exact against the two-pass path on the same inputs (kda_short_conv,
  then kda_prefill on its outputs, both on the split kernel): o, the final
  state and the conv state out.  The fused producers convolve with the same
  arithmetic and rounding as kda_short_conv, so the prefill sees the same
  bf16 values; any difference is a fault of the fusion (a halo row, a chunk
  boundary, a sequence boundary, the conv state);
- against the fp64 oracle (the convolutions, then the recurrence): o and the
  final state at 2e-2 relative Frobenius, the conv state bit-exact (a copy of
  inputs).
The cases cover several chunks per sequence (halo rows from the previous
chunk), ragged tails, an empty sequence, sequences shorter than W-1 (the conv
state out then mixes conv state in and inputs), widths 1 to 4, with and
without SiLU and a conv state in, and the equal split without cu_seqlens."""
import numpy as np
import pytest
import torch

import kimi_delta_attention_12_gb300 as kda
from kimi_delta_attention_12_gb300 import inputs
from metrics import BF16_TOL, rel_fro

pytestmark = pytest.mark.gpu

DEV = "cuda"
D = 128


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    kda.lib()


def _case(lens, H, W, seed, with_state=True, nonzero_state=True):
    x = inputs.make_prefill_inputs(lens, H, D, D, torch.bfloat16, seed=seed,
                                   nonzero_state=nonzero_state)
    w, s0 = inputs.make_conv_params(len(lens), H, D, D, W, torch.bfloat16, seed=seed,
                                    with_state=with_state)
    return x, w, s0


def _fused(x, w, s0, silu, equal_split=False):
    N = x.cu_seqlens.numel() - 1
    H = x.q.shape[1]
    W = w.shape[-1]
    xd = x.to(DEV)
    s_out = torch.full((N, H, W - 1, 3 * D), float("nan"), dtype=torch.bfloat16, device=DEV)
    ws = torch.empty(kda.prefill_conv_workspace_bytes(N, x.q.shape[0], H, D, D, torch.bfloat16),
                     dtype=torch.uint8, device=DEV)
    o, S = kda.kda_prefill_conv(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, w.to(DEV),
                                None if s0 is None else s0.to(DEV), s_out, xd.initial_state,
                                None if equal_split else xd.cu_seqlens,
                                None if equal_split else x.cu_seqlens, silu=silu,
                                workspace=ws)
    torch.cuda.synchronize()
    assert kda.workspace_status(ws) == kda.KDA_OK
    return o, S, s_out


def _two_pass(x, w, s0, silu):
    N = x.cu_seqlens.numel() - 1
    H = x.q.shape[1]
    W = w.shape[-1]
    xd = x.to(DEV)
    s_out = torch.full((N, H, W - 1, 3 * D), float("nan"), dtype=torch.bfloat16, device=DEV)
    qc, kc, vc = kda.kda_short_conv(xd.q, xd.k, xd.v, w.to(DEV),
                                    None if s0 is None else s0.to(DEV), s_out,
                                    xd.cu_seqlens, x.cu_seqlens, silu=silu)
    ws = kda.alloc_workspace(N, x.q.shape[0], H, D, D, torch.bfloat16, DEV)
    o, S = kda.kda_prefill(qc, kc, vc, xd.z, xd.beta, xd.A, xd.initial_state, xd.cu_seqlens,
                           cu_seqlens_host=x.cu_seqlens, workspace=ws)
    torch.cuda.synchronize()
    assert kda.workspace_status(ws) == kda.KDA_OK
    return o, S, s_out


@pytest.mark.parametrize("W,silu,with_state", [(4, True, True), (4, False, False),
                                               (3, True, True), (2, False, True),
                                               (1, True, False)])
def test_prefill_conv_bit_exact_vs_two_pass(W, silu, with_state):
    lens = [200, 0, 64, 130, 1, 2, 67]
    x, w, s0 = _case(lens, 3, W, seed=600 + W, with_state=with_state)
    fo, fS, fs = _fused(x, w, s0, silu)
    to, tS, ts = _two_pass(x, w, s0, silu)
    assert torch.equal(fo, to), "o differs from the two-pass path"
    assert torch.equal(fS, tS), "final state differs from the two-pass path"
    if W > 1:
        assert torch.equal(fs, ts), "conv state differs from the two-pass path"


@pytest.mark.parametrize("W,silu", [(4, True), (3, False)])
def test_prefill_conv_matches_oracle(oracle_mod, W, silu):
    lens = [150, 0, 2, 64, 97]
    x, w, s0 = _case(lens, 2, W, seed=620 + W)
    o, S, s_out = _fused(x, w, s0, silu)
    ro, rS, rs = oracle_mod.kda_reference_conv(x.q, x.k, x.v, x.z, x.beta, x.A, w, s0,
                                               x.initial_state, x.cu_seqlens, silu=silu)
    assert rel_fro(o, ro) <= BF16_TOL
    assert rel_fro(S, rS) <= BF16_TOL
    got = s_out.cpu().double().numpy()
    assert np.array_equal(got, rs), "conv state out is not the last W-1 inputs"


def test_prefill_conv_equal_split_long():
    """One sequence of 2,000 tokens (32 chunks, ragged tail) without
    cu_seqlens."""
    lens = [2000]
    x, w, s0 = _case(lens, 2, 4, seed=640)
    fo, fS, fs = _fused(x, w, s0, True, equal_split=True)
    to, tS, ts = _two_pass(x, w, s0, True)
    assert torch.equal(fo, to) and torch.equal(fS, tS) and torch.equal(fs, ts)


def test_prefill_conv_many_pairs_two_pass():
    """80 (sequence, head) pairs, more than one batch of the split kernel: the
    call takes the two passes through its own workspace, same bits."""
    lens = [100, 50]
    x, w, s0 = _case(lens, 40, 4, seed=650)
    fo, fS, fs = _fused(x, w, s0, True)
    to, tS, ts = _two_pass(x, w, s0, True)
    assert torch.equal(fo, to) and torch.equal(fS, tS) and torch.equal(fs, ts)
