"""The split kernel's producer/consumer hand-over across many schedules.

With the full workspace kda_prefill runs the split kernel (producer CTAs
publish each chunk's operand tiles through ring slots in L2, one consumer CTA
per unit carries the state); with the minimal workspace it runs the
single-pass kernel. Both execute the same per-chunk arithmetic, so any slip
in the hand-over (a slot read before it was published, or overwritten before
it was copied out) shows up as a bitwise difference. Seeded random shapes
vary the number of batches, the ragged last batch, empty and one-token
sequences and the ring positions. Each case also checks kda_prefill_conv
(the convolutions fused into the producers when the units fit one batch)
against kda_short_conv followed by kda_prefill, bit for bit, with the conv
states. Oracle parity of these paths is in test_gpu_chunked.py and
test_gpu_prefill_conv.py."""
import random

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


def _cases(seed, n):
    rng = random.Random(seed)
    out = []
    for i in range(n):
        N = rng.randint(1, 24)
        H = rng.choice([1, 2, 3, 5, 8, 16, 24, 48])
        lens = [rng.choice([0, 1, 17, 63, 64, 65, rng.randint(0, 2000)]) for _ in range(N)]
        if sum(lens) == 0:
            lens[0] = 100
        out.append((i, lens, H, rng.random() < 0.5))
    return out


@pytest.mark.parametrize("case", _cases(11, 8), ids=lambda c: f"case{c[0]}")
def test_split_schedule_bitwise(case):
    i, lens, H, with_state = case
    N = len(lens)
    x = inputs.make_prefill_inputs(lens, H, 128, 128, torch.bfloat16, seed=300 + i,
                                   nonzero_state=with_state)
    xd = x.to(DEV)
    T = x.q.shape[0]
    big = kda.alloc_workspace(N, T, H, 128, 128, torch.bfloat16)
    small = torch.empty(256 + N * H * 4 + 256, dtype=torch.uint8, device=DEV)
    outs = []
    for ws in (big, small):
        o, S = kda.kda_prefill(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, xd.initial_state,
                               xd.cu_seqlens, cu_seqlens_host=x.cu_seqlens, workspace=ws)
        torch.cuda.synchronize()
        assert kda.workspace_status(ws) == kda.KDA_OK
        outs.append((o, S))
    assert torch.equal(outs[0][0], outs[1][0])
    assert torch.equal(outs[0][1], outs[1][1])

    w, cs0 = inputs.make_conv_params(N, H, 128, 128, 4, torch.bfloat16, seed=400 + i)
    w, cs_in = w.to(DEV), cs0.to(DEV)
    cs_fused, cs_two = torch.empty_like(cs_in), torch.empty_like(cs_in)
    wsf = torch.empty(kda.prefill_conv_workspace_bytes(N, T, H, 128, 128, torch.bfloat16),
                      dtype=torch.uint8, device=DEV)
    of, Sf = kda.kda_prefill_conv(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, w, cs_in, cs_fused,
                                  initial_state=xd.initial_state, cu_seqlens=xd.cu_seqlens,
                                  cu_seqlens_host=x.cu_seqlens, silu=True, workspace=wsf)
    qc, kc, vc = kda.kda_short_conv(xd.q, xd.k, xd.v, w, cs_in, cs_two,
                                    cu_seqlens=xd.cu_seqlens, cu_seqlens_host=x.cu_seqlens,
                                    silu=True)
    o2, S2 = kda.kda_prefill(qc, kc, vc, xd.z, xd.beta, xd.A, xd.initial_state, xd.cu_seqlens,
                             cu_seqlens_host=x.cu_seqlens, workspace=big)
    torch.cuda.synchronize()
    assert kda.workspace_status(wsf) == kda.KDA_OK
    assert kda.workspace_status(big) == kda.KDA_OK
    assert torch.equal(of, o2)
    assert torch.equal(Sf, S2)
    assert torch.equal(cs_fused, cs_two)
