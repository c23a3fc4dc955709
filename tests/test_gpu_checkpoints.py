"""GPU parity of prefill state checkpoints (kda_prefill_checkpointed) against
the fp64 oracle, through the C ABI.  For sequence n and m >= 1 with
m * interval <= its length, the state after its first m * interval tokens goes
to pool row slots[i] (default i) for checkpoint i = (checkpoints of earlier
sequences) + m - 1.  Bars: relative Frobenius <= 2e-2 per checkpoint (bf16
chunked kernels), max relative <= 1e-4 (fp32 recurrent kernel)."""
import numpy as np
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


def _run(x, interval, d, dtype, pool_rows=None, slots=None, minimal_ws=False):
    xd = x.to(DEV)
    N = x.cu_seqlens.numel() - 1
    T, H = x.q.shape[0], x.q.shape[1]
    count = kda.checkpoint_count(x.cu_seqlens, N, T, interval)
    rows = count if pool_rows is None else pool_rows
    pool = torch.full((max(rows, 1), H, d, d), float("nan"), device=DEV)
    ws = (torch.empty(512, dtype=torch.uint8, device=DEV) if minimal_ws
          else kda.alloc_workspace(N, T, H, d, d, dtype))
    o, S = kda.kda_prefill(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, xd.initial_state,
                           xd.cu_seqlens, cu_seqlens_host=x.cu_seqlens, workspace=ws,
                           ckpt_interval=interval, ckpt_pool=pool,
                           ckpt_slots=None if slots is None else slots.to(DEV))
    assert kda.workspace_status(ws) == kda.KDA_OK
    return o, S, pool, count


def _oracle_ckpts(x, interval):
    import oracle
    o, S, ck, _ = oracle.kda_reference_checkpoints(x.q, x.k, x.v, x.z, x.beta, x.A,
                                                   x.initial_state, x.cu_seqlens,
                                                   interval=interval)
    return ck


LENS = [300, 0, 77, 256, 129, 640]


@pytest.mark.parametrize("interval", [64, 192])
def test_bf16_chunked_checkpoints_match_oracle(interval):
    x = inputs.make_prefill_inputs(LENS, 4, 128, 128, torch.bfloat16, seed=31,
                                   nonzero_state=True)
    _, S, pool, count = _run(x, interval, 128, torch.bfloat16)
    counts = [l // interval for l in LENS]
    assert count == sum(counts)
    ref = _oracle_ckpts(x, interval)
    got = pool.cpu().numpy()
    assert np.isfinite(got[:count]).all()
    for i in range(count):
        assert rel_fro(got[i], ref[i]) <= BF16_TOL, (i, rel_fro(got[i], ref[i]))
    # a length that is a multiple of the interval ends with its final state
    base = np.concatenate([[0], np.cumsum(counts)])
    for n, l in enumerate(LENS):
        if l and l % interval == 0:
            assert torch.equal(pool[base[n + 1] - 1].cpu(), S[n].cpu())


def test_split_and_single_pass_checkpoints_bitwise():
    x = inputs.make_prefill_inputs(LENS, 4, 128, 128, torch.bfloat16, seed=32,
                                   nonzero_state=True)
    _, S_a, pool_a, _ = _run(x, 64, 128, torch.bfloat16)
    _, S_b, pool_b, _ = _run(x, 64, 128, torch.bfloat16, minimal_ws=True)
    assert torch.equal(pool_a, pool_b)
    assert torch.equal(S_a, S_b)


def test_checkpoint_equals_prefix_final_state():
    """Checkpoint m of a sequence is, bit for bit, the final state of a prefill
    over its first m * interval tokens (the same chunks are computed)."""
    lens = [640]
    x = inputs.make_prefill_inputs(lens, 3, 128, 128, torch.bfloat16, seed=33,
                                   nonzero_state=True)
    _, _, pool, count = _run(x, 128, 128, torch.bfloat16)
    assert count == 5
    for m in (1, 3):
        n_tok = 128 * m
        xp = inputs.PrefillInputs(x.q[:n_tok], x.k[:n_tok], x.v[:n_tok], x.z[:n_tok],
                                  x.beta[:n_tok], x.A, x.initial_state,
                                  torch.tensor([0, n_tok], dtype=torch.int32))
        xd = xp.to(DEV)
        _, Sp = kda.kda_prefill(xd.q, xd.k, xd.v, xd.z, xd.beta, xd.A, xd.initial_state,
                                xd.cu_seqlens)
        assert torch.equal(pool[m - 1].cpu(), Sp[0].cpu()), m


def test_f32_recurrent_checkpoints_match_oracle():
    lens = [130, 64, 200]
    x = inputs.make_prefill_inputs(lens, 2, 64, 64, torch.float32, seed=34, nonzero_state=True)
    _, _, pool, count = _run(x, 64, 64, torch.float32)
    assert count == 2 + 1 + 3
    ref = _oracle_ckpts(x, 64)
    assert max_rel(pool.cpu().numpy()[:count], ref) <= F32_TOL


@pytest.mark.parametrize("minimal_ws", [False, True])
def test_slot_mapping_and_skipped_rows(minimal_ws):
    """Checkpoints land in the rows the slots name; rows outside the pool are
    skipped and nothing else is written."""
    x = inputs.make_prefill_inputs(LENS, 2, 128, 128, torch.bfloat16, seed=35,
                                   nonzero_state=True)
    _, _, ident, count = _run(x, 64, 128, torch.bfloat16, minimal_ws=minimal_ws)
    pool_rows = count + 3
    slots = torch.arange(count, dtype=torch.int32).flip(0) + 2   # rows 2 .. count+1, reversed
    slots[0] = -1                                                # skipped
    slots[5] = pool_rows + 7                                     # skipped
    _, _, pool, _ = _run(x, 64, 128, torch.bfloat16, pool_rows=pool_rows, slots=slots,
                         minimal_ws=minimal_ws)
    written = set()
    for i in range(count):
        r = int(slots[i])
        if 0 <= r < pool_rows:
            assert torch.equal(pool[r], ident[i]), i
            written.add(r)
    for r in range(pool_rows):
        if r not in written:
            assert torch.isnan(pool[r]).all(), r
