"""Error measures used by the parity tests.

max_rel   max|x - y| / max|y| over a tensor (the fp32 bar: <= 1e-4)
rel_fro   ||x - y||_F / ||y||_F            (the bf16 bar: <= 2e-2)
max_rel_stored  as max_rel, after allowing each value the rounding of its
          storage dtype (unit roundoff u * |y|), for outputs stored in bf16.
"""
import numpy as np
import torch

F32_TOL = 1e-4
BF16_TOL = 2e-2
BF16_UNIT_ROUNDOFF = 2.0 ** -8


def _np(x):
    if isinstance(x, torch.Tensor):
        x = x.detach().float().cpu().numpy() if x.dtype != torch.float64 else x.cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def max_rel(x, y):
    x, y = _np(x), _np(y)
    return float(np.max(np.abs(x - y)) / max(float(np.max(np.abs(y))), 1e-30))


def rel_fro(x, y):
    x, y = _np(x), _np(y)
    return float(np.linalg.norm(x - y) / max(float(np.linalg.norm(y)), 1e-30))


def max_rel_stored(x, y, unit_roundoff=BF16_UNIT_ROUNDOFF):
    x, y = _np(x), _np(y)
    excess = np.abs(x - y) - unit_roundoff * np.abs(y)
    return float(max(float(excess.max()), 0.0) / max(float(np.max(np.abs(y))), 1e-30))
