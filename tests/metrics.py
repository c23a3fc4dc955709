"""Error measures used by the parity tests.

max_rel   max|x - y| / max|y| over a tensor (the fp32 bar: <= 1e-4)
rel_fro   ||x - y||_F / ||y||_F            (the bf16 bar: <= 2e-2)
max_rel_stored  as max_rel, after allowing each value the rounding of its
          storage dtype (unit roundoff u * |y|), for outputs stored in bf16.
check_dA  the bf16 bar for dL/dA, a sum of per-token shares (see below).
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


# A head's dL/dA is one number, the sum over its tokens of the shares
# s_t = sum_c dx_tc x_tc = sum_c dz_tc z_tc (x = e^A z, dz = dx e^A).  Its
# relative error is bounded only through its terms: a sum that cancels by a
# factor kappa = sum_t |s_t| / |sum_t s_t| turns a relative error e of the
# shares into up to kappa * e of the sum.  So the bf16 bar applies to the
# vector of shares (as to every other gradient), the scalar must be the sum
# of its own shares, and the relative bar is also held on the scalar where
# the sum does not cancel by more than DA_KAPPA_MAX.
DA_KAPPA_MAX = 100.0


def check_dA(dA_got, dz_got, dA_ref, dz_ref, z, tol=BF16_TOL):
    """dA_got, dA_ref [H]; dz_got, dz_ref, z [T, H, d_k].  Raises
    AssertionError naming the head and the failed test."""
    dA_got, dz_got, dA_ref, dz_ref, z = (_np(t) for t in (dA_got, dz_got, dA_ref, dz_ref, z))
    s_got = (dz_got * z).sum(-1)
    s_ref = (dz_ref * z).sum(-1)
    for h in range(dA_ref.shape[0]):
        e = rel_fro(s_got[:, h], s_ref[:, h])
        assert e <= tol, (h, "per-token shares", e)
        # (the kernel forms the shares from x = e^A z in fp32: fp32 rounding of
        # every term, against the sum of the terms' magnitudes)
        scale = float(np.abs(dz_got[:, h] * z[:, h]).sum())
        assert abs(dA_got[h] - s_got[:, h].sum()) <= 1e-5 * max(scale, 1e-30), (
            h, "dA is not the sum of its shares", float(dA_got[h]), float(s_got[:, h].sum()))
        kappa = float(np.abs(s_ref[:, h]).sum()) / max(abs(float(dA_ref[h])), 1e-30)
        if kappa <= DA_KAPPA_MAX:
            rel = abs(float(dA_got[h]) - float(dA_ref[h])) / abs(float(dA_ref[h]))
            assert rel <= tol, (h, "relative dA", rel, kappa)
