"""Host-side checks of the C ABI (no GPU needed, nothing is launched).

The library must load, export every symbol include/kda.h declares, and turn
every host-detectable argument error into its status code before touching
the device.  Fake device pointers are plain aligned integers: validation
never dereferences device memory, and every call below fails validation.
"""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import kimi_delta_attention_12_gb300 as kda


@pytest.fixture(scope="module")
def L():
    from kimi_delta_attention_12_gb300 import build
    build.build()
    return kda.lib()


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "kda.h")).read()
    return sorted(set(re.findall(r"KDA_API\s+[\w\s\*]+?\b(kda_\w+)\s*\(", text)))


def test_exports_every_declared_symbol(L):
    declared = _declared_symbols()
    assert set(declared) == set(kda.EXPORTED_SYMBOLS), declared
    for name in declared:
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def test_status_strings(L):
    for code, name in [(0, "KDA_OK"), (-1, "KDA_ERR_INVALID_ARG"), (-2, "KDA_ERR_UNSUPPORTED"),
                       (-3, "KDA_ERR_ALIGNMENT"), (-4, "KDA_ERR_WORKSPACE"),
                       (-5, "KDA_ERR_CUDA"), (-6, "KDA_ERR_TIMEOUT"), (7, "KDA_ERR_UNKNOWN")]:
        assert kda.status_string(code) == name
    assert L.kda_version() >= 100


def test_workspace_bytes(L):
    # fp32 always runs the single-pass kernels: header + one int per unit
    a = L.kda_prefill_workspace_bytes(1, 4096, 32, 128, 128, kda.KDA_F32)
    b = L.kda_prefill_workspace_bytes(16, 100000, 64, 128, 128, kda.KDA_F32)
    assert 0 < a < b
    assert a % 256 == 0 and b % 256 == 0
    assert b >= 16 * 64 * 4
    # bf16 d=128 may ask for more (room for the split kernel on a GPU host)
    c = L.kda_prefill_workspace_bytes(1, 4096, 32, 128, 128, kda.KDA_BF16)
    assert c >= a and c % 256 == 0


BASE = 0x7f0000000000  # a 256-byte aligned fake device address
WS_BYTES = 1 << 20


def _prefill_args(**over):
    a = dict(q=BASE, k=BASE + 0x100000, v=BASE + 0x200000, z=BASE + 0x300000,
             beta=BASE + 0x400000, A=BASE + 0x500000, S0=None, cu=None, cu_host=None,
             N=1, T=64, H=2, dk=32, dv=32, dt=kda.KDA_F32, scale=1.0, flags=1,
             o=BASE + 0x600000, Sf=None, ws=BASE + 0x700000, ws_bytes=WS_BYTES)
    a.update(over)
    return a


def _call_prefill(L, a):
    vp = ctypes.c_void_p
    return L.kda_prefill(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["z"]), vp(a["beta"]),
                         vp(a["A"]), vp(a["S0"]), vp(a["cu"]), a["cu_host"],
                         a["N"], a["T"], a["H"], a["dk"], a["dv"], a["dt"], a["scale"],
                         a["flags"], vp(a["o"]), vp(a["Sf"]), vp(a["ws"]), a["ws_bytes"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=48), kda.KDA_ERR_UNSUPPORTED),
    (dict(dv=256), kda.KDA_ERR_UNSUPPORTED),
    (dict(dt=7), kda.KDA_ERR_UNSUPPORTED),
    (dict(N=0), kda.KDA_ERR_INVALID_ARG),
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(T=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(q=None), kda.KDA_ERR_INVALID_ARG),
    (dict(o=None), kda.KDA_ERR_INVALID_ARG),
    (dict(A=None), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=8), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=32), kda.KDA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), kda.KDA_ERR_INVALID_ARG),
    (dict(N=3, T=64), kda.KDA_ERR_INVALID_ARG),      # 64 % 3 != 0 without cu_seqlens
    (dict(ws=None), kda.KDA_ERR_WORKSPACE),
    (dict(ws_bytes=16), kda.KDA_ERR_WORKSPACE),
    (dict(q=BASE + 8), kda.KDA_ERR_ALIGNMENT),
    (dict(o=BASE + 0x600004), kda.KDA_ERR_ALIGNMENT),
    (dict(Sf=BASE + 0x800008), kda.KDA_ERR_ALIGNMENT),
    (dict(beta=BASE + 0x400002), kda.KDA_ERR_ALIGNMENT),   # fp32 beta must be 4-aligned
    (dict(ws=BASE + 0x700010), kda.KDA_ERR_ALIGNMENT),
])
def test_prefill_validation(L, over, expect):
    assert _call_prefill(L, _prefill_args(**over)) == expect


@pytest.mark.parametrize("cu,expect", [
    ([1, 64], kda.KDA_ERR_INVALID_ARG),        # must start at 0
    ([0, 63], kda.KDA_ERR_INVALID_ARG),        # must end at total_T
    ([0, 40, 30, 64], kda.KDA_ERR_INVALID_ARG),  # non-decreasing
])
def test_prefill_host_cu_seqlens_validation(L, cu, expect):
    arr = (ctypes.c_int32 * len(cu))(*cu)
    a = _prefill_args(N=len(cu) - 1, cu=BASE + 0x900000, cu_host=arr)
    assert _call_prefill(L, a) == expect


def _call_decode(L, **over):
    a = dict(q=BASE, k=BASE + 0x100000, v=BASE + 0x200000, z=BASE + 0x300000,
             beta=BASE + 0x400000, A=BASE + 0x500000, state=BASE + 0x600000, slots=None,
             pool=4, B=4, H=2, dk=128, dv=128, dt=kda.KDA_BF16, scale=1.0, flags=1,
             o=BASE + 0x700000)
    a.update(over)
    vp = ctypes.c_void_p
    return L.kda_decode_step(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["z"]), vp(a["beta"]),
                             vp(a["A"]), vp(a["state"]), vp(a["slots"]), a["pool"], a["B"],
                             a["H"], a["dk"], a["dv"], a["dt"], a["scale"], a["flags"],
                             vp(a["o"]), None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=16), kda.KDA_ERR_UNSUPPORTED),
    (dict(dt=3), kda.KDA_ERR_UNSUPPORTED),
    (dict(H=0), kda.KDA_ERR_INVALID_ARG),
    (dict(B=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(pool=2), kda.KDA_ERR_INVALID_ARG),    # identity slots need pool >= B
    (dict(state=None), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=2), kda.KDA_ERR_INVALID_ARG),   # the recurrent flag is prefill-only
    (dict(flags=8), kda.KDA_ERR_INVALID_ARG),
    (dict(k=BASE + 0x100004), kda.KDA_ERR_ALIGNMENT),
    (dict(state=BASE + 0x600008), kda.KDA_ERR_ALIGNMENT),
    (dict(slots=BASE + 0x800002), kda.KDA_ERR_ALIGNMENT),
    (dict(B=0), kda.KDA_OK),                    # nothing to do, nothing launched
])
def test_decode_validation(L, over, expect):
    assert _call_decode(L, **over) == expect


def test_state_io_validation(L):
    vp = ctypes.c_void_p
    f = L.kda_state_io
    assert f(kda.KDA_STATE_ZERO, vp(BASE), None, None, 1, 1, 2, 100, 128, None) == kda.KDA_ERR_UNSUPPORTED
    assert f(kda.KDA_STATE_GATHER, vp(BASE), vp(BASE + 0x1000), None, 1, 1, 2, 128, 128, None) == kda.KDA_ERR_INVALID_ARG
    assert f(kda.KDA_STATE_SCATTER, vp(BASE), None, vp(BASE + 0x2000), 1, 1, 2, 128, 128, None) == kda.KDA_ERR_INVALID_ARG
    assert f(kda.KDA_STATE_COPY, vp(BASE), vp(BASE + 0x1000), vp(BASE + 0x2000), 1, 1, 2, 128, 128, None) == kda.KDA_ERR_INVALID_ARG
    assert f(kda.KDA_STATE_COPY, vp(BASE + 4), vp(BASE + 0x1000), None, 1, 1, 2, 128, 128, None) == kda.KDA_ERR_ALIGNMENT
    assert f(9, vp(BASE), vp(BASE + 0x1000), None, 1, 1, 2, 128, 128, None) == kda.KDA_ERR_INVALID_ARG
    assert f(kda.KDA_STATE_ZERO, vp(BASE), None, None, 0, 0, 2, 128, 128, None) == kda.KDA_OK


def test_product_path_has_no_cpu_fallback():
    """The binding refuses CPU tensors instead of computing on the host."""
    import torch
    q = torch.zeros(4, 1, 32)
    with pytest.raises((ValueError, RuntimeError)):
        kda.kda_prefill(q, q, q, q, torch.zeros(4, 1), torch.zeros(1))


def test_package_does_not_import_oracle():
    """The product package never imports the test oracle."""
    import ast
    pkg = os.path.join(ROOT, "kimi_delta_attention_12_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith(".py"):
                tree = ast.parse(open(os.path.join(dirpath, f)).read())
                for node in ast.walk(tree):
                    if isinstance(node, ast.Import):
                        assert all(not a.name.startswith("oracle") for a in node.names), f
                    if isinstance(node, ast.ImportFrom):
                        assert not (node.module or "").startswith("oracle"), f


def test_checkpoint_count(L):
    cu = (ctypes.c_int32 * 5)(0, 300, 300, 377, 633)
    assert L.kda_checkpoint_count(cu, 4, 633, 64) == 4 + 0 + 1 + 4
    assert L.kda_checkpoint_count(cu, 4, 633, 128) == 2 + 0 + 0 + 2
    assert L.kda_checkpoint_count(None, 2, 256, 64) == 4
    assert L.kda_checkpoint_count(None, 3, 256, 64) < 0      # 256 % 3 != 0
    assert L.kda_checkpoint_count(cu, 4, 633, 0) < 0
    assert L.kda_checkpoint_count(cu, 4, 600, 64) < 0        # does not end at total_T


def _call_ckpt(L, interval, pool, slots=None, pool_size=4, **over):
    a = _prefill_args(**over)
    vp = ctypes.c_void_p
    return L.kda_prefill_checkpointed(
        vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["z"]), vp(a["beta"]), vp(a["A"]),
        vp(a["S0"]), vp(a["cu"]), a["cu_host"], a["N"], a["T"], a["H"], a["dk"], a["dv"],
        a["dt"], a["scale"], a["flags"], vp(a["o"]), vp(a["Sf"]), interval, vp(pool),
        vp(slots), pool_size, vp(a["ws"]), a["ws_bytes"], None)


@pytest.mark.parametrize("interval,pool,slots,pool_size,expect", [
    (32, BASE + 0xA00000, None, 4, kda.KDA_ERR_INVALID_ARG),       # not a multiple of 64
    (-64, BASE + 0xA00000, None, 4, kda.KDA_ERR_INVALID_ARG),
    (64, None, None, 4, kda.KDA_ERR_INVALID_ARG),                  # no pool
    (64, BASE + 0xA00000, None, 0, kda.KDA_ERR_INVALID_ARG),       # empty pool
    (64, BASE + 0xA00008, None, 4, kda.KDA_ERR_ALIGNMENT),
    (64, BASE + 0xA00000, BASE + 0xB00002, 4, kda.KDA_ERR_ALIGNMENT),
])
def test_checkpoint_validation(L, interval, pool, slots, pool_size, expect):
    assert _call_ckpt(L, interval, pool, slots, pool_size) == expect


def test_checkpoint_zero_interval_is_plain_prefill_validation(L):
    # interval 0 takes the plain path: the other arguments are validated as usual
    assert _call_ckpt(L, 0, None, None, 0, dk=48) == kda.KDA_ERR_UNSUPPORTED


def _call_conv(L, **over):
    # q, k, v, outputs and states far apart; T=64, H=2, d=32 (bf16): 8 KB each
    a = dict(q=BASE, k=BASE + 0x100000, v=BASE + 0x200000, w=BASE + 0x300000,
             s_in=BASE + 0x400000, s_out=BASE + 0x500000, cu=None, cu_host=None, N=1, T=64,
             H=2, dk=32, dv=32, W=4, dt=kda.KDA_BF16, flags=0, qo=BASE + 0x600000,
             ko=BASE + 0x700000, vo=BASE + 0x800000)
    a.update(over)
    vp = ctypes.c_void_p
    return L.kda_short_conv(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["w"]), vp(a["s_in"]),
                            vp(a["s_out"]), vp(a["cu"]), a["cu_host"], a["N"], a["T"], a["H"],
                            a["dk"], a["dv"], a["W"], a["dt"], a["flags"], vp(a["qo"]),
                            vp(a["ko"]), vp(a["vo"]), None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=48), kda.KDA_ERR_UNSUPPORTED),
    (dict(dt=5), kda.KDA_ERR_UNSUPPORTED),
    (dict(W=0), kda.KDA_ERR_INVALID_ARG),
    (dict(W=5), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=1), kda.KDA_ERR_INVALID_ARG),          # only KDA_FLAG_CONV_SILU applies
    (dict(N=0), kda.KDA_ERR_INVALID_ARG),
    (dict(T=-1), kda.KDA_ERR_INVALID_ARG),
    (dict(w=None), kda.KDA_ERR_INVALID_ARG),
    (dict(vo=None), kda.KDA_ERR_INVALID_ARG),
    (dict(N=3), kda.KDA_ERR_INVALID_ARG),              # 64 % 3 without cu_seqlens
    (dict(qo=BASE), kda.KDA_ERR_INVALID_ARG),          # output on top of its input
    (dict(ko=BASE + 0x201000), kda.KDA_ERR_INVALID_ARG),   # output inside v
    (dict(vo=BASE + 0x601000), kda.KDA_ERR_INVALID_ARG),   # two outputs overlap
    (dict(s_out=BASE + 0x400100), kda.KDA_ERR_INVALID_ARG),  # state out overlaps state in
    (dict(s_out=BASE + 0x800100), kda.KDA_ERR_INVALID_ARG),  # state out overlaps an output
    (dict(q=BASE + 8), kda.KDA_ERR_ALIGNMENT),
    (dict(s_in=BASE + 0x400008), kda.KDA_ERR_ALIGNMENT),
    (dict(w=BASE + 0x300002), kda.KDA_ERR_ALIGNMENT),
    (dict(w=BASE + 0x300004), kda.KDA_ERR_ALIGNMENT),      # taps are read as 16-byte vectors
])
def test_short_conv_validation(L, over, expect):
    assert _call_conv(L, **over) == expect


def test_short_conv_host_cu_seqlens_validation(L):
    arr = (ctypes.c_int32 * 3)(0, 70, 64)
    assert _call_conv(L, N=2, cu=BASE + 0x900000, cu_host=arr) == kda.KDA_ERR_INVALID_ARG


def _call_decode_conv(L, **over):
    a = dict(q=BASE, k=BASE + 0x100000, v=BASE + 0x200000, z=BASE + 0x300000,
             beta=BASE + 0x400000, A=BASE + 0x500000, state=BASE + 0x600000, slots=None,
             pool=4, w=BASE + 0x800000, cs=BASE + 0x900000, W=4, B=4, H=2, dk=128, dv=128,
             dt=kda.KDA_BF16, scale=1.0, flags=1, o=BASE + 0x700000, ws=BASE + 0xa00000,
             ws_bytes=1 << 20)
    a.update(over)
    vp = ctypes.c_void_p
    return L.kda_decode_step_conv(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["z"]),
                                  vp(a["beta"]), vp(a["A"]), vp(a["state"]), vp(a["slots"]),
                                  a["pool"], vp(a["w"]), vp(a["cs"]), a["W"], a["B"], a["H"],
                                  a["dk"], a["dv"], a["dt"], a["scale"], a["flags"], vp(a["o"]),
                                  vp(a["ws"]), a["ws_bytes"], None)


@pytest.mark.parametrize("over,expect", [
    (dict(W=0), kda.KDA_ERR_INVALID_ARG),
    (dict(W=5), kda.KDA_ERR_INVALID_ARG),
    (dict(w=None), kda.KDA_ERR_INVALID_ARG),
    (dict(cs=None), kda.KDA_ERR_INVALID_ARG),          # W > 1 needs a conv state
    (dict(flags=2), kda.KDA_ERR_INVALID_ARG),          # the recurrent flag is prefill-only
    (dict(flags=32), kda.KDA_ERR_INVALID_ARG),
    (dict(dk=16), kda.KDA_ERR_UNSUPPORTED),
    (dict(pool=2), kda.KDA_ERR_INVALID_ARG),
    (dict(w=BASE + 0x800002), kda.KDA_ERR_ALIGNMENT),
    (dict(w=BASE + 0x800008), kda.KDA_ERR_ALIGNMENT),
    (dict(cs=BASE + 0x900008), kda.KDA_ERR_ALIGNMENT),
    (dict(ws=None), kda.KDA_ERR_WORKSPACE),
    (dict(ws_bytes=1024), kda.KDA_ERR_WORKSPACE),     # 3 x 4 x 2 x 128 bf16 = 6 KB needed
    (dict(ws=BASE + 0xa00008), kda.KDA_ERR_ALIGNMENT),
    (dict(ws=BASE + 0x700100), kda.KDA_ERR_INVALID_ARG),   # workspace overlapping o
    (dict(B=70000, pool=70000), kda.KDA_ERR_UNSUPPORTED),
    (dict(B=0, flags=1 | 4 | 8), kda.KDA_OK),          # nothing to do, nothing launched
])
def test_decode_conv_validation(L, over, expect):
    assert _call_decode_conv(L, **over) == expect


def test_decode_conv_workspace_bytes(L):
    f = L.kda_decode_conv_workspace_bytes
    assert f(4, 2, 128, 128, kda.KDA_BF16) == 3 * 4 * 2 * 128 * 2
    assert f(3, 1, 32, 64, kda.KDA_F32) == 512 + 512 + 768     # each part rounded up to 256 B
    assert f(-1, 2, 128, 128, kda.KDA_BF16) == 0


def _call_backward(L, **over):
    a = dict(q=BASE, k=BASE + 0x100000, v=BASE + 0x200000, z=BASE + 0x300000,
             beta=BASE + 0x400000, A=BASE + 0x500000, S0=None, cu=None, cu_host=None, N=1, T=64,
             H=2, dk=32, dv=32, dt=kda.KDA_F32, scale=1.0, flags=1, dO=BASE + 0x600000,
             dSf=None, dq=BASE + 0x700000, dk_=BASE + 0x800000, dv_=BASE + 0x900000,
             dz=BASE + 0xa00000, db=BASE + 0xb00000, dA=BASE + 0xc00000, dS0=BASE + 0xd00000,
             ws=BASE + 0x1000000, ws_bytes=64 << 20)
    a.update(over)
    vp = ctypes.c_void_p
    return L.kda_backward(vp(a["q"]), vp(a["k"]), vp(a["v"]), vp(a["z"]), vp(a["beta"]),
                          vp(a["A"]), vp(a["S0"]), vp(a["cu"]), a["cu_host"], a["N"], a["T"],
                          a["H"], a["dk"], a["dv"], a["dt"], a["scale"], a["flags"], vp(a["dO"]),
                          vp(a["dSf"]), vp(a["dq"]), vp(a["dk_"]), vp(a["dv_"]), vp(a["dz"]),
                          vp(a["db"]), vp(a["dA"]), vp(a["dS0"]), vp(a["ws"]), a["ws_bytes"],
                          None)


@pytest.mark.parametrize("over,expect", [
    (dict(dk=48), kda.KDA_ERR_UNSUPPORTED),
    (dict(dt=4), kda.KDA_ERR_UNSUPPORTED),
    (dict(N=0), kda.KDA_ERR_INVALID_ARG),
    (dict(flags=2), kda.KDA_ERR_INVALID_ARG),      # the recurrent flag is a forward choice
    (dict(flags=8), kda.KDA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), kda.KDA_ERR_INVALID_ARG),
    (dict(dO=None), kda.KDA_ERR_INVALID_ARG),
    (dict(dA=None), kda.KDA_ERR_INVALID_ARG),
    (dict(dS0=None), kda.KDA_ERR_INVALID_ARG),
    (dict(db=None), kda.KDA_ERR_INVALID_ARG),
    (dict(N=3), kda.KDA_ERR_INVALID_ARG),          # 64 % 3 without cu_seqlens
    (dict(ws=None), kda.KDA_ERR_WORKSPACE),
    (dict(ws_bytes=4096), kda.KDA_ERR_WORKSPACE),
    (dict(dS0=BASE + 0xd00008), kda.KDA_ERR_ALIGNMENT),
    (dict(dq=BASE + 0x700002), kda.KDA_ERR_ALIGNMENT),
    (dict(ws=BASE + 0x1000008), kda.KDA_ERR_ALIGNMENT),
    (dict(ws=BASE + 0x1000080), kda.KDA_ERR_ALIGNMENT),   # the forward's part needs 256 B
])
def test_backward_validation(L, over, expect):
    assert _call_backward(L, **over) == expect


def test_backward_workspace_bytes(L):
    f = L.kda_backward_workspace_bytes
    r256 = lambda x: (x + 255) // 256 * 256
    SS = 32 * 32 * 4
    prefill = r256(L.kda_prefill_workspace_bytes(1, 64, 2, 32, 32, kda.KDA_F32))
    want = (prefill + r256(64 * 2 * 32 * 4)        # forward o
            + 1 * 2 * SS                           # one checkpoint (64 tokens) per head
            + 2 * 64 * SS                          # 64 scratch states per head
            + r256(64 * 2 * 97 * 4)                # one column group of partials
            + 64 * 2 * 4)                          # per-token dA shares
    assert f(1, 64, 2, 32, 32, kda.KDA_F32) == want
    assert f(0, 64, 2, 32, 32, kda.KDA_F32) == 0 and f(1, 64, 2, 48, 32, kda.KDA_F32) == 0
