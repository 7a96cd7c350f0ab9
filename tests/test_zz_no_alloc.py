"""nm_forward_mlp2_noalloc: the MLP memory forward for callers that cannot
allocate device memory (a host that owns the whole device through its own
pool, or a loop that cannot take cudaMalloc's device-wide synchronisation).

It runs the fp32 FFMA MLP kernel with its workspace in a fixed file-scope
device array instead of a handle's allocation.  The kernel and its arithmetic
are the same as nm_forward's on the fp32 FFMA path, so the tests call it
through the C ABI and require the result to equal nm_forward's bit for bit
(a workspace-offset mistake that perturbs the result slightly would not pass
a tolerance-free comparison): two calls in a row on different inputs (the
second over the array left behind by the first), then a deeper (3-layer)
memory.  They also check that calls needing more than the array return
NM_ERR_TOO_LARGE, for the two- and the three-layer sizes.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import test_neural_memory_titans_b300 as nm
from test_neural_memory_titans_b300 import workloads as W

pytestmark = pytest.mark.gpu

NM_ERR_TOO_LARGE = 9
SCRATCH_BYTES = 16 << 20


def _entry():
    fn = nm.load_library().nm_forward_mlp2_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(nm._Config), ctypes.c_int, ctypes.c_int, ctypes.c_int] + [vp] * 13
    fn.restype = ctypes.c_int
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc(cfg, x, M0, S0):
    B, H, T, d = x["q"].shape
    y = torch.empty((B, H, T, d), dtype=torch.bfloat16, device="cuda")
    MT = torch.empty_like(M0)
    ST = torch.empty_like(S0)
    stream = torch.cuda.current_stream()
    rc = _entry()(ctypes.byref(cfg), B, H, T, _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["alpha"]), _p(x["eta"]),
                  _p(x["beta"]), None, _p(M0), _p(S0), _p(y), _p(MT), _p(ST), ctypes.c_void_p(stream.cuda_stream))
    assert rc == nm.NM_OK, nm.status_string(rc)
    torch.cuda.synchronize()
    return y, MT, ST


def _deep_state(B, H, d, hidden, layers, seed):
    """W_l ~ N(0, 0.5 / fan_in), S_l ~ 0.1 of that, packed W1, W2 .. W_L."""
    g = torch.Generator("cuda").manual_seed(seed)
    n = B * H
    ms, ss = [], []
    for li in range(layers):
        out_f = d if li == layers - 1 else hidden
        in_f = d if li == 0 else hidden
        std = (0.5 / in_f) ** 0.5
        ms.append(std * torch.randn((n, out_f * in_f), generator=g, device="cuda"))
        ss.append(0.1 * std * torch.randn((n, out_f * in_f), generator=g, device="cuda"))
    P = nm.param_count(nm.MLP2, d, hidden, layers)
    return (torch.cat(ms, 1).reshape(B, H, P).contiguous(), torch.cat(ss, 1).reshape(B, H, P).contiguous())


def _assert_bit_equal(got, ref, what):
    for name, g, r in zip(("y", "M_T", "S_T"), got, ref):
        assert torch.equal(g, r), "%s: %s differs from nm_forward (max |diff| %.3e)" % (
            what, name, (g.float() - r.float()).abs().max().item())


def test_noalloc_matches_nm_forward_twice():
    wl = W.WORKLOADS[1]
    cfg = nm._Config(nm.MLP2, wl.d, wl.hidden, wl.chunk, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO)
    mem = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk, in_dtype=wl.dtype, path=nm.PATH_SIMT)
    for call, (B, H, T, seed) in enumerate([(1, 3, 150, 1), (2, 2, 200, 2)]):
        w = wl.with_sizes(B=B, H=H, T=T)
        x = W.make_inputs(w, "cuda", seed=seed)
        M0, S0 = W.random_state(w, "cuda", seed=10 + seed)
        got = _noalloc(cfg, x, M0, S0)
        ref = mem.forward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], M0, S0)
        assert mem.synchronize() == nm.NM_OK
        _assert_bit_equal(got, ref, "call %d" % call)
    mem.close()


def test_noalloc_deep_memory_matches_nm_forward():
    """A 3-layer memory (64 -> 128 -> 128 -> 64) through the same entry point."""
    d, hidden, chunk, layers = 64, 128, 64, 3
    cfg = nm._Config(nm.MLP2, d, hidden, chunk, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO, nm.LOSS_L2, 0.0, layers)
    mem = nm.NeuralMemory(nm.MLP2, d, hidden, chunk, in_dtype=torch.bfloat16, path=nm.PATH_SIMT, layers=layers)
    w = W.WORKLOADS[1].with_sizes(B=1, H=3, T=130)
    x = W.make_inputs(w, "cuda", seed=5)
    x["eta"] *= 0.5
    M0, S0 = _deep_state(1, 3, d, hidden, layers, seed=6)
    got = _noalloc(cfg, x, M0, S0)
    ref = mem.forward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], M0, S0)
    assert mem.synchronize() == nm.NM_OK
    mem.close()
    assert torch.isfinite(got[0].float()).all()
    _assert_bit_equal(got, ref, "3-layer memory")


def _round4(n):
    return (n + 3) // 4 * 4


@pytest.mark.parametrize("layers", [2, 3])
def test_noalloc_rejects_calls_beyond_its_workspace(layers):
    d, hidden, b = 64, 256 if layers == 2 else 128, 64
    P = nm.param_count(nm.MLP2, d, hidden, layers)
    per_unit = 4 * (2 * _round4(b * b) + 2 * _round4(b) + 4 * b * d + (3 * layers - 1) * b * hidden + 2 * P)
    H = SCRATCH_BYTES // per_unit + 1
    w = W.WORKLOADS[1].with_sizes(B=1, H=H, T=1)
    x = W.make_inputs(w, "cuda", seed=3)
    P = nm.param_count(nm.MLP2, d, hidden, layers)
    M0 = torch.zeros((1, H, P), device="cuda")
    S0 = torch.zeros_like(M0)
    y = torch.empty(x["q"].shape, dtype=torch.bfloat16, device="cuda")
    MT = torch.empty_like(M0)
    ST = torch.empty_like(S0)
    cfg = nm._Config(nm.MLP2, d, hidden, b, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO, nm.LOSS_L2, 0.0,
                     0 if layers == 2 else layers)
    args = (_p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["alpha"]), _p(x["eta"]), _p(x["beta"]), None)
    rc = _entry()(ctypes.byref(cfg), 1, H, 1, *args, _p(M0), _p(S0), _p(y), _p(MT), _p(ST), None)
    assert rc == NM_ERR_TOO_LARGE
    assert "workspace" in nm.status_string(rc)
    # one unit fewer fits
    rc = _entry()(ctypes.byref(cfg), 1, H - 1, 1, *args, _p(M0[:, :H - 1]), _p(S0[:, :H - 1]), _p(y[:, :H - 1]),
                  _p(MT[:, :H - 1]), _p(ST[:, :H - 1]), None)
    assert rc == nm.NM_OK, nm.status_string(rc)
    torch.cuda.synchronize()
