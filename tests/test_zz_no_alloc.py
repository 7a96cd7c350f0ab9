"""nm_forward_mlp2_noalloc: the MLP memory forward for callers that cannot
allocate device memory (a host that owns the whole device through its own
pool, or a loop that cannot take cudaMalloc's device-wide synchronisation).

It runs the fp32 FFMA MLP kernel with its workspace in a fixed file-scope
device array instead of a handle's allocation.  The test calls it through the
C ABI and checks it against the handle-based nm_forward on the same inputs,
within the bf16 tolerances the parity tests use, on two calls in a row (the
second on other inputs, over the array left behind by the first).  It also
checks that a call needing more than the array returns NM_ERR_TOO_LARGE.

This file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

import test_neural_memory_titans_b300 as nm
from test_neural_memory_titans_b300 import workloads as W

from _helpers import TOL, rel_l2

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


def test_noalloc_matches_nm_forward_twice():
    wl = W.WORKLOADS[1]
    cfg = nm._Config(nm.MLP2, wl.d, wl.hidden, wl.chunk, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO)
    mem = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk, in_dtype=wl.dtype, path=nm.PATH_SIMT)
    tol = TOL[torch.bfloat16]
    for call, (B, H, T, seed) in enumerate([(1, 3, 150, 1), (2, 2, 200, 2)]):
        w = wl.with_sizes(B=B, H=H, T=T)
        x = W.make_inputs(w, "cuda", seed=seed)
        M0, S0 = W.random_state(w, "cuda", seed=10 + seed)
        got = _noalloc(cfg, x, M0, S0)
        ref = mem.forward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], M0, S0)
        assert mem.synchronize() == nm.NM_OK
        for name, g, r in zip(("y", "M_T", "S_T"), got, ref):
            err = rel_l2(g.double().cpu().numpy(), r.double().cpu().numpy())
            assert err <= tol[name], "call %d: %s rel L2 %.3e" % (call, name, err)
    mem.close()


def test_noalloc_rejects_calls_beyond_its_workspace():
    wl = W.WORKLOADS[1]
    per_unit = 4 * (2 * wl.chunk ** 2 + 2 * wl.chunk + 4 * wl.chunk * wl.d + 4 * wl.chunk * wl.hidden)
    H = SCRATCH_BYTES // per_unit + 1
    w = wl.with_sizes(B=1, H=H, T=1)
    x = W.make_inputs(w, "cuda", seed=3)
    y = torch.empty(x["q"].shape, dtype=torch.bfloat16, device="cuda")
    MT = torch.empty_like(x["M0"])
    ST = torch.empty_like(x["S0"])
    cfg = nm._Config(nm.MLP2, wl.d, wl.hidden, wl.chunk, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO)
    rc = _entry()(ctypes.byref(cfg), 1, H, 1, _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["alpha"]), _p(x["eta"]),
                  _p(x["beta"]), None, _p(x["M0"]), _p(x["S0"]), _p(y), _p(MT), _p(ST), None)
    assert rc == NM_ERR_TOO_LARGE
    assert "workspace" in nm.status_string(rc)
