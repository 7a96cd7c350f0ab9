"""nm_backward against the fp64 reference gradients (oracle/backward.py, pinned
to central differences of the C oracle's forward in
tests/test_oracle_backward.py), element by element on the same seeded
inputs: every gradient (q, k, v, alpha, eta, beta, c, M0, S0) of
L = <Gy, y> + <GM, M_T> + <GS, S_T> for random upstream gradients.

Tolerance.  Both sides differentiate the same function of the same (bf16-
rounded, where the inputs are bf16) values; the GPU works in fp32.  Each
gradient is a sum over a chunk of products of fp32-rounded terms (unit
roundoff 6e-8) carried through ceil(T / chunk) chunks of the reverse sweep,
whose adjoint recursion contracts by the forgetting factor, so a relative L2
error of a few 1e-7 is expected (measured: 8e-8 to 1.3e-6 over these cases);
the bound is 1e-5, ten times tighter than the fp32 forward's 1e-4.

On a tensor-core handle (NM_PATH_TC) the reverse sweep's contractions run as
tf32 tensor-core products (operands rounded to 11 significant bits, fp32
accumulation), and for the linear memory with d = 128, chunk 64 the
chunk-start states come from the tensor-core forward (bf16 copies of the
state as operands): those cases are held to the bf16-input tolerances of the
forward (relative L2 1e-2 on the state's gradients dM0, dS0, 2e-2 on the
others).
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from oracle import backward as ob
import test_neural_memory_titans_b300 as nm
from test_neural_memory_titans_b300 import workloads as W

from _helpers import f64, rel_l2

pytestmark = pytest.mark.gpu

TOL = 1e-5
TOL_TC = {"M0": 1e-2, "S0": 1e-2}  # every other gradient: 2e-2
NAMES = ("q", "k", "v", "alpha", "eta", "beta", "M0", "S0")


def _tol(path, name):
    return TOL if path == nm.PATH_SIMT else TOL_TC.get(name, 2e-2)


def _handle(path, *args, **kw):
    """A handle on the given path, or a skip where that path is not built for the shape."""
    try:
        return nm.NeuralMemory(*args, path=path, **kw)
    except nm.NMError as e:
        if e.status == nm.NM_ERR_UNSUPPORTED and path == nm.PATH_TC:
            pytest.skip("no tensor-core kernel for this shape")
        raise


def _case(wid, d, T, chunk, dtype, seed, c_mode, units=2):
    wl = dataclasses.replace(W.WORKLOADS[wid], d=d, chunk=chunk, dtype=dtype).with_sizes(B=1, H=units, T=T,
                                                                                           segment=0)
    x = W.make_inputs(wl, "cuda", seed=seed)
    M0, S0 = W.random_state(wl, "cuda", seed=seed + 1, scale=0.5)
    x["M0"], x["S0"] = M0, S0
    if c_mode == nm.C_PER_TOKEN:
        x["c"] = torch.rand(x["alpha"].shape, device="cuda", generator=torch.Generator("cuda").manual_seed(seed + 2))
    g = torch.Generator("cuda").manual_seed(seed + 3)
    up = {"Gy": torch.randn((1, units, T, d), generator=g, device="cuda"),
          "GM": torch.randn((1, units, d * d), generator=g, device="cuda"),
          "GS": torch.randn((1, units, d * d), generator=g, device="cuda")}
    return wl, x, up


@pytest.mark.parametrize("wid,d,T,chunk,dtype,c_mode,delta", [
    (0, 16, 37, 8, torch.float32, nm.C_ONE, None),
    (0, 64, 200, 16, torch.float32, nm.C_ONE, None),
    (2, 64, 130, 64, torch.bfloat16, nm.C_ONE, None),
    (4, 64, 300, 256, torch.bfloat16, nm.C_PER_TOKEN, None),
    (2, 128, 130, 64, torch.bfloat16, nm.C_ONE_MINUS_BETA, 0.08),
    (2, 32, 75, 32, torch.float32, nm.C_PER_TOKEN, 0.05),
])
@pytest.mark.parametrize("path", [nm.PATH_SIMT, nm.PATH_TC])
def test_backward_linear_matches_reference(wid, d, T, chunk, dtype, c_mode, delta, path):
    wl, x, up = _case(wid, d, T, chunk, dtype, seed=200 + T, c_mode=c_mode)
    loss = nm.LOSS_L2 if delta is None else nm.LOSS_HUBER
    mem = _handle(path, nm.LINEAR, d, 0, chunk, in_dtype=dtype, c_mode=c_mode, loss=loss,
                  huber_delta=0.0 if delta is None else delta)
    got = mem.backward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"],
                       up["Gy"], up["GM"], up["GS"], c=x.get("c"))
    assert mem.synchronize() == nm.NM_OK
    mem.close()
    names = NAMES + (("c",) if c_mode == nm.C_PER_TOKEN else ())
    errs = {}
    for u in range(wl.H):
        sel = lambda t: None if t is None else f64(t[0, u])
        ref = ob.backward(oracle.LINEAR, d, 0, chunk, c_mode, sel(x["q"]), sel(x["k"]), sel(x["v"]),
                          sel(x["alpha"]), sel(x["eta"]), sel(x["beta"]), sel(x.get("c")), sel(x["M0"]),
                          sel(x["S0"]), sel(up["Gy"]), sel(up["GM"]), sel(up["GS"]),
                          oracle.LOSS_L2 if delta is None else oracle.LOSS_HUBER,
                          np.inf if delta is None else delta)
        for n_ in names:
            errs[(n_, u)] = rel_l2(f64(got[n_][0, u]), ref[n_])
    print({k_: "%.2e" % v_ for k_, v_ in errs.items()})
    bad = {k_: v_ for k_, v_ in errs.items() if not v_ <= _tol(path, k_[0])}
    assert not bad, bad


def test_backward_zero_tokens_passes_the_state_adjoints():
    wl, x, up = _case(2, 64, 1, 64, torch.bfloat16, seed=7, c_mode=nm.C_ONE)
    for key in ("q", "k", "v", "alpha", "eta", "beta"):
        x[key] = x[key][:, :, :0].contiguous()
    up["Gy"] = up["Gy"][:, :, :0].contiguous()
    mem = nm.NeuralMemory(nm.LINEAR, 64, 0, 64, in_dtype=torch.bfloat16)
    got = mem.backward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"],
                       up["Gy"], up["GM"], up["GS"])
    assert mem.synchronize() == nm.NM_OK
    assert torch.equal(got["M0"], up["GM"]) and torch.equal(got["S0"], up["GS"])


@pytest.mark.parametrize("d,hidden,T,chunk,dtype,c_mode,delta", [
    (16, 32, 37, 8, torch.float32, nm.C_ONE, None),
    (64, 128, 130, 64, torch.bfloat16, nm.C_PER_TOKEN, None),
    (64, 256, 100, 64, torch.bfloat16, nm.C_ONE_MINUS_BETA, 0.5),
    (32, 64, 75, 16, torch.float32, nm.C_ONE, 0.3),
    (128, 256, 70, 64, torch.bfloat16, nm.C_ONE, None),
])
@pytest.mark.parametrize("path", [nm.PATH_SIMT, nm.PATH_TC])
def test_backward_mlp_matches_reference(d, hidden, T, chunk, dtype, c_mode, delta, path):
    """The 2-layer SiLU MLP memory (the workloads' recipe at these sizes, from
    random states W ~ N(0, 0.5 / fan_in), step eta halved)."""
    wl = dataclasses.replace(W.WORKLOADS[1], d=d, hidden=hidden, chunk=chunk, dtype=dtype).with_sizes(B=1, H=2, T=T)
    seed = 300 + T
    x = W.make_inputs(wl, "cuda", seed=seed)
    x["eta"] *= 0.5
    x["M0"], x["S0"] = W.random_state(wl, "cuda", seed=seed + 1, scale=0.5)
    if c_mode == nm.C_PER_TOKEN:
        x["c"] = torch.rand(x["alpha"].shape, device="cuda", generator=torch.Generator("cuda").manual_seed(seed + 2))
    g = torch.Generator("cuda").manual_seed(seed + 3)
    up = {"Gy": torch.randn((1, 2, T, d), generator=g, device="cuda"),
          "GM": torch.randn((1, 2, wl.P), generator=g, device="cuda"),
          "GS": torch.randn((1, 2, wl.P), generator=g, device="cuda")}
    loss = nm.LOSS_L2 if delta is None else nm.LOSS_HUBER
    mem = _handle(path, nm.MLP2, d, hidden, chunk, in_dtype=dtype, c_mode=c_mode, loss=loss,
                  huber_delta=0.0 if delta is None else delta)
    got = mem.backward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"],
                       up["Gy"], up["GM"], up["GS"], c=x.get("c"))
    assert mem.synchronize() == nm.NM_OK
    mem.close()
    names = NAMES + (("c",) if c_mode == nm.C_PER_TOKEN else ())
    errs = {}
    for u in range(2):
        sel = lambda t: None if t is None else f64(t[0, u])
        ref = ob.backward(oracle.MLP2, d, hidden, chunk, c_mode, sel(x["q"]), sel(x["k"]), sel(x["v"]),
                          sel(x["alpha"]), sel(x["eta"]), sel(x["beta"]), sel(x.get("c")), sel(x["M0"]),
                          sel(x["S0"]), sel(up["Gy"]), sel(up["GM"]), sel(up["GS"]),
                          oracle.LOSS_L2 if delta is None else oracle.LOSS_HUBER,
                          np.inf if delta is None else delta)
        for n_ in names:
            errs[(n_, u)] = rel_l2(f64(got[n_][0, u]), ref[n_])
    print({k_: "%.2e" % v_ for k_, v_ in errs.items()})
    bad = {k_: v_ for k_, v_ in errs.items() if not v_ <= _tol(path, k_[0])}
    assert not bad, bad


def test_backward_deeper_mlp_is_not_built():
    wl = W.WORKLOADS[1].with_sizes(B=1, H=1, T=64)
    x = W.make_inputs(wl, "cuda")
    mem = nm.NeuralMemory(nm.MLP2, 64, 128, 64, in_dtype=torch.bfloat16, layers=3)
    P = nm.param_count(nm.MLP2, 64, 128, 3)
    Gy = torch.zeros((1, 1, 64, 64), device="cuda")
    G = torch.zeros((1, 1, P), device="cuda")
    M0 = torch.zeros((1, 1, P), device="cuda")
    with pytest.raises(nm.NMError) as ei:
        mem.backward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], M0, M0, Gy, G, G)
    assert ei.value.status == nm.NM_ERR_UNSUPPORTED
