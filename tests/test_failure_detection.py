"""Device-side failure detection, tested without a GPU fault.

Every wait of the tensor-core kernels (TMA tiles, tensor-core completion, the
peers' bytes of an exchange inside a cluster) is bounded (2 s).  The test hook
nm_inject_missing_load makes the next launch skip its first tile loads, so
that wait expires: the kernel must record
NM_ERR_DEVICE_TIMEOUT in the handle's status word, skip the rest of its
tensor-core work, exit normally, and leave the context usable, so that the
next call on the same handle is correct again.
"""
import time

import pytest
import torch

import test_neural_memory_titans_b300 as nm
from test_neural_memory_titans_b300 import workloads as W

from _helpers import compare, oracle_forward

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid", [2, 1, 3], ids=["linear_d128", "mlp_64x256_cluster", "mlp_128x512_cluster"])
def test_missing_tile_load_times_out_and_the_handle_recovers(wid):
    wl = W.WORKLOADS[wid].with_sizes(B=1, H=2, T=192)
    x = W.make_inputs(wl, "cuda", seed=3)
    M0, S0 = W.random_state(wl, "cuda", seed=4, scale=0.5)
    mem = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk, in_dtype=wl.dtype, path=nm.PATH_TC)
    args = (x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], M0, S0)
    assert mem.inject_missing_load() == nm.NM_OK
    t0 = time.time()
    mem.forward(*args)
    assert mem.synchronize() == nm.NM_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 60
    # the status word was cleared by synchronize, and the same handle works again
    y, MT, ST = mem.forward(*args)
    assert mem.synchronize() == nm.NM_OK
    compare(wl, (y, MT, ST), oracle_forward(wl, x, M0=M0, S0=S0))
    mem.close()


def test_missing_load_deep_memory_times_out_and_the_handle_recovers():
    """The deeper-memory kernel (3 layers, tf32 tensor cores): the hook makes
    its copy thread issue nothing for the call's first product, so the MMA
    thread's wait for those operands gives up after 2 s."""
    import dataclasses
    import numpy as np
    import oracle
    from _helpers import TOL, f64, rel_l2
    d, hidden, layers, T = 64, 128, 3, 130
    wl = dataclasses.replace(W.WORKLOADS[1], hidden=hidden, layers=layers).with_sizes(B=1, H=2, T=T)
    x = W.make_inputs(wl, "cuda", seed=5)
    x["eta"] *= 0.5
    g = torch.Generator("cuda").manual_seed(6)
    M0 = (0.5 / hidden) ** 0.5 * torch.randn((1, 2, wl.P), generator=g, device="cuda")
    S0 = 0.1 * M0.flip(-1).contiguous()
    mem = nm.NeuralMemory(nm.MLP2, d, hidden, 64, in_dtype=torch.bfloat16, layers=layers, path=nm.PATH_TC)
    args = (x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], M0, S0)
    assert mem.inject_missing_load() == nm.NM_OK
    t0 = time.time()
    mem.forward(*args)
    assert mem.synchronize() == nm.NM_ERR_DEVICE_TIMEOUT
    assert time.time() - t0 < 60
    y, MT, ST = mem.forward(*args)
    assert mem.synchronize() == nm.NM_OK
    mem.close()
    ref = oracle.forward(oracle.MLP2, d, hidden, 64, oracle.C_ONE,
                         *(f64(x[k_]) for k_ in ("q", "k", "v", "alpha", "eta", "beta")), None, f64(M0), f64(S0),
                         layers=layers)
    tol = TOL[torch.bfloat16]
    assert rel_l2(f64(y), ref[0]) <= tol["y"]
    assert rel_l2(f64(MT), ref[1]) <= tol["M_T"]
    assert rel_l2(f64(ST), ref[2]) <= tol["S_T"]


def test_injection_needs_the_tensor_core_path():
    wl = W.WORKLOADS[0]
    mem = nm.NeuralMemory(wl.kind, wl.d, 0, wl.chunk, in_dtype=torch.float32, path=nm.PATH_SIMT)
    assert mem.inject_missing_load() == nm.NM_ERR_UNSUPPORTED
    mem.close()
