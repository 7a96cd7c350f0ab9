"""Host-side logic of bench.py, on the CPU: the work model behind the roofline
fractions, the staleness rule of the ncu traffic table, and the workload
selection (sizes and depth overrides)."""
import argparse
import dataclasses
import importlib.util
import os

import pytest

from test_neural_memory_titans_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _args(**over):
    base = dict(workload=1, B=None, H=None, T=None, layers=None)
    base.update(over)
    return argparse.Namespace(**base)


def test_flop_model_matches_the_per_token_formulas():
    b = _bench()
    for wid in range(5):
        wl = W.WORKLOADS[wid]
        alg = b.algorithmic(wl)
        d, h, c = wl.d, wl.hidden, wl.chunk
        per_tok = 10 * d * d + 2 * (c + 1) * d if wl.kind == W.LINEAR else 22 * d * h + 2 * (c + 1) * (d + h)
        assert alg["flops"] == pytest.approx(per_tok * wl.B * wl.H * wl.T, rel=1e-12)
        assert alg["tokens"] == wl.B * wl.H * wl.T
        assert alg["bound"] == ("hbm" if wl.kind == W.LINEAR else "tensor")
    # an L-layer memory: 11 flops per parameter and token plus the causal products of every layer input
    wl3 = dataclasses.replace(W.WORKLOADS[1], layers=3)
    d, h, c = wl3.d, wl3.hidden, wl3.chunk
    P = 2 * h * d + h * h
    assert wl3.P == P
    assert b.algorithmic(wl3)["flops"] == pytest.approx((11 * P + 2 * (c + 1) * (d + 2 * h)) * wl3.tokens, rel=1e-12)


def test_bytes_model_counts_inputs_outputs_gates_and_state():
    b = _bench()
    wl = W.WORKLOADS[2]
    alg = b.algorithmic(wl)
    per_tok = 3 * wl.d * 2 + 12 + wl.d * 2
    assert alg["bytes"] == per_tok * wl.tokens + 4 * wl.P * 4 * wl.B * wl.H
    wl4 = W.WORKLOADS[4]  # streamed: the state crosses HBM once per segment call
    calls = wl4.T // wl4.segment
    assert b.algorithmic(wl4)["calls"] == calls


def test_ncu_traffic_only_for_the_captured_source():
    b = _bench()
    for name, (files, digest, nbytes) in b.NCU_TRAFFIC.items():
        got = b.ncu_traffic(name)
        assert got in (None, nbytes)
    saved = dict(b.NCU_TRAFFIC)
    try:
        name = next(iter(saved))
        files, digest, nbytes = saved[name]
        b.NCU_TRAFFIC[name] = (files, "0" * 16, nbytes)  # a capture of some other source
        assert b.ncu_traffic(name) is None
    finally:
        b.NCU_TRAFFIC.clear()
        b.NCU_TRAFFIC.update(saved)
    assert b.ncu_traffic("no such workload") is None


def test_workload_overrides():
    b = _bench()
    assert b.workload(_args()) is W.WORKLOADS[1]
    small = b.workload(_args(B=1, H=2, T=128))
    assert (small.B, small.H, small.T) == (1, 2, 128) and small.name != W.WORKLOADS[1].name
    deep = b.workload(_args(layers=4))
    assert deep.layers == 4 and deep.name.endswith("_L4") and deep.P == 2 * 64 * 256 + 2 * 256 * 256
    short = b.workload(_args(workload=4, T=4096))  # a streamed workload below one segment runs as one call
    assert short.segment == 0
    with pytest.raises(SystemExit):
        b.workload(_args(workload=2, layers=3))


def test_roofline_takes_the_peak_of_the_products_operand_type():
    """The 2-layer tensor-core kernels' products are bf16 (the measured bf16
    peak); the deeper memory's are tf32 (that peak times 1.1 / 2.25, the
    nominal dense tf32 / bf16 ratio of a B300); the fp32 FFMA path of an MLP
    memory is still measured against the tensor roofline of the workload."""
    b = _bench()
    peaks = {"hbm_gbs": 6500.0, "bf16_tflops": 1750.0, "bf16_tflops_sustained": 1350.0}
    wl1 = W.WORKLOADS[1]
    r = b.roofline(wl1, 0.6, True, peaks, "measured", None)
    assert r["bound"] == "tensor" and r["peak"] == 1750.0
    assert r["frac"] == pytest.approx(b.algorithmic(wl1)["flops"] / 0.6e-3 / 1e12 / 1750.0, rel=1e-12)
    wl3 = dataclasses.replace(W.WORKLOADS[1], layers=3)
    r3 = b.roofline(wl3, 14.0, True, peaks, "measured", None)
    assert r3["peak"] == pytest.approx(1750.0 * 1.1 / 2.25, rel=1e-12) and "tf32" in r3["peak_source"]
    assert r3["frac"] == pytest.approx(r3["achieved"] / r3["peak"], rel=1e-12)
    r3f = b.roofline(wl3, 147.0, False, peaks, "measured", None)
    assert r3f["peak"] == 1750.0
    r2 = b.roofline(W.WORKLOADS[2], 1.14, True, peaks, "measured", 2.17e9)
    assert r2["bound"] == "hbm" and r2["peak"] == 6500.0 and r2["traffic"] == 2.17e9


def test_deep_traffic_entry_names_the_deep_kernel_sources():
    b = _bench()
    files, digest, nbytes = b.NCU_TRAFFIC["mlp_64x256_bf16_b4h8_t4096_c64_L3"]
    assert files[0] == "nm_tc_deep.cu" and len(digest) == 16 and nbytes > 0


def test_backward_traffic_entry_names_the_sweep_sources():
    """The backward line's traffic is the reverse sweep's (nm_backward.cu), keyed
    apart from the forward kernel's entry of the same workload."""
    b = _bench()
    files, digest, nbytes = b.NCU_TRAFFIC["linear_d128_bf16_b8h16_t16384_c64@backward_tc"]
    assert files[0] == "nm_backward.cu" and len(digest) == 16
    assert nbytes > b.NCU_TRAFFIC["linear_d128_bf16_b8h16_t16384_c64"][2]
