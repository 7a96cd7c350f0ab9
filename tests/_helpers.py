"""Shared test plumbing: run the CUDA path and the oracle on the same inputs.

Tolerances (relative L2 over the whole compared tensor,
||x - x_ref||_2 / ||x_ref||_2):
  fp32 inputs:                 y 1e-4, M_T 1e-4, S_T 1e-4
  bf16 inputs, fp32 state:     y 2e-2, M_T 1e-2, S_T 1e-2
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import test_neural_memory_titans_b300 as nm
from test_neural_memory_titans_b300 import workloads as W

TOL = {torch.float32: {"y": 1e-4, "M_T": 1e-4, "S_T": 1e-4},
       torch.bfloat16: {"y": 2e-2, "M_T": 1e-2, "S_T": 1e-2}}


def rel_l2(x, ref) -> float:
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref)
    num = np.linalg.norm(x - ref)
    if den == 0.0:
        return float(num)
    return float(num / den)


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def gpu_forward(wl: W.Workload, x: dict, path: int = nm.PATH_AUTO, M0=None, S0=None, c_mode=nm.C_ONE,
                chunk=None, out_dtype=None, huber_delta=None):
    mem = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk if chunk is None else chunk, in_dtype=wl.dtype,
                          out_dtype=out_dtype, c_mode=c_mode, path=path,
                          loss=nm.LOSS_L2 if huber_delta is None else nm.LOSS_HUBER,
                          huber_delta=0.0 if huber_delta is None else huber_delta)
    dev = torch.device("cuda", 0)
    g = lambda t: None if t is None else t.to(dev).contiguous()
    y, MT, ST = mem.forward(g(x["q"]), g(x["k"]), g(x["v"]), g(x["alpha"]), g(x["eta"]), g(x["beta"]),
                            g(x["M0"] if M0 is None else M0), g(x["S0"] if S0 is None else S0), c=g(x.get("c")))
    st = mem.synchronize()
    assert st == nm.NM_OK, nm.status_string(st)
    sel = mem.path
    mem.close()
    return y, MT, ST, sel


def oracle_forward(wl: W.Workload, x: dict, units=None, M0=None, S0=None, c_mode=oracle.C_ONE, chunk=None,
                   T=None, huber_delta=None):
    """Oracle on the selected flat (batch*head) units and first T tokens."""
    B, H = wl.B, wl.H
    T = x["q"].shape[2] if T is None else T

    def sel(t, tok=True):
        if t is None:
            return None
        a = t.reshape(B * H, *t.shape[2:])
        if units is not None:
            a = a[list(units)]
        if tok:
            a = a[:, :T]
        return f64(a).reshape(1, a.shape[0], *a.shape[1:])

    M0 = x["M0"] if M0 is None else M0
    S0 = x["S0"] if S0 is None else S0
    return oracle.forward(wl.kind, wl.d, wl.hidden, wl.chunk if chunk is None else chunk, c_mode,
                          sel(x["q"]), sel(x["k"]), sel(x["v"]), sel(x["alpha"]), sel(x["eta"]), sel(x["beta"]),
                          sel(x.get("c")), sel(M0, False), sel(S0, False),
                          oracle.LOSS_L2 if huber_delta is None else oracle.LOSS_HUBER,
                          np.inf if huber_delta is None else huber_delta)


def pick(t: torch.Tensor, wl: W.Workload, units=None, T=None) -> np.ndarray:
    a = t.reshape(wl.B * wl.H, *t.shape[2:])
    if units is not None:
        a = a[list(units)]
    if T is not None and a.dim() == 3:
        a = a[:, :T]
    return f64(a)[None]


def rel_l2_per_unit(x, ref) -> np.ndarray:
    """Relative L2 of each unit (axis 1 of [1, U, ...] arrays) on its own."""
    x = np.asarray(x, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    x = x.reshape(x.shape[0] * x.shape[1], -1)
    ref = ref.reshape(ref.shape[0] * ref.shape[1], -1)
    den = np.linalg.norm(ref, axis=1)
    num = np.linalg.norm(x - ref, axis=1)
    return np.where(den == 0.0, num, num / np.where(den == 0.0, 1.0, den))


def compare(wl, gpu, ref, units=None, T=None, tol=None):
    """Relative L2 of y, M_T, S_T over the whole tensor and for the worst
    unit (batch, head) on its own; returns both and asserts the tolerances
    on each, so one bad unit cannot hide inside a whole-tensor norm."""
    tol = TOL[wl.dtype] if tol is None else tol
    y, MT, ST = gpu[:3]
    got = {"y": pick(y, wl, units, T), "M_T": pick(MT, wl, units), "S_T": pick(ST, wl, units)}
    refs = {"y": ref[0], "M_T": ref[1], "S_T": ref[2]}
    out = {key: rel_l2(got[key], refs[key]) for key in got}
    worst = {}
    for key in got:
        per = rel_l2_per_unit(got[key], refs[key])
        i = int(np.nanargmax(per)) if per.size and not np.all(np.isnan(per)) else 0
        worst[key] = (float(per[i]) if per.size else 0.0, i)
    out["worst_unit"] = worst
    for key in ("y", "M_T", "S_T"):
        assert out[key] <= tol[key], "%s rel L2 %.3e > %.1e (%s)" % (key, out[key], tol[key], out)
        assert worst[key][0] <= tol[key], "%s worst-unit rel L2 %.3e (unit %d) > %.1e (%s)" % (
            key, worst[key][0], worst[key][1], tol[key], out)
    return out


def chunks_as_units(wl: W.Workload, x: dict, chunk_ids, span: int, seed: int = 77):
    """Teacher-forced units: the tokens [c*b, c*b + span) of unit u, for each
    (u, c) in chunk_ids, each started from its own random nondegenerate state."""
    b = wl.chunk
    parts = {key: [] for key in ("q", "k", "v", "alpha", "eta", "beta")}
    flat = {key: x[key].reshape(wl.B * wl.H, *x[key].shape[2:]) for key in parts}
    for (u, c) in chunk_ids:
        for key in parts:
            parts[key].append(flat[key][u, c * b: c * b + span])
    n = len(chunk_ids)
    out = {key: torch.stack(v).reshape(1, n, *v[0].shape) for key, v in parts.items()}
    wl2 = wl.with_sizes(B=1, H=n, T=span)
    M0, S0 = W.random_state(wl2, device=x["q"].device, seed=seed)
    out["M0"], out["S0"], out["c"] = M0, S0, None
    return wl2, out


class ParityAccumulator:
    """Relative L2 accumulated over pieces of a large comparison (groups of
    units, or successive segments of the same units), so that the oracle can
    run piece by piece: per unit the squared error and squared reference norm
    are summed; ``check`` asserts the whole-tensor and worst-unit values."""

    def __init__(self, n_units: int):
        self.n = n_units
        self.num = {}
        self.den = {}

    def add(self, key: str, got, ref, unit_ids) -> None:
        got = np.asarray(got, dtype=np.float64)
        ref = np.asarray(ref, dtype=np.float64)
        u = len(unit_ids)
        g = got.reshape(u, -1)
        r = ref.reshape(u, -1)
        if key not in self.num:
            self.num[key] = np.zeros(self.n)
            self.den[key] = np.zeros(self.n)
        idx = np.asarray(unit_ids)
        self.num[key][idx] += np.sum((g - r) ** 2, axis=1)
        self.den[key][idx] += np.sum(r ** 2, axis=1)

    def check(self, tol: dict) -> dict:
        out, worst = {}, {}
        for key in self.num:
            num, den = self.num[key], self.den[key]
            out[key] = float(np.sqrt(num.sum() / den.sum())) if den.sum() > 0 else float(np.sqrt(num.sum()))
            per = np.sqrt(num / np.where(den > 0, den, 1.0))
            i = int(np.argmax(per))
            worst[key] = (float(per[i]), i)
        out["worst_unit"] = worst
        for key in self.num:
            assert out[key] <= tol[key], "%s rel L2 %.3e > %.1e (%s)" % (key, out[key], tol[key], out)
            assert worst[key][0] <= tol[key], "%s worst-unit rel L2 %.3e (unit %d) > %.1e (%s)" % (
                key, worst[key][0], worst[key][1], tol[key], out)
        return out
