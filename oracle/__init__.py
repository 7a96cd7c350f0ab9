"""Plain fp64 CPU oracle for the Titans neural-memory forward pass.

TEST INFRASTRUCTURE ONLY: tests/, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
package.  The product library (``test_neural_memory_titans_b300``) never does,
and this package imports nothing from it.

The arithmetic lives in ``nm_oracle.c`` (double precision, one token at a
time, gradients at the chunk-start weights); this module only compiles it and
marshals numpy arrays.  See that file's header for the equations and the pages
they come from ("Titans: Imparare a Memorizzare al Tempo di Test", sections
"Meccanismo di Aggiornamento della Memoria", "Meccanismo di Dimenticanza",
"Funzione Obiettivo", "Addestramento Parallelizzato"; and the 0h-n0.github.io
explainer, sections "メモリ読み出し", "モメンタム機構", "適応的重み減衰").

Every function here is pinned by tests/test_oracle.py against things other than
itself: hand-worked examples, finite differences, an autograd gradient, the
delta rule, linear attention and a closed-form geometric scan.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

LINEAR = 0
MLP2 = 1
C_ONE = 0
C_ONE_MINUS_BETA = 1
C_PER_TOKEN = 2
LOSS_L2 = 0
LOSS_HUBER = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nm_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile nm_oracle.c into liboracle.so (gcc, -O2, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp.%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        i = ctypes.c_int
        dd = ctypes.c_double
        lib.oracle_forward.argtypes = [i, i, i, i, i, i, i, dd, i, i, i] + [dp] * 13
        lib.oracle_forward.restype = i
        lib.oracle_grad.argtypes = [i, i, i, i, i, dd, dp, dp, dp, dp, dp]
        lib.oracle_grad.restype = None
        lib.oracle_loss.argtypes = [i, i, i, i, i, dd, dp, dp, dp, dp]
        lib.oracle_loss.restype = ctypes.c_double
        lib.oracle_memory_apply.argtypes = [i, i, i, i, dp, dp, dp, dp]
        lib.oracle_memory_apply.restype = None
        lib.oracle_param_count.argtypes = [i, i, i, i]
        lib.oracle_param_count.restype = ctypes.c_long
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def param_count(kind: int, d: int, hidden: int = 0, layers: int = 2) -> int:
    return int(_load().oracle_param_count(kind, d, hidden, layers))


def memory_apply(kind: int, d: int, hidden: int, W, x, layers: int = 2) -> np.ndarray:
    """y = M_W(x) for one memory (linear: M x; MLP2: W_L silu(... silu(W1 x)), L = layers)."""
    W, x = _f64(W), _f64(x)
    y = np.zeros(d)
    work = np.zeros(2 * max(hidden, 1) + 8)
    _load().oracle_memory_apply(kind, d, hidden, layers, _ptr(W), _ptr(x), _ptr(y), _ptr(work))
    return y


def loss(kind: int, d: int, hidden: int, W, k, v, loss_kind: int = LOSS_L2, huber_delta: float = np.inf,
         layers: int = 2) -> float:
    """||M_W(k) - v||^2, or the element-wise Huber sum (rho(r) = r^2 inside delta,
    2 delta |r| - delta^2 beyond)."""
    W, k, v = _f64(W), _f64(k), _f64(v)
    work = np.zeros(d + 2 * max(hidden, 1) + 8)
    return float(_load().oracle_loss(kind, d, hidden, layers, loss_kind, float(huber_delta), _ptr(W), _ptr(k),
                                     _ptr(v), _ptr(work)))


def grad(kind: int, d: int, hidden: int, W, k, v, loss_kind: int = LOSS_L2, huber_delta: float = np.inf,
         layers: int = 2) -> np.ndarray:
    """grad_W of the loss above by explicit backprop."""
    W, k, v = _f64(W), _f64(k), _f64(v)
    g = np.zeros(param_count(kind, d, hidden, layers))
    work = np.zeros((2 * layers + 2) * max(hidden, 1) + 2 * d + 8)
    _load().oracle_grad(kind, d, hidden, layers, loss_kind, float(huber_delta), _ptr(W), _ptr(k), _ptr(v), _ptr(g),
                        _ptr(work))
    return g


def mag_gate(y_mem, y_attn) -> np.ndarray:
    """The Memory-as-Gate combination of the memory's output with another
    branch's output, element by element: o = sigmoid(y_mem) * y_attn with the
    logistic sigmoid 1 / (1 + exp(-y)), in fp64 (0h-n0.github.io explainer,
    "3つのアーキテクチャ変種", MAG: o_t = sigma(y_t^mem) (.) y_t^attn;
    "Titans: Imparare a Memorizzare al Tempo di Test", "Varianti
    dell'Architettura Titans", "Memory as Gate (MAG)")."""
    y_mem, y_attn = _f64(y_mem), _f64(y_attn)
    assert y_mem.shape == y_attn.shape
    with np.errstate(over="ignore"):
        return y_attn / (1.0 + np.exp(-y_mem))


def forward(kind: int, d: int, hidden: int, chunk: int, c_mode: int,
            q, k, v, alpha, eta, beta, c, M0, S0, loss_kind: int = LOSS_L2, huber_delta: float = np.inf,
            surprise: bool = False, layers: int = 2):
    """The chunked forward on [B, H, T, d] inputs and [B, H, T] gates.

    Returns (y [B,H,T,d], M_T [B,H,P], S_T [B,H,P]) as float64 arrays, and with
    surprise=True also the per-token gradient norms [B,H,T].
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, T, dd = q.shape
    assert dd == d and k.shape == q.shape and v.shape == q.shape
    alpha, eta, beta = _f64(alpha), _f64(eta), _f64(beta)
    assert alpha.shape == (B, H, T) and eta.shape == (B, H, T) and beta.shape == (B, H, T)
    P = param_count(kind, d, hidden, layers)
    M0 = _f64(M0).reshape(B, H, P)
    S0 = _f64(S0).reshape(B, H, P)
    if c_mode == C_PER_TOKEN:
        c = _f64(c)
        assert c.shape == (B, H, T)
        cp = _ptr(c)
    else:
        c = None
        cp = None
    y = np.zeros((B, H, T, d))
    MT = np.zeros((B, H, P))
    ST = np.zeros((B, H, P))
    sp = np.zeros((B, H, T)) if surprise else None
    rc = _load().oracle_forward(kind, d, hidden, layers, chunk, c_mode, loss_kind, float(huber_delta), B, H, T,
                                _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta), _ptr(beta),
                                cp, _ptr(M0), _ptr(S0), _ptr(y), _ptr(MT), _ptr(ST),
                                _ptr(sp) if surprise else None)
    if rc != 0:
        raise ValueError("oracle_forward rejected its arguments")
    return (y, MT, ST, sp) if surprise else (y, MT, ST)
