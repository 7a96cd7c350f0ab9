"""Titans neural long-term memory forward pass on B300 (sm_103a).

A thin ctypes binding over ``libnm.so`` (C ABI in ``include/nm.h``).  This
module only marshals arguments: it checks dtypes, shapes and devices of torch
tensors, allocates outputs with torch, and passes raw pointers plus the
current CUDA stream.  Every step of the method runs in the library's CUDA
kernels; there is no CPU or PyTorch fallback, and a missing or unloadable
library raises.

The operation ("Titans: Imparare a Memorizzare al Tempo di Test", sections
"Meccanismo di Aggiornamento della Memoria", "Meccanismo di Dimenticanza",
"Funzione Obiettivo", "Addestramento Parallelizzato"; 0h-n0.github.io
explainer, "メモリ読み出し", "モメンタム機構", "適応的重み減衰"): per (batch, head)
and per chunk of ``chunk`` tokens with W0 the chunk-start memory,
``S = beta_t S + c_t grad||M_W0(k_t) - v_t||^2``,
``M = (1 - alpha_t) M - eta_t S``, ``y_t = M(q_t)``.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

LINEAR = 0
MLP2 = 1
F32 = 0
BF16 = 1
C_ONE = 0
C_ONE_MINUS_BETA = 1
C_PER_TOKEN = 2
PATH_AUTO = 0
PATH_SIMT = 1
PATH_TC = 2
LOSS_L2 = 0
LOSS_HUBER = 1

NM_OK = 0
NM_ERR_ARG = 1
NM_ERR_ALIGN = 2
NM_ERR_UNSUPPORTED = 3
NM_ERR_ALIAS = 4
NM_ERR_CUDA = 5
NM_ERR_NOMEM = 6
NM_ERR_DEVICE_TIMEOUT = 7
NM_ERR_DEVICE_CHECK = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnm.so")
EXPORTED = ("nm_create", "nm_forward", "nm_forward_host", "nm_synchronize", "nm_destroy",
            "nm_status_string", "nm_selected_path", "nm_launch_count", "nm_inject_missing_load",
            "nm_forward_mlp2_noalloc", "nm_forward_surprise", "nm_forward_gated", "nm_backward")

_DT = {torch.float32: F32, torch.bfloat16: BF16}
_TORCH_DT = {F32: torch.float32, BF16: torch.bfloat16}


class NMError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


class _Config(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("d", ctypes.c_int), ("hidden", ctypes.c_int),
                ("chunk", ctypes.c_int), ("in_dtype", ctypes.c_int), ("out_dtype", ctypes.c_int),
                ("c_mode", ctypes.c_int), ("path", ctypes.c_int), ("loss", ctypes.c_int),
                ("huber_delta", ctypes.c_float), ("layers", ctypes.c_int)]


_lib = None


def load_library() -> ctypes.CDLL:
    """Load the in-tree libnm.so; raise if it is missing (no fallback)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError("libnm.so is not built (run __graft_entry__.build() or "
                              "python test_neural_memory_titans_b300/build.py)")
        lib = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p
        lib.nm_create.argtypes = [ctypes.POINTER(_Config), i, ctypes.POINTER(vp)]
        lib.nm_create.restype = i
        fwd = [vp, i, i, i, vp, vp, vp, f, f, f, f, f, f, vp, f, f, vp]
        lib.nm_forward.argtypes = fwd
        lib.nm_forward.restype = i
        lib.nm_forward_host.argtypes = fwd
        lib.nm_forward_host.restype = i
        lib.nm_forward_surprise.argtypes = fwd[:-1] + [vp, vp]
        lib.nm_forward_surprise.restype = i
        lib.nm_forward_gated.argtypes = fwd[:13] + [vp, vp, f, f, vp]
        lib.nm_forward_gated.restype = i
        lib.nm_backward.argtypes = [vp, i, i, i] + [vp] * 22
        lib.nm_backward.restype = i
        lib.nm_synchronize.argtypes = [vp]
        lib.nm_synchronize.restype = i
        lib.nm_destroy.argtypes = [vp]
        lib.nm_destroy.restype = i
        lib.nm_status_string.argtypes = [i]
        lib.nm_status_string.restype = ctypes.c_char_p
        lib.nm_selected_path.argtypes = [vp]
        lib.nm_selected_path.restype = i
        lib.nm_launch_count.argtypes = [vp]
        lib.nm_launch_count.restype = ctypes.c_longlong
        lib.nm_inject_missing_load.argtypes = [vp]
        lib.nm_inject_missing_load.restype = i
        _lib = lib
    return _lib


def status_string(status: int) -> str:
    return load_library().nm_status_string(status).decode()


def param_count(kind: int, d: int, hidden: int = 0, layers: int = 2) -> int:
    return d * d if kind == LINEAR else 2 * hidden * d + (max(layers, 2) - 2) * hidden * hidden


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


class NeuralMemory:
    """One configured forward kernel (a handle of the C ABI)."""

    def __init__(self, kind: int, d: int, hidden: int = 0, chunk: int = 64,
                 in_dtype: torch.dtype = torch.bfloat16, out_dtype: Optional[torch.dtype] = None,
                 c_mode: int = C_ONE, path: int = PATH_AUTO, device: int = 0,
                 loss: int = LOSS_L2, huber_delta: float = 0.0, layers: int = 0):
        lib = load_library()
        out_dtype = in_dtype if out_dtype is None else out_dtype
        self.cfg = _Config(kind, d, hidden, chunk, _DT[in_dtype], _DT[out_dtype], c_mode, path, loss, huber_delta,
                           layers)
        self.kind, self.d, self.hidden, self.chunk = kind, d, hidden, chunk
        self.in_dtype, self.out_dtype, self.c_mode = in_dtype, out_dtype, c_mode
        self.device = device
        self.P = param_count(kind, d, hidden, layers)
        h = ctypes.c_void_p()
        rc = lib.nm_create(ctypes.byref(self.cfg), device, ctypes.byref(h))
        if rc != NM_OK:
            raise NMError(rc, "nm_create")
        self._h = h

    @property
    def path(self) -> int:
        return load_library().nm_selected_path(self._h)

    @property
    def launches(self) -> int:
        return int(load_library().nm_launch_count(self._h))

    def close(self):
        if getattr(self, "_h", None):
            load_library().nm_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _check(self, q, k, v, alpha, eta, beta, c, M0, S0, host: bool):
        B, H, T, d = q.shape
        if d != self.d or k.shape != q.shape or v.shape != q.shape:
            raise ValueError("q, k, v must all be [B, H, T, %d]" % self.d)
        for t in (q, k, v):
            if t.dtype != self.in_dtype:
                raise TypeError("q, k, v must be %s" % self.in_dtype)
        for t in (alpha, eta, beta) + ((c,) if c is not None else ()):
            if t.shape != (B, H, T) or t.dtype != torch.float32:
                raise ValueError("gates must be float32 [B, H, T]")
        for t in (M0, S0):
            if t.shape != (B, H, self.P) or t.dtype != torch.float32:
                raise ValueError("M0, S0 must be float32 [B, H, %d]" % self.P)
        ts = [q, k, v, alpha, eta, beta, M0, S0] + ([c] if c is not None else [])
        for t in ts:
            if not t.is_contiguous():
                raise ValueError("all tensors must be contiguous")
            if host and t.is_cuda:
                raise ValueError("forward_host takes host tensors")
            if not host and (not t.is_cuda or t.device.index != self.device):
                raise ValueError("forward takes tensors on cuda:%d" % self.device)
        return B, H, T

    def forward(self, q, k, v, alpha, eta, beta, M0, S0, c=None, y=None, M_T=None, S_T=None,
                stream: Optional[torch.cuda.Stream] = None):
        """Device tensors in, device tensors out: returns (y, M_T, S_T).

        M_T may be M0 and S_T may be S0 (in-place state carry)."""
        B, H, T = self._check(q, k, v, alpha, eta, beta, c, M0, S0, host=False)
        dev = q.device
        if y is None:
            y = torch.empty((B, H, T, self.d), dtype=self.out_dtype, device=dev)
        if M_T is None:
            M_T = torch.empty_like(M0)
        if S_T is None:
            S_T = torch.empty_like(S0)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = load_library().nm_forward(self._h, B, H, T, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta),
                                       _ptr(beta), _ptr(c), _ptr(M0), _ptr(S0), _ptr(y), _ptr(M_T), _ptr(S_T),
                                       ctypes.c_void_p(s.cuda_stream))
        if rc != NM_OK:
            raise NMError(rc, "nm_forward")
        return y, M_T, S_T

    def forward_surprise(self, q, k, v, alpha, eta, beta, M0, S0, c=None, y=None, M_T=None, S_T=None,
                         surprise=None, stream: Optional[torch.cuda.Stream] = None):
        """forward() that also returns each token's surprise, the norm of the
        loss gradient at the chunk-start weights: (y, M_T, S_T, surprise [B,H,T])."""
        B, H, T = self._check(q, k, v, alpha, eta, beta, c, M0, S0, host=False)
        dev = q.device
        if y is None:
            y = torch.empty((B, H, T, self.d), dtype=self.out_dtype, device=dev)
        if M_T is None:
            M_T = torch.empty_like(M0)
        if S_T is None:
            S_T = torch.empty_like(S0)
        if surprise is None:
            surprise = torch.empty((B, H, T), dtype=torch.float32, device=dev)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = load_library().nm_forward_surprise(self._h, B, H, T, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha),
                                                _ptr(eta), _ptr(beta), _ptr(c), _ptr(M0), _ptr(S0), _ptr(y),
                                                _ptr(M_T), _ptr(S_T), _ptr(surprise), ctypes.c_void_p(s.cuda_stream))
        if rc != NM_OK:
            raise NMError(rc, "nm_forward_surprise")
        return y, M_T, S_T, surprise

    def forward_gated(self, q, k, v, alpha, eta, beta, M0, S0, y_attn, c=None, o=None, M_T=None, S_T=None,
                      stream: Optional[torch.cuda.Stream] = None):
        """forward() whose output is combined with another branch's output by
        the Memory-as-Gate rule, o = sigmoid(y) * y_attn (y_attn of the output
        dtype and y's shape; o may be y_attn itself): returns (o, M_T, S_T)."""
        B, H, T = self._check(q, k, v, alpha, eta, beta, c, M0, S0, host=False)
        dev = q.device
        if y_attn.shape != (B, H, T, self.d) or y_attn.dtype != self.out_dtype or not y_attn.is_contiguous():
            raise ValueError("y_attn must be a contiguous %s [B, H, T, %d] tensor" % (self.out_dtype, self.d))
        if not y_attn.is_cuda or y_attn.device.index != self.device:
            raise ValueError("forward_gated takes tensors on cuda:%d" % self.device)
        if o is None:
            o = torch.empty((B, H, T, self.d), dtype=self.out_dtype, device=dev)
        if M_T is None:
            M_T = torch.empty_like(M0)
        if S_T is None:
            S_T = torch.empty_like(S0)
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = load_library().nm_forward_gated(self._h, B, H, T, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta),
                                             _ptr(beta), _ptr(c), _ptr(M0), _ptr(S0), _ptr(y_attn), _ptr(o),
                                             _ptr(M_T), _ptr(S_T), ctypes.c_void_p(s.cuda_stream))
        if rc != NM_OK:
            raise NMError(rc, "nm_forward_gated")
        return o, M_T, S_T

    def backward(self, q, k, v, alpha, eta, beta, M0, S0, Gy, GM, GS, c=None,
                 stream: Optional[torch.cuda.Stream] = None) -> dict:
        """Gradients of a loss with upstream gradients Gy = dL/dy [B,H,T,d],
        GM = dL/dM_T, GS = dL/dS_T [B,H,P] (fp32 device tensors) with respect
        to every input of forward() on the same inputs: a dict with q, k, v,
        alpha, eta, beta, M0, S0 (and c for C_PER_TOKEN), all fp32."""
        B, H, T = self._check(q, k, v, alpha, eta, beta, c, M0, S0, host=False)
        dev = q.device
        if Gy.shape != (B, H, T, self.d) or Gy.dtype != torch.float32 or not Gy.is_contiguous():
            raise ValueError("Gy must be a contiguous float32 [B, H, T, %d] tensor" % self.d)
        for t in (GM, GS):
            if t.shape != (B, H, self.P) or t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError("GM, GS must be contiguous float32 [B, H, %d] tensors" % self.P)
        for t in (Gy, GM, GS):
            if not t.is_cuda or t.device.index != self.device:
                raise ValueError("backward takes tensors on cuda:%d" % self.device)
        f = lambda shape: torch.empty(shape, dtype=torch.float32, device=dev)
        out = {"q": f((B, H, T, self.d)), "k": f((B, H, T, self.d)), "v": f((B, H, T, self.d)),
               "alpha": f((B, H, T)), "eta": f((B, H, T)), "beta": f((B, H, T)),
               "c": f((B, H, T)) if self.c_mode == C_PER_TOKEN else None,
               "M0": f((B, H, self.P)), "S0": f((B, H, self.P))}
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        rc = load_library().nm_backward(self._h, B, H, T, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta),
                                        _ptr(beta), _ptr(c), _ptr(M0), _ptr(S0), _ptr(Gy), _ptr(GM), _ptr(GS),
                                        _ptr(out["q"]), _ptr(out["k"]), _ptr(out["v"]), _ptr(out["alpha"]),
                                        _ptr(out["eta"]), _ptr(out["beta"]), _ptr(out["c"]), _ptr(out["M0"]),
                                        _ptr(out["S0"]), ctypes.c_void_p(s.cuda_stream))
        if rc != NM_OK:
            raise NMError(rc, "nm_backward")
        if out["c"] is None:
            del out["c"]
        return out

    def forward_host(self, q, k, v, alpha, eta, beta, M0, S0, c=None, y=None, M_T=None, S_T=None,
                     stream: Optional[torch.cuda.Stream] = None):
        """Host tensors in (pinned for asynchronous copies), host tensors out.

        Copies in, runs and copies out on the handle's device; returns when
        the results are on the host."""
        B, H, T = self._check(q, k, v, alpha, eta, beta, c, M0, S0, host=True)
        pin = q.is_pinned()
        if y is None:
            y = torch.empty((B, H, T, self.d), dtype=self.out_dtype, pin_memory=pin)
        if M_T is None:
            M_T = torch.empty(M0.shape, dtype=torch.float32, pin_memory=pin)
        if S_T is None:
            S_T = torch.empty(S0.shape, dtype=torch.float32, pin_memory=pin)
        s = stream if stream is not None else torch.cuda.current_stream(torch.device("cuda", self.device))
        rc = load_library().nm_forward_host(self._h, B, H, T, _ptr(q), _ptr(k), _ptr(v), _ptr(alpha), _ptr(eta),
                                            _ptr(beta), _ptr(c), _ptr(M0), _ptr(S0), _ptr(y), _ptr(M_T),
                                            _ptr(S_T), ctypes.c_void_p(s.cuda_stream))
        if rc != NM_OK:
            raise NMError(rc, "nm_forward_host")
        return y, M_T, S_T

    def inject_missing_load(self) -> int:
        """Test hook: the next forward runs without its first tile loads, so
        its bounded wait expires and nm_synchronize reports
        NM_ERR_DEVICE_TIMEOUT (see nm_inject_missing_load in include/nm.h)."""
        return int(load_library().nm_inject_missing_load(self._h))

    def synchronize(self) -> int:
        """Wait for the device; return (and clear) the device status word."""
        return int(load_library().nm_synchronize(self._h))
