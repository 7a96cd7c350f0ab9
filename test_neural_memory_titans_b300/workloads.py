"""Seeded synthetic inputs for the neural-memory forward pass.

This module holds random-number recipes only (no step of the method): it is
the one module that both the CUDA path's tests/bench and the oracle's tests
use.  The pages measure on datasets that are not available here (FineWeb-Edu,
RULER S-NIAH, BABILong); the recipes below stand in for them with the shapes,
value ranges and structure the workloads need:

  0  linear memory d=64, fp32 inputs, B=H=1, T=256, chunk 16
  1  2-layer SiLU MLP memory 64->256->64, bf16, B=4, H=8, T=4096, chunk 64
  2  linear memory d=128, bf16, B=8, H=16, T=16384, chunk 64; v = k R + noise
  3  MLP 128->512->128, bf16, B=2, H=16, T=131072, chunk 64; Zipf codebook keys
  4  linear memory d=64, bf16, B=1, H=8, T=2,097,152, chunk 256, streamed in
     64K-token segments; 1% needle tokens whose key reappears as a later query

Inputs are drawn in fp32, L2-normalised in fp32 where the recipe says so, and
then rounded to the input dtype (round-to-nearest-even).  Both sides consume
the rounded values.  Gates and states are fp32.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

LINEAR = 0
MLP2 = 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: int
    d: int
    hidden: int
    chunk: int
    dtype: torch.dtype
    B: int
    H: int
    T: int
    alpha: tuple
    eta: tuple
    beta: tuple
    keys: str          # "gauss" | "orth_map" | "codebook" | "needles"
    segment: int = 0   # >0: processed as T/segment calls carrying (M, S)
    w_init_std: float = 0.0
    layers: int = 2    # MLP depth (W1, L - 2 hidden-to-hidden layers, W_L); 2 for the configured workloads

    @property
    def P(self) -> int:
        if self.kind == LINEAR:
            return self.d * self.d
        return 2 * self.hidden * self.d + (self.layers - 2) * self.hidden * self.hidden

    @property
    def tokens(self) -> int:
        return self.B * self.H * self.T

    def with_sizes(self, B=None, H=None, T=None, segment=None) -> "Workload":
        return dataclasses.replace(self, B=self.B if B is None else B, H=self.H if H is None else H,
                                   T=self.T if T is None else T,
                                   segment=self.segment if segment is None else segment)


_G0 = ((0.0, 0.05), (0.01, 0.1), (0.8, 0.95))

WORKLOADS = {
    0: Workload("linear_d64_fp32_b1h1_t256_c16", LINEAR, 64, 0, 16, torch.float32, 1, 1, 256, *_G0, keys="gauss"),
    1: Workload("mlp_64x256_bf16_b4h8_t4096_c64", MLP2, 64, 256, 64, torch.bfloat16, 4, 8, 4096, *_G0,
                keys="gauss", w_init_std=0.02),
    2: Workload("linear_d128_bf16_b8h16_t16384_c64", LINEAR, 128, 0, 64, torch.bfloat16, 8, 16, 16384, *_G0,
                keys="orth_map"),
    3: Workload("mlp_128x512_bf16_b2h16_t131072_c64", MLP2, 128, 512, 64, torch.bfloat16, 2, 16, 131072,
                (0.0, 0.02), (0.01, 0.05), (0.9, 0.99), keys="codebook", w_init_std=0.02),
    4: Workload("linear_d64_bf16_b1h8_t2097152_c256_seg65536", LINEAR, 64, 0, 256, torch.bfloat16, 1, 8, 2097152,
                *_G0, keys="needles", segment=65536),
}

CODEBOOK_SIZE = 4096
ZIPF_S = 1.1
NEEDLE_FRACTION = 0.01


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normalise(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True).clamp_min(1e-30)


def _uniform(shape, lo, hi, g, device):
    return lo + (hi - lo) * torch.rand(shape, generator=g, device=device, dtype=torch.float32)


def _orthogonal(n_mats: int, d: int, g, device) -> torch.Tensor:
    """Random orthogonal matrices (QR of a Gaussian, signs fixed by diag(R))."""
    a = torch.randn((n_mats, d, d), generator=g, device=device, dtype=torch.float32)
    qm, r = torch.linalg.qr(a)
    return qm * torch.sign(torch.diagonal(r, dim1=-2, dim2=-1)).unsqueeze(-2)


def make_inputs(wl: Workload, device="cpu", seed: Optional[int] = None) -> dict:
    """Build one workload's inputs on ``device``.

    Returns a dict with q, k, v [B,H,T,d] (wl.dtype), alpha, eta, beta [B,H,T]
    (fp32), c (None: the workloads use c = 1), M0, S0 [B,H,P] (fp32) and, for
    the needle recipe, ``needles`` = (positions, probe positions) per head.
    Each tensor has its own generator stream derived from ``seed`` in a fixed
    order, so a smaller variant of a workload draws the same kind of values.
    """
    seed = 1000 if seed is None else seed
    B, H, T, d = wl.B, wl.H, wl.T, wl.d
    dev = torch.device(device)
    out = {}
    shape = (B, H, T, d)
    if wl.keys == "gauss" or wl.keys == "needles":
        q = _normalise(torch.randn(shape, generator=_gen(dev, seed + 1), device=dev))
        k = _normalise(torch.randn(shape, generator=_gen(dev, seed + 2), device=dev))
        v = torch.randn(shape, generator=_gen(dev, seed + 3), device=dev)
        if wl.keys == "needles":
            v = _normalise(v)
            pos, probe = _place_needles(B * H, T, _gen(dev, seed + 7), dev)
            qf = q.reshape(B * H, T, d)
            kf = k.reshape(B * H, T, d)
            rows = torch.arange(B * H, device=dev).unsqueeze(1).expand_as(pos)
            qf[rows, probe] = kf[rows, pos]
            out["needles"] = (pos.reshape(B, H, -1), probe.reshape(B, H, -1))
    elif wl.keys == "orth_map":
        k = _normalise(torch.randn(shape, generator=_gen(dev, seed + 2), device=dev))
        q = _normalise(torch.randn(shape, generator=_gen(dev, seed + 1), device=dev))
        R = _orthogonal(B * H, d, _gen(dev, seed + 4), dev).reshape(B, H, d, d)
        v = k @ R + 0.1 * torch.randn(shape, generator=_gen(dev, seed + 3), device=dev)
    elif wl.keys == "codebook":
        cb = torch.randn((CODEBOOK_SIZE, d), generator=_gen(dev, seed + 5), device=dev)
        emb = _normalise(torch.randn((CODEBOOK_SIZE, d), generator=_gen(dev, seed + 6), device=dev))
        Pm = _orthogonal(1, d, _gen(dev, seed + 4), dev)[0]
        ranks = torch.arange(1, CODEBOOK_SIZE + 1, device=dev, dtype=torch.float64)
        probs = (ranks ** (-ZIPF_S)).to(torch.float32)
        kid = torch.multinomial(probs, B * H * T, replacement=True, generator=_gen(dev, seed + 2)).reshape(B, H, T)
        qid = torch.multinomial(probs, B * H * T, replacement=True, generator=_gen(dev, seed + 1)).reshape(B, H, T)
        k = _normalise(cb[kid] + 0.05 * torch.randn(shape, generator=_gen(dev, seed + 8), device=dev))
        q = _normalise(cb[qid] + 0.05 * torch.randn(shape, generator=_gen(dev, seed + 9), device=dev))
        v = emb[kid] @ Pm.T
        out["ids"] = kid
    else:
        raise ValueError(wl.keys)
    out["q"] = q.to(wl.dtype).contiguous()
    out["k"] = k.to(wl.dtype).contiguous()
    out["v"] = v.to(wl.dtype).contiguous()
    g = _gen(dev, seed + 10)
    out["alpha"] = _uniform((B, H, T), *wl.alpha, g, dev)
    out["eta"] = _uniform((B, H, T), *wl.eta, g, dev)
    out["beta"] = _uniform((B, H, T), *wl.beta, g, dev)
    out["c"] = None
    if wl.kind == MLP2:
        M0 = wl.w_init_std * torch.randn((B, H, wl.P), generator=_gen(dev, seed + 11), device=dev)
    else:
        M0 = torch.zeros((B, H, wl.P), device=dev)
    out["M0"] = M0.contiguous()
    out["S0"] = torch.zeros((B, H, wl.P), device=dev)
    return out


def _place_needles(units: int, T: int, g, dev):
    """1% of positions p (uniform, p < T-1); each gets a later probe p' in
    [p+1, T-1] whose query is set to k_p, so the target there is v_p."""
    n = max(1, int(T * NEEDLE_FRACTION)) if T >= 2 else 0
    pos = torch.randint(0, max(T - 1, 1), (units, n), generator=g, device=dev)
    u = torch.rand((units, n), generator=g, device=dev, dtype=torch.float64)
    span = (T - 1 - pos).to(torch.float64)
    probe = pos + 1 + torch.clamp((u * span).floor().to(torch.long), max=(T - 2 - pos).clamp_min(0))
    return pos, probe


def random_state(wl: Workload, device="cpu", seed: int = 77, scale: float = 1.0) -> tuple:
    """Chunk-start states at a nondegenerate scale: W ~ N(0, scale/fan_in),
    S ~ 0.1 N(0, scale/fan_in), for teacher-forced per-chunk checks."""
    B, H, d, h = wl.B, wl.H, wl.d, wl.hidden
    g = _gen(torch.device(device), seed)
    if wl.kind == LINEAR:
        std = (scale / d) ** 0.5
        M = std * torch.randn((B, H, d * d), generator=g, device=device)
        S = 0.1 * std * torch.randn((B, H, d * d), generator=g, device=device)
    else:
        s1 = (scale / d) ** 0.5
        s2 = (scale / h) ** 0.5
        W1 = s1 * torch.randn((B, H, h * d), generator=g, device=device)
        W2 = s2 * torch.randn((B, H, d * h), generator=g, device=device)
        M = torch.cat([W1, W2], dim=-1)
        S1 = 0.1 * s1 * torch.randn((B, H, h * d), generator=g, device=device)
        S2 = 0.1 * s2 * torch.randn((B, H, d * h), generator=g, device=device)
        S = torch.cat([S1, S2], dim=-1)
    return M.contiguous(), S.contiguous()
