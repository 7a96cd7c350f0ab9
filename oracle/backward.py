"""Reference gradients of the chunked forward, for outer-loop training: fp64
PyTorch on the CPU.

TEST INFRASTRUCTURE ONLY, like the rest of this package: tests/ may import it;
the product library never does, and it imports nothing from the product.

The pages train the memory's surroundings (projections, gates) through the
memory ("Titans: Imparare a Memorizzare al Tempo di Test", "Addestramento
Parallelizzato": the inner loop is written with matmuls so that the outer
loop trains fast).  That needs the gradient of a loss of the forward's
outputs with respect to its inputs.  This module restates the forward with
torch operations in the pages' order -- per chunk the snapshot W0, per token
the explicit gradient g_t at W0 (2 (M_W0(k) - v) ... by hand-written
backprop, so that it can itself be differentiated), S = beta S + c g,
M = (1 - alpha) M - eta S, y_t = M(q_t) -- and lets torch.autograd
differentiate the functional
    L = <Gy, y> + <GM, M_T> + <GS, S_T>
for given upstream gradients Gy, GM, GS.  No blocking and no chunked-parallel
reformulation: the same sequence of steps as nm_oracle.c, whose forward it
must reproduce (pinned in tests/test_oracle_backward.py, together with
central differences of that C forward).
"""
from __future__ import annotations

import numpy as np
import torch

from . import C_ONE, C_ONE_MINUS_BETA, C_PER_TOKEN, LINEAR, LOSS_HUBER, LOSS_L2, MLP2


def _dloss(r, loss_kind, delta):
    """d rho / d r: 2 r, or 2 clip(r, -delta, delta) for the Huber loss."""
    if loss_kind == LOSS_HUBER:
        return 2.0 * torch.clamp(r, -delta, delta)
    return 2.0 * r


def _sizes(kind, d, hidden, layers):
    """(out, in) of every weight matrix, in packing order."""
    if kind == LINEAR:
        return [(d, d)]
    return [(hidden, d)] + [(hidden, hidden)] * (layers - 2) + [(d, hidden)]


def _split(W, sizes):
    out, off = [], 0
    for r, c in sizes:
        out.append(W[off: off + r * c].reshape(r, c))
        off += r * c
    return out


def _apply(Ws, x):
    """M_W(x): silu after every layer but the last."""
    h = x
    for li, Wl in enumerate(Ws):
        h = Wl @ h
        if li < len(Ws) - 1:
            h = torch.nn.functional.silu(h)
    return h


def _grad(Ws, k, v, loss_kind, delta):
    """g = grad_W l(W; k, v) by explicit backprop (differentiable in W, k, v)."""
    xs, zs = [k], []
    h = k
    for Wl in Ws[:-1]:
        z = Wl @ h
        zs.append(z)
        h = torch.nn.functional.silu(z)
        xs.append(h)
    e = _dloss(Ws[-1] @ h - v, loss_kind, delta)
    grads = [None] * len(Ws)
    delta_l = e
    for li in range(len(Ws) - 1, -1, -1):
        grads[li] = torch.outer(delta_l, xs[li])
        if li > 0:
            s = torch.sigmoid(zs[li - 1])
            delta_l = (Ws[li].T @ delta_l) * (s * (1.0 + zs[li - 1] * (1.0 - s)))
    return torch.cat([g.reshape(-1) for g in grads])


def forward_torch(kind, d, hidden, chunk, c_mode, q, k, v, alpha, eta, beta, c, M0, S0,
                  loss_kind=LOSS_L2, huber_delta=np.inf, layers=2):
    """The chunked forward of one (batch, head) unit on torch fp64 tensors:
    q, k, v [T, d], gates [T], M0, S0 [P].  Returns (y [T, d], M_T, S_T)."""
    sizes = _sizes(kind, d, hidden, layers)
    T = q.shape[0]
    M, S = M0, S0
    ys = []
    for t0 in range(0, T, chunk):
        W0s = _split(M, sizes)  # the chunk-start weights
        for t in range(t0, min(t0 + chunk, T)):
            g = _grad(W0s, k[t], v[t], loss_kind, huber_delta)
            if c_mode == C_ONE_MINUS_BETA:
                ct = 1.0 - beta[t]
            elif c_mode == C_PER_TOKEN:
                ct = c[t]
            else:
                ct = 1.0
            S = beta[t] * S + ct * g
            M = (1.0 - alpha[t]) * M - eta[t] * S
            ys.append(_apply(_split(M, sizes), q[t]))
    y = torch.stack(ys) if ys else q.new_zeros((0, d))
    return y, M, S


def backward(kind, d, hidden, chunk, c_mode, q, k, v, alpha, eta, beta, c, M0, S0, Gy, GM, GS,
             loss_kind=LOSS_L2, huber_delta=np.inf, layers=2):
    """Gradients of <Gy, y> + <GM, M_T> + <GS, S_T> with respect to every
    input of one unit (numpy arrays in, a dict of numpy arrays out: q, k, v,
    alpha, eta, beta, M0, S0, and c for C_PER_TOKEN)."""
    names = ["q", "k", "v", "alpha", "eta", "beta", "M0", "S0"] + (["c"] if c_mode == C_PER_TOKEN else [])
    vals = dict(q=q, k=k, v=v, alpha=alpha, eta=eta, beta=beta, M0=M0, S0=S0, c=c)
    ts = {n: torch.tensor(np.asarray(vals[n], dtype=np.float64), requires_grad=True) for n in names}
    y, MT, ST = forward_torch(kind, d, hidden, chunk, c_mode, ts["q"], ts["k"], ts["v"], ts["alpha"], ts["eta"],
                              ts["beta"], ts.get("c"), ts["M0"], ts["S0"], loss_kind, huber_delta, layers)
    L = ((y * torch.tensor(Gy, dtype=torch.float64)).sum() + (MT * torch.tensor(GM, dtype=torch.float64)).sum()
         + (ST * torch.tensor(GS, dtype=torch.float64)).sum())
    grads = torch.autograd.grad(L, [ts[n] for n in names], allow_unused=True)
    return {n: (np.zeros_like(np.asarray(vals[n], dtype=np.float64)) if g is None else g.numpy())
            for n, g in zip(names, grads)}
