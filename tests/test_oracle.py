"""Pins for the fp64 oracle: each test checks it against something other than
itself (hand-worked values, finite differences, a library gradient, the delta
rule, linear attention, a closed-form geometric scan, the two momentum forms
exactly as the pages write them, and invariants).

Sources, by page title and section:
  "Titans: Imparare a Memorizzare al Tempo di Test" (lowest.today) - update,
      momentum (form A), forgetting, loss, parallel (chunked) training;
  0h-n0.github.io Titans explainer - retrieval, momentum (form B), weight
      decay, relation to DeltaNet / Gated DeltaNet and linear attention
      ("関連研究", "ニューラル長期メモリモジュール").
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = [Fraction(x) for x in vals]
    return out


def _fl(vals):
    return np.array([float(x) for x in vals])


def _run(kind, d, hidden, chunk, c_mode, q, k, v, a, e, b, c=None, M0=None, S0=None):
    """Oracle on a single (batch, head) given [T, d] arrays."""
    T = q.shape[0]
    P = oracle.param_count(kind, d, hidden)
    M0 = np.zeros(P) if M0 is None else M0
    S0 = np.zeros(P) if S0 is None else S0
    y, MT, ST = oracle.forward(kind, d, hidden, chunk, c_mode,
                               q.reshape(1, 1, T, d), k.reshape(1, 1, T, d), v.reshape(1, 1, T, d),
                               np.asarray(a, float).reshape(1, 1, T), np.asarray(e, float).reshape(1, 1, T),
                               np.asarray(b, float).reshape(1, 1, T),
                               None if c is None else np.asarray(c, float).reshape(1, 1, T),
                               M0.reshape(1, 1, P), S0.reshape(1, 1, P))
    return y[0, 0], MT[0, 0], ST[0, 0]


# ---------------------------------------------------------------- worked examples

@pytest.mark.parametrize("chunk", [2, 1])
def test_scalar_worked_example(chunk):
    g = _read_golden("linear_scalar_worked.txt")
    k, v, q = (_fl(g[n]).reshape(3, 1) for n in ("k", "v", "q"))
    y, MT, ST = _run(oracle.LINEAR, 1, 0, chunk, oracle.C_ONE, q, k, v,
                     _fl(g["alpha"]), _fl(g["eta"]), _fl(g["beta"]))
    key = "chunk%d" % chunk
    # dyadic rationals: exact in binary floating point
    assert np.array_equal(y[:, 0], _fl(g[key + ".y"]))
    assert np.array_equal(MT, _fl(g[key + ".M_T"]))
    assert np.array_equal(ST, _fl(g[key + ".S_T"]))


def test_2x2_worked_example():
    g = _read_golden("linear_2x2_worked.txt")
    k, v, q = (_fl(g[n]).reshape(3, 2) for n in ("k", "v", "q"))
    y, MT, ST = _run(oracle.LINEAR, 2, 0, int(g["chunk"][0]), oracle.C_ONE, q, k, v,
                     _fl(g["alpha"]), _fl(g["eta"]), _fl(g["beta"]))
    assert np.array_equal(y.reshape(-1), _fl(g["y"]))
    assert np.array_equal(MT, _fl(g["M_T"]))
    assert np.array_equal(ST, _fl(g["S_T"]))


# ---------------------------------------------------------------- gradients

def _torch_memory(kind, d, hidden, W, x):
    """The memory map written with library ops (matmul, F.silu)."""
    if kind == oracle.LINEAR:
        return W.reshape(d, d) @ x
    W1 = W[: hidden * d].reshape(hidden, d)
    W2 = W[hidden * d:].reshape(d, hidden)
    return W2 @ torch.nn.functional.silu(W1 @ x)


def _autograd_grad(kind, d, hidden, W, k, v):
    Wt = torch.tensor(W, dtype=torch.float64, requires_grad=True)
    kt = torch.tensor(k, dtype=torch.float64)
    vt = torch.tensor(v, dtype=torch.float64)
    loss = ((_torch_memory(kind, d, hidden, Wt, kt) - vt) ** 2).sum()
    (g,) = torch.autograd.grad(loss, Wt)
    return g.numpy()


@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 2, 0), (oracle.LINEAR, 4, 0),
                                           (oracle.MLP2, 2, 3), (oracle.MLP2, 3, 8),
                                           (oracle.MLP2, 4, 5)])
def test_grad_finite_differences(kind, d, hidden):
    rng = np.random.default_rng(7 + d + hidden)
    P = oracle.param_count(kind, d, hidden)
    for _ in range(3):
        W = rng.normal(0, 0.7, P)
        k = rng.normal(0, 1, d)
        v = rng.normal(0, 1, d)
        g = oracle.grad(kind, d, hidden, W, k, v)
        h = 1e-6
        fd = np.zeros(P)
        for p in range(P):
            Wp = W.copy(); Wp[p] += h
            Wm = W.copy(); Wm[p] -= h
            fd[p] = (oracle.loss(kind, d, hidden, Wp, k, v) - oracle.loss(kind, d, hidden, Wm, k, v)) / (2 * h)
        assert np.linalg.norm(g - fd) <= 1e-7 * np.linalg.norm(fd)


@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 5, 0), (oracle.MLP2, 4, 7), (oracle.MLP2, 6, 16)])
def test_grad_and_apply_match_library(kind, d, hidden):
    rng = np.random.default_rng(11)
    P = oracle.param_count(kind, d, hidden)
    W = rng.normal(0, 0.5, P)
    k = rng.normal(0, 1, d)
    v = rng.normal(0, 1, d)
    np.testing.assert_allclose(oracle.grad(kind, d, hidden, W, k, v),
                               _autograd_grad(kind, d, hidden, W, k, v), rtol=1e-12, atol=1e-13)
    ref = _torch_memory(kind, d, hidden, torch.tensor(W), torch.tensor(k)).numpy()
    np.testing.assert_allclose(oracle.memory_apply(kind, d, hidden, W, k), ref, rtol=1e-13, atol=1e-14)
    ref_loss = float(((ref - v) ** 2).sum())
    assert abs(oracle.loss(kind, d, hidden, W, k, v) - ref_loss) <= 1e-12 * max(1.0, ref_loss)


@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 3, 0), (oracle.MLP2, 3, 5)])
def test_single_chunk_sums_gradients_at_chunk_start(kind, d, hidden):
    """One chunk with beta = 1, c = 1: S_T is the sum of every token's gradient
    at the chunk-start weights, i.e. the gradient of the summed loss there
    ("Addestramento Parallelizzato": mini-batch gradient descent in a chunk)."""
    rng = np.random.default_rng(3)
    T = 6
    P = oracle.param_count(kind, d, hidden)
    W0 = rng.normal(0, 0.5, P)
    S0 = rng.normal(0, 0.1, P)
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.3, T); eta = rng.uniform(0.01, 0.2, T)
    _, _, ST = _run(kind, d, hidden, T, oracle.C_ONE, q, k, v, alpha, eta, np.ones(T), M0=W0, S0=S0)
    Wt = torch.tensor(W0, requires_grad=True)
    total = sum(((_torch_memory(kind, d, hidden, Wt, torch.tensor(k[i])) - torch.tensor(v[i])) ** 2).sum()
                for i in range(T))
    (gsum,) = torch.autograd.grad(total, Wt)
    np.testing.assert_allclose(ST, S0 + gsum.numpy(), rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- the pages' own forms

@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 3, 0), (oracle.MLP2, 3, 4)])
def test_chunk1_equals_form_A_sequential(kind, d, hidden):
    """Form A ("Meccanismo di Aggiornamento della Memoria" + "Meccanismo di
    Dimenticanza"): S_t = eta_t S_{t-1} - theta_t grad l(M_{t-1}; x_t),
    M_t = (1 - alpha_t) M_{t-1} + S_t, written token by token with an autograd
    gradient.  It equals the oracle at chunk 1 with c = theta (per token), the
    oracle's beta = the page's eta, the oracle's eta = 1 and S_oracle = -S_A."""
    rng = np.random.default_rng(5)
    T = 9
    P = oracle.param_count(kind, d, hidden)
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.2, T)
    eta_A = rng.uniform(0.5, 0.9, T)     # surprise decay
    theta = rng.uniform(0.01, 0.1, T)    # scale of instantaneous surprise
    M = rng.normal(0, 0.3, P)
    S = np.zeros(P)
    M0 = M.copy()
    ys = []
    for t in range(T):
        g = _autograd_grad(kind, d, hidden, M, k[t], v[t])
        S = eta_A[t] * S - theta[t] * g
        M = (1 - alpha[t]) * M + S
        ys.append(_torch_memory(kind, d, hidden, torch.tensor(M), torch.tensor(q[t])).numpy())
    y, MT, ST = _run(kind, d, hidden, 1, oracle.C_PER_TOKEN, q, k, v, alpha, np.ones(T), eta_A,
                     c=theta, M0=M0)
    np.testing.assert_allclose(y, np.array(ys), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(MT, M, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ST, -S, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 4, 0), (oracle.MLP2, 2, 6)])
def test_chunk1_equals_form_B_sequential(kind, d, hidden):
    """Form B ("モメンタム機構", "適応的重み減衰"): s_t = beta s_{t-1} +
    (1 - beta) grad L(x_t; theta_t), theta_{t+1} = (1 - alpha_t) theta_t -
    eta_t s_t, constant beta, gradient at the current weights; retrieval here
    reads the weights after the update.  It equals the oracle at chunk 1 with
    c = 1 - beta."""
    rng = np.random.default_rng(6)
    T = 8
    P = oracle.param_count(kind, d, hidden)
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.2, T); eta = rng.uniform(0.05, 0.3, T); beta = 0.7
    theta = rng.normal(0, 0.3, P); s = rng.normal(0, 0.05, P)
    M0, S0 = theta.copy(), s.copy()
    ys = []
    for t in range(T):
        g = _autograd_grad(kind, d, hidden, theta, k[t], v[t])
        s = beta * s + (1 - beta) * g
        theta = (1 - alpha[t]) * theta - eta[t] * s
        ys.append(_torch_memory(kind, d, hidden, torch.tensor(theta), torch.tensor(q[t])).numpy())
    y, MT, ST = _run(kind, d, hidden, 1, oracle.C_ONE_MINUS_BETA, q, k, v, alpha, eta,
                     np.full(T, beta), M0=M0, S0=S0)
    np.testing.assert_allclose(y, np.array(ys), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(MT, theta, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(ST, s, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- special cases

def test_delta_rule():
    """alpha = 0, beta = 0, c = 1, chunk 1, linear memory: the delta rule
    M_t = M_{t-1} - 2 eta_t (M_{t-1} k_t - v_t) k_t^T (explainer, "関連研究":
    Titans generalises the DeltaNet update)."""
    rng = np.random.default_rng(8)
    T, d = 12, 5
    k = rng.normal(0, 1, (T, d)); k /= np.linalg.norm(k, axis=1, keepdims=True)
    v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    eta = rng.uniform(0.05, 0.4, T)
    M = rng.normal(0, 0.3, (d, d)); M0 = M.copy()
    ys = []
    for t in range(T):
        M = M - 2 * eta[t] * np.outer(M @ k[t] - v[t], k[t])
        ys.append(M @ q[t])
    y, MT, _ = _run(oracle.LINEAR, d, 0, 1, oracle.C_ONE, q, k, v, np.zeros(T), eta, np.zeros(T),
                    M0=M0.reshape(-1))
    np.testing.assert_allclose(y, np.array(ys), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(MT.reshape(d, d), M, rtol=1e-12, atol=1e-13)


def test_decayed_delta_rule():
    """beta = 0, c = 1, chunk 1: M_t = M_{t-1} ((1 - alpha_t) I - 2 eta_t k k^T)
    + 2 eta_t v k^T (decay applies to M only, not to the erase/write term)."""
    rng = np.random.default_rng(9)
    T, d = 10, 4
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.5, T); eta = rng.uniform(0.01, 0.2, T)
    M = rng.normal(0, 0.3, (d, d)); M0 = M.copy()
    ys = []
    for t in range(T):
        M = M @ ((1 - alpha[t]) * np.eye(d) - 2 * eta[t] * np.outer(k[t], k[t])) + 2 * eta[t] * np.outer(v[t], k[t])
        ys.append(M @ q[t])
    y, MT, _ = _run(oracle.LINEAR, d, 0, 1, oracle.C_ONE, q, k, v, alpha, eta, np.zeros(T),
                    M0=M0.reshape(-1))
    np.testing.assert_allclose(y, np.array(ys), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(MT.reshape(d, d), M, rtol=1e-12, atol=1e-13)


def test_linear_attention():
    """One chunk, M0 = S0 = 0, alpha = beta = 0: the memory is an outer-product
    sum and retrieval is causal linear attention,
    y_t = sum_{i<=t} 2 eta_i c_i (k_i . q_t) v_i (explainer: linear attention
    stores an outer-product sum)."""
    rng = np.random.default_rng(10)
    T, d = 16, 6
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    eta = rng.uniform(0.01, 0.1, T); c = rng.uniform(0.5, 1.5, T)
    y, MT, ST = _run(oracle.LINEAR, d, 0, T, oracle.C_PER_TOKEN, q, k, v, np.zeros(T), eta, np.zeros(T), c=c)
    mask = np.tril(np.ones((T, T)))
    expect = (mask * (q @ k.T)) @ (2 * (eta * c)[:, None] * v)
    np.testing.assert_allclose(y, expect, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(MT.reshape(d, d), (2 * (eta * c)[:, None] * v).T @ k, rtol=1e-12, atol=1e-13)
    # beta = 0: only the last token's gradient survives in S
    np.testing.assert_allclose(ST.reshape(d, d), c[-1] * (-2) * np.outer(v[-1], k[-1]), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("alpha,eta,beta,c", [(0.1, 0.05, 0.8, 1.0), (0.3, 0.2, 0.5, 0.7), (0.02, 0.1, 0.95, 1.0)])
def test_closed_form_geometric_scan(alpha, eta, beta, c):
    """Constant gates, M0 = S0 = 0, one chunk: every gradient is -2 v_i k_i^T and
    the weight of token i in M_t is the geometric sum
    G(t, i) = c eta sum_{j=i}^{t} (1-alpha)^{t-j} beta^{j-i}
            = c eta ((1-alpha)^{n+1} - beta^{n+1}) / ((1-alpha) - beta),  n = t - i,
    so y_t = sum_i 2 G(t, i) (k_i . q_t) v_i."""
    rng = np.random.default_rng(12)
    T, d = 20, 3
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    cm = oracle.C_PER_TOKEN
    y, MT, ST = _run(oracle.LINEAR, d, 0, T, cm, q, k, v, np.full(T, alpha), np.full(T, eta),
                     np.full(T, beta), c=np.full(T, c))
    a = 1 - alpha
    n = np.arange(T)[:, None] - np.arange(T)[None, :]
    G = np.where(n >= 0, c * eta * (a ** (n + 1) - beta ** (np.maximum(n, 0) + 1)) / (a - beta), 0.0)
    expect = (G * (q @ k.T)) @ (2 * v)
    np.testing.assert_allclose(y, expect, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(MT.reshape(d, d), (2 * G[-1][:, None] * v).T @ k, rtol=1e-11, atol=1e-12)
    U = c * beta ** (T - 1 - np.arange(T))  # momentum weight of token i at the end
    np.testing.assert_allclose(ST.reshape(d, d), -(2 * U[:, None] * v).T @ k, rtol=1e-11, atol=1e-12)


# ---------------------------------------------------------------- invariants

@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 4, 0), (oracle.MLP2, 3, 6)])
def test_eta_zero_is_pure_decay(kind, d, hidden):
    rng = np.random.default_rng(13)
    T = 10
    P = oracle.param_count(kind, d, hidden)
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.3, T); beta = rng.uniform(0.5, 0.9, T)
    W0 = rng.normal(0, 0.5, P)
    y, MT, _ = _run(kind, d, hidden, 4, oracle.C_ONE, q, k, v, alpha, np.zeros(T), beta, M0=W0)
    A = np.cumprod(1 - alpha)
    np.testing.assert_allclose(MT, A[-1] * W0, rtol=1e-13, atol=1e-14)
    for t in range(T):
        ref = _torch_memory(kind, d, hidden, torch.tensor(A[t] * W0), torch.tensor(q[t])).numpy()
        np.testing.assert_allclose(y[t], ref, rtol=1e-12, atol=1e-13)


def test_alpha_one_wipes_memory():
    rng = np.random.default_rng(14)
    T, d = 7, 3
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.2, T); alpha[-1] = 1.0
    eta = rng.uniform(0.05, 0.2, T); beta = rng.uniform(0.5, 0.9, T)
    _, MT, ST = _run(oracle.LINEAR, d, 0, 3, oracle.C_ONE, q, k, v, alpha, eta, beta,
                     M0=rng.normal(0, 1, d * d))
    np.testing.assert_allclose(MT, -eta[-1] * ST, rtol=1e-14, atol=1e-15)


def test_linear_memory_is_homogeneous():
    """Linear memory: scaling (V, M0, S0) by lambda scales y, M_T, S_T by lambda."""
    rng = np.random.default_rng(15)
    T, d, lam = 11, 4, 3.0
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.1, T); eta = rng.uniform(0.01, 0.1, T); beta = rng.uniform(0.8, 0.95, T)
    M0 = rng.normal(0, 0.3, d * d); S0 = rng.normal(0, 0.1, d * d)
    y1, M1, S1 = _run(oracle.LINEAR, d, 0, 4, oracle.C_ONE, q, k, v, alpha, eta, beta, M0=M0, S0=S0)
    y2, M2, S2 = _run(oracle.LINEAR, d, 0, 4, oracle.C_ONE, q, k, lam * v, alpha, eta, beta,
                      M0=lam * M0, S0=lam * S0)
    np.testing.assert_allclose(y2, lam * y1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(M2, lam * M1, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S2, lam * S1, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 4, 0), (oracle.MLP2, 3, 5)])
def test_segment_carry_equals_one_call(kind, d, hidden):
    """Carrying (M, S) from one call into the next equals one long call when the
    first segment is a whole number of chunks (segment carry between windows,
    engineer-news notes, "Titans 的核心想法：測試時記憶")."""
    rng = np.random.default_rng(16)
    T, chunk, split = 24, 4, 12
    P = oracle.param_count(kind, d, hidden)
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.1, T); eta = rng.uniform(0.01, 0.1, T); beta = rng.uniform(0.8, 0.95, T)
    M0 = rng.normal(0, 0.2, P)
    y, MT, ST = _run(kind, d, hidden, chunk, oracle.C_ONE, q, k, v, alpha, eta, beta, M0=M0)
    s1 = slice(0, split); s2 = slice(split, T)
    ya, Ma, Sa = _run(kind, d, hidden, chunk, oracle.C_ONE, q[s1], k[s1], v[s1], alpha[s1], eta[s1], beta[s1], M0=M0)
    yb, Mb, Sb = _run(kind, d, hidden, chunk, oracle.C_ONE, q[s2], k[s2], v[s2], alpha[s2], eta[s2], beta[s2],
                      M0=Ma, S0=Sa)
    assert np.array_equal(np.concatenate([ya, yb]), y)
    assert np.array_equal(Mb, MT) and np.array_equal(Sb, ST)


def test_units_are_independent_and_parallel_safe():
    """B x H units are independent: a batched call equals per-unit calls."""
    rng = np.random.default_rng(17)
    B, H, T, d, h = 2, 3, 9, 3, 4
    P = oracle.param_count(oracle.MLP2, d, h)
    q, k, v = (rng.normal(0, 1, (B, H, T, d)) for _ in range(3))
    a = rng.uniform(0, .05, (B, H, T)); e = rng.uniform(.01, .1, (B, H, T)); b = rng.uniform(.8, .95, (B, H, T))
    M0 = rng.normal(0, .3, (B, H, P)); S0 = rng.normal(0, .03, (B, H, P))
    y, MT, ST = oracle.forward(oracle.MLP2, d, h, 4, oracle.C_ONE, q, k, v, a, e, b, None, M0, S0)
    for bi in range(B):
        for hi in range(H):
            y1, M1, S1 = _run(oracle.MLP2, d, h, 4, oracle.C_ONE, q[bi, hi], k[bi, hi], v[bi, hi],
                              a[bi, hi], e[bi, hi], b[bi, hi], M0=M0[bi, hi], S0=S0[bi, hi])
            assert np.array_equal(y[bi, hi], y1) and np.array_equal(MT[bi, hi], M1)
            assert np.array_equal(ST[bi, hi], S1)


def test_ragged_last_chunk_and_empty():
    rng = np.random.default_rng(18)
    d = 3
    # T = 0: state passes through unchanged
    y, MT, ST = _run(oracle.LINEAR, d, 0, 4, oracle.C_ONE, np.zeros((0, d)), np.zeros((0, d)), np.zeros((0, d)),
                     [], [], [], M0=np.arange(9.0), S0=np.ones(9))
    assert y.shape == (0, d) and np.array_equal(MT, np.arange(9.0)) and np.array_equal(ST, np.ones(9))
    # T = 7, chunk 4: a full chunk and a ragged one of 3 equal two calls of 4 and 3 tokens
    T = 7
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    a = rng.uniform(0, .1, T); e = rng.uniform(.01, .2, T); b = rng.uniform(.5, .9, T)
    y, MT, ST = _run(oracle.LINEAR, d, 0, 4, oracle.C_ONE, q, k, v, a, e, b)
    ya, Ma, Sa = _run(oracle.LINEAR, d, 0, 4, oracle.C_ONE, q[:4], k[:4], v[:4], a[:4], e[:4], b[:4])
    yb, Mb, Sb = _run(oracle.LINEAR, d, 0, 3, oracle.C_ONE, q[4:], k[4:], v[4:], a[4:], e[4:], b[4:], M0=Ma, S0=Sa)
    assert np.array_equal(y, np.concatenate([ya, yb])) and np.array_equal(MT, Mb) and np.array_equal(ST, Sb)


# ---------------------------------------------------------------- Huber loss (YAAD) and surprise norm
# The YAAD variant uses a Huber loss (0h-n0.github.io explainer, "MIRASフレームワーク",
# "3つの変種"; es.news.hada.io, "Modelos basados en MIRAS"); the pages give no formula
# or threshold.  Reading: element-wise on r = M(k) - v with a given delta,
# rho(r) = r^2 for |r| <= delta and 2 delta |r| - delta^2 beyond.  The surprise of a
# token is the norm of the loss gradient with respect to the memory's parameters
# (the same explainer, "Surprise機構"), here the Frobenius norm of the gradient the
# update uses, taken at the chunk-start weights.

def _huber_torch(r, delta):
    a = r.abs()
    return torch.where(a <= delta, r * r, 2 * delta * a - delta * delta).sum()


@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 3, 0), (oracle.MLP2, 3, 5), (oracle.MLP2, 4, 8)])
def test_huber_grad_finite_differences_and_library(kind, d, hidden):
    """The Huber gradient against central differences of the Huber loss and
    against torch autograd of the same loss written independently; delta is
    set so that some residuals are clipped and none lies near the kink."""
    rng = np.random.default_rng(31 + d + hidden)
    P = oracle.param_count(kind, d, hidden)
    checked_clip = False
    for trial in range(6):
        W = rng.normal(0, 0.7, P)
        k = rng.normal(0, 1, d)
        v = rng.normal(0, 1, d)
        r = oracle.memory_apply(kind, d, hidden, W, k) - v
        delta = float(np.median(np.abs(r)))
        if np.min(np.abs(np.abs(r) - delta)) < 1e-3:
            delta *= 1.01
        if np.min(np.abs(np.abs(r) - delta)) < 1e-3:
            continue
        checked_clip |= bool(np.any(np.abs(r) > delta))
        g = oracle.grad(kind, d, hidden, W, k, v, oracle.LOSS_HUBER, delta)
        h = 1e-6
        fd = np.zeros(P)
        for p in range(P):
            Wp = W.copy(); Wp[p] += h
            Wm = W.copy(); Wm[p] -= h
            fd[p] = (oracle.loss(kind, d, hidden, Wp, k, v, oracle.LOSS_HUBER, delta)
                     - oracle.loss(kind, d, hidden, Wm, k, v, oracle.LOSS_HUBER, delta)) / (2 * h)
        assert np.linalg.norm(g - fd) <= 1e-7 * np.linalg.norm(fd)
        Wt = torch.tensor(W, requires_grad=True)
        lt = _huber_torch(_torch_memory(kind, d, hidden, Wt, torch.tensor(k)) - torch.tensor(v), delta)
        (gt,) = torch.autograd.grad(lt, Wt)
        np.testing.assert_allclose(g, gt.numpy(), rtol=1e-12, atol=1e-13)
        lv = float(lt.detach())
        assert abs(oracle.loss(kind, d, hidden, W, k, v, oracle.LOSS_HUBER, delta) - lv) <= 1e-12 * abs(lv)
    assert checked_clip


def test_huber_single_token_closed_form():
    """Linear memory, M0 = S0 = 0, one token: r = -v, so
    y = -eta c 2 clip(-v, -delta, delta) (k . q), M_T = -eta c 2 clip(-v) k^T."""
    rng = np.random.default_rng(5)
    d, delta = 4, 0.3
    q, k = rng.normal(0, 1, (1, d)), rng.normal(0, 1, (1, d))
    v = np.array([[0.1, -0.2, 0.9, -1.4]])
    eta = 0.25
    out = oracle.forward(oracle.LINEAR, d, 0, 1, oracle.C_ONE, q.reshape(1, 1, 1, d), k.reshape(1, 1, 1, d),
                         v.reshape(1, 1, 1, d), np.full((1, 1, 1), 0.1), np.full((1, 1, 1), eta),
                         np.full((1, 1, 1), 0.5), None, np.zeros((1, 1, d * d)), np.zeros((1, 1, d * d)),
                         oracle.LOSS_HUBER, delta)
    e = 2.0 * np.clip(-v[0], -delta, delta)        # [ -0.2, 0.4, -0.6, 0.6 ]
    np.testing.assert_allclose(e, [-0.2, 0.4, -0.6, 0.6], rtol=0, atol=1e-15)
    np.testing.assert_allclose(out[0][0, 0, 0], -eta * e * float(k[0] @ q[0]), rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(out[1][0, 0].reshape(d, d), -eta * np.outer(e, k[0]), rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("kind,d,hidden", [(oracle.LINEAR, 4, 0), (oracle.MLP2, 3, 6)])
def test_huber_large_threshold_is_the_squared_loss(kind, d, hidden):
    rng = np.random.default_rng(17)
    T = 23
    q, k, v = (rng.normal(0, 1, (1, 1, T, d)) for _ in range(3))
    a, e, b = rng.uniform(0, .05, (1, 1, T)), rng.uniform(.01, .1, (1, 1, T)), rng.uniform(.8, .95, (1, 1, T))
    P = oracle.param_count(kind, d, hidden)
    M0 = rng.normal(0, 0.3, (1, 1, P))
    S0 = np.zeros((1, 1, P))
    ref = oracle.forward(kind, d, hidden, 5, oracle.C_ONE, q, k, v, a, e, b, None, M0, S0)
    hub = oracle.forward(kind, d, hidden, 5, oracle.C_ONE, q, k, v, a, e, b, None, M0, S0, oracle.LOSS_HUBER, 1e30)
    for x, y in zip(ref, hub):
        np.testing.assert_array_equal(x, y)


@pytest.mark.parametrize("kind,d,hidden,loss_kind", [(oracle.LINEAR, 4, 0, oracle.LOSS_L2),
                                                     (oracle.LINEAR, 4, 0, oracle.LOSS_HUBER),
                                                     (oracle.MLP2, 3, 6, oracle.LOSS_L2),
                                                     (oracle.MLP2, 3, 6, oracle.LOSS_HUBER)])
def test_surprise_is_the_gradient_norm_at_chunk_start(kind, d, hidden, loss_kind):
    """Surprise of the first chunk's tokens against the norm of torch
    autograd's gradient at M0 (the chunk-start weights); for the linear memory
    also against the closed form ||rho'(M0 k - v)|| ||k||."""
    rng = np.random.default_rng(23)
    T, chunk, delta = 9, 6, 0.4
    q, k, v = (rng.normal(0, 1, (1, 1, T, d)) for _ in range(3))
    a, e, b = rng.uniform(0, .05, (1, 1, T)), rng.uniform(.01, .1, (1, 1, T)), rng.uniform(.8, .95, (1, 1, T))
    P = oracle.param_count(kind, d, hidden)
    M0 = rng.normal(0, 0.5, (1, 1, P))
    out = oracle.forward(kind, d, hidden, chunk, oracle.C_ONE, q, k, v, a, e, b, None, M0, np.zeros((1, 1, P)),
                         loss_kind, delta if loss_kind == oracle.LOSS_HUBER else np.inf, surprise=True)
    sur = out[3][0, 0]
    assert sur.shape == (T,)
    for t in range(chunk):
        Wt = torch.tensor(M0[0, 0], requires_grad=True)
        r = _torch_memory(kind, d, hidden, Wt, torch.tensor(k[0, 0, t])) - torch.tensor(v[0, 0, t])
        lt = _huber_torch(r, delta) if loss_kind == oracle.LOSS_HUBER else (r * r).sum()
        (gt,) = torch.autograd.grad(lt, Wt)
        assert abs(sur[t] - float(gt.norm())) <= 1e-12 * float(gt.norm())
        if kind == oracle.LINEAR:
            rr = M0[0, 0].reshape(d, d) @ k[0, 0, t] - v[0, 0, t]
            ee = 2 * (np.clip(rr, -delta, delta) if loss_kind == oracle.LOSS_HUBER else rr)
            assert abs(sur[t] - np.linalg.norm(ee) * np.linalg.norm(k[0, 0, t])) <= 1e-12 * sur[t]
    # the later tokens take their gradients at the second chunk's start weights
    assert np.all(sur[chunk:] > 0)


# ---------------------------------------------------------------- deeper memories (L >= 3 layers)
# The memory is an MLP of L_M >= 1 layers (0h-n0.github.io explainer, "ニューラル長期メモリモジュール");
# here M(x) = W_L silu(W_{L-1} ... silu(W1 x)), W1 h x d, W2 .. W_{L-1} h x h, W_L d x h, no bias,
# packed in that order.

def _torch_deep(d, hidden, layers, W, x):
    """The L-layer memory written with library ops, independently of the oracle."""
    sizes = [(hidden, d)] + [(hidden, hidden)] * (layers - 2) + [(d, hidden)]
    off, h = 0, x
    for li, (r, c) in enumerate(sizes):
        Wl = W[off: off + r * c].reshape(r, c)
        off += r * c
        h = Wl @ h
        if li < layers - 1:
            h = torch.nn.functional.silu(h)
    assert off == W.shape[0]
    return h


@pytest.mark.parametrize("d,hidden,layers", [(2, 3, 3), (3, 4, 4), (2, 5, 5)])
def test_deep_grad_finite_differences_and_library(d, hidden, layers):
    rng = np.random.default_rng(50 + layers)
    P = oracle.param_count(oracle.MLP2, d, hidden, layers)
    assert P == 2 * hidden * d + (layers - 2) * hidden * hidden
    for _ in range(3):
        W = rng.normal(0, 0.8, P)
        k, v = rng.normal(0, 1, d), rng.normal(0, 1, d)
        g = oracle.grad(oracle.MLP2, d, hidden, W, k, v, layers=layers)
        h = 1e-6
        fd = np.zeros(P)
        for p in range(P):
            Wp = W.copy(); Wp[p] += h
            Wm = W.copy(); Wm[p] -= h
            fd[p] = (oracle.loss(oracle.MLP2, d, hidden, Wp, k, v, layers=layers)
                     - oracle.loss(oracle.MLP2, d, hidden, Wm, k, v, layers=layers)) / (2 * h)
        assert np.linalg.norm(g - fd) <= 1e-7 * np.linalg.norm(fd)
        Wt = torch.tensor(W, requires_grad=True)
        yt = _torch_deep(d, hidden, layers, Wt, torch.tensor(k))
        (gt,) = torch.autograd.grad(((yt - torch.tensor(v)) ** 2).sum(), Wt)
        np.testing.assert_allclose(g, gt.numpy(), rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(oracle.memory_apply(oracle.MLP2, d, hidden, W, k, layers=layers),
                                   yt.detach().numpy(), rtol=1e-13, atol=1e-14)


@pytest.mark.parametrize("layers", [3, 4])
def test_deep_chunk1_equals_sequential_and_chunk_sums_gradients(layers):
    """b = 1: the token-by-token rule (S = beta S + c g, M = (1 - alpha) M - eta S,
    y = M(q) after the update) with autograd gradients of the L-layer memory;
    one chunk with beta = 1: S_T is the gradient of the summed loss at the
    chunk-start weights."""
    rng = np.random.default_rng(60 + layers)
    d, hidden, T = 3, 4, 7
    P = oracle.param_count(oracle.MLP2, d, hidden, layers)
    k = rng.normal(0, 1, (T, d)); v = rng.normal(0, 1, (T, d)); q = rng.normal(0, 1, (T, d))
    alpha = rng.uniform(0, 0.2, T); eta = rng.uniform(0.05, 0.3, T); beta = rng.uniform(0.5, 0.9, T)
    M = rng.normal(0, 0.5, P); S = rng.normal(0, 0.05, P)
    M0, S0 = M.copy(), S.copy()

    def grad_at(Wnp, t):
        Wt = torch.tensor(Wnp, requires_grad=True)
        l_ = ((_torch_deep(d, hidden, layers, Wt, torch.tensor(k[t])) - torch.tensor(v[t])) ** 2).sum()
        return torch.autograd.grad(l_, Wt)[0].numpy()

    ys = []
    for t in range(T):
        S = beta[t] * S + grad_at(M, t)
        M = (1 - alpha[t]) * M - eta[t] * S
        ys.append(_torch_deep(d, hidden, layers, torch.tensor(M), torch.tensor(q[t])).numpy())
    out = oracle.forward(oracle.MLP2, d, hidden, 1, oracle.C_ONE, q[None, None], k[None, None], v[None, None],
                         alpha[None, None], eta[None, None], beta[None, None], None, M0[None, None], S0[None, None],
                         layers=layers)
    np.testing.assert_allclose(out[0][0, 0], np.array(ys), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out[1][0, 0], M, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out[2][0, 0], S, rtol=1e-11, atol=1e-12)
    # one chunk of all T tokens with beta = 1, alpha = eta = 0: S_T = S0 + sum_t g_t(M0)
    out = oracle.forward(oracle.MLP2, d, hidden, T, oracle.C_ONE, q[None, None], k[None, None], v[None, None],
                         np.zeros((1, 1, T)), np.zeros((1, 1, T)), np.ones((1, 1, T)), None, M0[None, None],
                         S0[None, None], layers=layers)
    gsum = sum(grad_at(M0, t) for t in range(T))
    np.testing.assert_allclose(out[2][0, 0], S0 + gsum, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(out[1][0, 0], M0, rtol=0, atol=0)


# ------------------------------------------------------------ Memory-as-Gate combination

def test_mag_gate_hand_worked():
    """Rational points of the sigmoid (y = ln r gives r / (r + 1)), worked by
    hand in tests/golden/mag_gate_worked.txt."""
    g = _read_golden("mag_gate_worked.txt")
    y = np.log(_fl(g["r"]))
    o = oracle.mag_gate(y, _fl(g["y_attn"]))
    assert np.allclose(o, _fl(g["o"]), rtol=1e-15, atol=0)


def test_mag_gate_symmetry_limits_and_library():
    """sigmoid(-y) = 1 - sigmoid(y), so o(y) + o(-y) = y_attn; o -> y_attn for
    y -> +inf and -> 0 for y -> -inf; and the library logistic function."""
    from scipy.special import expit
    rng = np.random.default_rng(0)
    y = rng.normal(size=(3, 5, 7)) * 4
    ya = rng.normal(size=y.shape)
    assert np.allclose(oracle.mag_gate(y, ya) + oracle.mag_gate(-y, ya), ya, rtol=1e-14, atol=1e-15)
    assert np.allclose(oracle.mag_gate(y, ya), expit(y) * ya, rtol=1e-14, atol=0)
    big = np.full(4, 800.0)
    assert np.array_equal(oracle.mag_gate(big, ya.ravel()[:4]), ya.ravel()[:4])
    assert np.array_equal(oracle.mag_gate(-big, np.ones(4)), np.zeros(4))
