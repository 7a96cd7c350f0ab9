"""Pins for oracle.backward, the fp64 reference gradients of the chunked
forward (for outer-loop training, "Titans: Imparare a Memorizzare al Tempo di
Test", "Addestramento Parallelizzato"): its torch restatement of the forward
reproduces the C oracle, and its gradients match central differences of the
C oracle's forward, input by input."""
import numpy as np
import pytest

import oracle
from oracle import backward as ob

CASES = [
    # kind, d, hidden, layers, chunk, c_mode, loss
    (oracle.LINEAR, 3, 0, 2, 3, oracle.C_ONE, oracle.LOSS_L2),
    (oracle.LINEAR, 4, 0, 2, 2, oracle.C_PER_TOKEN, oracle.LOSS_HUBER),
    (oracle.MLP2, 3, 4, 2, 3, oracle.C_ONE_MINUS_BETA, oracle.LOSS_L2),
    (oracle.MLP2, 2, 3, 3, 2, oracle.C_ONE, oracle.LOSS_L2),
]


def _case(kind, d, hidden, layers, chunk, c_mode, seed):
    rng = np.random.default_rng(seed)
    T = 7
    P = oracle.param_count(kind, d, hidden, layers)
    x = dict(q=rng.normal(0, 1, (T, d)), k=rng.normal(0, 1, (T, d)), v=rng.normal(0, 1, (T, d)),
             alpha=rng.uniform(0.05, 0.2, T), eta=rng.uniform(0.05, 0.3, T), beta=rng.uniform(0.3, 0.9, T),
             M0=rng.normal(0, 0.5, P), S0=rng.normal(0, 0.1, P),
             c=rng.uniform(0.2, 1.0, T) if c_mode == oracle.C_PER_TOKEN else None)
    up = dict(Gy=rng.normal(0, 1, (T, d)), GM=rng.normal(0, 1, P), GS=rng.normal(0, 1, P))
    return x, up


def _c_forward(kind, d, hidden, layers, chunk, c_mode, loss, delta, x):
    T = x["q"].shape[0]
    P = x["M0"].shape[0]
    r = lambda a: np.asarray(a, dtype=np.float64).reshape((1, 1) + np.shape(a))
    return oracle.forward(kind, d, hidden, chunk, c_mode, r(x["q"]), r(x["k"]), r(x["v"]), r(x["alpha"]),
                          r(x["eta"]), r(x["beta"]), None if x["c"] is None else r(x["c"]), r(x["M0"]), r(x["S0"]),
                          loss, delta, layers=layers)


@pytest.mark.parametrize("kind,d,hidden,layers,chunk,c_mode,loss", CASES)
def test_torch_restatement_reproduces_the_c_oracle(kind, d, hidden, layers, chunk, c_mode, loss):
    import torch
    x, _ = _case(kind, d, hidden, layers, chunk, c_mode, seed=3)
    delta = 0.7 if loss == oracle.LOSS_HUBER else np.inf
    y, MT, ST = _c_forward(kind, d, hidden, layers, chunk, c_mode, loss, delta, x)
    t = {n: None if a is None else torch.tensor(a, dtype=torch.float64) for n, a in x.items()}
    yt, MTt, STt = ob.forward_torch(kind, d, hidden, chunk, c_mode, t["q"], t["k"], t["v"], t["alpha"], t["eta"],
                                    t["beta"], t["c"], t["M0"], t["S0"], loss, delta, layers)
    np.testing.assert_allclose(yt.numpy(), y[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(MTt.numpy(), MT[0, 0], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(STt.numpy(), ST[0, 0], rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("kind,d,hidden,layers,chunk,c_mode,loss", CASES)
def test_gradients_match_central_differences_of_the_c_forward(kind, d, hidden, layers, chunk, c_mode, loss):
    x, up = _case(kind, d, hidden, layers, chunk, c_mode, seed=11)
    delta = 0.7 if loss == oracle.LOSS_HUBER else np.inf

    def functional(xx):
        y, MT, ST = _c_forward(kind, d, hidden, layers, chunk, c_mode, loss, delta, xx)
        return float((y[0, 0] * up["Gy"]).sum() + (MT[0, 0] * up["GM"]).sum() + (ST[0, 0] * up["GS"]).sum())

    g = ob.backward(kind, d, hidden, chunk, c_mode, x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"],
                    x["c"], x["M0"], x["S0"], up["Gy"], up["GM"], up["GS"], loss, delta, layers)
    rng = np.random.default_rng(5)
    h = 1e-6
    for name, grad in g.items():
        flat = np.asarray(x[name], dtype=np.float64).reshape(-1)
        for idx in rng.choice(flat.size, size=min(6, flat.size), replace=False):
            xp = dict(x); xm = dict(x)
            ap = flat.copy(); ap[idx] += h
            am = flat.copy(); am[idx] -= h
            xp[name] = ap.reshape(np.shape(x[name]))
            xm[name] = am.reshape(np.shape(x[name]))
            fd = (functional(xp) - functional(xm)) / (2 * h)
            got = grad.reshape(-1)[idx]
            assert abs(got - fd) <= 1e-6 * max(1.0, abs(fd)), (name, idx, got, fd)
