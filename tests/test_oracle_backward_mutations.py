"""Planted mistakes in the reference gradients (oracle/backward.py): each one is
a plausible error in its torch restatement of the forward or in the functional
it differentiates (a wrong derivative, the gradient or the retrieval at the
wrong weights, an ignored coefficient, a wrong sign, a transposed layer
gradient, an unclipped Huber gradient, a dropped or swapped upstream term).
The test loads a copy of the module's source with the mistake as a module of
its own, points the pins of tests/test_oracle_backward.py at it, and checks
that they catch it.  Mistakes are planted only in that in-memory copy, on the
CPU."""
import types

import pytest

import oracle
from oracle import backward as ob
import test_oracle_backward as pins

MUTATIONS = {
    "wrong silu derivative": ("(s * (1.0 + zs[li - 1] * (1.0 - s)))", "(s * (1.0 + zs[li - 1] * s))"),
    "gradient at the current weights": ("g = _grad(W0s, k[t], v[t], loss_kind, huber_delta)",
                                        "g = _grad(_split(M, sizes), k[t], v[t], loss_kind, huber_delta)"),
    "retrieval at the chunk-start weights": ("ys.append(_apply(_split(M, sizes), q[t]))",
                                             "ys.append(_apply(W0s, q[t]))"),
    "coefficient 1 - beta ignored": ("ct = 1.0 - beta[t]", "ct = 1.0"),
    "wrong sign of the step": ("M = (1.0 - alpha[t]) * M - eta[t] * S", "M = (1.0 - alpha[t]) * M + eta[t] * S"),
    "transposed layer gradient": ("grads[li] = torch.outer(delta_l, xs[li])",
                                  "grads[li] = torch.outer(xs[li], delta_l)"),
    "Huber gradient not clipped": ("return 2.0 * torch.clamp(r, -delta, delta)", "return 2.0 * r"),
    "upstream of S_T dropped": ("\n         + (ST * torch.tensor(GS, dtype=torch.float64)).sum())", ")"),
    "upstream of M_T used for S_T": ("(ST * torch.tensor(GS, dtype=torch.float64))",
                                     "(ST * torch.tensor(GM, dtype=torch.float64))"),
    "momentum decay dropped": ("S = beta[t] * S + ct * g", "S = S + ct * g"),
}

PIN_CALLS = [(fn, case) for case in pins.CASES
             for fn in (pins.test_torch_restatement_reproduces_the_c_oracle,
                        pins.test_gradients_match_central_differences_of_the_c_forward)]


def _load(source, tag):
    """The module's source (maybe mutated) as a fresh module of the oracle package."""
    mod = types.ModuleType("oracle.backward_" + tag)
    mod.__dict__["__package__"] = "oracle"
    exec(compile(source, ob.__file__ + " [" + tag + "]", "exec"), mod.__dict__)
    return mod


def _caught(mod, monkeypatch):
    failed = []
    with monkeypatch.context() as m:
        m.setattr(pins, "ob", mod)
        for fn, case in PIN_CALLS:
            try:
                fn(*case)
            except AssertionError:
                failed.append((fn.__name__, case))
    return failed


def test_unmodified_reference_passes_the_pin_set(monkeypatch):
    oracle.build()
    assert _caught(_load(open(ob.__file__).read(), "copy"), monkeypatch) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, monkeypatch):
    old, new = MUTATIONS[name]
    src = open(ob.__file__).read()
    assert src.count(old) == 1, "the mutation site moved: %s" % name
    failed = _caught(_load(src.replace(old, new), "mutated"), monkeypatch)
    assert failed, "no pin caught: %s" % name
