"""Planted mistakes: each one is a plausible error in the oracle (a dropped
factor, a wrong sign, the wrong weights, a transposed operand, an ignored
coefficient, a wrong derivative, a wrong layer offset, a wrong surprise norm,
a wrong gate).  For the C oracle the test compiles a copy of nm_oracle.c with
the mistake and points the oracle at it; for the Memory-as-Gate combination
(numpy) it builds a copy of the function with the mistake.  Either way it
checks that the pins of tests/test_oracle.py catch it.  Mistakes are planted
only in those temporary copies, on the CPU."""
import os
import subprocess
import tempfile

import pytest

import oracle
import test_oracle as pins

SRC = oracle._SRC

MUTATIONS = {
    "dropped factor 2 of the squared loss": ("    return 2.0 * r;\n}", "    return r;\n}"),
    "gradient at the current weights": (
        "oracle_grad(kind, d, h, layers, loss, delta, W0, k + (long)t * d",
        "oracle_grad(kind, d, h, layers, loss, delta, M, k + (long)t * d"),
    "wrong sign of the step": ("M[p] = (1.0 - alpha[t]) * M[p] - eta[t] * S[p];",
                               "M[p] = (1.0 - alpha[t]) * M[p] + eta[t] * S[p];"),
    "retrieval before the update": ("oracle_memory_apply(kind, d, h, layers, M, q + (long)t * d",
                                    "oracle_memory_apply(kind, d, h, layers, W0, q + (long)t * d"),
    "transposed linear gradient": ("g[(long)o * d + i] = e[o] * k[i];", "g[(long)o * d + i] = e[i] * k[o];"),
    "per-token c ignored": ("else if (c_mode == OR_C_PER_TOKEN) ct = c[t];", "else if (c_mode == OR_C_PER_TOKEN) ct = 1.0;"),
    "wrong silu derivative": ("return s * (1.0 + z * (1.0 - s));", "return s * (1.0 + z * s);"),
    "Huber gradient not clipped": ("if (r > delta) return 2.0 * delta;", "if (r > delta) return 2.0 * r;"),
    "wrong offset of the hidden layers": ("off[l] = off[l - 1] + (long)h * h;", "off[l] = off[l - 1] + (long)h * d;"),
    "momentum decay dropped": ("S[p] = beta[t] * S[p] + ct * g[p];", "S[p] = S[p] + ct * g[p];"),
    "coefficient 1 - beta taken as beta": ("if (c_mode == OR_C_ONE_MINUS_BETA) ct = 1.0 - beta[t];",
                                           "if (c_mode == OR_C_ONE_MINUS_BETA) ct = beta[t];"),
    "forgetting factor taken as alpha": ("M[p] = (1.0 - alpha[t]) * M[p] - eta[t] * S[p];",
                                         "M[p] = alpha[t] * M[p] - eta[t] * S[p];"),
    "surprise as the squared norm": ("surprise[t] = sqrt(n2);", "surprise[t] = n2;"),
    "surprise from absolute values": ("n2 += g[p] * g[p];", "n2 += fabs(g[p]);"),
}

PIN_CALLS = [
    (pins.test_scalar_worked_example, (2,)),
    (pins.test_scalar_worked_example, (1,)),
    (pins.test_2x2_worked_example, ()),
    (pins.test_grad_finite_differences, (oracle.LINEAR, 2, 0)),
    (pins.test_grad_finite_differences, (oracle.MLP2, 2, 3)),
    (pins.test_grad_and_apply_match_library, (oracle.LINEAR, 5, 0)),
    (pins.test_grad_and_apply_match_library, (oracle.MLP2, 4, 7)),
    (pins.test_single_chunk_sums_gradients_at_chunk_start, (oracle.MLP2, 3, 5)),
    (pins.test_chunk1_equals_form_A_sequential, (oracle.LINEAR, 3, 0)),
    (pins.test_chunk1_equals_form_B_sequential, (oracle.MLP2, 2, 6)),
    (pins.test_huber_grad_finite_differences_and_library, (oracle.LINEAR, 3, 0)),
    (pins.test_deep_grad_finite_differences_and_library, (2, 3, 3)),
    (pins.test_deep_chunk1_equals_sequential_and_chunk_sums_gradients, (3,)),
    (pins.test_surprise_is_the_gradient_norm_at_chunk_start, (oracle.LINEAR, 4, 0, oracle.LOSS_L2)),
    (pins.test_surprise_is_the_gradient_norm_at_chunk_start, (oracle.MLP2, 3, 6, oracle.LOSS_HUBER)),
]


def _caught(lib_path):
    saved = (oracle._LIB, oracle._lib)
    oracle._LIB, oracle._lib = lib_path, None
    failed = []
    try:
        for fn, args in PIN_CALLS:
            try:
                fn(*args)
            except AssertionError:
                failed.append(fn.__name__)
    finally:
        oracle._LIB, oracle._lib = saved
    return failed


def test_unmodified_oracle_passes_the_pin_set():
    oracle.build()
    assert _caught(oracle._LIB) == []


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTATIONS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, "the mutation site moved: %s" % name
    mutated = tmp_path / "nm_oracle_mutated.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mutated.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-o", str(so), str(mutated),
                           "-lm"])
    failed = _caught(str(so))
    assert failed, "no pin caught: %s" % name


# The Memory-as-Gate combination is plain numpy in oracle/__init__.py: its mistakes are planted in an
# in-memory copy of that function, which the pins then call in place of the original.
GATE_MUTATIONS = {
    "sigmoid of -y": ("y_attn / (1.0 + np.exp(-y_mem))", "y_attn / (1.0 + np.exp(y_mem))"),
    "operands swapped": ("y_attn / (1.0 + np.exp(-y_mem))", "y_mem / (1.0 + np.exp(-y_attn))"),
    "tanh for the sigmoid": ("y_attn / (1.0 + np.exp(-y_mem))", "y_attn * np.tanh(y_mem)"),
}
GATE_PINS = [pins.test_mag_gate_hand_worked, pins.test_mag_gate_symmetry_limits_and_library]


def _gate_caught(fn, monkeypatch):
    failed = []
    with monkeypatch.context() as m:
        m.setattr(oracle, "mag_gate", fn)
        for pin in GATE_PINS:
            try:
                pin()
            except AssertionError:
                failed.append(pin.__name__)
    return failed


def _gate_from(source):
    import inspect
    ns = dict(oracle.__dict__)
    exec(compile(source, inspect.getsourcefile(oracle) + " [mag_gate]", "exec"), ns)
    return ns["mag_gate"]


def test_unmodified_gate_passes_its_pins(monkeypatch):
    import inspect
    assert _gate_caught(_gate_from(inspect.getsource(oracle.mag_gate)), monkeypatch) == []


@pytest.mark.parametrize("name", sorted(GATE_MUTATIONS))
def test_planted_gate_mistake_is_caught(name, monkeypatch):
    import inspect
    old, new = GATE_MUTATIONS[name]
    src = inspect.getsource(oracle.mag_gate)
    assert src.count(old) == 1, "the mutation site moved: %s" % name
    assert _gate_caught(_gate_from(src.replace(old, new)), monkeypatch), "no pin caught: %s" % name
