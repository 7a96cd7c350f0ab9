"""Planted mistakes: each one is a plausible error in the oracle (a dropped
factor, a wrong sign, the wrong weights, a transposed operand, an ignored
coefficient, a wrong derivative, a wrong layer offset).  The test compiles a
copy of nm_oracle.c with the mistake, points the oracle at it, and checks that
the pins of tests/test_oracle.py catch it.  Mistakes are planted only in this
temporary copy of the oracle, on the CPU."""
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
