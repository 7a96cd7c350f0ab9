"""The C-ABI boundary: the library loads without a GPU, exports every entry
point include/nm.h declares, and (on a GPU) rejects bad arguments on the host
with the documented status and nothing launched."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

import test_neural_memory_titans_b300 as nm
from test_neural_memory_titans_b300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in sorted(os.listdir(os.path.join(ROOT, "include")))
           if f.endswith(".h")]


def _declared():
    names = set()
    for h in HEADERS:
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[\w\s\*]+?\b(nm_\w+)\s*\(", src, flags=re.M):
            names.add(m.group(1))
    return names


def test_library_loads_and_exports_header_symbols():
    lib = nm.load_library()
    declared = _declared()
    assert {"nm_create", "nm_forward", "nm_destroy", "nm_synchronize", "nm_status_string"} <= declared
    for name in declared:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", nm.LIB_PATH], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (nm_\w+)", out))
    assert declared <= exported, declared - exported
    assert set(nm.EXPORTED) <= exported


@pytest.mark.parametrize("lang,std", [("c", "-std=c99"), ("c++", "-std=c++11")])
def test_headers_compile_as_plain_c_and_cpp(lang, std):
    """The boundary is a C ABI: its headers take no CUDA, torch or C++-only
    type and compile on their own, warning-free, from C and from C++."""
    for h in HEADERS:
        r = subprocess.run(["gcc", "-fsyntax-only", std, "-Wall", "-Wextra", "-Werror", "-x", lang, h],
                           capture_output=True, text=True)
        assert r.returncode == 0, (h, r.stderr)


def test_status_strings_without_gpu():
    for code in range(0, 9):
        s = nm.status_string(code)
        assert isinstance(s, str) and s
    assert nm.status_string(12345) == "unknown status"


def test_status_codes_match_header():
    src = open(os.path.join(ROOT, "include", "nm.h")).read()
    defs = dict((k, int(v)) for k, v in re.findall(r"#define\s+(NM_\w+)\s+(-?\d+)", src))
    for name in ("NM_OK", "NM_ERR_ARG", "NM_ERR_ALIGN", "NM_ERR_UNSUPPORTED", "NM_ERR_ALIAS", "NM_ERR_CUDA",
                 "NM_ERR_NOMEM", "NM_ERR_DEVICE_TIMEOUT", "NM_ERR_DEVICE_CHECK"):
        assert getattr(nm, name) == defs[name]
    for name, py in (("NM_LINEAR", "LINEAR"), ("NM_MLP2", "MLP2"), ("NM_F32", "F32"), ("NM_BF16", "BF16"),
                     ("NM_C_ONE", "C_ONE"), ("NM_C_ONE_MINUS_BETA", "C_ONE_MINUS_BETA"),
                     ("NM_C_PER_TOKEN", "C_PER_TOKEN"), ("NM_PATH_AUTO", "PATH_AUTO"),
                     ("NM_PATH_SIMT", "PATH_SIMT"), ("NM_PATH_TC", "PATH_TC"), ("NM_LOSS_L2", "LOSS_L2"),
                     ("NM_LOSS_HUBER", "LOSS_HUBER")):
        assert getattr(nm, py) == defs[name]


def test_null_handle_and_bad_config_without_gpu():
    lib = nm.load_library()
    assert lib.nm_forward(None, 1, 1, 1, *([None] * 12), None) == nm.NM_ERR_ARG
    assert lib.nm_forward_surprise(None, 1, 1, 1, *([None] * 13), None) == nm.NM_ERR_ARG
    assert lib.nm_forward_gated(None, 1, 1, 1, *([None] * 13), None) == nm.NM_ERR_ARG
    assert lib.nm_synchronize(None) == nm.NM_ERR_ARG
    assert lib.nm_destroy(None) == nm.NM_OK
    h = ctypes.c_void_p()
    bad = nm._Config(7, 64, 0, 64, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO)
    assert lib.nm_create(ctypes.byref(bad), 0, ctypes.byref(h)) == nm.NM_ERR_ARG
    unsupported = nm._Config(nm.LINEAR, 48, 0, 64, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_SIMT)
    assert lib.nm_create(ctypes.byref(unsupported), 0, ctypes.byref(h)) == nm.NM_ERR_UNSUPPORTED
    big_chunk = nm._Config(nm.LINEAR, 64, 0, 1024, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO)
    assert lib.nm_create(ctypes.byref(big_chunk), 0, ctypes.byref(h)) == nm.NM_ERR_UNSUPPORTED
    assert lib.nm_create(None, 0, ctypes.byref(h)) == nm.NM_ERR_ARG
    # the depth: only an MLP memory has layers, 2..16
    for kind, layers in ((nm.LINEAR, 3), (nm.MLP2, 1), (nm.MLP2, 17), (nm.MLP2, -2)):
        cfg = nm._Config(kind, 64, 128, 64, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO, nm.LOSS_L2, 0.0, layers)
        assert lib.nm_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == nm.NM_ERR_ARG
    # the loss: an unknown kind, or a Huber threshold that is not finite and positive
    for loss, delta in ((2, 1.0), (nm.LOSS_HUBER, 0.0), (nm.LOSS_HUBER, -1.0), (nm.LOSS_HUBER, float("inf")),
                        (nm.LOSS_HUBER, float("nan"))):
        cfg = nm._Config(nm.LINEAR, 64, 0, 64, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO, loss, delta)
        assert lib.nm_create(ctypes.byref(cfg), 0, ctypes.byref(h)) == nm.NM_ERR_ARG
        assert lib.nm_forward_mlp2_noalloc(ctypes.byref(cfg), 1, 1, 1, *([None] * 12), None) in (
            nm.NM_ERR_ARG, nm.NM_ERR_UNSUPPORTED)


def _shape_taken(lib, kind, d, hidden, chunk, dtype, path, layers=0):
    """Whether nm_create's path selection takes the shape: it decides before any
    CUDA call, so without a GPU a taken shape fails later, at the device query
    (NM_ERR_CUDA, or NM_ERR_ARG when no device is listed), and a shape no
    kernel of the path takes returns NM_ERR_UNSUPPORTED."""
    h = ctypes.c_void_p()
    cfg = nm._Config(kind, d, hidden, chunk, dtype, nm.BF16, nm.C_ONE, path, nm.LOSS_L2, 0.0, layers)
    rc = lib.nm_create(ctypes.byref(cfg), 0, ctypes.byref(h))
    if rc == nm.NM_OK:  # (a run with a GPU)
        lib.nm_destroy(h)
    assert rc in (nm.NM_OK, nm.NM_ERR_CUDA, nm.NM_ERR_ARG, nm.NM_ERR_UNSUPPORTED), rc
    return rc != nm.NM_ERR_UNSUPPORTED


def test_shapes_each_path_takes_without_gpu():
    """The shape table of nm_config's documentation, path by path."""
    lib = nm.load_library()
    L, M, B16, F32, TC, SIMT = nm.LINEAR, nm.MLP2, nm.BF16, nm.F32, nm.PATH_TC, nm.PATH_SIMT
    tc_taken = [(L, 128, 0, 64), (L, 64, 0, 64), (L, 64, 0, 128), (L, 64, 0, 256),  # linear d = 128; d = 64
                (M, 64, 128, 64), (M, 64, 256, 64),                                  # MLP d = 64
                (M, 128, 128, 64), (M, 128, 256, 64), (M, 128, 512, 64)]             # MLP d = 128
    tc_not = [(L, 128, 0, 32), (L, 64, 0, 32), (L, 32, 0, 64), (L, 16, 0, 64),
              (M, 64, 512, 64), (M, 64, 256, 32), (M, 128, 1024, 64), (M, 32, 128, 64)]
    for kind, d, hid, ch in tc_taken:
        assert _shape_taken(lib, kind, d, hid, ch, B16, TC), (kind, d, hid, ch)
        assert not _shape_taken(lib, kind, d, hid, ch, F32, TC), (kind, d, hid, ch)  # bf16 inputs only
    for kind, d, hid, ch in tc_not:
        assert not _shape_taken(lib, kind, d, hid, ch, B16, TC), (kind, d, hid, ch)
    # deeper memories on the tensor cores: d 64 or 128, hidden a multiple of 64 up to 512, chunk <= 64
    for d, hid, ch, ok in ((64, 256, 64, True), (128, 512, 64, True), (64, 64, 1, True), (64, 256, 32, True),
                           (64, 96, 64, False), (64, 576, 64, False), (64, 256, 128, False), (32, 256, 64, False)):
        assert _shape_taken(lib, M, d, hid, ch, B16, TC, layers=3) == ok, (d, hid, ch)
    # the fp32 FFMA path: d in {16, 32, 64, 128}, chunk 1..256, hidden a multiple of 32 up to 1024
    for kind, d, hid, ch, ok in ((L, 16, 0, 1, True), (L, 128, 0, 256, True), (L, 48, 0, 64, False),
                                 (L, 64, 0, 257, False), (M, 32, 1024, 16, True), (M, 64, 1056, 64, False),
                                 (M, 64, 48, 64, False)):
        for dt in (F32, B16):
            assert _shape_taken(lib, kind, d, hid, ch, dt, SIMT) == ok, (kind, d, hid, ch, dt)
    assert _shape_taken(lib, M, 64, 96, 8, F32, SIMT, layers=5)


@pytest.mark.skipif(torch.cuda.is_available(), reason="fake addresses are for a machine without a GPU")
def test_noalloc_host_checks_without_gpu():
    """nm_forward_mlp2_noalloc checks alignment, overlaps, the c argument and
    the workspace bound on the host, before any CUDA call.  Every call below
    breaks one of those rules, so the addresses (fake, never dereferenced) are
    only compared; the test does not run where a GPU is visible."""
    fn = nm.load_library().nm_forward_mlp2_noalloc
    vp = ctypes.c_void_p
    fn.argtypes = [ctypes.POINTER(nm._Config), ctypes.c_int, ctypes.c_int, ctypes.c_int] + [vp] * 13
    fn.restype = ctypes.c_int
    d, hidden, chunk, B, H, T = 64, 128, 64, 1, 2, 100
    cfg = nm._Config(nm.MLP2, d, hidden, chunk, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_AUTO)
    P = nm.param_count(nm.MLP2, d, hidden)
    MB = 1 << 20
    # disjoint, 16-byte-aligned ranges: inputs (bf16 [B,H,T,d]), gates, states, y, M_T, S_T
    base = dict(q=1 * MB, k=2 * MB, v=3 * MB, alpha=4 * MB, eta=5 * MB, beta=6 * MB, c=None, M0=8 * MB,
                S0=9 * MB, y=10 * MB, M_T=11 * MB, S_T=12 * MB)
    order = ("q", "k", "v", "alpha", "eta", "beta", "c", "M0", "S0", "y", "M_T", "S_T")

    def call(cf=cfg, units=(B, H, T), **over):
        p = dict(base)
        p.update(over)
        return fn(ctypes.byref(cf), *units, *(None if p[n] is None else vp(p[n]) for n in order), None)

    assert call(q=1 * MB + 2) == nm.NM_ERR_ALIGN
    assert call(S_T=12 * MB + 8) == nm.NM_ERR_ALIGN
    assert call(y=1 * MB + 64) == nm.NM_ERR_ALIAS                 # y inside q
    assert call(M_T=8 * MB + 16) == nm.NM_ERR_ALIAS               # M_T partly over M0
    assert call(S_T=11 * MB + 4 * P - 16) == nm.NM_ERR_ALIAS      # S_T's start inside M_T
    assert call(c=7 * MB) == nm.NM_ERR_ARG                        # c given without NM_C_PER_TOKEN
    per_token = nm._Config(nm.MLP2, d, hidden, chunk, nm.BF16, nm.BF16, nm.C_PER_TOKEN, nm.PATH_AUTO)
    assert call(cf=per_token) == nm.NM_ERR_ARG                    # c missing with it
    assert call(y=None) == nm.NM_ERR_ARG
    assert call(units=(1, 1 << 16, T)) == 9                       # NM_ERR_TOO_LARGE: beyond the fixed workspace
    tc = nm._Config(nm.MLP2, d, hidden, chunk, nm.BF16, nm.BF16, nm.C_ONE, nm.PATH_TC)
    assert call(cf=tc) == nm.NM_ERR_UNSUPPORTED                   # the fp32 FFMA kernel only


# ------------------------------------------------------------------ on a GPU

def _args(wl, dev="cuda"):
    x = W.make_inputs(wl, dev)
    y = torch.empty(x["q"].shape, dtype=wl.dtype, device=dev)
    MT = torch.empty_like(x["M0"])
    ST = torch.empty_like(x["S0"])
    return x, y, MT, ST


def _call(mem, B, H, T, x, yo, MTo, STo, **over):
    p = dict(q=x["q"], k=x["k"], v=x["v"], alpha=x["alpha"], eta=x["eta"], beta=x["beta"], c=None,
             M0=x["M0"], S0=x["S0"], y=yo, M_T=MTo, S_T=STo)
    p.update(over)

    def ptr(t):
        if t is None:
            return None
        if isinstance(t, int):
            return ctypes.c_void_p(t)
        return ctypes.c_void_p(t.data_ptr())
    return nm.load_library().nm_forward(mem._h, B, H, T, *(ptr(p[k]) for k in
                                        ("q", "k", "v", "alpha", "eta", "beta", "c", "M0", "S0", "y", "M_T",
                                         "S_T")), None)


@pytest.mark.gpu
def test_host_validation_launches_nothing():
    wl = W.WORKLOADS[2].with_sizes(B=2, H=2, T=128)
    x, y, MT, ST = _args(wl)
    mem = nm.NeuralMemory(wl.kind, wl.d, 0, wl.chunk, in_dtype=wl.dtype)
    n0 = mem.launches
    B, H, T = wl.B, wl.H, wl.T
    assert _call(mem, B, H, T, x, y, MT, ST, q=None) == nm.NM_ERR_ARG
    assert _call(mem, -1, H, T, x, y, MT, ST) == nm.NM_ERR_ARG
    assert _call(mem, B, H, T, x, y, MT, ST, c=x["alpha"]) == nm.NM_ERR_ARG  # c given but c_mode is ONE
    assert _call(mem, B, H, T, x, y, MT, ST, k=x["k"].data_ptr() + 2) == nm.NM_ERR_ALIGN
    assert _call(mem, B, H, T, x, y, MT, ST, M_T=x["S0"]) == nm.NM_ERR_ALIAS          # M_T on S0
    assert _call(mem, B, H, T, x, y, MT, ST, y=x["q"]) == nm.NM_ERR_ALIAS             # y on an input
    assert _call(mem, B, H, T, x, y, MT, ST, S_T=MT) == nm.NM_ERR_ALIAS               # outputs overlap
    part = x["M0"].data_ptr() + 16 * 4
    assert _call(mem, B, H, T, x, y, MT, ST, M_T=part) == nm.NM_ERR_ALIAS             # partial overlap
    assert mem.launches == n0
    assert _call(mem, 0, H, T, x, y, MT, ST) == nm.NM_OK and mem.launches == n0     # empty batch
    # exact aliasing of the state is allowed
    M = x["M0"].clone()
    S = x["S0"].clone()
    assert _call(mem, B, H, T, x, y, M, S, M0=M, S0=S) == nm.NM_OK
    assert mem.synchronize() == nm.NM_OK
    assert mem.launches == n0 + 1


@pytest.mark.gpu
def test_per_token_c_required():
    wl = W.WORKLOADS[2].with_sizes(B=1, H=1, T=64)
    x, y, MT, ST = _args(wl)
    mem = nm.NeuralMemory(wl.kind, wl.d, 0, wl.chunk, in_dtype=wl.dtype, c_mode=nm.C_PER_TOKEN)
    assert _call(mem, 1, 1, 64, x, y, MT, ST) == nm.NM_ERR_ARG
    assert _call(mem, 1, 1, 64, x, y, MT, ST, c=x["beta"]) == nm.NM_OK
    assert mem.synchronize() == nm.NM_OK


@pytest.mark.gpu
def test_binding_rejects_wrong_tensors():
    wl = W.WORKLOADS[2].with_sizes(B=1, H=1, T=64)
    x = W.make_inputs(wl, "cuda")
    mem = nm.NeuralMemory(wl.kind, wl.d, 0, wl.chunk, in_dtype=wl.dtype)
    with pytest.raises(TypeError):
        mem.forward(x["q"].float(), x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"])
    with pytest.raises(ValueError):
        mem.forward(x["q"].cpu(), x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"])
    with pytest.raises(ValueError):
        mem.forward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"][..., :-1], x["S0"])


@pytest.mark.gpu
def test_gated_validation():
    """nm_forward_gated: y_attn required, aligned, and apart from the outputs
    except o == y_attn (gating in place); nothing launched on an error."""
    wl = W.WORKLOADS[2].with_sizes(B=2, H=2, T=128)
    x, y, MT, ST = _args(wl)
    ya = torch.randn(y.shape, device="cuda").to(wl.dtype)
    mem = nm.NeuralMemory(wl.kind, wl.d, 0, wl.chunk, in_dtype=wl.dtype)
    lib = nm.load_library()
    n0 = mem.launches

    def call(y_attn, o, M_T=MT, S_T=ST):
        p = lambda t: None if t is None else ctypes.c_void_p(t if isinstance(t, int) else t.data_ptr())
        return lib.nm_forward_gated(mem._h, 2, 2, 128, p(x["q"]), p(x["k"]), p(x["v"]), p(x["alpha"]),
                                    p(x["eta"]), p(x["beta"]), None, p(x["M0"]), p(x["S0"]), p(y_attn), p(o),
                                    p(M_T), p(S_T), None)
    assert call(None, y) == nm.NM_ERR_ARG
    assert call(ya.data_ptr() + 2, y) == nm.NM_ERR_ALIGN
    assert call(ya, ya.data_ptr() + 16) == nm.NM_ERR_ALIAS        # o partly over y_attn
    assert call(ya, y, M_T=ya) == nm.NM_ERR_ALIAS                 # a state output over y_attn
    assert call(x["q"], x["q"]) == nm.NM_ERR_ALIAS                # o over q (even as y_attn)
    assert mem.launches == n0
    assert call(ya, ya) == nm.NM_OK                               # in place
    assert mem.synchronize() == nm.NM_OK
    assert mem.launches == n0 + 1
