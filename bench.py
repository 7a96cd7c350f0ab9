"""Benchmark of the neural-memory forward pass: one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

A step is one full forward over the workload (for the streamed workload, all
of its segment calls, carrying the state in place).  Inputs are resident in
HBM before timing; L2 is flushed (a 256 MB write) between timed steps, outside
each step's CUDA-event pair.  ``value`` is B*H*T tokens per second over all
ranks (weak scaling: every rank runs its own copy of the workload with its own
seed, no collective on the data path).  ``e2e`` measures the same metric
through nm_forward_host with pinned host buffers (host->device copies of the
inputs and device->host copies of y, M_T, S_T inside the timed region).

``--impl reference`` times the fp64 CPU oracle (the reference arm here) on
the host cores, on a bounded sample of the same workload.

Extra fields: ``roofline`` (the dominant kernel's algorithmic rate against the
measured peak, with ``traffic`` from an ncu capture while the captured kernel
source is unchanged), ``cpu_baseline`` (the oracle on a bounded sample),
``clocks`` (SM clock and throttle reasons sampled during the timed region),
``gpu_launches`` (this library's kernel launches in the timed region) and
``variants`` (the same workload with the Huber loss and with the surprise
output, a few steps each; ``--no-variants`` skips them).  ``--layers L`` runs
an MLP workload with an L-layer memory.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "memory-layer fwd tokens/sec (B*H*T/s) and % of roofline (TC FLOPs vs HBM)"

# DRAM bytes (read + write) per launch of the dominant kernel, from ncu captures summarised under
# profiles/: workload -> (kernel sources, sha256 prefix of those sources when captured, bytes).
# A capture describes the kernel it was taken on only: when the sources differ, traffic is null.
NCU_TRAFFIC = {
    "mlp_64x256_bf16_b4h8_t4096_c64": (("nm_tc_mlp.cu", "tc_common.cuh"), "90384118f1d61292", 61.86e6),
    "linear_d128_bf16_b8h16_t16384_c64": (("nm_tc_linear.cu", "tc_common.cuh"), "a2afbc7a0329e8ae", 2.116e9),
}


def ncu_traffic(workload_name: str):
    """DRAM bytes per launch from the table above, or None if absent or stale."""
    import hashlib
    entry = NCU_TRAFFIC.get(workload_name)
    if entry is None:
        return None
    files, digest, nbytes = entry
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "test_neural_memory_titans_b300", "csrc", f),
                  "rb") as fh:
            h.update(fh.read())
    return nbytes if h.hexdigest()[:16] == digest else None
DEFAULT_WORKLOAD = 1
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}


# --------------------------------------------------------------------- model of the work

def algorithmic(wl) -> dict:
    """Algorithmic tensor-core flops and HBM bytes of one full forward.

    flops per token: linear 10 d^2 + 2 (b+1) d, MLP 22 d h + 2 (b+1)(d+h)
    (the b x b causal products counted as lower-triangular); an MLP of L
    layers: 11 P + 2 (b+1)(d + (L-1) h) with P = 2 d h + (L-2) h^2 (11 flops
    per parameter and token, as for two layers).
    bytes per token: q, k, v in, y out, three fp32 gates; plus per unit the
    fp32 state read (M0, S0) and written (M_T, S_T) once per call.
    """
    d, h, b = wl.d, wl.hidden, wl.chunk
    if wl.kind == 0:
        f_tok = 10 * d * d + 2 * (b + 1) * d
    else:
        f_tok = 11 * wl.P + 2 * (b + 1) * (d + (wl.layers - 1) * h)
    eb = 2 if wl.dtype == torch.bfloat16 else 4
    bytes_tok = 3 * d * eb + 12 + d * eb
    calls = (wl.T // wl.segment) if wl.segment else 1
    state_bytes = 4 * wl.P * 4 * wl.B * wl.H * calls
    tokens = wl.B * wl.H * wl.T
    return {"flops": float(f_tok) * tokens, "bytes": float(bytes_tok) * tokens + state_bytes,
            "tokens": tokens, "calls": calls, "bound": "tensor" if wl.kind == 1 else "hbm"}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


# --------------------------------------------------------------------- clocks

class ClockSampler:
    """Samples the SM clock and the clock-event (throttle) reasons while the
    timed region runs: through NVML when pynvml imports, else by running
    ``nvidia-smi --query-gpu=... -lms 100`` for the device in a subprocess."""

    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown", 0x1: "gpu_idle",
               0x2: "applications_clocks_setting", 0x100: "sync_boost", 0x10: "display_clock_setting"}
    SMI_FIELDS = ("clocks.sm", "clocks.max.sm", "power.draw", "clocks_event_reasons.hw_slowdown",
                  "clocks_event_reasons.hw_thermal_slowdown", "clocks_event_reasons.sw_thermal_slowdown",
                  "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int, period_s: float = 0.01):
        self.samples = []
        self.reasons = set()
        self.max_mhz = None
        self.period = period_s
        self.err = None
        self.source = None
        self._stop = threading.Event()
        self._t = None
        self._proc = None
        self.nv = None
        props = torch.cuda.get_device_properties(device_index)
        self.pci = "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
        try:
            import pynvml
            pynvml.nvmlInit()
            try:
                self.h = pynvml.nvmlDeviceGetHandleByPciBusId(self.pci.encode())
            except Exception:
                self.h = pynvml.nvmlDeviceGetHandleByIndex(device_index)
            self.max_mhz = pynvml.nvmlDeviceGetMaxClockInfo(self.h, pynvml.NVML_CLOCK_SM)
            self.nv = pynvml
            self.source = "nvml"
        except Exception as e:
            self.err = "%s: %s" % (type(e).__name__, e)

    def _run(self):
        while not self._stop.is_set():
            try:
                self.samples.append(self.nv.nvmlDeviceGetClockInfo(self.h, self.nv.NVML_CLOCK_SM))
                mask = self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h)
                for bit, name in self.REASONS.items():
                    if mask & bit:
                        self.reasons.add(name)
            except Exception:
                pass
            time.sleep(self.period)

    def __enter__(self):
        if self.nv is not None:
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        else:
            import shutil
            import subprocess
            smi = shutil.which("nvidia-smi")
            if smi:
                self._proc = subprocess.Popen(
                    [smi, "-i", self.pci, "--query-gpu=" + ",".join(self.SMI_FIELDS), "--format=csv,noheader,nounits",
                     "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
                self.source = "nvidia-smi"
                time.sleep(0.3)  # let the first sample land before the timed work starts
            else:
                self.err = (self.err or "") + "; nvidia-smi not found"
        return self

    def __exit__(self, *exc):
        self._stop.set()
        if self._t is not None:
            self._t.join()
        if self._proc is not None:
            self._proc.terminate()
            out, _ = self._proc.communicate(timeout=10)
            names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
            for line in out.splitlines():
                f = [s.strip() for s in line.split(",")]
                if len(f) != len(self.SMI_FIELDS):
                    continue
                try:
                    self.samples.append(float(f[0]))
                    self.max_mhz = float(f[1])
                except ValueError:
                    continue
                for name, val in zip(names, f[3:]):
                    if val.lower() == "active":
                        self.reasons.add(name)

    def summary(self):
        if not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": sorted(self.reasons),
                    "note": "no clock samples (%s)" % (self.err or self.source)}
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "reasons": sorted(self.reasons - {"gpu_idle"}), "samples": len(self.samples),
                "source": self.source}


# --------------------------------------------------------------------- oracle timing

def time_oracle(wl, x, budget_s: float = 15.0):
    """The fp64 oracle, as it stands, on a bounded sample of the workload
    sized to about ``budget_s`` seconds: whole units (all T tokens when one
    round of units fits the budget, else a prefix of T), as many units as
    fit up to B*H, repeated while the budget allows.  Returns tokens/s (all
    units and repeats over the summed wall time), cores and the sample."""
    import oracle

    cores = len(os.sched_getaffinity(0))
    BH = wl.B * wl.H

    def prep(units, T):
        f = lambda t: t.reshape(BH, *t.shape[2:])[:units, :T].to("cpu", torch.float64).numpy()[None]
        g = lambda t: t.reshape(BH, -1)[:units].to("cpu", torch.float64).numpy()[None]
        return (f(x["q"]), f(x["k"]), f(x["v"]), f(x["alpha"]), f(x["eta"]), f(x["beta"]), None,
                g(x["M0"]), g(x["S0"]))

    def run(args):
        t0 = time.perf_counter()
        oracle.forward(wl.kind, wl.d, wl.hidden, wl.chunk, oracle.C_ONE, *args, layers=wl.layers)
        return time.perf_counter() - t0

    # calibrate on one round of units (one per core) over a few chunks
    units = min(BH, cores)
    Tc = min(wl.T, max(wl.chunk, 256))
    per_tok = run(prep(units, Tc)) / (units * Tc)  # wall seconds per token at this parallelism
    if per_tok * units * wl.T > budget_s:  # a prefix of T for one round of units
        T = max(wl.chunk, int(budget_s / (per_tok * units)) // wl.chunk * wl.chunk)
        T = min(T, wl.T)
    else:  # whole units: more rounds of units, then repeats
        T = wl.T
        rounds = max(1, min(-(-BH // units), int(budget_s / (per_tok * units * T))))
        units = min(BH, rounds * units)
    args = prep(units, T)
    dt, reps = 0.0, 0
    while reps == 0 or dt < 0.8 * budget_s:  # the calibration overestimates; repeat to the budget
        dt += run(args)
        reps += 1
    tokens = units * T * reps
    return {"value": tokens / dt, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": "%d units x %d tokens of the workload, %d run(s) (fp64, OpenMP over units), %.1f s"
                      % (units, T, reps, dt),
            "seconds": dt, "tokens": tokens}


# --------------------------------------------------------------------- our arm

def workload(args):
    """The selected workload, with --B / --H / --T overrides applied (a
    streamed workload overridden to T below one segment runs as one call)."""
    from test_neural_memory_titans_b300 import workloads as W

    wl = W.WORKLOADS[args.workload]
    if args.layers is not None and args.layers != wl.layers:
        import dataclasses
        if wl.kind != W.MLP2:
            raise SystemExit("--layers applies to the MLP workloads (1 and 3)")
        wl = dataclasses.replace(wl, layers=args.layers, name="%s_L%d" % (wl.name, args.layers))
    if args.B is None and args.H is None and args.T is None:
        return wl
    wl = wl.with_sizes(B=args.B, H=args.H, T=args.T)
    if wl.segment and (wl.T % wl.segment or wl.T < wl.segment):
        wl = wl.with_sizes(segment=0)
    import dataclasses
    return dataclasses.replace(wl, name="%s@B%dH%dT%d" % (wl.name, wl.B, wl.H, wl.T))


def run_ours(args, rank, world, local_rank):
    import test_neural_memory_titans_b300 as nm
    from test_neural_memory_titans_b300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    wl = workload(args)
    x = W.make_inputs(wl, dev, seed=1000 + args.workload + 100 * rank)
    mem = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk, in_dtype=wl.dtype, path=args.path, device=local_rank,
                          layers=wl.layers if wl.kind == nm.MLP2 else 0)
    stream = torch.cuda.current_stream(dev)
    y = torch.empty(x["q"].shape, dtype=wl.dtype, device=dev)
    M = torch.empty_like(x["M0"])
    S = torch.empty_like(x["S0"])
    seg = wl.segment if wl.segment else wl.T

    def step():
        if seg == wl.T:
            mem.forward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"],
                        y=y, M_T=M, S_T=S, stream=stream)
        else:
            M.copy_(x["M0"])
            S.copy_(x["S0"])
            for s0 in range(0, wl.T, seg):
                sl = lambda t: t[:, :, s0:s0 + seg]
                mem.forward(segs["q"][s0], segs["k"][s0], segs["v"][s0], segs["alpha"][s0], segs["eta"][s0],
                            segs["beta"][s0], M, S, y=segs["y"][s0], M_T=M, S_T=S, stream=stream)

    segs = {}
    if seg != wl.T:  # contiguous per-segment views prepared once, outside timing
        for key in ("q", "k", "v", "alpha", "eta", "beta"):
            segs[key] = {s0: x[key][:, :, s0:s0 + seg].contiguous() for s0 in range(0, wl.T, seg)}
        segs["y"] = {s0: torch.empty((wl.B, wl.H, seg, wl.d), dtype=wl.dtype, device=dev)
                     for s0 in range(0, wl.T, seg)}
        del x["q"], x["k"], x["v"]

    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        step()
    st = mem.synchronize()
    if st != nm.NM_OK:
        raise RuntimeError("device status after warm-up: %s" % nm.status_string(st))

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    l0 = mem.launches
    with ClockSampler(local_rank) as clocks:
        for i in range(args.steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    launches = mem.launches - l0
    st = mem.synchronize()
    if st != nm.NM_OK:
        raise RuntimeError("device status after timing: %s" % nm.status_string(st))
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = sum(step_ms) / len(step_ms)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())

    alg = algorithmic(wl)
    tokens = alg["tokens"]
    value = world * tokens / (ms * 1e-3)

    # the same workload through the two optional forms of the method (Huber loss; surprise output),
    # single-call workloads only, a few steps each, same L2 flush and event timing
    variants = None
    if seg == wl.T and not args.no_variants:
        def time_calls(fn, n_steps):
            for _ in range(2):
                fn()
            ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
            for a_, b_ in ev:
                flush.zero_()
                a_.record(stream)
                fn()
                b_.record(stream)
            torch.cuda.synchronize(dev)
            return sum(a_.elapsed_time(b_) for a_, b_ in ev) / n_steps

        n_var = max(3, min(args.steps, 30))
        args8 = (x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"])
        sur = torch.empty(x["alpha"].shape, dtype=torch.float32, device=dev)
        mem_h = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk, in_dtype=wl.dtype, path=args.path,
                                device=local_rank, loss=nm.LOSS_HUBER, huber_delta=0.1,
                                layers=wl.layers if wl.kind == nm.MLP2 else 0)
        v_h = time_calls(lambda: mem_h.forward(*args8, y=y, M_T=M, S_T=S, stream=stream), n_var)
        v_s = time_calls(lambda: mem.forward_surprise(*args8, y=y, M_T=M, S_T=S, surprise=sur, stream=stream), n_var)
        for m_ in (mem, mem_h):
            st = m_.synchronize()
            if st != nm.NM_OK:
                raise RuntimeError("device status after the variants: %s" % nm.status_string(st))
        mem_h.close()
        variants = {"huber_loss": {"ms_per_step": v_h, "value": world * tokens / (v_h * 1e-3), "delta": 0.1},
                    "surprise_output": {"ms_per_step": v_s, "value": world * tokens / (v_s * 1e-3)},
                    "steps": n_var, "note": "nm_config.loss = NM_LOSS_HUBER; nm_forward_surprise"}

    # e2e through the host-buffer entry point (pinned), copies inside the timed region
    e2e = None
    if not args.no_e2e and seg == wl.T:
        hx = {k: x[k].cpu().pin_memory() for k in ("q", "k", "v", "alpha", "eta", "beta", "M0", "S0")}
        hy = torch.empty(y.shape, dtype=wl.dtype, pin_memory=True)
        hM = torch.empty(M.shape, dtype=torch.float32, pin_memory=True)
        hS = torch.empty(S.shape, dtype=torch.float32, pin_memory=True)
        hargs = (hx["q"], hx["k"], hx["v"], hx["alpha"], hx["eta"], hx["beta"], hx["M0"], hx["S0"])
        for _ in range(max(1, min(args.warmup, 3))):
            mem.forward_host(*hargs, y=hy, M_T=hM, S_T=hS, stream=stream)
        e_steps = max(3, min(args.steps, 20))
        t0 = time.perf_counter()
        for _ in range(e_steps):
            mem.forward_host(*hargs, y=hy, M_T=hM, S_T=hS, stream=stream)
        e_s = (time.perf_counter() - t0) / e_steps
        h2d = sum(t.numel() * t.element_size() for t in hargs)
        d2h = hy.numel() * hy.element_size() + hM.numel() * 4 + hS.numel() * 4
        e2e = {"value": world * tokens / e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_s * 1e3}
    elif not args.no_e2e:
        # streamed: one host-buffer call per segment, the state carried on the host from call to call
        keys = ("q", "k", "v", "alpha", "eta", "beta")
        hseg = {k: {s0: segs[k][s0].cpu().pin_memory() for s0 in segs[k]} for k in keys}
        hy = {s0: torch.empty(segs["y"][s0].shape, dtype=wl.dtype, pin_memory=True) for s0 in segs["y"]}
        hM0 = x["M0"].cpu().pin_memory()
        hS0 = x["S0"].cpu().pin_memory()
        hM = [torch.empty(hM0.shape, dtype=torch.float32, pin_memory=True) for _ in range(2)]
        hS = [torch.empty(hS0.shape, dtype=torch.float32, pin_memory=True) for _ in range(2)]

        def host_step():
            m, sv = hM0, hS0
            for n_, s0 in enumerate(range(0, wl.T, seg)):
                mo, so = hM[n_ & 1], hS[n_ & 1]
                mem.forward_host(*(hseg[k][s0] for k in keys), m, sv, y=hy[s0], M_T=mo, S_T=so, stream=stream)
                m, sv = mo, so

        host_step()
        e_steps = max(1, min(args.steps, 3))
        t0 = time.perf_counter()
        for _ in range(e_steps):
            host_step()
        e_s = (time.perf_counter() - t0) / e_steps
        n_seg = wl.T // seg
        h2d = sum(t.numel() * t.element_size() for k in keys for t in hseg[k].values())
        h2d += n_seg * (hM0.numel() + hS0.numel()) * 4
        d2h = sum(t.numel() * t.element_size() for t in hy.values()) + n_seg * (hM0.numel() + hS0.numel()) * 4
        e2e = {"value": world * tokens / e_s, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e_s * 1e3,
               "note": "one host-buffer call per segment; the state is carried on the host"}

    peaks, peak_src = load_peaks()
    per_launch_ms = ms / alg["calls"]
    if alg["bound"] == "tensor":
        achieved = alg["flops"] / alg["calls"] / (per_launch_ms * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"])
        unit = "TFLOP/s"
    else:
        achieved = alg["bytes"] / alg["calls"] / (per_launch_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        unit = "GB/s"
    roof = {"bound": "hbm" if alg["bound"] == "hbm" else "tensor", "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak,
            "traffic": args.traffic if args.traffic is not None else
            (ncu_traffic(wl.name) if mem.path == nm.PATH_TC and (args.B, args.H, args.T) == (None, None, None) else None),
            "peak_source": peak_src + " (burst)",
            "kernel": "nm_forward (%s path)" % ("tcgen05" if mem.path == nm.PATH_TC else "fp32 FFMA"),
            "per_launch_ms": per_launch_ms,
            "frac_tensor": alg["flops"] / (per_launch_ms * alg["calls"] * 1e-3) / (float(peaks["bf16_tflops"]) * 1e12),
            "frac_hbm": alg["bytes"] / (per_launch_ms * alg["calls"] * 1e-3) / (float(peaks["hbm_gbs"]) * 1e9),
            "frac_tensor_sustained": (alg["flops"] / (per_launch_ms * alg["calls"] * 1e-3)
                                      / (float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * 1e12))}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        if seg != wl.T:
            x["q"], x["k"], x["v"] = (torch.cat([segs[k][s] for s in sorted(segs[k])], dim=2) for k in ("q", "k", "v"))
        cpu = time_oracle(wl, x)
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16" if mem.path == nm.PATH_TC else "f32", "data": "synthetic",
           "config": {"workload": wl.name, "memory": "linear" if wl.kind == 0 else "mlp2", "B": wl.B, "H": wl.H,
                      "T": wl.T, "d": wl.d, "hidden": wl.hidden, "chunk": wl.chunk,
                      "layers": wl.layers if wl.kind == 1 else None, "segment": wl.segment or None, "in_dtype": str(wl.dtype).replace("torch.", ""),
                      "parallelism": "dp%d" % world,
                      "l2": "flushed between timed steps (256 MB write, outside the step's events)"},
           "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
           "clocks": clocks.summary(), "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms), "max": max(step_ms)},
           "variants": variants}
    return out


# --------------------------------------------------------------------- reference arm (oracle)

def run_reference(args, rank, world):
    if rank != 0:
        return None
    from test_neural_memory_titans_b300 import workloads as W

    wl = workload(args)
    x = W.make_inputs(wl, "cpu", seed=1000 + args.workload)
    budget = args.cpu_budget if args.cpu_budget else max(1.0, 150.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        time_oracle(wl, x, budget_s=budget)
    runs = [time_oracle(wl, x, budget_s=budget) for _ in range(args.steps)]
    secs = sum(r["seconds"] for r in runs)
    toks = sum(r["tokens"] for r in runs)
    value = toks / secs
    cpu = {"value": value, "unit": "tokens/s", "cores": runs[0]["cores"], "kind": "oracle",
           "sample": runs[0]["sample"].rsplit(",", 1)[0] + " per step"}
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(runs),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": wl.name, "memory": "linear" if wl.kind == 0 else "mlp2", "B": wl.B, "H": wl.H,
                       "T": wl.T, "d": wl.d, "hidden": wl.hidden, "chunk": wl.chunk,
                       "layers": wl.layers if wl.kind == 1 else None},
            "cpu_baseline": cpu,
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=[0, 1, 2, 3, 4])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", type=int, default=0, help="0 auto, 1 fp32 FFMA, 2 tcgen05")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the dominant kernel from an ncu capture")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-variants", action="store_true", help="skip timing the Huber-loss and surprise forms")
    ap.add_argument("--layers", type=int, default=None,
                    help="MLP workloads: a memory of this many layers instead of 2 (fp32 FFMA kernel for > 2)")
    ap.add_argument("--cpu-budget", type=float, default=None,
                    help="seconds of oracle work per step of the reference arm (default: about 150 s in all)")
    ap.add_argument("--B", type=int, default=None, help="override the workload's batch (small profiling cases)")
    ap.add_argument("--H", type=int, default=None, help="override the workload's heads")
    ap.add_argument("--T", type=int, default=None, help="override the workload's tokens per unit")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            out = run_reference(args, rank, world)
        else:
            out = run_ours(args, rank, world, local_rank)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
