"""Benchmark of the neural-memory forward pass: one JSON line on stdout.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl ours|reference]

The headline workload is the largest configuration (2-layer MLP memory
128 -> 512 -> 128, B=2, H=16, T=131072, chunk 64).  A step is one full forward
over the workload (for the streamed workload, all of its segment calls,
carrying the state in place).  Inputs are resident in HBM before timing; L2 is
flushed (a 256 MB write) between timed steps, outside each step's CUDA-event
pair.  ``value`` is B*H*T tokens per second over all ranks (weak scaling:
every rank runs its own copy of the workload with its own seed, no collective
on the data path).  ``e2e`` measures the same metric through nm_forward_host
with pinned host buffers (host->device copies of the inputs and device->host
copies of y, M_T, S_T inside the timed region), with ``e2e.link`` the pinned
copy bandwidth of the same byte counts measured alone in the same run.

``--impl reference`` times the fp64 CPU oracle (the reference arm here) on
the host cores, on a bounded sample of the same workload.

Extra fields: ``roofline`` (the dominant kernel's algorithmic rate against the
measured peak, with ``traffic`` from an ncu capture while the captured kernel
source is unchanged), ``cpu_baseline`` (the oracle on a bounded sample),
``clocks`` (SM clock and throttle reasons sampled during the timed region),
``gpu_launches`` (this library's kernel launches in the timed region),
``variants`` (the same workload with the Huber loss, with the surprise
output and with the Memory-as-Gate output, a few steps each;
``--no-variants`` skips them) and ``per_workload``
(the other configurations timed in the same run, each with its own roofline
fraction and clocks; the streamed one adds the needle-retrieval cosine;
``--no-per-workload`` skips them).  ``--layers L`` runs an MLP workload with an
L-layer memory.

``--gpus N`` without a launcher starts N ranks itself (torch.distributed.run on
127.0.0.1); under a launcher, N must equal WORLD_SIZE.
"""
from __future__ import annotations

import argparse
import dataclasses
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
# The 128->512->128 figure is scaled from a capture of a 16384-token slice of the workload (token
# traffic x 8, plus the state read and written once per call); the streamed workload's is one
# 65536-token segment call, which is what one launch of its bench step processes; the 3-layer memory's
# from a 512-token capture (8 of the 64 chunks: its per-chunk traffic x 64, plus the state once); the
# backward sweep's from a 512-token capture (8 of the 256 chunks: x 32, its traffic being per chunk).
NCU_TRAFFIC = {
    "mlp_64x256_bf16_b4h8_t4096_c64": (("nm_tc_mlp.cu", "tc_common.cuh", "nm_internal.h"), "810ad16e5ee50003",
                                       62.45e6),
    "linear_d128_bf16_b8h16_t16384_c64": (("nm_tc_linear.cu", "tc_common.cuh", "nm_internal.h"), "54eb102664576f30",
                                          2.172e9),
    "mlp_128x512_bf16_b2h16_t131072_c64": (("nm_tc_mlp_wide.cu", "tc_common.cuh", "nm_internal.h"),
                                           "d70d351ebd9b6b93", 4.178e9),
    "linear_d64_bf16_b1h8_t2097152_c256_seg65536": (("nm_tc_linear64.cu", "tc_common.cuh", "nm_internal.h"),
                                                    "cd0494a3b25f3211", 254.6e6),
    "mlp_64x256_bf16_b4h8_t4096_c64_L3": (("nm_tc_deep.cu", "tc_common.cuh", "nm_internal.h"), "f471c769b7e276b8",
                                          8.442e9),
    # the backward pass's reverse sweep on tensor-core contractions (bwd_linear_kernel), one launch
    "linear_d128_bf16_b8h16_t16384_c64@backward_tc": (("nm_backward.cu", "tc_common.cuh", "nm_internal.h"),
                                                      "eaf54753b26663c9", 71.8e9),
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
DEFAULT_WORKLOAD = 3
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


def backward_algorithmic(wl) -> dict:
    """Algorithmic fp32 flops of one nm_backward call: the reverse sweep's
    products (linear: 13 d^2 + 5 b d multiply-adds per token; 2-layer MLP:
    29 d h + 3 b (d + h) per token) plus the checkpointing forward that
    records the chunk-start states (linear 3 d^2, MLP 11 d h per token)."""
    d, h, b = wl.d, wl.hidden, wl.chunk
    if wl.kind == 0:
        fma_tok = 13 * d * d + 5 * b * d + 3 * d * d
    else:
        fma_tok = 29 * d * h + 3 * b * (d + h) + 11 * d * h
    return {"flops": 2.0 * fma_tok * wl.tokens, "tokens": wl.tokens}


# the fp32 FFMA peak of a B300 from its unit counts and clock: 148 SMs x 128 fp32 lanes x 2 flops x 2032 MHz
FP32_PEAK_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


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
        if wl.kind != W.MLP2:
            raise SystemExit("--layers applies to the MLP workloads (1 and 3)")
        wl = dataclasses.replace(wl, layers=args.layers, name="%s_L%d" % (wl.name, args.layers))
    if args.B is None and args.H is None and args.T is None:
        return wl
    wl = wl.with_sizes(B=args.B, H=args.H, T=args.T)
    if wl.segment and (wl.T % wl.segment or wl.T < wl.segment):
        wl = wl.with_sizes(segment=0)
    return dataclasses.replace(wl, name="%s@B%dH%dT%d" % (wl.name, wl.B, wl.H, wl.T))


class Runner:
    """One workload on one device: inputs resident in HBM, a handle, and a
    ``step`` that runs one full forward (all segment calls of a streamed
    workload, the state carried in place)."""

    def __init__(self, wl, dev, stream, seed, path, layers):
        import test_neural_memory_titans_b300 as nm
        from test_neural_memory_titans_b300 import workloads as W

        self.wl, self.dev, self.stream = wl, dev, stream
        x = W.make_inputs(wl, dev, seed=seed)
        self.x = x
        self.mem = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk, in_dtype=wl.dtype, path=path,
                                   device=dev.index, layers=layers if wl.kind == nm.MLP2 else 0)
        self.y = torch.empty(x["q"].shape, dtype=wl.dtype, device=dev)
        self.M = torch.empty_like(x["M0"])
        self.S = torch.empty_like(x["S0"])
        self.seg = wl.segment if wl.segment else wl.T
        self.segs = {}
        if self.seg != wl.T:  # contiguous per-segment views prepared once, outside timing
            for key in ("q", "k", "v", "alpha", "eta", "beta"):
                self.segs[key] = {s0: x[key][:, :, s0:s0 + self.seg].contiguous() for s0 in range(0, wl.T, self.seg)}
            self.segs["y"] = {s0: torch.empty((wl.B, wl.H, self.seg, wl.d), dtype=wl.dtype, device=dev)
                              for s0 in range(0, wl.T, self.seg)}
            del x["q"], x["k"], x["v"]

    def step(self):
        x, wl, segs = self.x, self.wl, self.segs
        if self.seg == wl.T:
            self.mem.forward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"],
                             y=self.y, M_T=self.M, S_T=self.S, stream=self.stream)
        else:
            self.M.copy_(x["M0"])
            self.S.copy_(x["S0"])
            for s0 in range(0, wl.T, self.seg):
                self.mem.forward(segs["q"][s0], segs["k"][s0], segs["v"][s0], segs["alpha"][s0], segs["eta"][s0],
                                 segs["beta"][s0], self.M, self.S, y=segs["y"][s0], M_T=self.M, S_T=self.S,
                                 stream=self.stream)

    def check_status(self, when: str):
        import test_neural_memory_titans_b300 as nm
        st = self.mem.synchronize()
        if st != nm.NM_OK:
            raise RuntimeError("device status %s: %s" % (when, nm.status_string(st)))

    def close(self):
        self.mem.close()


def time_steps(step, steps, warmup, flush, stream, dev, world, local_rank, check, launches):
    """W untimed warm-up steps, then K steps each bracketed by CUDA events on
    the launching stream (L2 flushed before each, outside the events), with a
    barrier and a device synchronisation on both sides of the timed region
    and the SM clock sampled during it.  Returns the per-step times (ms), the
    clock summary and the library's kernel launches inside the timed region
    (``launches()`` reads the handle's counter)."""
    for _ in range(warmup):
        step()
    check("after warm-up")
    l0 = launches()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        for i in range(steps):
            flush.zero_()
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        torch.cuda.synchronize(dev)
    n_launch = launches() - l0
    if world > 1:
        torch.distributed.barrier()
    check("after timing")
    return [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)], clocks.summary(), n_launch


# Nominal dense tf32 / bf16 tensor rate of a B300 (1.1 / 2.25 PFLOP/s): the
# tf32 peak is the measured bf16 peak times this ratio.
TF32_PER_BF16 = 1.1 / 2.25


def roofline(wl, ms, path_tc, peaks, peak_src, traffic):
    """The dominant kernel's algorithmic rate per launch against the measured
    peak of its own operand type (the deeper-memory kernel's products are
    tf32, the other tensor-core kernels' bf16)."""
    alg = algorithmic(wl)
    per_launch_ms = ms / alg["calls"]
    tf32 = path_tc and wl.kind == 1 and wl.layers > 2  # the MLP memory
    if alg["bound"] == "tensor":
        achieved = alg["flops"] / alg["calls"] / (per_launch_ms * 1e-3) / 1e12
        peak = float(peaks["bf16_tflops"]) * (TF32_PER_BF16 if tf32 else 1.0)
        unit = "TFLOP/s"
    else:
        achieved = alg["bytes"] / alg["calls"] / (per_launch_ms * 1e-3) / 1e9
        peak = float(peaks["hbm_gbs"])
        unit = "GB/s"
    secs = per_launch_ms * alg["calls"] * 1e-3
    return {"bound": "hbm" if alg["bound"] == "hbm" else "tensor", "achieved": achieved, "peak": peak, "unit": unit,
            "frac": achieved / peak, "traffic": traffic,
            "peak_source": peak_src + (" (burst bf16 x 1.1/2.25, the nominal tf32 ratio)" if tf32 else " (burst)"),
            "kernel": "nm_forward (%s path)" % ("tcgen05" if path_tc else "fp32 FFMA"),
            "per_launch_ms": per_launch_ms,
            "algorithmic_flops_per_launch": alg["flops"] / alg["calls"],
            "algorithmic_bytes_per_launch": alg["bytes"] / alg["calls"],
            "frac_tensor": alg["flops"] / secs / (float(peaks["bf16_tflops"]) * 1e12),
            "frac_hbm": alg["bytes"] / secs / (float(peaks["hbm_gbs"]) * 1e9),
            "frac_tensor_sustained": (alg["flops"] / secs
                                      / (float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * 1e12))}


def needle_cosine(r) -> dict:
    """Retrieval diagnostic of the streamed workload: for every needle
    (position p, later probe p' whose query is k_p), the cosine between the
    memory's output y_{p'} and the stored value v_p, from the last step's y."""
    pos, probe = r.x["needles"]
    wl = r.wl
    y = torch.cat([r.segs["y"][s0] for s0 in sorted(r.segs["y"])], dim=2).reshape(wl.B * wl.H, wl.T, wl.d)
    v = torch.cat([r.segs["v"][s0] for s0 in sorted(r.segs["v"])], dim=2).reshape(wl.B * wl.H, wl.T, wl.d)
    pos = pos.reshape(wl.B * wl.H, -1)
    probe = probe.reshape(wl.B * wl.H, -1)
    rows = torch.arange(wl.B * wl.H, device=y.device).unsqueeze(1).expand_as(pos)
    yp = y[rows, probe].float()
    vp = v[rows, pos].float()
    cos = torch.nn.functional.cosine_similarity(yp, vp, dim=-1)
    # the same cosine against a value that was never stored at that key (a random other needle's value)
    perm = torch.roll(torch.arange(pos.shape[1], device=y.device), 1)
    cos0 = torch.nn.functional.cosine_similarity(yp, vp[:, perm], dim=-1)
    dist = (probe - pos).float()
    near = dist <= 256
    out = {"needles": int(cos.numel()), "mean_cosine": float(cos.mean()), "median_cosine": float(cos.median()),
           "mean_cosine_unrelated_value": float(cos0.mean()), "mean_probe_distance": float(dist.mean()),
           "near_needles": int(near.sum()),
           "note": "with the workload's forgetting (alpha ~ U(0, 0.05) per token) a stored value decays within "
                   "a few hundred tokens; near_* covers probes at most 256 tokens after their needle"}
    if int(near.sum()) > 0:
        out["near_mean_cosine"] = float(cos[near].mean())
        out["near_mean_cosine_unrelated_value"] = float(cos0[near].mean())
    return out


def link_bandwidth(dev, stream, h2d_bytes, d2h_bytes, reps=3):
    """Pinned host <-> device copy rate for the e2e byte counts, measured alone:
    one cudaMemcpyAsync per direction (torch copy_ from / to pinned memory),
    each direction alone and both at once on two streams."""
    hsrc = torch.empty(h2d_bytes, dtype=torch.uint8, pin_memory=True)
    ddst = torch.empty(h2d_bytes, dtype=torch.uint8, device=dev)
    dsrc = torch.empty(d2h_bytes, dtype=torch.uint8, device=dev)
    hdst = torch.empty(d2h_bytes, dtype=torch.uint8, pin_memory=True)
    s2 = torch.cuda.Stream(dev)

    def timed(fn):
        best = None
        for _ in range(reps):
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            fn()
            torch.cuda.synchronize(dev)
            dt = time.perf_counter() - t0
            best = dt if best is None else min(best, dt)
        return best

    def h2d():
        with torch.cuda.stream(stream):
            ddst.copy_(hsrc, non_blocking=True)

    def d2h():
        with torch.cuda.stream(s2):
            hdst.copy_(dsrc, non_blocking=True)

    def both():
        h2d()
        d2h()

    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d_gbs": h2d_bytes / t_in / 1e9, "d2h_gbs": d2h_bytes / t_out / 1e9,
            "both_directions_ms": t_both * 1e3, "h2d_ms": t_in * 1e3, "d2h_ms": t_out * 1e3,
            "note": "pinned copies of the e2e byte counts alone (best of %d); the e2e step cannot be faster "
                    "than both_directions_ms" % reps}


def run_backward(args, rank, world, local_rank):
    """Times nm_backward (gradients of <Gy, y> + <GM, M_T> + <GS, S_T> with
    respect to every input) on the selected workload: one step = one call
    over the whole workload (a streamed workload as one call over T)."""
    import test_neural_memory_titans_b300 as nm
    from test_neural_memory_titans_b300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    wl = workload(args)
    x = W.make_inputs(wl, dev, seed=1000 + args.workload + 100 * rank)
    g = torch.Generator(device=dev).manual_seed(7)
    Gy = torch.randn((wl.B, wl.H, wl.T, wl.d), generator=g, device=dev)
    GM = torch.randn((wl.B, wl.H, wl.P), generator=g, device=dev)
    GS = torch.randn((wl.B, wl.H, wl.P), generator=g, device=dev)
    mem = nm.NeuralMemory(wl.kind, wl.d, wl.hidden, wl.chunk, in_dtype=wl.dtype, device=local_rank, path=args.path)
    tc = mem.path == nm.PATH_TC  # the reverse sweep's contractions on the tensor cores (tf32)
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    def step():
        mem.backward(x["q"], x["k"], x["v"], x["alpha"], x["eta"], x["beta"], x["M0"], x["S0"], Gy, GM, GS,
                     stream=stream)

    def check(when):
        st = mem.synchronize()
        if st != nm.NM_OK:
            raise RuntimeError("device status %s: %s" % (when, nm.status_string(st)))

    step_ms, clocks, launches = time_steps(step, args.steps, args.warmup, flush, stream, dev, world, local_rank,
                                           check, lambda: mem.launches)
    ms = sum(step_ms) / len(step_ms)
    if world > 1:
        t = torch.tensor([ms], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        ms = float(t.item())
    alg = backward_algorithmic(wl)
    achieved = alg["flops"] / (ms * 1e-3) / 1e12
    mem.close()
    if tc:
        peaks, peak_src = load_peaks()
        peak = float(peaks["bf16_tflops"]) * TF32_PER_BF16
        sweep_bytes = ncu_traffic(wl.name + "@backward_tc")
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "traffic": sweep_bytes, "peak_source": peak_src + " (burst bf16 x 1.1/2.25, the nominal tf32 ratio)",
                "kernel": "nm_backward (checkpointing forward, tcgen05 for the linear d=128 memory, else fp32 FFMA; "
                          "reverse sweep with tcgen05 tf32 contractions)"}
        if sweep_bytes is not None:
            roof["traffic_kernel"] = "bwd_linear_kernel (the reverse sweep), DRAM bytes of one launch"
    else:
        roof = {"bound": "alu", "achieved": achieved, "peak": FP32_PEAK_TFLOPS, "unit": "TFLOP/s",
                "frac": achieved / FP32_PEAK_TFLOPS, "traffic": None,
                "peak_source": "derived: 148 SMs x 128 fp32 lanes x 2 flops x 2032 MHz",
                "kernel": "nm_backward (fp32 FFMA checkpointing forward + reverse sweep)"}
    return {"metric": "memory-layer backward tokens/sec (B*H*T/s)", "value": world * alg["tokens"] / (ms * 1e-3),
            "unit": "tokens/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "tf32" if tc else "f32",
            "data": "synthetic",
            "config": {"workload": wl.name, "pass": "backward", "B": wl.B, "H": wl.H, "T": wl.T, "d": wl.d,
                       "hidden": wl.hidden, "chunk": wl.chunk, "parallelism": "dp%d" % world,
                       "l2": "flushed between timed steps (256 MB write, outside the step's events)"},
            "roofline": roof, "gpu_launches": launches, "clocks": clocks,
            "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms), "max": max(step_ms)}}


def run_ours(args, rank, world, local_rank):
    import test_neural_memory_titans_b300 as nm
    from test_neural_memory_titans_b300 import workloads as W

    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    wl = workload(args)
    r = Runner(wl, dev, stream, 1000 + args.workload + 100 * rank, args.path, wl.layers)
    mem, x, y, M, S, seg = r.mem, r.x, r.y, r.M, r.S, r.seg
    flush = torch.empty(256 * 1024 * 1024, dtype=torch.uint8, device=dev)

    step_ms, clocks, launches = time_steps(r.step, args.steps, args.warmup, flush, stream, dev, world, local_rank,
                                           r.check_status, lambda: mem.launches)
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
        y_attn = torch.randn(y.shape, device=dev).to(y.dtype)
        v_g = time_calls(lambda: mem.forward_gated(*args8, y_attn, o=y, M_T=M, S_T=S, stream=stream), n_var)
        for m_ in (mem, mem_h):
            st = m_.synchronize()
            if st != nm.NM_OK:
                raise RuntimeError("device status after the variants: %s" % nm.status_string(st))
        mem_h.close()
        del sur, y_attn
        variants = {"huber_loss": {"ms_per_step": v_h, "value": world * tokens / (v_h * 1e-3), "delta": 0.1},
                    "surprise_output": {"ms_per_step": v_s, "value": world * tokens / (v_s * 1e-3)},
                    "mag_gate": {"ms_per_step": v_g, "value": world * tokens / (v_g * 1e-3)},
                    "steps": n_var,
                    "note": "nm_config.loss = NM_LOSS_HUBER; nm_forward_surprise; nm_forward_gated (o = sigmoid(y) * "
                            "y_attn written in place of y)"}

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
               "d2h_bytes_per_step": d2h, "ms_per_step": e_s * 1e3,
               "link": link_bandwidth(dev, stream, h2d, d2h)}
        del hx, hy, hM, hS, hargs
    elif not args.no_e2e:
        # streamed: one host-buffer call per segment, the state carried on the host from call to call
        segs = r.segs
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
               "note": "one host-buffer call per segment; the state is carried on the host",
               "link": link_bandwidth(dev, stream, h2d, d2h)}
        del hseg, hy

    peaks, peak_src = load_peaks()
    full_size = (args.B, args.H, args.T) == (None, None, None)
    traffic = args.traffic if args.traffic is not None else (
        ncu_traffic(wl.name) if mem.path == nm.PATH_TC and full_size else None)
    roof = roofline(wl, ms, mem.path == nm.PATH_TC, peaks, peak_src, traffic)
    needles = needle_cosine(r) if wl.keys == "needles" and seg != wl.T else None
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        if seg != wl.T:
            x["q"], x["k"], x["v"] = (torch.cat([r.segs[k][s] for s in sorted(r.segs[k])], dim=2)
                                      for k in ("q", "k", "v"))
        cpu = time_oracle(wl, x)
    out = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "bf16" if mem.path == nm.PATH_TC else "f32", "data": "synthetic",
           "config": {"workload": wl.name, "memory": "linear" if wl.kind == 0 else "mlp2", "B": wl.B, "H": wl.H,
                      "T": wl.T, "d": wl.d, "hidden": wl.hidden, "chunk": wl.chunk,
                      "layers": wl.layers if wl.kind == 1 else None, "segment": wl.segment or None,
                      "in_dtype": str(wl.dtype).replace("torch.", ""),
                      "parallelism": "dp%d" % world,
                      "l2": "flushed between timed steps (256 MB write, outside the step's events)"},
           "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
           "clocks": clocks, "step_ms": {"min": min(step_ms), "median": statistics.median(step_ms),
                                         "max": max(step_ms)},
           "variants": variants}
    if needles is not None:
        out["needle_retrieval"] = needles
    r.close()
    del r, x, y, M, S, mem

    # the other configurations, timed in the same run (full size, same timing rules), rank 0 alone at N = 1
    if world == 1 and not args.no_per_workload and full_size and args.layers is None:
        per = []
        for wid in sorted(W.WORKLOADS):
            if wid == args.workload:
                continue
            wl2 = W.WORKLOADS[wid]
            torch.cuda.empty_cache()
            r2 = Runner(wl2, dev, stream, 1000 + wid, args.path, wl2.layers)
            n_steps = max(3, min(args.steps, 200 if not wl2.segment else 10))
            ms2, clk2, n2 = time_steps(r2.step, n_steps, max(3, min(args.warmup, 5)), flush, stream, dev, 1,
                                       local_rank, r2.check_status, lambda: r2.mem.launches)
            m2 = sum(ms2) / len(ms2)
            entry = {"workload": wl2.name, "ms_per_step": m2, "value": wl2.tokens / (m2 * 1e-3), "unit": "tokens/s",
                     "steps": n_steps, "gpu_launches": n2,
                     "roofline": roofline(wl2, m2, r2.mem.path == nm.PATH_TC, peaks, peak_src,
                                          ncu_traffic(wl2.name) if r2.mem.path == nm.PATH_TC else None),
                     "clocks": clk2, "path": "tcgen05" if r2.mem.path == nm.PATH_TC else "fp32 FFMA"}
            if wl2.keys == "needles" and r2.seg != wl2.T:
                entry["needle_retrieval"] = needle_cosine(r2)
            per.append(entry)
            r2.close()
            del r2
        # the deeper memory (3 layers) on the 64 -> 256 -> 64 workload's shape and inputs
        wl3 = dataclasses.replace(W.WORKLOADS[1], layers=3, name=W.WORKLOADS[1].name + "_L3")
        torch.cuda.empty_cache()
        r3 = Runner(wl3, dev, stream, 1001, args.path, 3)
        n3 = max(3, min(args.steps, 20))
        ms3, clk3, l3 = time_steps(r3.step, n3, max(3, min(args.warmup, 5)), flush, stream, dev, 1, local_rank,
                                   r3.check_status, lambda: r3.mem.launches)
        m3 = sum(ms3) / len(ms3)
        per.append({"workload": wl3.name, "ms_per_step": m3, "value": wl3.tokens / (m3 * 1e-3), "unit": "tokens/s",
                    "steps": n3, "gpu_launches": l3,
                    "roofline": roofline(wl3, m3, r3.mem.path == nm.PATH_TC, peaks, peak_src,
                                         ncu_traffic(wl3.name) if r3.mem.path == nm.PATH_TC else None),
                    "clocks": clk3, "path": "tcgen05 tf32" if r3.mem.path == nm.PATH_TC else "fp32 FFMA"})
        r3.close()
        del r3
        out["per_workload"] = per
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
    ap.add_argument("--no-per-workload", action="store_true", help="skip timing the other configurations")
    ap.add_argument("--backward", action="store_true",
                    help="time nm_backward (gradients of every input) on the workload instead of the forward")
    ap.add_argument("--layers", type=int, default=None,
                    help="MLP workloads: a memory of this many layers instead of 2")
    ap.add_argument("--cpu-budget", type=float, default=None,
                    help="seconds of oracle work per step of the reference arm (default: about 150 s in all)")
    ap.add_argument("--B", type=int, default=None, help="override the workload's batch (small profiling cases)")
    ap.add_argument("--H", type=int, default=None, help="override the workload's heads")
    ap.add_argument("--T", type=int, default=None, help="override the workload's tokens per unit")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3

    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        # no launcher: start one rank per GPU on this node and wait for them
        import socket
        import subprocess
        with socket.socket() as so:
            so.bind(("127.0.0.1", 0))
            port = so.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", str(args.gpus),
               "--master-addr", "127.0.0.1", "--master-port", str(port), os.path.abspath(__file__)] + sys.argv[1:]
        raise SystemExit(subprocess.call(cmd))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if world != args.gpus:
        raise SystemExit("bench.py: --gpus %d but the launcher started %d rank(s) (WORLD_SIZE)" % (args.gpus, world))
    if world > 1:
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            out = run_reference(args, rank, world)
        elif args.backward:
            out = run_backward(args, rank, world, local_rank)
        else:
            out = run_ours(args, rank, world, local_rank)
        if rank == 0 and out is not None:
            print(json.dumps(out), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
