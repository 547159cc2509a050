"""Benchmark of the deterministic fused linear-logp operator on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline (one JSON line on rank 0): the fused forward on the Qwen3-8B-shaped LM head,
T=4096 rows, H=4096, V=151936 bf16, tau=0.7, logp + LSE + entropy, in tokens/s, with
the tensor-core roofline of the fused GEMM kernel. The other hot-path rows are timed
alongside in "paths": the tiny configuration (T=64, H=256, V=1000), the headline's shapes
at micro-batch sizes (T=128, 512 and 1024), logits reuse
(T=8192 x 151936 bf16 logits, HBM-bound) and the gradient with respect to those logits,
compact top-p replay (T=8192, 4 shards) from x.W and from the logits, and the
vocabulary-sharded forward + backward (T=4096, V=151936 padded to 152064 in 4 shards,
bias). Each leg carries its own clock record and roofline, and (unless --no-cpu-baseline)
the fp64 oracle timed on a bounded row sample of the same workload with the GPU's largest
deviation from it on those rows.

Every input is synthetic and seeded; the weights and logits are larger than the
129 MB L2, so no flush is needed between timed steps. --impl reference times the fp64
CPU oracle on the host cores on a bounded row sample of the same workload (under
torchrun, rank 0 alone runs it).

One GPU only: the benchmark times the one-GPU hot path. The GPU arm refuses a run with
more than one rank (or --gpus > 1) before it touches a GPU; the multi-GPU vocabulary-parallel
path (lm_head_linear_tcgen05_gb300.vocab_parallel) is tested but not timed here.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused linear-logp tokens/s (T×4096→151936 bf16) and % of dense bf16 tensor peak"
UNIT = "tokens/s"
T_FWD, H, V = 4096, 4096, 151936
TAU = 0.7
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
CSRC = os.path.join(ROOT, "lm_head_linear_tcgen05_gb300", "csrc")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "traffic.json")


# ----------------------------------------------------------------- utilities

def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# device sources each timed kernel is compiled from
KERNEL_SOURCES = {
    "fused_forward": ("lp_fused_forward.cu", "lp_tcgemm.cuh", "lp_device.cuh"),
    "stream_logits": ("lp_stream.cu", "lp_device.cuh", "lp_f32x2.cuh"),
    "replay": ("lp_replay.cu", "lp_device.cuh"),
    "logits_backward": ("lp_logits_backward.cu", "lp_device.cuh", "lp_f32x2.cuh"),
}


def source_hash(kernel: str) -> str:
    """Hash of a kernel's sources: a stored ncu traffic figure is valid only for this hash."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(CSRC, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def stored_traffic(kernel: str):
    """DRAM bytes per launch from profiles/traffic.json, or None if the kernel changed since."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
        e = d.get(kernel)
        if e and e.get("source_hash") == source_hash(kernel):
            return float(e["bytes_per_launch"])
    except Exception:
        pass
    return None


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (read-only queries) every
    `period` seconds by a background thread while the timed region runs. Raises on entry if
    NVML cannot be used; ClockSampler (nvidia-smi) is the fallback."""
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown"}

    def __init__(self, device, period: float = 0.005):
        import ctypes
        import threading
        import torch
        self.ct, self.threading, self.period = ctypes, threading, period
        lib = None
        for name in ("libnvidia-ml.so.1", "libnvidia-ml.so"):
            try:
                lib = ctypes.CDLL(name)
                break
            except OSError:
                continue
        if lib is None or lib.nvmlInit_v2() != 0:
            raise RuntimeError("NVML unavailable")
        self.nvml = lib
        props = torch.cuda.get_device_properties(device)
        h = ctypes.c_void_p()
        bus = getattr(props, "pci_bus_id", None)
        ok = False
        if bus is not None:
            busid = f"{getattr(props, 'pci_domain_id', 0):08X}:{bus:02X}:{getattr(props, 'pci_device_id', 0):02X}.0"
            ok = lib.nvmlDeviceGetHandleByPciBusId_v2(busid.encode(), ctypes.byref(h)) == 0
        if not ok and lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(torch.cuda.current_device()),
                                                         ctypes.byref(h)) != 0:
            raise RuntimeError("NVML device handle unavailable")
        self.h = h
        self.get_reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            getattr(lib, "nvmlDeviceGetCurrentClocksThrottleReasons")
        self.samples, self.reason_bits = [], 0

    def _read(self):
        c = self.ct.c_uint()
        r = self.ct.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, self.ct.byref(c)) == 0:  # 1: SM clock
            self.samples.append(c.value)
        if self.get_reasons(self.h, self.ct.byref(r)) == 0:
            self.reason_bits |= r.value

    def _loop(self):
        while not self.stop.is_set():
            self._read()
            self.stop.wait(self.period)

    def __enter__(self):
        self.stop = self.threading.Event()
        self.thread = self.threading.Thread(target=self._loop, daemon=True)
        self.thread.start()
        return self

    def __exit__(self, *exc):
        self.stop.set()
        self.thread.join(timeout=5)

    def summary(self):
        if not self.samples:
            return None
        mx = self.ct.c_uint()
        max_mhz = float(mx.value) if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, self.ct.byref(mx)) == 0 else None
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": max_mhz,
                "sm_min_mhz": float(min(self.samples)),
                "reasons": sorted(n for b, n in self.REASONS.items() if self.reason_bits & b),
                "samples": len(self.samples), "source": f"NVML, every {self.period * 1e3:.0f} ms of the timed region"}


def clock_sampler(device):
    try:
        return NvmlClockSampler(device)
    except Exception:
        return ClockSampler(torch_index(device))


def torch_index(device) -> int:
    return device.index if getattr(device, "index", None) is not None else 0


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.FIELDS,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or self.path is None:
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        try:
            with open(self.path) as f:
                for line in f:
                    c = [x.strip() for x in line.split(",")]
                    if len(c) < 9:
                        continue
                    try:
                        sm.append(float(c[1]))
                        mx.append(float(c[2]))
                    except ValueError:
                        continue
                    for n, v in zip(names, c[5:9]):
                        if v.lower() == "active":
                            reasons.add(n)
            os.unlink(self.path)
        except Exception:
            return None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


ONE_GPU_ONLY = ("bench.py times the one-GPU hot path only (the vocabulary-parallel multi-GPU path is tested, "
                "not timed); run it with one rank and --gpus 1")


def refuse_multi_gpu(args, world: int) -> bool:
    """The GPU arm runs on one GPU only: with more than one rank (or --gpus > 1) it prints one
    JSON line saying why and returns True, before any GPU or process-group work."""
    if args.impl == "ours" and (world > 1 or args.gpus > 1):
        if int(os.environ.get("RANK", "0")) == 0:
            print(json.dumps({"impl": "ours", "n_gpus": max(world, args.gpus), "error": ONE_GPU_ONLY}), flush=True)
        return True
    return False


def time_steps(fn, steps, warmup, stream, sampler=None):
    """Average ms per step over `steps` calls of fn(), CUDA events on `stream`; `sampler`
    (a context manager) runs around the timed calls only, after the warm-up."""
    import contextlib
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with sampler if sampler is not None else contextlib.nullcontext():
        start.record(stream)
        for _ in range(steps):
            fn()
        end.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


def time_graph(fn, steps, warmup, stream, sampler=None):
    """Average ms per call of fn() replayed from one CUDA graph holding `steps` calls, for
    kernels shorter than the binding's per-call host overhead (events on `stream`)."""
    import contextlib
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(steps):
            fn()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    with sampler if sampler is not None else contextlib.nullcontext():
        start.record(stream)
        g.replay()
        end.record(stream)
        torch.cuda.synchronize()
    return start.elapsed_time(end) / steps


# -------------------------------------------------------------- our GPU arm

def run_ours(args):
    import numpy as np
    import torch

    import lm_head_linear_tcgen05_gb300 as lp
    import synth

    from lm_head_linear_tcgen05_gb300 import _build
    _build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    if not lp.lp_device_supported():
        raise RuntimeError("this GPU cannot run liblp.so (sm_103a build)")
    stream = torch.cuda.current_stream(dev)
    peaks, peak_src = load_peaks()

    if args.skip_headline:
        paths = time_other_paths(args, lp, synth, dev, stream, peaks)
        print(json.dumps({"paths": paths}), flush=True)
        return

    # ---- headline: fused forward, T=4096, H=4096, V=151936, tau=0.7, no bias
    T_FWD, V = args.rows, args.vocab
    part = synth.even_partition(V, 1)
    P = lp.VocabPartition(part.vocab_real, part.vocab_padded, part.ranges)
    X, W, _, y = synth.device_forward_inputs(T_FWD, H, part, TAU, dev, seed=0)
    ws = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD, T_FWD, H, P), dtype=torch.uint8, device=dev)
    step = lambda: lp.lp_forward(X, W, None, P, y, TAU, workspace=ws)
    clk = clock_sampler(dev)
    ms = time_steps(step, args.steps, args.warmup, stream, sampler=clk)
    if lp.lp_get_device_error() != 0:
        raise RuntimeError("device error during the timed forward")
    flops = 2.0 * T_FWD * H * V
    tflops = flops / (ms * 1e-3) / 1e12
    value = T_FWD / (ms * 1e-3)

    # ---- end to end through the C entry point lp_forward_host: pinned host X, y in; host logp,
    # lse, entropy out. The call copies the inputs in, runs the forward and copies the outputs
    # back on the stream; the binding synchronises before returning, so each step is timed on
    # the host clock.
    hX = torch.empty((T_FWD, H), dtype=torch.bfloat16, pin_memory=True)
    hX.copy_(X.cpu())
    hy = y.cpu().pin_memory()
    ws_host = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD_HOST, T_FWD, H, P), dtype=torch.uint8, device=dev)
    host_out = {k: torch.empty(T_FWD, dtype=torch.float32, pin_memory=True) for k in ("logp", "lse", "entropy")}
    for _ in range(args.warmup):
        lp.lp_forward_host(hX, W, None, P, hy, TAU, workspace=ws_host, out=host_out)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        lp.lp_forward_host(hX, W, None, P, hy, TAU, workspace=ws_host, out=host_out)
    ms_e2e = (time.perf_counter() - t0) * 1e3 / args.steps
    ref = lp.lp_forward(X, W, None, P, y, TAU, workspace=ws)
    if not torch.equal(host_out["logp"], ref["logp"].cpu()):
        raise RuntimeError("host-staged forward differs from the device forward")
    del hX, ws_host
    # ---- bitwise checks on the timed workload (outside the timed region): a repeat of the
    # call, and the same rows as 8 batches of T/8, give the same bits
    base = lp.lp_forward(X, W, None, P, y, TAU, workspace=ws)
    again = lp.lp_forward(X, W, None, P, y, TAU, workspace=ws)
    bit_repeat = all(torch.equal(base[k], again[k]) for k in ("logp", "lse", "entropy"))
    chunk = max(1, T_FWD // 8)
    parts = [lp.lp_forward(X[s0:s0 + chunk].contiguous(), W, None, P, y[s0:s0 + chunk].contiguous(), TAU)
             for s0 in range(0, T_FWD, chunk)]
    bit_batch = all(torch.equal(torch.cat([q[k] for q in parts]), base[k]) for k in ("logp", "lse", "entropy"))
    del again, parts
    paths = {}
    if not args.headline_only:
        paths = time_other_paths(args, lp, synth, dev, stream, peaks)
    # ---- the headline call held for about half a second, long enough for the power cap to
    # set the clock: the figure to hold against the sustained tensor peak. Measured last, so
    # that it does not change the state the other legs start from.
    sus_steps = max(args.steps, args.sustained_steps)
    clk_sus = clock_sampler(dev)
    ms_sus = time_steps(step, sus_steps, 0, stream, sampler=clk_sus)

    traffic = stored_traffic("fused_forward")
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"Qwen3-8B-shaped LM-head fused forward, T={T_FWD} rows, H={H}, V={V}, "
                               "tau=0.7, no bias, logp+LSE+entropy",
                   "T": T_FWD, "H": H, "V": V, "tau": TAU, "shards": 1,
                   "l2": "inputs larger than L2 (W 1.245 GB > 129 MB); no flush",
                   "parallelism": "one GPU"},
        "clocks": clk.summary(),
        "e2e": {"value": T_FWD / (ms_e2e * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": T_FWD * H * 2 + T_FWD * 4, "d2h_bytes_per_step": 3 * T_FWD * 4,
                "ms_per_step": ms_e2e, "timed": "host clock around the C entry point lp_forward_host (H2D, "
                                                  "forward, D2H, synchronised every step)"},
        "gpu_launches": 2 * args.steps,  # per timed lp_forward call: projection GEMM + merge
        "roofline": {"bound": "tensor", "achieved": tflops, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                     "frac": tflops / peaks["bf16_tflops"], "traffic": traffic,
                     "peak_source": f"{peak_src} bf16 dense burst",
                     "timed": "whole lp_forward call (fused GEMM kernel + row merge kernel)",
                     "sustained": {"steps": sus_steps, "ms_per_step": ms_sus,
                                   "achieved": flops / (ms_sus * 1e-3) / 1e12,
                                   "peak": peaks["bf16_tflops_sustained"],
                                   "frac": flops / (ms_sus * 1e-3) / 1e12 / peaks["bf16_tflops_sustained"],
                                   "clocks": clk_sus.summary()}},
        "paths": paths,
        "bitwise": {"repeat": bit_repeat, f"1x{T_FWD}_vs_{-(-T_FWD // chunk)}x{chunk}": bit_batch},
        "build": lp.build_info(),
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"], line["parity"] = cpu_baseline_forward(X, W, y, base, rows=1536)
    print(json.dumps(line), flush=True)


def _host_bits(t):
    """A CUDA bf16 tensor's bits as a host uint16 array (oracle input)."""
    import numpy as np
    import torch
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _sample_rows(T: int, n: int):
    import numpy as np
    return np.unique(np.linspace(0, T - 1, min(n, T)).round().astype(np.int64))


def _oracle_leg(run, rows: int, sample: str, compare):
    """Time `run()` (an oracle call on a bounded row sample) on the host cores; compare(result)
    returns the GPU outputs' largest deviations on those rows."""
    t0 = time.perf_counter()
    res = run()
    dt = time.perf_counter() - t0
    return {"value": rows / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{sample}; {dt:.1f} s", "parity": compare(res)}


def _maxdev(gpu, ref):
    import numpy as np
    a = np.asarray(gpu, dtype=np.float64)
    b = np.asarray(ref, dtype=np.float64)
    both = np.isinf(a) & np.isinf(b) & (np.sign(a) == np.sign(b))
    return float(np.max(np.abs(np.where(both, 0.0, a) - np.where(both, 0.0, b)))) if a.size else 0.0


def _relfro(gpu, ref):
    import numpy as np
    a = np.asarray(gpu, dtype=np.float64)
    b = np.asarray(ref, dtype=np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))


def time_other_paths(args, lp, synth, dev, stream, peaks):
    """The other hot-path rows, each on its own workload (vocabulary args.vocab), each timed
    with its own clock record."""
    import torch
    out = {}
    Vp = args.vocab
    TP = args.path_rows  # rows of the logits and replay workloads

    def timed(fn, steps):
        clk = clock_sampler(dev)
        ms = time_steps(fn, steps, args.warmup, stream, sampler=clk)
        return ms, clk.summary()

    def hbm_roofline(nbytes, ms, kernel, **extra):
        gbs = nbytes / (ms * 1e-3) / 1e9
        r = {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
             "frac": gbs / peaks["hbm_gbs"], "algorithmic_bytes": nbytes}
        if kernel is not None:
            r["traffic"] = stored_traffic(kernel)
        r.update(extra)
        return r

    wanted = set(args.paths.split(","))
    oracle_on = not args.no_cpu_baseline
    tau32 = float(__import__("numpy").float32(TAU))
    if oracle_on:
        import oracle
    if "tiny" in wanted:
        # the tiny configuration (T=64, H=256, V=1000, tau 1): launch-bound, timed from a graph
        pt = synth.even_partition(1000, 1)
        Pt = lp.VocabPartition(pt.vocab_real, pt.vocab_padded, pt.ranges)
        inp = synth.forward_inputs(64, 256, pt, tau=1.0, seed=0)
        import numpy as np
        import torch
        Xt = torch.from_numpy(inp.X.view(np.int16)).to(dev).view(torch.bfloat16)
        Wt = [torch.from_numpy(inp.W[0].view(np.int16)).to(dev).view(torch.bfloat16)]
        yt = torch.from_numpy(inp.y).to(dev)
        clk_t = clock_sampler(dev)
        ms = time_graph(lambda: lp.lp_forward(Xt, Wt, None, Pt, yt, inp.tau), args.steps, args.warmup, stream,
                        sampler=clk_t)
        leg = {"workload": "T=64, H=256, V=1000, one shard, no bias, tau=1.0", "ms": ms,
               "tokens_per_s": 64 / (ms * 1e-3), "steps": args.steps, "clocks": clk_t.summary(),
               "timed": "one CUDA graph of the timed calls (a call is launch-bound)"}
        if oracle_on:
            got = lp.lp_forward(Xt, Wt, None, Pt, yt, inp.tau)
            leg["cpu_baseline"] = _oracle_leg(
                lambda: oracle.forward(inp.X, inp.W, None, pt, inp.y, inp.tau), 64, "all 64 rows, fp64 numpy oracle",
                lambda r: {"max_abs_dlogp": _maxdev(got["logp"].cpu(), r.logp),
                           "max_abs_dentropy": _maxdev(got["entropy"].cpu(), r.entropy)})
        out["tiny"] = leg
    if "batches" in wanted:
        # the headline workload at micro-batch sizes (T = 128, 512, 1024 rows of the same X, W):
        # one read of W (1.245 GB) is spread over fewer rows, so the call is bound by the tensor
        # pipe or by streaming W, whichever is slower (W at T = 128, a single row block); both
        # fractions are reported
        pb = synth.even_partition(Vp, 1)
        Pb = lp.VocabPartition(pb.vocab_real, pb.vocab_padded, pb.ranges)
        Xb, Wb, _, yb = synth.device_forward_inputs(1024, H, pb, TAU, dev, seed=6)
        w_bytes = float(sum(w.numel() * 2 for w in Wb))
        legs = {}
        for T in (128, 512, 1024):
            Xt, yt = Xb[:T].contiguous(), yb[:T].contiguous()
            wst = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD, T, H, Pb), dtype=torch.uint8, device=dev)
            ms, clk = timed(lambda: lp.lp_forward(Xt, Wb, None, Pb, yt, TAU, workspace=wst), args.steps)
            tf = 2.0 * T * H * Vp / (ms * 1e-3) / 1e12
            w_gbs = (w_bytes + Xt.numel() * 2) / (ms * 1e-3) / 1e9
            leg = {"ms": ms, "tokens_per_s": T / (ms * 1e-3), "steps": args.steps, "clocks": clk,
                   "roofline": {"bound": "tensor", "achieved": tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                                "frac": tf / peaks["bf16_tflops"],
                                "w_stream_gbs": w_gbs, "w_stream_frac": w_gbs / peaks["hbm_gbs"]}}
            if oracle_on:
                import numpy as np
                got = lp.lp_forward(Xt, Wb, None, Pb, yt, TAU, workspace=wst)
                idx = _sample_rows(T, 64)
                idx_d = torch.from_numpy(idx).to(dev)
                Xh, Wh, yh = _host_bits(Xt[idx_d]), [_host_bits(w) for w in Wb], yt[idx_d].cpu().numpy()
                leg["cpu_baseline"] = _oracle_leg(
                    lambda: oracle.forward(Xh, Wh, None, pb, yh, tau32), len(idx),
                    f"{len(idx)} of {T} rows (full H, V), fp64 numpy oracle",
                    lambda r: {"max_abs_dlogp": _maxdev(got["logp"][idx_d].cpu(), r.logp),
                               "max_abs_dentropy": _maxdev(got["entropy"][idx_d].cpu(), r.entropy)})
                del Wh
            legs[f"T{T}"] = leg
        out["fused_forward_batches"] = {
            "workload": f"T=128, 512 and 1024 rows, H=4096, V={Vp}, tau=0.7, no bias (the headline's shapes "
                        "at micro-batch sizes)", **legs}
        del Xb, Wb
        torch.cuda.empty_cache()
    if wanted & {"logits", "replay"}:
        part = synth.even_partition(Vp, 1)
        P = lp.VocabPartition(part.vocab_real, part.vocab_padded, part.ranges)
        L, y = synth.device_logits(TP, part, dev, seed=4)
        part4 = synth.even_partition(Vp, 4)
        P4 = lp.VocabPartition(part4.vocab_real, part4.vocab_padded, part4.ranges)
        ids, yr = synth.replay_ids(TP, part4, seed=5)
        ids_d = torch.from_numpy(ids).to(dev)
        yr_d = torch.from_numpy(yr).to(dev)
        uniq = sum(len(set(r[r >= 0].tolist())) for r in ids)
        if "logits" in wanted:
            # logits reuse: T=TP x V bf16 logits
            ms, clk = timed(lambda: lp.lp_forward_from_logits(L, P, y, TAU), args.steps)
            nbytes = TP * Vp * 2
            out["logits_reuse"] = {
                "workload": f"T={TP}, V={Vp} bf16 logits N(0,9), 1% peaked, tau=0.7",
                "tokens_per_s": TP / (ms * 1e-3), "ms": ms, "steps": args.steps, "clocks": clk,
                "roofline": hbm_roofline(nbytes, ms, "stream_logits",
                                         frac_of_8tbs=nbytes / (ms * 1e-3) / 1e9 / 8000.0)}
            fl = lp.lp_forward_from_logits(L, P, y, TAU)
            if oracle_on:
                idx = _sample_rows(TP, 1024)
                idx_d = torch.from_numpy(idx).to(dev)
                Lb = [_host_bits(L[0][idx_d])]
                ys = y[idx_d].cpu().numpy()
                out["logits_reuse"]["cpu_baseline"] = _oracle_leg(
                    lambda: oracle.forward_from_logits(Lb, part, ys, tau32), len(idx),
                    f"{len(idx)} of {TP} rows (full V), fp64 numpy oracle",
                    lambda r: {"max_abs_dlogp": _maxdev(fl["logp"][idx_d].cpu(), r.logp),
                               "max_abs_dlse": _maxdev(fl["lse"][idx_d].cpu(), r.lse),
                               "max_abs_dentropy": _maxdev(fl["entropy"][idx_d].cpu(), r.entropy)})
            # its backward: the gradient with respect to those logits, bf16, out of place
            gl = torch.randn(TP, generator=torch.Generator(device=dev).manual_seed(4), device=dev)
            dL = [torch.empty_like(L[0])]
            ms, clk = timed(lambda: lp.lp_backward_from_logits(L, P, y, TAU, fl["lse"], gl, entropy=fl["entropy"],
                                                               grad_entropy=gl, out=dL), args.steps)
            out["logits_backward"] = {
                "workload": f"gradient w.r.t. the T={TP} x V={Vp} logits above (logp + entropy terms), bf16 out",
                "tokens_per_s": TP / (ms * 1e-3), "ms": ms, "steps": args.steps, "clocks": clk,
                "roofline": hbm_roofline(2 * TP * Vp * 2, ms, "logits_backward")}
            if oracle_on:
                idx = _sample_rows(TP, 256)
                idx_d = torch.from_numpy(idx).to(dev)
                Lb = [_host_bits(L[0][idx_d])]
                ys, gs = y[idx_d].cpu().numpy(), gl[idx_d].cpu().numpy()
                got = dL[0][idx_d].float().cpu().numpy()
                out["logits_backward"]["cpu_baseline"] = _oracle_leg(
                    lambda: oracle.backward_from_logits(Lb, part, ys, tau32, gs, h=gs), len(idx),
                    f"{len(idx)} of {TP} rows (full V), fp64 numpy oracle",
                    lambda r: {"rel_fro_dlogits": _relfro(got, r[0])})
            del dL, fl
        if "replay" in wanted:
            # the compact replay scored from the reused logits above: per row its 64 id slots
            # and one logit per distinct id, each logit alone in a 32-byte DRAM sector
            L4 = [L[0][:, s:e] for s, e in part4.ranges]
            clk_g = clock_sampler(dev)
            ms = time_graph(lambda: lp.lp_top_p_replay_from_logits(L4, P4, ids_d, yr_d, TAU), args.steps,
                            args.warmup, stream, sampler=clk_g)
            clk = clk_g.summary()
            sector_bytes = TP * (64 * 4 + 4) + uniq * 32
            if oracle_on:
                got = lp.lp_top_p_replay_from_logits(L4, P4, ids_d, yr_d, TAU)
                idx = _sample_rows(TP, TP)
                idx_d = torch.from_numpy(idx).to(dev)
                L4b = [_host_bits(t[idx_d]) for t in L4]
                replay_from_logits_cpu = _oracle_leg(
                    lambda: oracle.top_p_replay_from_logits(L4b, part4, ids[idx], yr[idx], tau32), len(idx),
                    f"{len(idx)} of {TP} rows, fp64 oracle (a Python loop over each row's ids)",
                    lambda r: {"max_abs_dlogp": _maxdev(got["logp"][idx_d].cpu(), r.logp),
                               "max_abs_dlse": _maxdev(got["lse"][idx_d].cpu(), r.lse)})
            out["top_p_replay_from_logits"] = {
                "workload": f"T={TP} rows of the logits above in 4 shards, 1-64 ids/row",
                "tokens_per_s": TP / (ms * 1e-3), "ms": ms, "steps": args.steps, "clocks": clk,
                "timed": "one CUDA graph of the timed calls (the kernel is shorter than the binding's per-call "
                         "host overhead)",
                "ids_scored": uniq,
                "roofline": hbm_roofline(sector_bytes, ms, None,
                                         note="bytes counted at DRAM sector granularity (32 B per gathered logit, "
                                              "plus the id slots and targets); bound by the rate of scattered sector "
                                              "reads and each row's dependent steps (ids, sort, gather, fold), not "
                                              "by bandwidth")}
            if oracle_on:
                out["top_p_replay_from_logits"]["cpu_baseline"] = replay_from_logits_cpu
        del L
        torch.cuda.empty_cache()
        if "replay" in wanted:
            # compact top-p replay: T=TP, 4 shards, ids as the nucleus recipe
            X, W, _, _ = synth.device_forward_inputs(TP, H, part4, TAU, dev, seed=5)
            ms, clk = timed(lambda: lp.lp_top_p_replay(X, W, None, P4, ids_d, yr_d, TAU), args.steps)
            distinct = len(set(ids[ids >= 0].tolist()))
            gathered = TP * H * 2 + uniq * H * 2
            distinct_b = TP * H * 2 + distinct * H * 2
            out["top_p_replay"] = {
                "workload": f"T={TP}, H=4096, V={Vp} in 4 shards, 1-64 ids/row (+10% dups), tau=0.7",
                "tokens_per_s": TP / (ms * 1e-3), "ms": ms, "steps": args.steps, "clocks": clk,
                "gathered_bytes": gathered, "distinct_bytes": distinct_b,
                "roofline": hbm_roofline(gathered, ms, "replay",
                                         frac_distinct=distinct_b / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"])}
            if oracle_on:
                got = lp.lp_top_p_replay(X, W, None, P4, ids_d, yr_d, TAU)
                idx = _sample_rows(TP, 4096)
                idx_d = torch.from_numpy(idx).to(dev)
                Xb, Wb = _host_bits(X), [_host_bits(w) for w in W]
                out["top_p_replay"]["cpu_baseline"] = _oracle_leg(
                    lambda: oracle.top_p_replay(Xb, Wb, None, part4, ids, yr, tau32, rows=idx), len(idx),
                    f"{len(idx)} of {TP} rows (full H), fp64 oracle (a Python loop over each row's ids)",
                    lambda r: {"max_abs_dlogp": _maxdev(got["logp"][idx_d].cpu(), r.logp),
                               "max_abs_dlse": _maxdev(got["lse"][idx_d].cpu(), r.lse)})
                del Xb, Wb
            del X, W
            torch.cuda.empty_cache()

    if "backward" in wanted:
        # vocabulary-sharded forward + backward: padded to a multiple of 4 x 64, 4 shards, bias
        Vpad = (Vp + 4 * 64 * 2 - 1) // (4 * 64 * 2) * (4 * 64 * 2) if Vp != V else 152064
        w4 = Vpad // 4
        part3 = synth.ranges_partition(Vp, Vpad, [0, w4, 2 * w4, 3 * w4, Vpad])
        P3 = lp.VocabPartition(part3.vocab_real, part3.vocab_padded, part3.ranges)
        X, W, b, y = synth.device_forward_inputs(T_FWD, H, part3, TAU, dev, seed=3, bias_std=0.01)
        g = torch.randn(T_FWD, generator=torch.Generator(device=dev).manual_seed(3), device=dev)
        wsf = torch.empty(lp.lp_workspace_size(lp.LP_OP_FORWARD, T_FWD, H, P3), dtype=torch.uint8, device=dev)
        wsb = torch.empty(lp.lp_workspace_size(lp.LP_OP_BACKWARD, T_FWD, H, P3), dtype=torch.uint8, device=dev)
        fwd = lp.lp_forward(X, W, b, P3, y, TAU, workspace=wsf)
        ms_f, clk_f = timed(lambda: lp.lp_forward(X, W, b, P3, y, TAU, workspace=wsf), args.steps)
        bwd = lambda: lp.lp_backward(X, W, b, P3, y, TAU, fwd["lse"], g, workspace=wsb)
        # a short burst first (5 calls, ~45 ms: the clock has not yet met the power cap), then
        # the 20-call figure, long enough for the power cap to set the clock
        ms_bb, clk_bb = timed(bwd, 5)
        bsteps = max(20, args.steps)
        ms_b, clk_b = timed(bwd, bsteps)
        f_fl = 2.0 * T_FWD * H * Vp
        b_tf = 3 * f_fl / (ms_b * 1e-3) / 1e12
        out["sharded_fwd_bwd"] = {
            "workload": f"T=4096, H=4096, V={Vp} padded to {Vpad}, 4 shards, bias, tau=0.7",
            "fwd_tokens_per_s": T_FWD / (ms_f * 1e-3), "fwd_ms": ms_f, "fwd_steps": args.steps, "fwd_clocks": clk_f,
            "bwd_tokens_per_s": T_FWD / (ms_b * 1e-3), "bwd_ms": ms_b, "bwd_steps": bsteps, "bwd_clocks": clk_b,
            "fwd_bwd_tokens_per_s": T_FWD / ((ms_f + ms_b) * 1e-3),
            "fwd_roofline": {"bound": "tensor", "achieved": f_fl / (ms_f * 1e-3) / 1e12,
                             "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": f_fl / (ms_f * 1e-3) / 1e12 / peaks["bf16_tflops"]},
            # three GEMMs of 2 T H V each (G recomputed, dW, dX); ~0.2 s of back-to-back GEMMs
            # runs into the power cap, so the sustained peak is reported beside the burst one
            "bwd_roofline": {"bound": "tensor", "achieved": b_tf, "peak": peaks["bf16_tflops"], "unit": "TFLOP/s",
                             "frac": b_tf / peaks["bf16_tflops"],
                             "frac_of_sustained": b_tf / peaks["bf16_tflops_sustained"],
                             "flops_per_call": 3 * f_fl},
            "bwd_burst": {"steps": 5, "ms": ms_bb, "clocks": clk_bb,
                          "achieved": 3 * f_fl / (ms_bb * 1e-3) / 1e12,
                          "frac": 3 * f_fl / (ms_bb * 1e-3) / 1e12 / peaks["bf16_tflops"]}}
        if oracle_on:
            import numpy as np
            Xb, Wb, bb = _host_bits(X), [_host_bits(w) for w in W], [_host_bits(t) for t in b]
            yb = y.cpu().numpy()
            idx = _sample_rows(T_FWD, 256)
            idx_d = torch.from_numpy(idx).to(dev)
            out["sharded_fwd_bwd"]["fwd_cpu_baseline"] = _oracle_leg(
                lambda: oracle.forward(Xb, Wb, bb, part3, yb, tau32, rows=idx), len(idx),
                f"{len(idx)} of {T_FWD} rows (full H, V), fp64 numpy oracle",
                lambda r: {"max_abs_dlogp": _maxdev(fwd["logp"][idx_d].cpu(), r.logp),
                           "max_abs_dentropy": _maxdev(fwd["entropy"][idx_d].cpu(), r.entropy)})
            bw_out = bwd()
            dx_rows = _sample_rows(T_FWD, 64)
            gb = g.cpu().numpy()
            out["sharded_fwd_bwd"]["bwd_cpu_baseline"] = _oracle_leg(
                lambda: oracle.backward_sampled(Xb, Wb, bb, part3, yb, tau32, gb, dx_rows,
                                                [np.zeros(0, np.int64)] * 4), len(dx_rows),
                f"dX of {len(dx_rows)} of {T_FWD} rows (full H, V), fp64 numpy oracle",
                lambda r: {"rel_fro_dX": _relfro(bw_out["dX"][torch.from_numpy(dx_rows).to(dev)].cpu(), r[0])})
            del Xb, Wb, bb, bw_out
    if lp.lp_get_device_error() != 0:
        raise RuntimeError("device error in the path timings")
    return out


# ------------------------------------------------------------ oracle (CPU) arm

def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline_forward(X, W, y, gpu_out, rows: int):
    """The fp64 oracle on `rows` rows of the timed workload itself (full H and V; rows spread
    evenly over T; 1536 rows are ~10 s of host work): its speed on the host cores, and the GPU
    outputs' largest deviation from it on those rows."""
    import numpy as np
    import torch

    import oracle
    import synth
    T, V = X.shape[0], W[0].shape[0]
    idx = torch.linspace(0, T - 1, rows).round().long().unique()
    Xb = X[idx.to(X.device)].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    Wb = [w.view(torch.int16).cpu().numpy().view(np.uint16) for w in W]
    yb = y[idx.to(y.device)].cpu().numpy()
    part = synth.even_partition(V, 1)
    tau32 = float(np.float32(TAU))  # the fp32 temperature the library receives
    t0 = time.perf_counter()
    ref = oracle.forward(Xb, Wb, None, part, yb, tau32)
    dt = time.perf_counter() - t0
    n = int(idx.numel())
    got = {k: gpu_out[k][idx.to(X.device)].cpu().numpy().astype(np.float64) for k in ("logp", "lse", "entropy")}
    parity = {"rows": n, "oracle": "fp64 numpy",
              "max_abs_dlogp": float(np.max(np.abs(got["logp"] - ref.logp))),
              "max_abs_dlse": float(np.max(np.abs(got["lse"] - ref.lse))),
              "max_abs_dentropy": float(np.max(np.abs(got["entropy"] - ref.entropy))),
              "tolerance": {"logp": 2e-3, "lse": 2e-3, "entropy": 5e-3}}
    base = {"value": n / dt, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
            "sample": f"{n} of {T} rows of the timed workload (full H={X.shape[1]}, V={V}), fp64 numpy oracle; "
                      f"{dt:.1f} s"}
    return base, parity


def run_reference(args, world):
    import oracle
    import synth
    rows = args.ref_rows
    part = synth.even_partition(V, 1)
    inp = synth.forward_inputs(rows, H, part, tau=TAU, seed=0)
    for _ in range(args.warmup):
        oracle.forward(inp.X, inp.W, None, part, inp.y, inp.tau)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.forward(inp.X, inp.W, None, part, inp.y, inp.tau)
    dt = (time.perf_counter() - t0) / args.steps
    value = rows / dt
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": "Qwen3-8B-shaped LM-head fused forward, T=4096 rows, H=4096, V=151936, "
                                   "tau=0.7, no bias, logp+LSE+entropy", "T": T_FWD, "H": H, "V": V, "tau": TAU,
                       "sample_rows_per_step": rows},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cpu_cores(), "kind": "oracle",
                             "sample": f"{rows} of {T_FWD} rows per step (full H, V), fp64 numpy oracle"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--headline-only", action="store_true", help="time only the fused forward")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-rows", type=int, default=256,
                    help="oracle rows per reference step (each call also decodes all of W, which a larger "
                         "sample amortises as the full 4096-row workload would)")
    ap.add_argument("--rows", type=int, default=T_FWD, help="headline rows T (profiling of smaller cases)")
    ap.add_argument("--path-rows", type=int, default=8192,
                    help="rows of the logits-reuse and replay workloads (profiling of smaller cases)")
    ap.add_argument("--vocab", type=int, default=V, help="vocabulary V of every path (profiling of smaller cases)")
    ap.add_argument("--paths", default="tiny,batches,logits,replay,backward",
                    help="comma list of the other paths to time: tiny, batches, logits, replay, backward")
    ap.add_argument("--skip-headline", action="store_true", help="time only --paths (profiling)")
    ap.add_argument("--sustained-steps", type=int, default=200,
                    help="calls of the headline held long enough for the power cap to set the clock")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if refuse_multi_gpu(args, world):
        return 2
    if args.impl == "reference":
        if rank == 0:  # under torchrun the other ranks exit without work
            run_reference(args, world)
    else:
        run_ours(args)
    return 0


if __name__ == "__main__":
    sys.exit(main())
