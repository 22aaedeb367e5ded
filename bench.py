"""Benchmark of the low-rank bottleneck hot path on GB300.

One step = forward + backward of the LLaMA-2-7B-shaped CoLA MLP
(T = 4 x 4096 tokens, d = 4096, r = 1024, ffn = 11008, S = 8 norm shards):
gate/up bottleneck (Online-RMSNorm statistics, folded gamma, grouped
down-projection with deferred 1/rms + SiLU, batched up-projection) -> SwiGLU ->
down bottleneck, then the backward with low-rank recompute. Inputs are the
seeded synthetic tensors of rank_bottleneck_online_gb300.inputs, resident in
HBM before the timed region; every large tensor the step touches (x 134 MB, the
gate/up activations 721 MB and their gradients) is larger than the 129 MB L2,
so no L2 flush is inserted between steps.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
One GPU only: the GEMMs load their operands with cluster-multicast TMA copies, which
may run only in single-GPU processes, so `--gpus N` with N > 1 (or a torchrun launch
with WORLD_SIZE > 1) prints an `unavailable` line and exits 0 without launching a
kernel. The reference arm (the CPU oracle) runs on rank 0 at any N.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "bottleneck-block fwd+bwd TFLOP/s & tokens/s on 1 GB300; % of roofline"
WORKLOAD = "llama2_7b_mlp"
CPU_SAMPLE_T = 1024          # tokens of the CPU-baseline sample (full d, r, ffn)
REF_STEP_T = 16              # tokens per step of the reference arm


def _flops(T, blocks):
    """Executed flops of one fwd + bwd step over bottleneck blocks (input width, k*r, n),
    the recompute of z included, and model flops (without it)."""
    exe = sum(8 * T * din * kr + 6 * T * kr * n for din, kr, n in blocks)
    model = sum(6 * T * din * kr + 6 * T * kr * n for din, kr, n in blocks)
    return exe, model


def mlp_flops(T, d, r, ffn):
    """Executed flops of one MLP step (recompute included) and model flops."""
    return _flops(T, [(d, 2 * r, ffn), (ffn, r, d)])


def workload_blocks(name):
    """(input width, k*r, n) of every bottleneck block in a step of a named workload."""
    from rank_bottleneck_online_gb300.inputs import CONFIGS

    c = CONFIGS[name]
    d, r = c["d"], c["r"]
    kind = c["kind"]
    if kind == "block":
        return [(d, c["k"] * r, c["n"])]
    if kind == "mlp":
        return [(d, 2 * r, c["ffn"]), (c["ffn"], r, d)]
    if kind == "layer":       # QKV, O (input: the attention stand-in V), gate/up, down
        return [(d, 3 * r, d), (d, r, d), (d, 2 * r, c["ffn"]), (c["ffn"], r, d)]
    if kind == "svd_pair":    # QKV and gate/up on one x
        return [(d, 3 * r, d), (d, 2 * r, c["ffn"])]
    raise KeyError(name)


def workload_flops(name, T):
    return _flops(T, workload_blocks(name))


def dense_mlp_flops(T, d, ffn):
    """Dense (full-rank) LLaMA MLP fwd + bwd: three [d, ffn]-sized GEMMs, each 2 flops per
    multiply-add, forward once and twice in backward (dgrad and wgrad)."""
    return 6.0 * T * 3 * d * ffn


def dense_mlp(T, d, ffn, device, seed=0, dtype=None, eps=1e-5):
    """The full-rank counterpart of the low-rank MLP at the same shapes, in plain torch
    (cuBLAS GEMMs, torch's RMSNorm and SiLU): out = (silu(n @ Wg) * (n @ Wu)) @ Wd with
    n = RMSNorm(x) * gamma. Context for the low-rank step, not part of the library.
    Returns (step, tensors); step() runs forward and backward once."""
    import torch
    import torch.nn.functional as F

    dtype = dtype or torch.bfloat16
    g = torch.Generator(device="cpu").manual_seed(seed)

    def randn(*shape, std=1.0):
        return (torch.randn(*shape, generator=g) * std).to(dtype).to(device)

    t = {"x": randn(T, d), "gamma": (1.0 + 0.1 * torch.randn(d, generator=g)).to(dtype).to(device),
         "Wg": randn(d, ffn, std=d ** -0.5), "Wu": randn(d, ffn, std=d ** -0.5),
         "Wd": randn(ffn, d, std=ffn ** -0.5), "dout": randn(T, d)}
    for k in ("x", "gamma", "Wg", "Wu", "Wd"):
        t[k].requires_grad_(True)

    def step():
        for k in ("x", "gamma", "Wg", "Wu", "Wd"):
            t[k].grad = None
        n = F.rms_norm(t["x"], (d,), t["gamma"], eps)
        h = F.silu(n @ t["Wg"]) * (n @ t["Wu"])
        out = h @ t["Wd"]
        out.backward(t["dout"])
        return out

    return step, t


def _dense_context(T, d, ffn, ms_ours, reps=10):
    """Time the full-rank MLP step on this GPU (CUDA events, after warm-up) against the
    low-rank step's ms_per_step: the one-GPU analogue of the pages' full-rank vs
    low-rank comparison."""
    import torch

    step, t = dense_mlp(T, d, ffn, "cuda")
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    del t, step
    torch.cuda.empty_cache()
    fl = dense_mlp_flops(T, d, ffn)
    return {"impl": "torch eager, cuBLAS bf16 GEMMs", "ms_per_step": ms,
            "tokens_per_s": T / (ms / 1e3), "tflops_per_s": fl / (ms / 1e3) / 1e12,
            "flops_per_step": fl, "lowrank_speedup": ms / ms_ours}


def _checkpoint_cuts(mlp, w, x, dout, T, d, r, ffn, S, ms_input, reps=10):
    """The step with the bottleneck checkpoint cut (only the gate/up block's r-wide
    activation kept; gate, up and h regenerated in backward) against the timed step,
    which keeps the blocks' inputs: time per step and bytes kept between forward and
    backward beyond x and the row scale."""
    import torch

    from rank_bottleneck_online_gb300.block import MLP

    m2 = MLP(T, d, r, ffn, S=S, weights=w, device=x.device, checkpoint="bottleneck")

    def step():
        m2.forward(x)
        m2.backward(x, dout)

    for _ in range(3):
        step()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / reps
    out = {"input": {"ms_per_step": ms_input, "saved_bytes": mlp.saved_bytes()},
           "bottleneck": {"ms_per_step": ms, "saved_bytes": m2.saved_bytes()}}
    del m2
    torch.cuda.empty_cache()
    return out


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except (OSError, KeyError, ValueError):
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


def _cfg(name=WORKLOAD):
    from rank_bottleneck_online_gb300.inputs import CONFIGS
    return CONFIGS[name]


# ------------------------------------------------------------- clocks

# NVML clock-event reason bits (nvmlClocksEventReason* in nvml.h) that the timing rules
# name; the others (idle, application clocks, sync boost, ...) are not reported.
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown"}


def summarize_clocks(samples, source, in_region=True):
    """Summary of clock samples (sm_mhz, sm_max_mhz, power_w, set of reason names) taken
    during the timed region: median SM clock, maximum clock and power, every reason seen,
    and the share of samples with the power cap active."""
    if not samples:
        return {"sm_mhz": None, "sm_max_mhz": None, "power_w_max": None, "reasons": [],
                "samples": 0, "power_cap_share": None, "source": source}
    sm = sorted(s[0] for s in samples)
    n = len(sm)
    med = sm[n // 2] if n % 2 else 0.5 * (sm[n // 2 - 1] + sm[n // 2])
    seen = set()
    for s in samples:
        seen |= set(s[3])
    out = {"sm_mhz": med, "sm_max_mhz": max(s[1] for s in samples),
           "power_w_max": max(s[2] for s in samples), "reasons": sorted(seen),
           "samples": n if in_region else 0,
           "power_cap_share": sum(1 for s in samples if "sw_power_cap" in s[3]) / n,
           "source": source}
    if not in_region:
        out["note"] = "no sample fell inside the timed region; nearest sample reported"
    return out


class _Nvml:
    """The few read-only NVML queries the sampler needs, through ctypes on the driver's
    libnvidia-ml (no Python NVML package on the GPU host)."""

    def __init__(self, cuda_index):
        import ctypes

        self.c = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        ok = False
        try:                                   # the CUDA device's own GPU, by UUID
            import torch
            uuid = str(torch.cuda.get_device_properties(cuda_index).uuid)
            key = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid).encode()
            ok = self.lib.nvmlDeviceGetHandleByUUID(key, ctypes.byref(self.h)) == 0
        except Exception:  # noqa: BLE001
            ok = False
        if not ok and self.lib.nvmlDeviceGetHandleByIndex_v2(
                ctypes.c_uint(cuda_index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle for the device")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.sm_max = self._uint(self.lib.nvmlDeviceGetMaxClockInfo, 1)

    def _uint(self, fn, *args):
        v = self.c.c_uint()
        if fn(self.h, *args, self.c.byref(v)) != 0:
            return None
        return float(v.value)

    def sample(self):
        sm = self._uint(self.lib.nvmlDeviceGetClockInfo, 1)          # NVML_CLOCK_SM
        mw = self._uint(self.lib.nvmlDeviceGetPowerUsage)
        bits = self.c.c_ulonglong()
        names = set()
        if self.reasons_fn(self.h, self.c.byref(bits)) == 0:
            names = {nm for b, nm in NVML_REASONS.items() if bits.value & b}
        if sm is None:
            return None
        return (sm, self.sm_max or sm, (mw or 0.0) / 1e3, names)

    def close(self):
        self.lib.nvmlShutdown()


class ClockSampler:
    """SM clock, power and clock-event reasons sampled while the timed region runs.

    Reads NVML every few milliseconds from a background thread (read-only queries);
    where NVML cannot be loaded, nvidia-smi's own loop (100 ms) stands in. Every sample
    carries its time, and only samples taken between mark_start() and mark_stop() are
    reported (the nearest one, marked as such, if none fell inside)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
    PERIOD_S = 0.005

    def __init__(self, index):
        self.index = index
        self.nvml = None
        self.thread = None
        self.samples = []          # (time, (sm, sm_max, power, reasons))
        self.stopping = False
        self.proc = None
        self.out = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.nvml = _Nvml(self.index)
        except Exception:  # noqa: BLE001
            self.nvml = None
        if self.nvml is not None:
            import threading

            def loop():
                while not self.stopping:
                    try:
                        s = self.nvml.sample()
                    except Exception:  # noqa: BLE001  (a failed read is a missing sample)
                        s = None
                    if s is not None:
                        self.samples.append((time.time(), s))
                    time.sleep(self.PERIOD_S)

            self.thread = threading.Thread(target=loop, daemon=True)
            self.thread.start()
            return
        try:
            self.out = tempfile.TemporaryFile(mode="w+")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.out, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def mark_start(self):
        self.t0 = time.time()

    def mark_stop(self):
        self.t1 = time.time()

    @staticmethod
    def _when(stamp):
        # "YYYY/MM/DD HH:MM:SS.mmm" in the host's local time
        try:
            whole, _, frac = stamp.partition(".")
            return time.mktime(time.strptime(whole, "%Y/%m/%d %H:%M:%S")) + \
                float("0." + (frac or "0"))
        except ValueError:
            return None

    def _smi_rows(self):
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.seek(0)
        rows = [[c.strip() for c in ln.split(",")] for ln in self.out.read().splitlines()
                if ln.strip()]
        rows = [r for r in rows if len(r) >= 10]
        if any(r[1] == str(self.index) for r in rows):
            rows = [r for r in rows if r[1] == str(self.index)]
        out = []
        for r in rows:
            try:
                s = (float(r[2]), float(r[3]), float(r[4]),
                     {nm for nm, v in zip(self.NAMES, r[6:10]) if v.lower() == "active"})
            except ValueError:
                continue
            w = self._when(r[0])
            if w is not None:
                out.append((w, s))
        return out

    def stop(self):
        if self.nvml is not None:
            self.stopping = True
            self.thread.join(timeout=5)
            self.nvml.close()
            timed, source = list(self.samples), "nvml"
        elif self.proc is not None:
            timed, source = self._smi_rows(), "nvidia-smi"
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clocks unavailable"],
                    "samples": 0, "power_cap_share": None, "source": None}
        return self.select(timed, self.t0, self.t1, source)

    @staticmethod
    def select(timed, t0, t1, source):
        """Summary of the (time, sample) pairs inside [t0, t1], else of the nearest one."""
        inside = [s for w, s in timed if t0 is not None and t1 is not None and t0 <= w <= t1]
        if inside or not timed:
            return summarize_clocks(inside, source)
        mid = 0.5 * (t0 + t1) if t0 is not None and t1 is not None else timed[-1][0]
        near = min(timed, key=lambda ws: abs(ws[0] - mid))[1]
        return summarize_clocks([near], source, in_region=False)


def choose_peak(peaks, clocks):
    """(kind, TFLOP/s) of the bf16 peak the dominant GEMM is set against.

    The burst peak is a dense GEMM timed alone at full clock; the sustained one the same
    GEMM held for seconds, where the 1.4 kW power cap pulls the SM clock down. A timed
    region whose clock samples show the power cap in at least half of them ran under the
    same conditions as the sustained measurement and takes that peak; any other region
    (also one with no sample) takes the burst peak, the stricter denominator."""
    share = (clocks or {}).get("power_cap_share")
    if share is not None and share >= 0.5:
        return "sustained", peaks["bf16_tflops_sustained"]
    return "burst", peaks["bf16_tflops"]


# ------------------------------------------------------------- oracle

def cpu_oracle_sample(T_sample, steps=1, workload=WORKLOAD):
    """Time the oracle (bf16 flow, fwd+bwd) on T_sample tokens of a workload.

    Runs in a fresh subprocess with every BLAS/OpenMP pool sized to the cores
    this process may use; returns seconds per step, tokens and thread count.
    """
    cores = len(os.sched_getaffinity(0))
    env = dict(os.environ)
    for k in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
        env[k] = str(cores)
    env["CUDA_VISIBLE_DEVICES"] = ""
    cmd = [sys.executable, os.path.abspath(__file__), "--_oracle-sample", str(T_sample),
           "--_oracle-steps", str(steps), "--workload", workload]
    r = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=1800)
    if r.returncode != 0:
        raise RuntimeError(f"oracle sample failed: {r.stderr[-2000:]}")
    res = json.loads(r.stdout.strip().splitlines()[-1])
    res["cores"] = cores
    return res


def _oracle_sample_main(T_sample, steps, workload=WORKLOAD):
    import oracle
    from rank_bottleneck_online_gb300 import inputs

    c = inputs.CONFIGS[workload]
    w = inputs.make_inputs(workload, T=T_sample, seed=0)

    def f64(v):
        return {k: f64(u) for k, u in v.items()} if isinstance(v, dict) else inputs.as_f64(v)

    f = {k: f64(v) for k, v in w.items()}
    S, kind = c["S"], c["kind"]

    def step():
        if kind == "mlp":
            args = (f["x"], f["gamma"], f["A1"], f["B1"], f["A2"], f["B2"])
            oracle.mlp_fwd(*args, S=S, flow="bf16")
            oracle.mlp_bwd(*args, f["dout"], S=S, flow="bf16")
        elif kind == "block":
            args = (f["x"], f["gamma"], f["A"], f["B"])
            oracle.block_fwd(*args, act=c["act"], S=S, flow="bf16")
            oracle.block_bwd(*args, f["dy"], act=c["act"], S=S, flow="bf16")
        elif kind == "layer":
            oracle.layer_fwd(f["x"], f["p"], S=S, flow="bf16")
            oracle.layer_bwd(f["x"], f["p"], f["dout"], f["dq"], f["dk"], S=S, flow="bf16")
        else:
            oracle.svd_pair_fwd(f["x"], f["p"], S=S, flow="bf16")
            oracle.svd_pair_bwd(f["x"], f["p"], f["dy_qkv"], f["dy_gu"], S=S, flow="bf16")

    times = []
    for _ in range(steps):
        t0 = time.perf_counter()
        step()
        times.append(time.perf_counter() - t0)
    print(json.dumps({"seconds": times, "tokens": T_sample}))


def reference_arm(args, rank, world):
    """The oracle, as it stands, on the host cores: rank 0 only.

    A step is REF_STEP_T tokens of the workload (full widths). The K timed steps'
    token samples are independent rows, so they are processed in one oracle pass of
    K * REF_STEP_T tokens (the oracle's per-call cost of rounding the weights would
    otherwise dominate); likewise the warm-up steps, untimed, before it.
    """
    if rank != 0:
        return 0
    c = _cfg()
    cpu_oracle_sample(args.warmup * REF_STEP_T, steps=1)
    res = cpu_oracle_sample(args.steps * REF_STEP_T, steps=1)
    per = res["seconds"][0] / args.steps
    T_s = REF_STEP_T
    value = T_s / per
    exe, _ = mlp_flops(T_s, c["d"], c["r"], c["ffn"])
    sample = (f"{T_s} of {c['T']} tokens of {WORKLOAD} per step (full d/r/ffn), the "
              f"{args.steps} timed steps in one pass of {args.steps * T_s} tokens; oracle bf16 "
              "flow fwd+bwd in numpy fp64")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "tokens": c["T"], "d": c["d"], "r": c["r"],
                       "ffn": c["ffn"], "S": c["S"], "l2": "inputs larger than L2"},
            "tflops_per_s": exe / per / 1e12,
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": res["cores"],
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------- ranks

def max_over_ranks(value, dist=None, device="cpu"):
    """The maximum of a per-rank float over all ranks (identity on one process)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def step_spread(ms):
    """Median and spread of per-step device times (ms), from events recorded between
    the timed steps; nearest-rank percentiles."""
    if not ms:
        return None
    v = sorted(ms)
    n = len(v)
    pick = lambda q: v[min(n - 1, max(0, int(round(q * (n - 1)))))]  # noqa: E731
    med = v[n // 2] if n % 2 else 0.5 * (v[n // 2 - 1] + v[n // 2])
    return {"median": med, "p10": pick(0.1), "p90": pick(0.9), "min": v[0], "max": v[-1],
            "samples": n}


def aggregate_rate(world, units_per_rank, seconds):
    """Whole-job rate under weak scaling: every rank processes the same units."""
    return world * units_per_rank / seconds


# ------------------------------------------------------------- ours

def csrc_digest():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "rank_bottleneck_online_gb300", "csrc")
    for fn in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def read_traffic(kernel, units):
    """DRAM bytes of one launch of `kernel` from the committed ncu summary, scaled from
    the captured case by units processed, or None when the kernel sources changed since
    the counters were taken (the summary records a digest of csrc/)."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.txt")
    if not os.path.exists(path):
        return None
    digest = csrc_digest()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if line.startswith("#") or len(parts) < 4 or parts[0] != kernel:
                continue
            if parts[1] != digest:
                return None
            return float(parts[2]) * units / float(parts[3])
    return None


def _workspaces(wl):
    """The distinct workspaces of a workload object and its blocks."""
    seen, out = set(), []
    stack = [wl]
    while stack:
        o = stack.pop()
        ws = getattr(o, "ws", None)
        if ws is not None and id(ws) not in seen:
            seen.add(id(ws))
            out.append(ws)
        for name in ("gu", "dn", "qkv", "o", "mlp"):
            sub = getattr(o, name, None)
            if sub is not None:
                stack.append(sub)
    return out


def _workload_step(name, wl, w, dev):
    """forward + backward of one step of a named workload on device inputs."""
    from rank_bottleneck_online_gb300.inputs import CONFIGS

    kind = CONFIGS[name]["kind"]
    x = w["x"].to(dev)
    if kind == "block":
        dy = w["dy"].to(dev)
        return lambda: (wl.forward(x), wl.backward(x, dy))
    if kind == "mlp":
        dout = w["dout"].to(dev)
        return lambda: (wl.forward(x), wl.backward(x, dout))
    if kind == "layer":
        # dq and dk stand in for the (excluded) attention core's gradients: placed once in
        # the stacked QKV gradient, where an attention backward would write them
        dout = w["dout"].to(dev)
        wl.dqkv[0].copy_(w["dq"])
        wl.dqkv[1].copy_(w["dk"])
        dq, dk = wl.dqkv[0], wl.dqkv[1]
        return lambda: (wl.forward(x), wl.backward(x, dout, dq, dk))
    dq, dg = w["dy_qkv"].to(dev), w["dy_gu"].to(dev)
    return lambda: (wl.forward(x), wl.backward(x, dq, dg))


def ours_arm(args):
    """The library's timed step on this process's one GPU (cuda:0)."""
    import torch

    from rank_bottleneck_online_gb300 import binding as B
    from rank_bottleneck_online_gb300 import build as build_mod
    from rank_bottleneck_online_gb300 import inputs
    from rank_bottleneck_online_gb300.block import MLP, build_workload

    build_mod.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    name = args.workload
    c = inputs.CONFIGS[name]
    T = args.tokens or c["T"]
    w = inputs.make_inputs(name, seed=0, T=T)
    stream = torch.cuda.current_stream()
    mlp = None
    if name == WORKLOAD:
        d, r, ffn, S = c["d"], c["r"], c["ffn"], c["S"]
        mlp = MLP(T, d, r, ffn, S=S, weights=w, device=dev)
        x = w["x"].to(dev)
        dout = w["dout"].to(dev)
        wl = mlp

        def step():
            mlp.forward(x)
            mlp.backward(x, dout)
    else:
        wl = build_workload(name, w, device=dev, T=T)
        step = _workload_step(name, wl, w, dev)
    workspaces = _workspaces(wl)

    def check():
        for ws in workspaces:
            B.check(ws)

    sampler = ClockSampler(0)
    sampler.start()                 # running before the timed region; samples filtered
    for _ in range(args.warmup):
        step()
    check()
    torch.cuda.synchronize()

    # Which operation dominates (the one whose kernel the roofline line reports): a short
    # pass with every operation timed. Timing an operation brackets it with events, and
    # each event makes its stream wait for the work before it (about 3% of the 7B step
    # with every operation timed), so the timed region below times that operation only.
    overlapped = set(OVERLAPPED_OPS) if _forked() else set()
    B.profile_only(None)
    B.profile_enable(True)
    for _ in range(min(args.steps, 3)):
        step()
    torch.cuda.synchronize()
    dom_name = dominant_kernel(B.profile_read(), overlapped)[0]
    B.profile_enable(False)

    # The timed region: the K steps captured into one CUDA graph and launched once (the
    # library's events around the dominant operation become graph nodes, one sample per
    # launch), or (--eager, or if the capture fails) issued as individual launches. Both
    # issue the same kernels in the same order from the same buffers; the graph removes
    # the host's launch gaps (7B MLP, 20 steps: 3.43 ms a step against 3.50 eager).
    B.profile_only(dom_name)
    B.profile_enable(True)
    graph = None
    if args.graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                for _ in range(args.steps):
                    step()
        except Exception as ex:  # noqa: BLE001
            print(f"graph capture failed, timing eagerly: {ex}", file=sys.stderr)
            graph = None
            B.profile_enable(False)        # drop what the failed capture recorded
            B.profile_enable(True)
    torch.cuda.synchronize()
    sampler.mark_start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    # (eager) an event between consecutive steps gives each step's own device time
    marks = ([torch.cuda.Event(enable_timing=True) for _ in range(args.steps - 1)]
             if graph is None else [])
    e0.record(stream)
    if graph is not None:
        graph.replay()
    else:
        for i in range(args.steps):
            step()
            if i < args.steps - 1:
                marks[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize()
    sampler.mark_stop()
    bounds = [e0, *marks, e1]
    args.step_ms = (step_spread([a.elapsed_time(b) for a, b in zip(bounds, bounds[1:])])
                    if graph is None else None)
    clocks = sampler.stop()
    dom = (dom_name, B.profile_read()[dom_name])
    B.profile_enable(False)
    args.timing = "cuda_graph" if graph is not None else "eager"
    del graph
    check()
    # The per-operation table: the same K steps once more, right after the timed region,
    # with every operation timed (its shares and kernel counts; the line's value and the
    # dominant kernel's rate come from the timed region itself).
    B.profile_only(None)
    B.profile_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize()
    prof = B.profile_read()
    prof_kernels = B.profile_kernels()
    B.profile_enable(False)
    check()
    ms_total = e0.elapsed_time(e1)
    if mlp is None:             # the other workloads: the timed step and its roofline only
        return _report(args, 1, prof, prof_kernels, clocks, ms_total, float("nan"), 0, 0,
                       T, c["d"], c["r"], c.get("ffn"), c["S"], dom=dom)

    aux = not args.skip_aux
    e2e_s, e2e_launch = _e2e(args, mlp, w, x, dout, T, d, dev) if aux else (float("nan"), None)
    btp = _btp_exchange(mlp, x, T, d, r, ffn, S) if aux else None
    dense = _dense_context(T, d, ffn, ms_total / args.steps) if aux else None
    cuts = (_checkpoint_cuts(mlp, w, x, dout, T, d, r, ffn, S, ms_total / args.steps)
            if aux else None)
    bi = 2 * T * d * 2          # x and dout, bf16
    bo = 2 * T * d * 2          # out and dx, bf16
    return _report(args, 1, prof, prof_kernels, clocks, ms_total, e2e_s, bi, bo, T, d, r,
                   ffn, S, btp, dense, cuts, dom=dom, e2e_launch=e2e_launch)


def _btp_exchange(mlp, x, T, d, r, ffn, S, reps=5):
    """The bottleneck-aware TP exchange emulated on this GPU (outside the timed step):
    per block, the S shards' partial products and sums of squares materialised as the
    payload S ranks would all-reduce, then reduced; against what vanilla low-rank TP
    all-reduces (each low-rank pair's d-wide output). Times are this GPU's cost of
    forming and reducing the payload, not a network's."""
    import torch

    from rank_bottleneck_online_gb300 import binding as B

    blocks = []
    S_dn = 4   # the down block's d = ffn = 11008 splits into 64-aligned shards for S = 4
    for name, blk, inp, s_blk in (("gate_up", mlp.gu, x, S), ("down", mlp.dn, mlp.h, S_dn)):
        desc = B.make_desc(T, blk.desc.d, r, blk.desc.k, blk.desc.n, S=s_blk,
                           has_norm=bool(blk.desc.has_norm))
        ws = B.Workspace(B.workspace_bytes(desc))
        pay = torch.empty(B.btp_payload_elems(desc), dtype=torch.float32, device=x.device)
        y = torch.empty_like(blk.y)

        def once():
            B.block_fwd_btp(desc, inp, blk.gamma, blk.A, blk.B, ws, y=y, payload=pay)
            B.block_fwd(desc, inp, blk.gamma, blk.A, blk.B, ws, y=y)

        once()
        torch.cuda.synchronize()
        B.profile_enable(True)
        for _ in range(reps):
            once()
        torch.cuda.synchronize()
        pr = B.profile_read()
        B.profile_enable(False)
        B.check(ws)
        kr = blk.desc.k * r
        pay_rank = T * (kr + (1 if desc.has_norm else 0))
        dwide_rank = T * blk.desc.k * blk.desc.n
        part, red, fused = pr["gemm_down_partials"], pr["btp_exchange_reduce"], pr["gemm_down_act"]
        blocks.append({
            "block": name, "S": s_blk, "payload_elems_per_rank": pay_rank,
            "vanilla_elems_per_rank": dwide_rank, "ratio": dwide_rank / pay_rank,
            "ms_partials": part[1] / reps, "partials_tflops": part[2] / (part[1] / 1e3) / 1e12,
            "ms_reduce": red[1] / reps, "reduce_gbs": red[3] / (red[1] / 1e3) / 1e9,
            "ms_fused_down": fused[1] / reps})
        del ws, pay
    tot_pay = sum(b["payload_elems_per_rank"] for b in blocks)
    tot_van = sum(b["vanilla_elems_per_rank"] for b in blocks)
    return {"blocks": blocks, "mlp_ratio": tot_van / tot_pay,
            "reading": "payload per rank: the bottleneck partials [T, k*r] (+1 column of "
                       "sums of squares for a normed block); vanilla low-rank TP: one "
                       "all-reduce of each low-rank pair's d-wide output ([T, k*n])"}


def _e2e(args, mlp, w, x, dout, T, d, dev):
    """(seconds, launch) for args.steps steps through the public API from pinned host
    buffers: each step copies its x and dout in, runs forward + backward and copies out
    and dx back. The copies are pipelined against the compute on two more streams (inputs
    of step i+1 in, results of step i-1 out, while step i computes) with double-buffered
    device tensors; every step's copies lie inside the timed region. Like the timed
    region, the K steps (copies included) are captured into one CUDA graph and launched
    once unless --eager is given or the capture fails; `launch` says which ran."""
    import torch

    from rank_bottleneck_online_gb300.block import MLP

    c = _cfg()
    r, ffn, S = c["r"], c["ffn"], c["S"]
    x_h = w["x"].pin_memory()
    dout_h = w["dout"].pin_memory()
    out_h = [torch.empty(T, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    dx_h = [torch.empty(T, d, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    # a second replica of the MLP (same weights) so that step i+1 does not overwrite the
    # results step i is still copying out
    mlps = [mlp, MLP(T, d, r, ffn, S=S, weights=w, device=dev)]
    xs = [x, torch.empty_like(x)]
    douts = [dout, torch.empty_like(dout)]
    h2d = torch.cuda.Stream()
    d2h = torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()   # noqa: E731
    in_ready = [ev(), ev()]
    computed = [ev(), ev()]
    copied_out = [ev(), ev()]

    def run(n, capturing=False):
        comp = torch.cuda.current_stream()
        if capturing:
            # the copy streams join the capture from the capturing stream; the first two
            # steps' buffers are free (everything before the capture has completed)
            h2d.wait_stream(comp)
            d2h.wait_stream(comp)
        for i in range(n):
            b = i % 2
            first = capturing and i < 2
            with torch.cuda.stream(h2d):
                if not first:
                    h2d.wait_event(computed[b])      # step i-2 finished with these inputs
                xs[b].copy_(x_h, non_blocking=True)
                douts[b].copy_(dout_h, non_blocking=True)
                in_ready[b].record(h2d)
            comp.wait_event(in_ready[b])
            if not first:
                comp.wait_event(copied_out[b])        # step i-2's results are out
            mlps[b].forward(xs[b])
            mlps[b].backward(xs[b], douts[b])
            computed[b].record(comp)
            with torch.cuda.stream(d2h):
                d2h.wait_event(computed[b])
                out_h[b].copy_(mlps[b].out, non_blocking=True)
                dx_h[b].copy_(mlps[b].gu.dx, non_blocking=True)
                copied_out[b].record(d2h)
        if capturing:
            comp.wait_stream(h2d)
            comp.wait_stream(d2h)

    run(2)
    torch.cuda.synchronize()
    graph = None
    if args.graph:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                run(args.steps, capturing=True)
        except Exception as ex:  # noqa: BLE001
            print(f"end-to-end graph capture failed, running eagerly: {ex}", file=sys.stderr)
            graph = None
        torch.cuda.synchronize()
    t0 = time.perf_counter()
    if graph is not None:
        graph.replay()
    else:
        run(args.steps)
    torch.cuda.synchronize()
    return time.perf_counter() - t0, ("cuda_graph" if graph is not None else "eager")


# Operations the library runs concurrently with other GEMMs when BOOST_FORK_STREAMS=1:
# dB and dA on forked streams beside dx on the caller's stream, the gamma fold beside
# the statistics. Their event intervals include time shared with the concurrent work,
# so they are not kernel durations.
OVERLAPPED_OPS = ("gemm_wgrad_B", "gemm_wgrad_A", "splitk_sum", "splitk_finalize_dA",
                  "dgamma_reduce", "gemm_dx", "gemm_dx_swiglu", "fold_gamma", "rmsnorm_stats")


def _env_flag(name, default):
    """The library's reading of an on/off environment switch (atoi: non-zero is on)."""
    try:
        return int(os.environ.get(name, str(default))) != 0
    except ValueError:
        return False


def _forked():
    return _env_flag("BOOST_FORK_STREAMS", 0)


def dominant_kernel(prof, overlapped):
    """(name, (launches, ms, flops, bytes)) of the operation with the largest event time
    among those that run alone (not in `overlapped`); all of them if none does."""
    serial = {k: v for k, v in prof.items() if k not in overlapped} or prof
    return max(serial.items(), key=lambda kv: kv[1][1])


def _report(args, world, prof, prof_kernels, clocks, ms_total, e2e_s, bi, bo, T, d, r, ffn,
            S, btp=None, dense=None, cuts=None, dom=None, e2e_launch=None):
    """The JSON line. `prof` / `prof_kernels`: every operation's events over K steps;
    `dom`: (name, (launches, ms, flops, bytes)) of the dominant operation timed alone over
    the timed region (None: taken from `prof`)."""
    ms_step = ms_total / args.steps
    tokens_per_s = aggregate_rate(world, T * args.steps, ms_total / 1e3)
    default = args.workload == WORKLOAD
    exe, model = workload_flops(args.workload, T)
    tflops = world * exe * args.steps / (ms_total / 1e3) / 1e12
    peaks = load_peaks()
    # dominant kernel: the largest share of the timed region among the operations timed
    # alone on the caller's stream (a forked operation's interval is not its duration)
    overlapped = set(OVERLAPPED_OPS) if _forked() else set()
    name, (launches, kms, kfl, kby) = dom if dom is not None else dominant_kernel(prof, overlapped)
    bound = "tensor" if kfl > 0 else "hbm"
    if bound == "tensor":
        achieved = kfl / (kms / 1e3) / 1e12
        peak_kind, peak = choose_peak(peaks, clocks)
        fracs = {"frac_burst": achieved / peaks["bf16_tflops"],
                 "frac_sustained": achieved / peaks["bf16_tflops_sustained"]}
        unit = "TFLOP/s"
        per_launch_units = kfl / launches
    else:
        achieved = kby / (kms / 1e3) / 1e9
        peak_kind, peak, fracs = "copy", peaks["hbm_gbs"], {}
        unit = "GB/s"
        per_launch_units = kby / launches
    # (the committed counters are for the default workload's shapes)
    traffic = read_traffic(name, per_launch_units) if default else None
    step_bytes = sum(v[3] for v in prof.values()) / args.steps
    roof_ms = max(exe / (peaks["bf16_tflops"] * 1e12),
                  step_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e3
    # the same against the sustained bf16 rate (a dense GEMM held for seconds under the
    # power cap), which is what a step that runs for a second sees
    roof_sus_ms = max(exe / (peaks["bf16_tflops_sustained"] * 1e12),
                      step_bytes / (peaks["hbm_gbs"] * 1e9)) * 1e3
    # kernels, not operations: a co-scheduled GEMM is two concurrent launches
    gpu_launches = sum(prof_kernels.get(k, v[0]) for k, v in prof.items())

    cpu = None
    if world == 1 and not args.skip_aux:
        # the wide workloads (13B layer, 40B pair) on 512 sampled tokens, the rest on 1024
        t_s = CPU_SAMPLE_T if _cfg(args.workload)["d"] <= 4096 else CPU_SAMPLE_T // 2
        try:
            res = cpu_oracle_sample(t_s, steps=1, workload=args.workload)
            cpu = {"value": t_s / res["seconds"][0], "unit": "tokens/s",
                   "cores": res["cores"], "kind": "oracle",
                   "sample": f"{t_s} of {T} tokens of {args.workload} (full widths), "
                             "oracle bf16 flow fwd+bwd in numpy fp64, one run"}
        except Exception as ex:  # noqa: BLE001
            cpu = {"value": None, "unit": "tokens/s", "cores": len(os.sched_getaffinity(0)),
                   "kind": "oracle", "sample": f"failed: {ex}"[:200]}

    total_ms = sum(u[1] for u in prof.values())
    kernels = {k: {"launches": v[0], "kernels": prof_kernels.get(k, v[0]),
                   "ms": round(v[1], 4), "share": round(v[1] / total_ms, 4),
                   "tflops": round(v[2] / (v[1] / 1e3) / 1e12, 1) if v[2] else None,
                   "gbs": round(v[3] / (v[1] / 1e3) / 1e9, 1),
                   **({"overlapped": True} if k in overlapped else {})}
               for k, v in sorted(prof.items(), key=lambda kv: -kv[1][1])}
    line = {
        "metric": METRIC, "value": tokens_per_s, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
        "step_ms": getattr(args, "step_ms", None),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": args.workload, "tokens": T, "d": d, "r": r,
                   **({"ffn": ffn} if ffn else {}), "S": S,
                   **({k: v for k, v in _cfg(args.workload).items() if k in ("k", "n", "kind")}),
                   "parallelism": "single",
                   "l2": "inputs larger than L2 (no flush)",
                   "launch": getattr(args, "timing", "eager"),
                   "kernel_launch": "programmatic" if _env_flag("BOOST_PDL", 1) else "plain",
                   "backward_streams": "forked" if _forked() else "one"},
        "tflops_per_s": tflops,
        "model_tflops_per_s": world * model * args.steps / (ms_total / 1e3) / 1e12,
        "pct_of_roofline": 100.0 * roof_ms / ms_step,
        "pct_of_roofline_sustained": 100.0 * roof_sus_ms / ms_step,
        "roofline_step": {"flops": exe, "bytes": step_bytes, "time_ms": roof_ms,
                          "peak_tflops": peaks["bf16_tflops"], "peak_gbs": peaks["hbm_gbs"],
                          "peaks": f"{peaks['source']} burst"},
        "roofline": {"kernel": name, "bound": bound, "achieved": achieved, "peak": peak,
                     "unit": unit, "frac": achieved / peak, **fracs, "traffic": traffic,
                     "launches_per_step": launches / args.steps,
                     "peak_kind": f"{peaks['source']} {peak_kind}",
                     "peak_choice": ("sustained when the power cap is active in at least "
                                     "half of the timed region's clock samples, else burst")
                     if bound == "tensor" else None},
        "kernels": kernels,
        "kernels_timing": ("every operation timed over the same K steps run again right after "
                           "the timed region; the timed region times only "
                           f"{name} (roofline.achieved)"),
        "gpu_launches": gpu_launches,
        "e2e": None if args.skip_aux or not default else {
            "value": aggregate_rate(world, T * args.steps, e2e_s), "unit": "tokens/s",
            "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
            **({"launch": e2e_launch} if e2e_launch else {})},
        "clocks": clocks,
        "cpu_baseline": cpu,
        "btp_exchange": btp,
        "dense_fullrank": dense,
        "checkpoint_cuts": cuts,
    }
    print(json.dumps(line), flush=True)
    return 0


def multi_gpu_unavailable(n):
    """The line printed instead of a measurement when more than one GPU is asked for."""
    return {"metric": METRIC, "n_gpus": n, "unavailable":
            "the GEMMs use cluster-multicast TMA loads: 1-GPU calls only"}


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)   # ~1 s timed: steady power and clocks
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload on fewer tokens (profiling captures)")
    ap.add_argument("--skip-aux", action="store_true",
                    help="skip the end-to-end and CPU-baseline legs (profiling captures)")
    ap.add_argument("--eager", dest="graph", action="store_false",
                    help="time the steps as individual launches instead of one CUDA graph")
    ap.add_argument("--graph", dest="graph", action="store_true",
                    help="time the K steps as one captured CUDA graph (the default)")
    ap.set_defaults(graph=True)
    ap.add_argument("--workload", default=WORKLOAD,
                    choices=["llama2_1b_attn_block", "llama2_7b_mlp", "llama2_13b_layer",
                             "svd_40b_pair", "tiny_block"],
                    help="the timed step's workload; the metric's own is the default, the "
                         "others report the step and its roofline only")
    ap.add_argument("--_oracle-sample", type=int, default=0, dest="oracle_sample")
    ap.add_argument("--_oracle-steps", type=int, default=1, dest="oracle_steps")
    args = ap.parse_args(argv)
    if args.oracle_sample:
        _oracle_sample_main(args.oracle_sample, args.oracle_steps, args.workload)
        return 0
    args.warmup = max(args.warmup, 3)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if args.workload != WORKLOAD:
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the oracle arm times the metric's own workload "
                                  f"({WORKLOAD}) only"}), flush=True)
            return 0
        return reference_arm(args, rank, world)
    if world > 1 or args.gpus > 1:
        # nothing is launched: the multicast GEMMs run in single-GPU processes only
        if rank == 0:
            print(json.dumps(multi_gpu_unavailable(max(world, args.gpus))), flush=True)
        return 0
    return ours_arm(args)


if __name__ == "__main__":
    sys.exit(main())
