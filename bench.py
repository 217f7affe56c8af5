#!/usr/bin/env python3
"""Throughput of the int4 routed-expert MoE layer on GB300 GPUs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl gb300|reference]

One step = one pass of the workload: for the default glm_decode workload, 256
independent tokens, each one moe_forward call (T = 1) of the GLM-5.2-shaped
layer (router, plan, 8 routed experts + shared expert, combine).  Inputs are
seeded synthetic tensors resident in HBM.  L2 is flushed (512 MiB read)
before every forward, outside the timed events, so that no expert weight is
served from L2.  `value` = tokens of all ranks / max-over-ranks device time.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(weak scaling, no data-path collective: the layer does not shard).
`--impl reference` times the CPU oracle (the reference arm) on rank 0.

Without --workload the run measures glm_decode (the headline line) and then,
at one GPU, glm_verify, glm_prefill, glm_stack, glm_prefill_uniform and
glm_decode_rowscale and glm_prefill_rowscale (one scale a row) as
sub-records of the same line, each timed for at least 1.5 s with its own
clock record.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s and achieved HBM GB/s (% of ~8 TB/s peak) on 1 GB300"
UNIT = "tokens/s"
FLUSH_BYTES = 512 << 20
NOMINAL_HBM_GBS = 8000.0


# ------------------------------------------------------------------ helpers --

def dist_env():
    return (int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)),
            int(os.environ.get("LOCAL_RANK", 0)))


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, summarised over a
    given window of the run (one timed region)."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.sw_power_cap,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-i", str(self.gpu)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 7:
                self.samples.append((time.monotonic(), parts))

    @staticmethod
    def now():
        return time.monotonic()

    def wait_first(self, timeout=10.0):
        end = time.monotonic() + timeout
        while not self.samples and time.monotonic() < end and self.proc is not None:
            time.sleep(0.05)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        """Median SM clock and the throttle reasons seen in [t0, t1]."""
        sm = []
        mx = None
        reasons = set()
        names = ("sw_power_cap", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")
        inside = [p for t, p in list(self.samples) if t0 <= t <= t1]
        for p in inside:
            try:
                sm.append(float(p[0]))
                mx = float(p[1])
            except ValueError:
                continue
            for n, v in zip(names, p[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def measured_tensor_peak():
    """Dense bf16 TFLOP/s (burst: the kernel is timed alone); f16 runs at the
    same rate on the tensor cores."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def phase_flops(phase, sh, T):
    """Tensor-core flops of one launch of a grouped-GEMM phase: 2 per
    multiply-add over every plan row and shared-expert row."""
    rows = T * sh.top_k
    srows = T if sh.n_shared else 0
    if phase == "tc_gate_up":
        return 2 * 2 * sh.hidden * (rows * sh.inter + srows * sh.i_shared)
    if phase == "tc_down":
        return 2 * sh.hidden * (rows * sh.inter + srows * sh.i_shared)
    return None


# Sources each profiled kernel is compiled from: its DRAM traffic in
# profiles/ncu_traffic.json is used only while these files are unchanged.
KERNEL_SOURCES = {
    "decode_fused": ("decode_fused.cuh", "decode_common.cuh", "decode_f1.cu", "decode_f2.cu",
                     "decode.cu", "stream_common.cuh", "router_math.cuh", "moe_internal.cuh"),
    "tc_gate_up": ("tc_gemm.cu", "tc_ptx.cuh", "stream_common.cuh", "moe_internal.cuh",
                   "smem_opt_in.cuh"),
    "tc_down": ("tc_gemm.cu", "tc_ptx.cuh", "stream_common.cuh", "moe_internal.cuh",
                "smem_opt_in.cuh"),
}


def kernel_source_hash(kernel: str):
    files = KERNEL_SOURCES.get(kernel)
    if files is None:
        return None
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "int4_routed_expert_gb300", "csrc")
    for name in sorted(files):
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the kernel's current sources."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            t = json.load(f)
    except (OSError, ValueError):
        return None
    hk = kernel_source_hash(kernel)
    if hk is None or t.get("source_hash", {}).get(kernel) != hk:
        return None
    return t.get("per_launch_bytes", {}).get(f"{workload}:{kernel}")


# ----------------------------------------------------- algorithmic bytes ----

def expert_gate_up_bytes(sh):
    """Gate and up weights with their scales, in the shape's format."""
    return 2 * sh.matrix_bytes(sh.inter, sh.hidden)


def expert_down_bytes(sh, inter=None):
    return sh.matrix_bytes(sh.hidden, inter or sh.inter)


def phase_bytes(phase, sh, T, n_act, x_bytes):
    """Algorithmic HBM bytes of one launch of a phase (weights read once,
    activations read once, outputs written once)."""
    H, E, k = sh.hidden, sh.n_experts, sh.top_k
    ns = 1 if sh.n_shared else 0
    router = E * H * 4 + E * 4
    hrows = (T * k + T * ns) * sh.inter * 4
    if phase == "decode_fused":
        # h stays between the kernel's two phases (L2), so it is not counted
        return (router + T * H * x_bytes + (n_act + ns) * expert_gate_up_bytes(sh)
                + n_act * expert_down_bytes(sh) + ns * expert_down_bytes(sh, sh.i_shared)
                + T * H * 4)
    if phase == "gate_up":
        return (n_act + ns) * expert_gate_up_bytes(sh) + T * H * 4 + hrows
    if phase == "down":
        return (n_act * expert_down_bytes(sh) + ns * expert_down_bytes(sh, sh.i_shared)
                + hrows + (T * k + T * ns) * H * 4)
    rows = T * k + T * ns  # plan rows + shared-expert rows of the f16 buffers
    if phase == "tc_prep":
        return T * H * 4 + rows * H * 2
    if phase == "tc_gate_up":
        return (n_act * expert_gate_up_bytes(sh) + ns * expert_gate_up_bytes(sh)
                + rows * H * 2 + rows * sh.inter * 2)
    if phase == "tc_down":
        return (n_act * expert_down_bytes(sh) + ns * expert_down_bytes(sh, sh.i_shared)
                + rows * sh.inter * 2 + rows * H * 4)
    return None


# ------------------------------------------------------------- workloads ----

def workload_key(wl, experts=None, tokens=None):
    key = f"{wl.name}_E{experts}" if experts else wl.name
    return f"{key}_T{tokens}" if tokens else key


def make_workload(name, experts=None, calls=None, tokens=None):
    from workloads import CONFIGS
    from workloads.configs import LayerShape, Workload
    wl = CONFIGS[name]
    if experts or calls or tokens:
        sh = wl.shape
        if experts:
            sh = LayerShape(sh.hidden, sh.inter, experts, sh.top_k, sh.n_group, sh.topk_group,
                            sh.routed_scaling_factor, sh.n_shared, sh.shared_inter,
                            sh.group_size)
        wl = Workload(wl.name, sh, tokens or wl.tokens_per_call, calls or wl.calls, wl.x_dtype,
                      wl.bias_kind, wl.seed, wl.layers, wl.correlated, wl.rmsnorm_eps,
                      wl.zipf_s)
    return wl


class DeviceRun:
    """Resident layers, inputs and outputs of one workload on one device."""

    def __init__(self, wl, dev, layers=None):
        import torch

        import int4_routed_expert_gb300 as m
        from workloads.gen import gen_activations, gen_layer, gen_norm_weight
        self.m, self.wl, self.dev = m, wl, dev
        sh = wl.shape
        self.T = wl.tokens_per_call
        self.calls = wl.calls
        self.n_layers = layers or wl.layers
        self.layers = [gen_layer(wl, layer=i, device=dev) for i in range(self.n_layers)]
        self.handles = [m.MoELayer(L, self.T) for L in self.layers]
        self.norm = wl.rmsnorm_eps > 0
        self.gammas = ([gen_norm_weight(wl, i).to(dev) for i in range(self.n_layers)]
                       if self.norm else [None] * self.n_layers)
        xs = [gen_activations(wl, self.T, call=c, dtype="f32" if self.norm else None)
              for c in range(self.calls)]
        self.x_host = torch.stack(xs).pin_memory()           # [calls, T, H]
        self.x = self.x_host.to(dev)
        self.x_bytes = self.x.element_size()
        self.y = torch.empty(self.calls, self.T, sh.hidden, dtype=torch.float32, device=dev)
        self.y_host = torch.empty_like(self.y, device="cpu").pin_memory()
        self.flush_buf = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.flush_buf.fill_(1.0)
        self.flush_out = torch.empty((), dtype=torch.float32, device=dev)
        self.stream = torch.cuda.current_stream()

    def flush(self):
        import torch
        torch.sum(self.flush_buf, dim=0, out=self.flush_out)

    def forward(self, c):
        """Layer stack on call c: y = MoE(x) (or the residual stack in place)."""
        if not self.norm:
            for h in self.handles:
                h.forward(self.x[c], y=self.y[c], stream=self.stream)
        else:
            y = self.y[c]
            y.copy_(self.x[c])
            for h, g in zip(self.handles, self.gammas):
                h.forward(y, y=y, gamma=g, eps=self.wl.rmsnorm_eps, accumulate=True,
                          stream=self.stream)

    def e2e_mode(self) -> str:
        """How the end-to-end pass moves x and y between host and device:
        "mapped" (x copied in by cudaMemcpyAsync, y written by the kernels
        straight into the pinned host buffer) for a small batch of one layer,
        "copy" (one cudaMemcpyAsync each way inside the events) for large
        batches and for the residual stack, whose layers update y in place."""
        return "mapped" if self.T <= 4 and not self.norm else "copy"

    def timed_pass(self, e2e=False, flush=True):
        """Device ms of one step: sum over calls of the forward's events."""
        import torch
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(self.calls)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(self.calls)]
        mapped = e2e and self.e2e_mode() == "mapped"
        for c in range(self.calls):
            if flush:
                self.flush()
            starts[c].record()
            if mapped:
                self.x[c].copy_(self.x_host[c], non_blocking=True)
                for h in self.handles:
                    h.forward(self.x[c], y=self.y_host[c], stream=self.stream)
            else:
                if e2e:
                    self.x[c].copy_(self.x_host[c], non_blocking=True)
                self.forward(c)
                if e2e:
                    self.y_host[c].copy_(self.y[c], non_blocking=True)
            ends[c].record()
        torch.cuda.synchronize()
        return sum(s.elapsed_time(e) for s, e in zip(starts, ends))

    def traced_pass(self):
        """Per-phase device ms (summed over the step) and launches per step."""
        import torch
        m = self.m
        for h in self.handles:
            m.moe_trace_enable(h.h, self.calls)
        for c in range(self.calls):
            self.flush()
            self.forward(c)
        torch.cuda.synchronize()
        phase_ms, launches, n_phase = {}, 0, {}
        for h in self.handles:
            names, rows = m.moe_trace_read(h.h, self.calls)
            for row in rows:
                for n, v in zip(names, row):
                    if v > 0:
                        phase_ms[n] = phase_ms.get(n, 0.0) + v
                        n_phase[n] = n_phase.get(n, 0) + 1
                        launches += 1
            m.moe_trace_enable(h.h, 0)
        return phase_ms, n_phase, launches

    def active_experts(self):
        """Mean distinct experts per call (from the plan of each call)."""
        import torch
        m = self.m
        sh = self.wl.shape
        tot = 0
        for c in range(min(self.calls, 32)):
            plan = m.Plan(self.T, sh.top_k, sh.n_experts, self.dev)
            x = self.x[c] if not self.norm else self.y[c]
            self.handles[0].route(x, gamma=self.gammas[0], eps=self.wl.rmsnorm_eps or 1e-5,
                                  plan=plan)
            tot += int(plan.n_active.item())
        torch.cuda.synchronize()
        return tot / min(self.calls, 32)

    def check_status(self):
        for h in self.handles:
            self.m.moe_device_status(h.h)


# ------------------------------------------------------------ oracle arm ----

class OracleArm:
    """The CPU oracle (single-thread C++) on sample tokens of the workload.

    Expert regeneration is input preparation, not the oracle's work: the
    experts the sample selects are generated before anything is timed."""

    def __init__(self, wl, n_calls):
        import numpy as np

        import oracle
        from workloads.gen import (SHARED_EXPERT, HostExpertCache, gen_activations,
                                   gen_norm_weight, gen_router)
        self.oracle, self.shared_id, self.wl = oracle, SHARED_EXPERT, wl
        sh = wl.shape
        self.norm = wl.rmsnorm_eps > 0
        # a bounded sample: at most 4 token rows of a call, at most 2 stacked layers
        self.rows = min(wl.tokens_per_call, 4)
        self.layers_run = 1 if not self.norm else min(wl.layers, 2)
        self.eps = float(np.float32(wl.rmsnorm_eps)) if self.norm else 0.0
        self.caches = [HostExpertCache(wl, i) for i in range(self.layers_run)]
        self.routers, self.gammas = [], []
        for i in range(self.layers_run):
            seed = wl.seed + i if wl.layers > 1 else wl.seed
            rw, rb = gen_router(sh, seed, i, wl.bias_kind, wl.zipf_s)
            self.routers.append((rw.numpy(), rb.numpy()))
            self.gammas.append(gen_norm_weight(wl, i).numpy() if self.norm else None)
        self.xs = [np.ascontiguousarray(
            gen_activations(wl, wl.tokens_per_call, call=c,
                            dtype="f32" if self.norm else None).float().numpy()[:self.rows])
            for c in range(n_calls)]
        for c in range(n_calls):
            h = self.xs[c]
            for i in range(self.layers_run):
                self._forward(i, h, warm=True)
                h = self._forward(i, h)

    def _forward(self, i, h, warm=False):
        if warm:
            _, _, ids, _ = self.oracle.route(self.wl.shape, *self.routers[i], h, self.eps,
                                             self.gammas[i])
            for e in set(ids.reshape(-1).tolist()) | {self.shared_id}:
                self.caches[i].expert(e)
            return None
        y, _, _, _ = self.oracle.moe_forward(
            self.wl.shape, *self.routers[i], self.caches[i].expert,
            self.caches[i].expert(self.shared_id), h, eps=self.eps, gamma=self.gammas[i],
            resid=h if self.norm else None)
        return y

    def run(self, c):
        """Seconds per token through the whole layer stack, for call c."""
        t0 = time.perf_counter()
        h = self.xs[c % len(self.xs)]
        for i in range(self.layers_run):
            h = self._forward(i, h)
        dt = time.perf_counter() - t0
        return dt / self.rows * (self.wl.layers / self.layers_run)

    def describe(self):
        return (f"{self.rows} token row(s) per call of {self.wl.name}, {self.layers_run} of "
                f"{self.wl.layers} layer(s) timed and scaled to the stack, single-thread C++ "
                "oracle, fp32 accumulation")


def max_over_ranks(values, world, device):
    """The per-rank timings reduced to their maximum over the ranks (the
    slowest rank sets the job's time); identity for one rank."""
    if world <= 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tokens_per_s(world, tokens_per_step, steps, ms):
    """Whole-job throughput: the tokens all ranks processed over the time."""
    return world * tokens_per_step * steps / (ms / 1000.0)


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    arm = OracleArm(wl, min(args.steps + args.warmup, 8))
    for w in range(args.warmup):
        arm.run(w)
    s_per_tok = 0.0
    for k in range(args.steps):
        s_per_tok += arm.run(args.warmup + k)
    value = args.steps / s_per_tok
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * s_per_tok / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "sample": arm.describe()},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": arm.describe()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------- main arm ----

# The workloads the default run measures after the headline (one process, one
# after another, each layer stack freed before the next is generated).
SUB_WORKLOADS = ("glm_verify", "glm_prefill", "glm_stack", "glm_prefill_uniform",
                 "glm_decode_rowscale", "glm_prefill_rowscale")
# A sub-record's timed region lasts at least this long, so that the 200 ms
# clock sampler sees several samples under load.
SUB_MIN_TIMED_S = 1.5

# Tokens a verify forward emits on average with the production MTP draft
# ("GLM-5.2 on a 32 GB Mac - native MLX port of the Colibri hierarchy", G4:
# 2.065 per forward; G5: 2.286).
ACCEPTED_PER_VERIFY = (("G4", 2.065), ("G5", 2.286))


def host_cpu():
    """The host's logical CPU count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu model")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return os.cpu_count(), model or "unknown"


def union_bytes_per_call(wl, n_act, x_bytes):
    """HBM bytes of one call that streams each selected expert once: the
    distinct experts of the call plus the shared one, the router, x and y."""
    sh = wl.shape
    T, H = wl.tokens_per_call, sh.hidden
    ns = 1 if sh.n_shared else 0
    return ((n_act + ns) * (expert_gate_up_bytes(sh) + expert_down_bytes(sh))
            + sh.n_experts * H * 4 + sh.n_experts * 4 + T * H * x_bytes + T * H * 4)


def measure(args, wl, dev, world, steps, warmup, clocks, min_timed_s=0.0, layers=None,
            experts=None, tokens=None):
    """One workload, timed: the fields of its bench line.

    steps: the timed steps (raised, when min_timed_s is given, until the timed
    region lasts at least that long, judged from the warm-up passes)."""
    import math

    import torch

    run = DeviceRun(wl, dev, layers)
    sh = wl.shape
    warm_ms = []
    for _ in range(max(warmup, 3)):
        warm_ms.append(run.timed_pass())
    run.check_status()
    if min_timed_s > 0:
        step_s = min(warm_ms) / 1000.0
        steps = max(steps, int(math.ceil(min_timed_s / max(step_s, 1e-6))))
    clocks.wait_first()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    barrier()
    t_start = clocks.now()
    dev_ms = 0.0
    for _ in range(steps):
        dev_ms += run.timed_pass()
    barrier()
    t_stop = clocks.now()
    run.check_status()

    # steady state without the L2 flush (weights of popular experts may stay in L2)
    unflushed_ms = run.timed_pass(flush=False)

    # end to end: inputs copied from pinned host memory and outputs read back
    # inside each forward's events
    e2e_ms = 0.0
    for _ in range(steps):
        e2e_ms += run.timed_pass(e2e=True)
    run.check_status()

    dev_ms, e2e_ms = max_over_ranks([dev_ms, e2e_ms], world, dev)

    tokens_step = wl.tokens_per_call * wl.calls
    value = job_tokens_per_s(world, tokens_step, steps, dev_ms)
    e2e_value = job_tokens_per_s(world, tokens_step, steps, e2e_ms)

    phase_ms, n_phase, launches_step = run.traced_pass()
    n_act = run.active_experts()
    peak, peak_kind = measured_peaks()
    dominant = max(phase_ms, key=phase_ms.get)
    per_launch_ms = phase_ms[dominant] / n_phase[dominant]
    T = wl.tokens_per_call
    kb = phase_bytes(dominant, sh, T, n_act, run.x_bytes)
    kernels = {}
    for name, ms in phase_ms.items():
        b = phase_bytes(name, sh, T, n_act, run.x_bytes)
        avg = ms / n_phase[name]
        kernels[name] = {"avg_us": round(1000 * avg, 3), "launches_per_step": n_phase[name],
                         "share": round(ms / sum(phase_ms.values()), 4)}
        if b:
            kernels[name]["algorithmic_bytes"] = b
            kernels[name]["achieved_gbs"] = round(b / (avg / 1000.0) / 1e9, 1)
        f = phase_flops(name, sh, T)
        if f:
            kernels[name]["tflops"] = round(f / (avg / 1000.0) / 1e12, 1)
    layer_bytes = sum(phase_bytes(n, sh, T, n_act, run.x_bytes) or 0 for n in phase_ms)
    ms_per_call = dev_ms / (steps * wl.calls * max(1, run.n_layers))
    layer_gbs = layer_bytes / (ms_per_call / 1000.0) / 1e9

    achieved = kb / (per_launch_ms / 1000.0) / 1e9
    roofline = {"bound": "hbm", "kernel": dominant,
                "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                "traffic": ncu_traffic(dominant, workload_key(wl, experts, tokens)),
                "algorithmic_bytes_per_launch": kb,
                "avg_launch_us": round(1000 * per_launch_ms, 3),
                "duration_source": "CUDA events between the kernels in a traced pass "
                                   "of the same step right after the timed region"}
    fl = phase_flops(dominant, sh, T)
    if wl.extra.get("bound") == "tensor" and fl:
        tpeak, tkind = measured_tensor_peak()
        tach = fl / (per_launch_ms / 1000.0) / 1e12
        roofline = {"bound": "tensor", "kernel": dominant, "achieved": round(tach, 1),
                    "peak": tpeak, "unit": "TFLOP/s", "frac": round(tach / tpeak, 4),
                    "peak_kind": tkind, "traffic": roofline["traffic"],
                    "algorithmic_flops_per_launch": fl,
                    "avg_launch_us": roofline["avg_launch_us"],
                    "duration_source": roofline["duration_source"],
                    "hbm": {"achieved": round(achieved, 1), "peak": peak, "unit": "GB/s"}}
    rec = {
        "value": value, "unit": UNIT, "steps": steps, "warmup": max(warmup, 3),
        "ms_per_step": dev_ms / steps, "timed_s": round(dev_ms / 1000.0, 3),
        "config": {
            "workload": wl.name, "hidden": sh.hidden, "inter": sh.inter,
            "n_experts": sh.n_experts, "top_k": sh.top_k, "layers": run.n_layers,
            "tokens_per_call": T, "calls_per_step": wl.calls,
            "tokens_per_step": tokens_step, "x_dtype": "f32" if run.norm else wl.x_dtype,
            "weights": "int4 offset-binary, group 32, fp16 scales",
            "l2": "flushed (512 MiB read) before every forward, outside the events",
            "unflushed_tokens_per_s": round(tokens_step / (unflushed_ms / 1000.0), 1),
            "parallelism": f"replicas x{world}",
        },
        "roofline": roofline,
        "layer_hbm": {"bytes_per_call": layer_bytes, "gbs": round(layer_gbs, 1),
                      "pct_of_8tbs": round(100 * layer_gbs / NOMINAL_HBM_GBS, 1),
                      "frac_of_measured": round(layer_gbs / peak, 4),
                      "mean_active_experts": n_act},
        "kernels": kernels,
        "e2e": {"value": e2e_value, "unit": UNIT,
                "h2d_bytes_per_step": int(run.x[0].numel() * run.x_bytes * wl.calls),
                "d2h_bytes_per_step": int(run.y[0].numel() * 4 * wl.calls),
                "method": ("x copied from pinned host memory (cudaMemcpyAsync), y written "
                           "by the kernels straight into pinned host memory, inside each "
                           "forward's events"
                           if run.e2e_mode() == "mapped" else
                           "x copied from and y copied to pinned host memory "
                           "(cudaMemcpyAsync) inside each forward's events")},
        "gpu_launches": launches_step * steps,
        "clocks": clocks.summary(t_start, t_stop),
    }
    if T > 1 and T <= 4:
        # a verify forward: bytes of the expert union it streams, per step,
        # per verified token and per emitted token
        ub = union_bytes_per_call(wl, n_act, run.x_bytes)
        calls_per_s = value / T
        rec["verify"] = {
            "union_bytes_per_call": ub, "bytes_per_step": ub * wl.calls,
            "bytes_per_verified_token": ub / T,
            "union_gbs": round(ub * calls_per_s / 1e9, 1),
            "union_frac_of_measured": round(ub * calls_per_s / 1e9 / peak, 4),
            "per_emitted_token": {
                f"{src} ({acc} tokens per forward)": {
                    "bytes": round(ub / acc, 1),
                    "emitted_tokens_per_s": round(calls_per_s * acc, 1)}
                for src, acc in ACCEPTED_PER_VERIFY},
            "source": "GLM-5.2 on a 32 GB Mac, G4 and G5 (accepted tokens per verify forward)",
        }
    del run
    torch.cuda.empty_cache()
    return rec


# The expert tier's record: glm_decode with the routed experts in pinned host
# memory and a quarter of them in HBM slots, some pinned.
TIER_SLOTS, TIER_PINNED = 64, 16


def measure_tier(dev, clocks, warmup, min_timed_s=SUB_MIN_TIMED_S, n_slots=TIER_SLOTS,
                 n_pinned=TIER_PINNED):
    """glm_decode through the expert tier (moe_tier_forward).

    The first warm-up step fills the slots and the use counts; the hot store
    is then seeded with the most-used experts (repin into free capacity, "GLM-
    5.2 on a 32 GB Mac", "What Colibri is actually doing", items 5-6).  A step
    is timed by the wall clock: each call routes, reads its union to the host,
    takes the slot decisions and copies its misses, so host time is part of
    it; the step ends with a device synchronisation."""
    import math

    import torch

    import int4_routed_expert_gb300 as m
    from workloads.gen import gen_activations, gen_layer

    wl = make_workload("glm_decode")
    sh = wl.shape
    L = gen_layer(wl, device=dev)
    x = torch.stack([gen_activations(wl, 1, call=c) for c in range(wl.calls)]).to(dev)
    y = torch.empty(wl.calls, 1, sh.hidden, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    tier = None

    def step():
        t0 = time.perf_counter()
        for c in range(wl.calls):
            tier.forward(x[c], y=y[c], stream=stream)
        torch.cuda.synchronize()
        return time.perf_counter() - t0

    # the same path with a slot for every expert: after one step every call
    # hits, so this is the cost of routing, read-back and the expert kernels
    tier = m.ExpertTier(L, max_tokens=1, n_slots=sh.n_experts)
    step()
    resident_s = min(step() for _ in range(2))
    tier.close()
    tier = None  # its pinned host copy is released before the next one is made
    tier = m.ExpertTier(L, max_tokens=1, n_slots=n_slots, n_pinned=n_pinned,
                        drop_device_routed=True)
    del L
    torch.cuda.empty_cache()
    # the host link: one routed array (all experts' gate weights) copied from
    # its page-locked host copy into HBM
    src = tier.host["gate_q"]
    dst = torch.empty(src.shape, dtype=src.dtype, device=dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    link_gbs = 0.0
    for _ in range(3):
        e0.record()
        dst.copy_(src, non_blocking=True)
        e1.record()
        e1.synchronize()
        link_gbs = max(link_gbs, src.numel() * src.element_size() / (e0.elapsed_time(e1) / 1e3)
                       / 1e9)
    del dst
    torch.cuda.empty_cache()
    step()
    pins = tier.repin(0)
    step_s = min(step() for _ in range(max(warmup, 3) - 1))
    steps = max(1, int(math.ceil(min_timed_s / max(step_s, 1e-6))))
    s0 = tier.query()[0]
    clocks.wait_first()
    t_start = clocks.now()
    secs = sum(step() for _ in range(steps))
    t_stop = clocks.now()
    s1 = tier.query()[0]
    d = {k: s1[k] - s0[k] for k in ("hits_pinned", "hits_lru", "misses", "loads", "evictions",
                                    "h2d_bytes")}
    tokens = steps * wl.calls
    admitted = d["hits_pinned"] + d["hits_lru"] + d["misses"]
    eb = sh.expert_bytes()
    rec = {
        "value": tokens / secs, "unit": UNIT, "steps": steps, "warmup": max(warmup, 3),
        "ms_per_step": 1000.0 * secs / steps, "timed_s": round(secs, 3),
        "config": {
            "workload": "glm_decode_tier", "hidden": sh.hidden, "inter": sh.inter,
            "n_experts": sh.n_experts, "top_k": sh.top_k, "tokens_per_call": 1,
            "calls_per_step": wl.calls, "tokens_per_step": wl.calls,
            "hbm_slots": n_slots, "pinned_slots": n_pinned,
            "host_store_bytes": sh.n_experts * eb, "hbm_slot_bytes": n_slots * eb,
            "weights": "int4 offset-binary, group 32, fp16 scales",
            "timing": "wall clock per step (routing, union read-back, slot decisions and "
                      "host-to-HBM expert copies inside), device synchronised at the end "
                      "of each step; L2 not flushed",
        },
        "tier": {
            "hit_rate": round((d["hits_pinned"] + d["hits_lru"]) / max(admitted, 1), 4),
            "pinned_hit_rate": round(d["hits_pinned"] / max(admitted, 1), 4),
            "experts_per_token": round(admitted / tokens, 3),
            "misses_per_token": round(d["misses"] / tokens, 3),
            "evictions_per_token": round(d["evictions"] / tokens, 3),
            "h2d_bytes_per_token": round(d["h2d_bytes"] / tokens, 1),
            "h2d_gbs": round(d["h2d_bytes"] / secs / 1e9, 1),
            "pins_seeded": pins,
            "host_link_h2d_gbs": round(link_gbs, 1),
            "copy_bound_tokens_per_s": round(link_gbs * 1e9 / max(d["h2d_bytes"] / tokens, 1), 1),
            "all_resident_tokens_per_s": round(wl.calls / resident_s, 1),
            "host_link_source": "cudaMemcpyAsync of one routed array (all experts' gate "
                                "weights) from page-locked host memory into HBM, CUDA events",
        },
        "clocks": clocks.summary(t_start, t_stop),
    }
    tier.close()
    del tier, x, y
    torch.cuda.empty_cache()
    return rec


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=None,
                    choices=["tiny", "glm_decode", "glm_verify", "glm_prefill", "glm_stack",
                             "glm_prefill_uniform", "glm_decode_rowscale",
                             "glm_prefill_rowscale", "glm_decode_tier"],
                    help="one workload only (default: glm_decode, then the other GLM "
                         "workloads as sub-records)")
    ap.add_argument("--experts", type=int, default=None, help="override E (profiling only)")
    ap.add_argument("--calls", type=int, default=None, help="override calls per step")
    ap.add_argument("--layers", type=int, default=None, help="override stacked layers")
    ap.add_argument("--tokens", type=int, default=None,
                    help="override tokens per call (profiling only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-records", action="store_true")
    ap.add_argument("--tier-slots", type=int, default=TIER_SLOTS,
                    help="HBM expert slots of the glm_decode_tier record")
    ap.add_argument("--tier-pinned", type=int, default=TIER_PINNED,
                    help="of which pinned (the hot store)")
    args = ap.parse_args()
    single = args.workload is not None
    name = args.workload or "glm_decode"
    if name == "glm_decode_tier":
        run_tier_only(args)
        return
    wl = make_workload(name, args.experts, args.calls, args.tokens)

    if args.impl == "reference":
        run_reference(args, wl)
        return

    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = f"cuda:{local}"
    torch.cuda.set_device(dev)

    import __graft_entry__
    __graft_entry__.build()

    clocks = ClockSampler(local)
    clocks.start()
    rec = measure(args, wl, dev, world, args.steps, args.warmup, clocks, layers=args.layers,
                  experts=args.experts, tokens=args.tokens)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        T = wl.tokens_per_call
        n_calls = 8 if T == 1 else 2
        arm = OracleArm(wl, n_calls)
        s_tok = sum(arm.run(c) for c in range(n_calls)) / n_calls
        nproc, model = host_cpu()
        cpu = {"value": 1.0 / s_tok, "unit": UNIT, "cores": 1, "host_nproc": nproc,
               "cpu_model": model, "kind": "oracle",
               "sample": f"{n_calls} call(s): " + arm.describe()}

    subs = None
    if not single and not args.no_sub_records and world == 1:
        subs = {}
        for sub in SUB_WORKLOADS:
            swl = make_workload(sub)
            subs[sub] = measure(args, swl, dev, world, 1, args.warmup, clocks,
                                min_timed_s=SUB_MIN_TIMED_S)
        try:
            subs["glm_decode_tier"] = measure_tier(dev, clocks, args.warmup)
        except Exception as e:  # the headline line must still be printed
            subs["glm_decode_tier"] = {"error": f"{type(e).__name__}: {e}"}
    clocks.stop()

    if rank == 0:
        line = {
            "metric": METRIC, "value": rec["value"], "unit": UNIT, "n_gpus": world,
            "steps": rec["steps"], "warmup": rec["warmup"], "ms_per_step": rec["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded int4 weights, fp16 scales, Zipf router bias)",
            "config": rec["config"],
            "roofline": rec["roofline"],
            "layer_hbm": rec["layer_hbm"],
            "kernels": rec["kernels"],
            "cpu_baseline": cpu,
            "e2e": rec["e2e"],
            "gpu_launches": rec["gpu_launches"],
            "clocks": rec["clocks"],
            "timed_s": rec["timed_s"],
        }
        if "verify" in rec:
            line["verify"] = rec["verify"]
        if subs is not None:
            line["sub_records"] = subs
        elif not single and world > 1:
            line["sub_records"] = "measured at one GPU only"
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_tier_only(args):
    """--workload glm_decode_tier: the tier's record alone, as one line."""
    import torch
    dev = "cuda:0"
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()
    clocks = ClockSampler(0)
    clocks.start()
    rec = measure_tier(dev, clocks, args.warmup, n_slots=args.tier_slots,
                       n_pinned=args.tier_pinned)
    clocks.stop()
    line = {"metric": METRIC, "n_gpus": 1, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32",
            "data": "synthetic (seeded int4 weights, fp16 scales, Zipf router bias)"}
    line.update(rec)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
