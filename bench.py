"""Throughput of the MoE layer on B300, one JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--no-configs] [--no-cpu]

A step is one forward pass of the whole layer (gate GEMM, softmax / top-k /
capacity / slots, dispatch, grouped expert FFN, combine) over one batch of
synthetic input, through the library's C ABI.  The headline workload is the
64-expert layer (S=16384, d=2048, E=64, f=5120, top-2, cf=1.25, bf16).  The
line also carries, under `configs`, the same measurement for every other
layer configuration (the tiny fp32 layer, the 8-expert layer, the skewed
16-expert layer with and without the capacity cap, and the 32-expert
training step, forward + backward), and the decode shape and the PR-MoE
forward of the 64-expert layer.

Each configuration reports tokens/s, per-stage times, the expert GEMMs'
TFLOP/s against the measured dense bf16 peak, the gate / dispatch / combine
GB/s against the measured HBM copy bandwidth (in the loop, and with L2
flushed before each launch), rows kept and tokens dropped, and -- in its
`cpu_baseline` leg, where the float64 oracle is timed on the whole batch --
how many tokens the oracle's own float64 routing sends elsewhere than the
GPU (routing flips) and the largest top-k margin among them.

Multi-GPU: the layer does not shard in this library, so N GPUs run N
independent replicas (one process per GPU under torchrun); `value` is the
tokens all ranks processed over the max-over-ranks time.

`--impl reference` times the float64 CPU oracle instead (rank 0 only), on a
bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s (bf16 fwd/fwd+bwd); % of BF16 TC peak and HBM GB/s"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.json")
GEMM_SOURCES = ["gemm_tc.cu", "tc_ptx.cuh", "common.cuh", "kernels.h"]
CONFIG_NAMES = ["tiny_fp32", "e8_bf16", "skew_e16_drop", "skew_e16_nodrop", "train_e32"]
# a timed region this long under the power cap is held against the sustained
# dense bf16 peak; shorter regions run at the burst clock
SUSTAINED_REGION_S = 2.0


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(PEAKS_FALLBACK), "fallback"


def gemm_source_sha() -> str:
    h = hashlib.sha256()
    for f in GEMM_SOURCES:
        with open(os.path.join(ROOT, "mixture_experts_layer_86_b300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per GEMM launch from the committed ncu summary; None if the
    kernel source changed since the capture."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    with open(TRAFFIC_FILE) as fh:
        d = json.load(fh)
    ent = d.get("tc_gemm_kernel")
    if not ent or ent.get("source_sha") != gemm_source_sha() or ent.get("workload") != workload:
        return None
    return int(ent["dram_bytes_per_launch"])


def workload_desc(wl) -> str:
    what = "forward+backward" if wl.backward else "forward"
    return (f"{wl.name}: MoE layer {what} S={wl.num_tokens} d={wl.hidden_size} "
            f"E={wl.num_experts} f={wl.ffn_size} top-{wl.k} cf={wl.capacity_factor} "
            f"min_cap={wl.min_capacity} drop={wl.drop_tokens} {wl.act} {wl.dtype}"
            + (f" skew={wl.skew}" if wl.skew else ""))


def forward_launches(wl, fused: bool, num_sms: int) -> int:
    """Kernels one forward pass launches: the gate -- one launch for bf16
    batches of at most 128 tokens per SM, else three (fused gate kernel, slot
    scan, slot assignment); four for fp32 (router GEMM, top-k, scan,
    assignment) -- the dispatch copy unless it is fused into the first expert
    GEMM, the two expert GEMMs and the combine."""
    if wl.dtype == "bf16":
        gate = 1 if wl.num_tokens <= 128 * num_sms else 3
    else:
        gate = 4
    return gate + (0 if fused else 1) + 2 + 1


# ------------------------------------------------------------------ clocks
class _NvmlCtypes:
    """The few read-only NVML queries the sampler needs, straight from
    libnvidia-ml through ctypes (for hosts without the pynvml module)."""
    NVML_CLOCK_SM = 1

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        self.lib = lib
        if lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit_v2 failed")
        self.handle = ctypes.c_void_p()
        bus = None
        try:
            import torch
            p = torch.cuda.get_device_properties(index)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0".encode()
        except Exception:  # noqa: BLE001
            bus = None
        if bus is None or lib.nvmlDeviceGetHandleByPciBusId_v2(bus, ctypes.byref(self.handle)):
            if lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle)) != 0:
                raise RuntimeError("no NVML handle")
        try:
            self._reasons_fn = lib.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self._reasons_fn = lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _u32(self, fn, *args):
        v = self.ct.c_uint()
        if fn(self.handle, *args, self.ct.byref(v)) != 0:
            raise RuntimeError(fn.__name__)
        return v.value

    def sm(self):
        return float(self._u32(self.lib.nvmlDeviceGetClockInfo, self.NVML_CLOCK_SM))

    def sm_max(self):
        return float(self._u32(self.lib.nvmlDeviceGetMaxClockInfo, self.NVML_CLOCK_SM))

    def power_w(self):
        return self._u32(self.lib.nvmlDeviceGetPowerUsage) / 1000.0

    def reasons(self):
        v = self.ct.c_ulonglong()
        if self._reasons_fn(self.handle, self.ct.byref(v)) != 0:
            raise RuntimeError("clock event reasons")
        return int(v.value)


class _NvmlPy:
    """The same queries through the pynvml module."""

    def __init__(self, index: int):
        import pynvml
        pynvml.nvmlInit()
        self.n = pynvml
        try:
            import torch
            p = torch.cuda.get_device_properties(index)
            bus = f"{p.pci_domain_id:08x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"
            self.handle = pynvml.nvmlDeviceGetHandleByPciBusId(bus)
        except Exception:  # noqa: BLE001
            self.handle = pynvml.nvmlDeviceGetHandleByIndex(index)

    def sm(self):
        return float(self.n.nvmlDeviceGetClockInfo(self.handle, self.n.NVML_CLOCK_SM))

    def sm_max(self):
        return float(self.n.nvmlDeviceGetMaxClockInfo(self.handle, self.n.NVML_CLOCK_SM))

    def power_w(self):
        return self.n.nvmlDeviceGetPowerUsage(self.handle) / 1000.0

    def reasons(self):
        try:
            return int(self.n.nvmlDeviceGetCurrentClocksEventReasons(self.handle))
        except Exception:  # noqa: BLE001
            return int(self.n.nvmlDeviceGetCurrentClocksThrottleReasons(self.handle))


class ClockSampler:
    """SM clock, power and clock-event reasons of one GPU, polled from a
    background thread while the timed region runs (read-only NVML queries,
    through pynvml or directly through libnvidia-ml; one nvidia-smi reading
    after the region when neither works)."""

    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40),
               ("sw_thermal_slowdown", 0x20), ("sw_power_cap", 0x4))

    def __init__(self, device_index: int, interval_s: float = 0.0002):
        self.index = device_index
        self.interval = interval_s
        self.rows = []
        self.stop_evt = threading.Event()
        self.thread = None
        self.nvml = None
        self.source = "none"
        self.nvml_error = None
        errors = []
        for name, cls in (("nvml (pynvml)", _NvmlPy), ("nvml (libnvidia-ml via ctypes)", _NvmlCtypes)):
            try:
                backend = cls(device_index)
                self.sm_max = backend.sm_max()
                backend.sm()
                backend.reasons()
                self.nvml, self.source = backend, name
                break
            except Exception as e:  # noqa: BLE001  (reported in the clocks record)
                errors.append(f"{name}: {type(e).__name__}: {e}")
        if self.nvml is None:
            self.nvml_error = "; ".join(errors)

    def _poll(self):
        n = self.nvml
        while not self.stop_evt.is_set():
            try:
                self.rows.append((n.sm(), n.power_w(), n.reasons()))
            except Exception:  # noqa: BLE001
                pass
            time.sleep(self.interval)

    def start(self):
        self.rows = []
        self.stop_evt.clear()
        if self.nvml is not None:
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()

    def stop(self):
        if self.thread is None:
            return self._smi_once()
        self.stop_evt.set()
        self.thread.join()
        self.thread = None
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": self.sm_max, "reasons": ["no samples"],
                    "samples": 0, "source": self.source}
        reasons = sorted({name for _, _, bits in rows for name, b in self.REASONS if bits & b})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_min_mhz": min(r[0] for r in rows),
                "sm_max_mhz": self.sm_max, "power_w_max": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows), "source": self.source}

    def _smi_once(self):
        rec = self._smi_query()
        if self.nvml_error:
            rec["nvml_error"] = self.nvml_error
        return rec

    def _smi_query(self):
        q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")
        try:
            out = subprocess.run(["nvidia-smi", "-i", str(self.index), f"--query-gpu={q}",
                                  "--format=csv,noheader,nounits"], capture_output=True,
                                 text=True, timeout=10).stdout.strip().split(",")
            v = [s.strip() for s in out]
            names = [n for n, _ in self.REASONS]
            return {"sm_mhz": float(v[0]), "sm_max_mhz": float(v[1]), "power_w_max": float(v[2]),
                    "reasons": [names[i] for i in range(4) if v[3 + i] == "Active"],
                    "samples": 1, "source": "nvidia-smi after the region"}
        except Exception:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock source"],
                    "samples": 0, "source": "none"}


# ------------------------------------------------------------- replica timing
def reduce_max(v: float, world: int, device) -> float:
    """The maximum of v over the ranks of the default process group (v itself
    on one rank): the job's time is its slowest replica's."""
    if world == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput of `world` replicas that each ran `steps` steps of
    `tokens_per_step` tokens in `ms` milliseconds (the max over ranks)."""
    return world * tokens_per_step * steps / (ms * 1e-3)


# ------------------------------------------------------------------ one layer
STAGES = ("gate", "dispatch", "expert_ffn", "combine")


class LayerRun:
    """Device state of one workload (inputs, buffers, workspaces) and its
    stage calls through the C ABI.  The forward runs the stage entry points,
    the kernels moe_forward launches in its order: moe_dispatch then
    moe_expert_ffn, or with fused=True the expert FFN reading the token rows
    straight from x (moe_expert_ffn_gather, no x_disp copy)."""

    def __init__(self, wl, dev, fused=None):
        import torch

        from mixture_experts_layer_86_b300 import _native as N
        from mixture_experts_layer_86_b300 import layer as L
        from mixture_experts_layer_86_b300.inputs import make_inputs
        self.N, self.torch = N, torch
        self.wl = wl
        self.cfg = N.config_from_workload(wl)
        self.inp_cpu = make_inputs(wl)
        self.d = self.inp_cpu.to(dev)
        self.train = wl.backward
        self.fused = False if fused is None else fused
        self.names = (("gate", "expert_ffn", "combine") if self.fused else STAGES) + \
            (("backward",) if self.train else ())
        self.bufs = L.alloc_buffers(self.cfg, dev, training=self.train,
                                    fused_dispatch=self.fused)
        self.bufs["logits"] = None      # optional output of the gate; nothing downstream reads it
        self.ws = L.alloc_workspace(self.cfg, dev)
        self.y = torch.empty_like(self.d.x)
        if self.train:
            d = self.d
            self.wsb = L.alloc_workspace(self.cfg, dev, for_backward=True)
            self.grads = {"dx": torch.empty_like(d.x), "dw_gate": torch.empty_like(d.w_gate),
                          "dw1": torch.empty_like(d.w1), "db1": torch.empty_like(d.b1),
                          "dw2": torch.empty_like(d.w2), "db2": torch.empty_like(d.b2)}

    def stage(self, name, st):
        N, d, b, c = self.N, self.d, self.bufs, self.cfg
        if name == "gate":
            N.moe_gate_topk(c, d.x, d.w_gate, d.logit_bias, b["logits"], b["probs"], b["topk_idx"],
                            b["topk_w"], b["slot"], b["routed_cnt"], b["kept_cnt"],
                            b["expert_offsets"], b["row_src"], b["l_aux"], self.ws, st)
        elif name == "dispatch":
            N.moe_dispatch(c, d.x, b["topk_idx"], b["slot"], b["expert_offsets"], b["x_disp"], st)
        elif name == "expert_ffn" and self.fused:
            N.moe_expert_ffn_gather(c, d.x, b["row_src"], b["expert_offsets"], d.w1, d.b1, d.w2,
                                    d.b2, b["h_pre"], b["h"], b["out_disp"], st)
        elif name == "expert_ffn":
            N.moe_expert_ffn(c, b["x_disp"], b["expert_offsets"], d.w1, d.b1, d.w2, d.b2,
                             b["h_pre"], b["h"], b["out_disp"], st)
        elif name == "combine":
            N.moe_combine(c, b["out_disp"], b["topk_idx"], b["slot"], b["expert_offsets"],
                          b["topk_w"], self.y, st)
        elif name == "backward":
            g = self.grads
            N.moe_backward(c, d.x, d.w_gate, d.w1, d.w2, b, d.dy, g["dx"], g["dw_gate"], g["dw1"],
                           g["db1"], g["dw2"], g["db2"], self.wsb, st)

    def step(self, st, ev=None, marks=()):
        """One step; ev[i] is recorded just before the i-th stage named in
        `marks` ("end": after the last stage)."""
        j = 0
        for name in self.names + ("end",):
            if ev is not None and name in marks:
                ev[j].record(st)
                j += 1
            if name != "end":
                self.stage(name, st)

    def rows(self) -> int:
        return int(self.bufs["expert_offsets"][-1].item())


def _events(torch, n_steps, n_ev):
    return [[torch.cuda.Event(enable_timing=True) for _ in range(n_ev)] for _ in range(n_steps)]


def timed(torch, st, steps, body, barrier=None):
    """Milliseconds of `steps` calls of body(i) between two events on st."""
    if barrier:
        barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for i in range(steps):
        body(i)
    e1.record(st)
    torch.cuda.synchronize()
    if barrier:
        barrier()
    return e0.elapsed_time(e1)


def host_link(torch, dev, x_host, y_host, reps=10):
    """Copy bandwidth of the host link for the end-to-end leg's own pinned
    buffers: host-to-device alone, device-to-host alone, and both at once on
    two streams (the pipeline's steady state), in GB/s per direction."""
    xd, yd = torch.empty_like(x_host, device=dev), torch.empty_like(y_host, device=dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    nbytes = x_host.numel() * x_host.element_size()

    def run(h2d, d2h):
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(s_in)
        ev[2].record(s_out)
        for _ in range(reps):
            if h2d:
                with torch.cuda.stream(s_in):
                    xd.copy_(x_host, non_blocking=True)
            if d2h:
                with torch.cuda.stream(s_out):
                    y_host.copy_(yd, non_blocking=True)
        ev[1].record(s_in)
        ev[3].record(s_out)
        torch.cuda.synchronize()
        return max(ev[0].elapsed_time(ev[1]) if h2d else 0.0,
                   ev[2].elapsed_time(ev[3]) if d2h else 0.0) / reps

    run(True, True)
    t_in, t_out, t_both = run(True, False), run(False, True), run(True, True)
    del xd, yd
    gbs = lambda ms: nbytes / (ms * 1e-3) / 1e9
    return {"bytes": nbytes, "h2d_gbs": gbs(t_in), "d2h_gbs": gbs(t_out),
            "both_gbs_per_direction": gbs(t_both), "both_ms": t_both}


def stage_bytes(wl, R, with_probs=False):
    """Algorithmic HBM bytes of the gate, dispatch and combine stages: each
    input read once, each output written once."""
    S, d, E, k = wl.num_tokens, wl.hidden_size, wl.num_experts, wl.k
    eb = 2 if wl.dtype == "bf16" else 4
    return {"gate": S * d * eb + E * d * eb + S * k * 12 + R * 4 + (S * E * 4 if with_probs else 0),
            "dispatch": S * d * eb + R * d * eb + S * k * 8,
            "combine": R * d * eb + S * d * eb + S * k * 12}


def step_roofline(wl, R, peaks, ms_per_step):
    """The step's floor: for every kernel of one step the larger of its
    tensor time (its FLOP at the burst bf16 peak) and its memory time (its
    algorithmic bytes at the measured copy bandwidth), summed.  Weights,
    activations and gradients are bf16, each read or written once.
    frac = floor / measured step time."""
    S, d, f, E, k = wl.num_tokens, wl.hidden_size, wl.ffn_size, wl.num_experts, wl.k
    eb = 2
    train = wl.backward
    byt = stage_bytes(wl, R, with_probs=train)
    gemm = 2.0 * R * d * f
    wb = E * d * f * eb  # one expert weight tensor (W1 or W2)
    ks = [("gate", 0.0, byt["gate"]), ("dispatch", 0.0, byt["dispatch"]),
          ("W1", gemm, wb + R * d * eb + (2 if train else 1) * R * f * eb),
          ("W2", gemm, wb + R * f * eb + R * d * eb),
          ("combine", 0.0, byt["combine"])]
    if train:
        ks += [("combine_bwd", 0.0, S * d * eb + 2 * R * d * eb + S * k * 4),
               ("dW2", gemm, R * d * eb + R * f * eb + wb),
               ("db2", 0.0, R * d * eb),
               ("dh", gemm, wb + R * d * eb + 2 * R * f * eb),
               ("dW1", gemm, R * f * eb + R * d * eb + wb),
               ("dx_disp", gemm, wb + R * f * eb + R * d * eb),
               # router backward: probs in, dW_g = dlogitsT x, and
               # dX = dlogits W_g + the gathered dx_disp rows
               ("router", 4.0 * S * d * E,
                S * E * 4 + S * d * eb + E * d * eb + R * d * eb + S * d * eb)]
    kern = {}
    for name, flops, nbytes in ks:
        t_tc = flops / (peaks["bf16_tflops"] * 1e12) * 1e6
        t_mem = nbytes / (peaks["hbm_gbs"] * 1e9) * 1e6
        kern[name] = {"us": round(max(t_tc, t_mem), 2), "bound": "tensor" if t_tc > t_mem else "hbm",
                      "flop": flops, "bytes": nbytes}
    floor_ms = sum(v["us"] for v in kern.values()) * 1e-3
    return {"floor_ms": floor_ms, "frac": floor_ms / ms_per_step, "kernels": kern,
            "peaks": "burst bf16 tensor, measured copy bandwidth"}


def stage_breakdown(run, st, steps, peaks):
    """Per-stage times from a loop with an event at every stage boundary (a
    separate loop from the headline one, so its events do not perturb it)."""
    torch = run.torch
    names = run.names
    evs = _events(torch, steps, len(names) + 1)
    timed(torch, st, steps, lambda i: run.step(st, evs[i], marks=names + ("end",)))
    ms = {n: statistics.mean(e[j].elapsed_time(e[j + 1]) for e in evs) for j, n in enumerate(names)}
    R = run.rows()
    wl = run.wl
    byt = stage_bytes(wl, R, with_probs=run.train)
    out = {}
    for n in names:
        ent = {"ms": ms[n]}
        if n in byt:
            gbs = byt[n] / (ms[n] * 1e-3) / 1e9
            ent.update({"bytes": byt[n], "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]})
        out[n] = ent
    ffn_flops = 4.0 * R * wl.hidden_size * wl.ffn_size
    out["expert_ffn"]["TFLOP/s"] = ffn_flops / (ms["expert_ffn"] * 1e-3) / 1e12
    if wl.dtype == "bf16":
        out["expert_ffn"]["frac_bf16_burst"] = out["expert_ffn"]["TFLOP/s"] / peaks["bf16_tflops"]
    return out


def stages_cold_l2(run, st, peaks, reps=10):
    """Gate, dispatch and combine launched alone with L2 flushed before each
    launch: their HBM bandwidth without help from data that an earlier stage
    left in the 126 MB L2.  The flush READS a 512 MB buffer, so the L2 holds
    clean lines and no write-back of the flush lands inside the timed
    launch."""
    torch = run.torch
    flush = torch.ones(512 << 20, dtype=torch.uint8, device=run.d.x.device)
    flush.max()
    R = run.rows()
    byt = stage_bytes(run.wl, R, with_probs=run.train)
    out = {}
    for n in ("gate", "dispatch", "combine"):
        if n not in run.names:
            continue
        t = []
        for i in range(reps):
            flush.max()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            run.stage(n, st)
            e1.record(st)
            torch.cuda.synchronize()
            t.append(e0.elapsed_time(e1))
        ms = statistics.median(t)
        gbs = byt[n] / (ms * 1e-3) / 1e9
        out[n] = {"ms": ms, "GB/s": gbs, "frac_hbm": gbs / peaks["hbm_gbs"]}
    del flush
    return out


def routing_stats(run):
    import numpy as np
    b = run.bufs
    slot = b["slot"].cpu().numpy()
    routed = b["routed_cnt"].cpu().numpy()
    kept = b["kept_cnt"].cpu().numpy()
    S, k = run.wl.num_tokens, run.wl.k
    R = int(kept.sum())
    return {"rows_kept": R, "dropped_choices": int(S * k - R),
            "fully_dropped_tokens": int(np.count_nonzero((slot < 0).all(axis=1))),
            "routed_max": int(routed.max()), "routed_min": int(routed.min()),
            "experts_used": int(np.count_nonzero(kept))}


# --------------------------------------------------------------------- GPU arm
def run_gpu(args):
    import torch
    import torch.distributed as dist

    from mixture_experts_layer_86_b300 import _native as N
    from mixture_experts_layer_86_b300 import layer as L
    from mixture_experts_layer_86_b300.inputs import WORKLOADS

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    def barrier():
        if world > 1:
            dist.barrier()

    def max_over_ranks(v: float) -> float:
        return reduce_max(v, world, dev)

    peaks, peak_src = load_peaks()
    wl = WORKLOADS[args.workload]
    run = LayerRun(wl, dev)
    cfg, d = run.cfg, run.d
    st = torch.cuda.current_stream()
    S, dm, f, E = wl.num_tokens, wl.hidden_size, wl.ffn_size, wl.num_experts
    eb = 2 if wl.dtype == "bf16" else 4

    for _ in range(max(args.warmup, 3)):
        run.step(st)
    torch.cuda.synchronize()
    R = run.rows()

    # ---- value: K forward steps, inputs resident in HBM.  The only events
    # inside are the two around the expert FFN (its two GEMM launches), which
    # give the dominant kernel's launch time for the roofline.
    ffn_ev = _events(torch, args.steps, 2)
    sampler = ClockSampler(local)
    sampler.start()
    ms = timed(torch, st, args.steps,
               lambda i: run.step(st, ffn_ev[i], marks=("expert_ffn", "combine")), barrier)
    clocks = sampler.stop()
    ms = max_over_ranks(ms)
    ffn_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ffn_ev)

    # ---- the same K steps through the single moe_forward call, and through
    # moe_forward with an x_disp buffer (the dispatch as its own copy kernel)
    fwd_call_ms = max_over_ranks(timed(torch, st, args.steps, lambda i: N.moe_forward(
        cfg, d.x, d.w_gate, d.logit_bias, d.w1, d.b1, d.w2, d.b2, run.y, run.bufs, run.ws, st)))
    bufs_fused = L.alloc_buffers(cfg, dev, fused_dispatch=True)
    bufs_fused["logits"] = None
    fused_ms = max_over_ranks(timed(torch, st, args.steps, lambda i: N.moe_forward(
        cfg, d.x, d.w_gate, d.logit_bias, d.w1, d.b1, d.w2, d.b2, run.y, bufs_fused, run.ws, st)))
    del bufs_fused
    stages = stage_breakdown(run, st, args.steps, peaks)
    cold = stages_cold_l2(run, st, peaks)
    rstats = routing_stats(run)

    # ---- e2e: host buffers, copies inside the timed region.  Each step
    # copies its batch host -> device, runs moe_forward and copies y, l_aux
    # and the expert counts back; HostPipeline overlaps the copies of
    # neighbouring steps with the forward (two slots, three streams).
    inp_cpu = run.inp_cpu
    x_host = [inp_cpu.x.pin_memory(), inp_cpu.x.clone().pin_memory()]
    y_host = [torch.empty_like(inp_cpu.x).pin_memory() for _ in range(2)]
    laux_host = [torch.empty((1,), dtype=torch.float32).pin_memory() for _ in range(2)]
    kept_host = [torch.empty((E,), dtype=torch.int32).pin_memory() for _ in range(2)]
    pipe = L.HostPipeline(cfg, d.w_gate, d.logit_bias, d.w1, d.b1, d.w2, d.b2, dev)

    def e2e_run(n):
        for i in range(n):
            pipe.submit(x_host[i % 2], y_host[i % 2], laux_host[i % 2], kept_host[i % 2])

    e2e_run(4)
    pipe.synchronize()
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.s_in)            # before the first copy in
    e2e_run(args.steps)
    e1.record(pipe.s_out)           # after the last copy out
    pipe.synchronize()
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1))
    barrier()
    # the last step's result really is on the host
    assert torch.equal(y_host[(args.steps - 1) % 2], run.y.cpu()), "e2e result differs"
    del pipe
    link = host_link(torch, dev, x_host[0], y_host[0])

    decode = decode_step(args, dev, max_over_ranks, world, peaks)
    residual = residual_step(args, dev, run, max_over_ranks, world)
    gpu_idx = run.bufs["topk_idx"].cpu().numpy()
    run_fused = run.fused
    num_sms = torch.cuda.get_device_properties(dev).multi_processor_count
    del run
    torch.cuda.empty_cache()
    configs = {}
    if not args.no_configs:
        for name in CONFIG_NAMES:
            configs[name] = config_line(WORKLOADS[name], args, dev, st, peaks, max_over_ranks,
                                        world, barrier, rank == 0 and not args.no_cpu)
            torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return

    # ---- roofline of the dominant kernel, the expert GEMM: 2 R d f FLOP per
    # launch over the average of its two launches (W1 and W2, equal FLOPs)
    flops_launch = 2.0 * R * dm * f
    gemm_launch_ms = ffn_ms / 2.0
    achieved = flops_launch / (gemm_launch_ms * 1e-3) / 1e12
    burst = peaks["bf16_tflops"]
    sustained = peaks.get("bf16_tflops_sustained", burst)
    long_capped = ms * 1e-3 >= SUSTAINED_REGION_S and "sw_power_cap" in clocks.get("reasons", [])
    peak = sustained if long_capped else burst
    roofline = {
        "bound": "tensor", "kernel": "tc_gemm_pair_kernel (expert GEMM; mean of its two launches)",
        "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
        "frac_burst": achieved / burst, "frac_sustained": achieved / sustained,
        "peak_source": (f"{peak_src} dense bf16 "
                        + ("sustained (timed region >= 2 s under the power cap)" if long_capped
                           else f"burst (timed region {ms:.1f} ms)")
                        + f"; burst {burst}, sustained {sustained} TFLOP/s"),
        "flops_per_launch": flops_launch, "launch_ms": gemm_launch_ms,
        "traffic": recorded_traffic(wl.name),
        "traffic_note": "DRAM bytes per launch from the committed ncu capture "
                        "(profiles/roofline_traffic.json) while the GEMM sources are unchanged, "
                        "else null"}
    cpu = cpu_baseline(wl, inp_cpu, gpu_idx) if not args.no_cpu else None
    line = {
        "metric": METRIC,
        "value": job_tokens_per_s(world, S, args.steps, ms),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype,
        "data": "synthetic (seeded N(0,1) activations, N(0,1/fan_in) weights)",
        "config": {"workload": workload_desc(wl), "capacity": N.moe_capacity(cfg),
                   **rstats,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": "no flush in the timed loop: each step streams 2.7 GB of expert "
                         "weights, 21x the 126 MB L2 (stages_cold_l2: gate, dispatch and "
                         "combine alone after a 512 MB flush)"},
        "roofline": roofline,
        "step_roofline": step_roofline(wl, R, peaks, ms / args.steps),
        "stages": stages,
        "stages_cold_l2": cold,
        "e2e": {"value": job_tokens_per_s(world, S, args.steps, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": S * dm * eb,
                "d2h_bytes_per_step": S * dm * eb + 4 * (1 + E),
                "ms_per_step": e2e_ms / args.steps,
                "timing": "CUDA events: before the first host-to-device copy, after the last "
                          "device-to-host copy",
                "host_link": link,
                # steady state of the pipeline: the slower of the forward and the
                # two copies running at once
                "floor_ms": max(ms / args.steps, link["both_ms"]),
                "frac_of_floor": max(ms / args.steps, link["both_ms"]) / (e2e_ms / args.steps)},
        "moe_forward_ms_per_step": fwd_call_ms / args.steps,
        "moe_forward_fused_dispatch_ms_per_step": fused_ms / args.steps,
        "dispatch": "fused into the first expert GEMM" if run_fused else "copy kernel",
        "gpu_launches": forward_launches(wl, run_fused, num_sms) * args.steps,
        "clocks": clocks,
        "configs": configs,
        "decode_step": decode,
        "residual_step": residual,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def config_line(wl, args, dev, st, peaks, max_over_ranks, world, barrier, with_cpu):
    """One layer configuration, measured like the headline workload."""
    import torch
    run = LayerRun(wl, dev)
    for _ in range(max(args.warmup, 3)):
        run.step(st)
    torch.cuda.synchronize()
    sampler = ClockSampler(dev.index or 0)
    sampler.start()
    ms = max_over_ranks(timed(torch, st, args.steps, lambda i: run.step(st), barrier))
    clocks = sampler.stop()
    stages = stage_breakdown(run, st, args.steps, peaks)
    R = run.rows()
    out = {"workload": workload_desc(wl),
           "value": job_tokens_per_s(world, wl.num_tokens, args.steps, ms), "unit": "tokens/s",
           "ms_per_step": ms / args.steps, "steps": args.steps, **routing_stats(run),
           "stages": stages, "clocks": {k: clocks.get(k) for k in ("sm_mhz", "reasons", "samples")}}
    gemm_flops = (12.0 if wl.backward else 4.0) * R * wl.hidden_size * wl.ffn_size
    step_tflops = gemm_flops / (ms / args.steps * 1e-3) / 1e12
    out["expert_gemm_TFLOP/s_over_step"] = step_tflops
    if wl.dtype == "bf16":
        out["expert_gemm_frac_bf16_burst_over_step"] = step_tflops / peaks["bf16_tflops"]
        out["stages_cold_l2"] = stages_cold_l2(run, st, peaks)
    if wl.backward:
        bwd_flops = 8.0 * R * wl.hidden_size * wl.ffn_size
        out["backward_TFLOP/s"] = bwd_flops / (stages["backward"]["ms"] * 1e-3) / 1e12
    if wl.dtype == "bf16":
        out["step_roofline"] = step_roofline(wl, R, peaks, ms / args.steps)
    if with_cpu:
        out["cpu_baseline"] = cpu_baseline(wl, run.inp_cpu, run.bufs["topk_idx"].cpu().numpy())
    del run
    return out


def residual_step(args, dev, run, max_over_ranks, world):
    """PR-MoE forward (moe_forward_residual: the layer plus a dense MLP of
    one expert's shape on every token) on the headline workload."""
    import torch

    from mixture_experts_layer_86_b300 import _native as N
    from mixture_experts_layer_86_b300 import layer as L
    from mixture_experts_layer_86_b300.inputs import make_residual_mix, make_residual_weights

    wl, cfg, d = run.wl, run.cfg, run.d
    rw = [t.to(dev) for t in make_residual_weights(wl)]
    mix_w, mix_b = [t.to(dev) for t in make_residual_mix(wl)]
    bufs = L.alloc_buffers(cfg, dev)
    bufs["logits"] = None
    ws = L.alloc_workspace(cfg, dev)
    y = torch.empty_like(d.x)
    res_h = torch.empty((wl.num_tokens, wl.ffn_size), dtype=d.x.dtype, device=dev)
    res_out = torch.empty_like(d.x)
    mix = torch.empty((wl.num_tokens, 2), dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()
    steps = max(1, min(args.steps, 100))

    def step(learned):
        N.moe_forward_residual(cfg, d.x, d.w_gate, d.logit_bias, d.w1, d.b1, d.w2, d.b2, *rw,
                               y, bufs, res_h, res_out, ws, st,
                               mix_w=mix_w if learned else None,
                               mix_b=mix_b if learned else None, mix=mix if learned else None)

    for _ in range(max(args.warmup, 3)):
        step(False)
        step(True)
    torch.cuda.synchronize()
    # the two forms run in alternating blocks (ABBA...), so a drift of the
    # power-capped clock over the run weighs on both alike
    blocks = 4
    per_block = max(1, steps // blocks)
    steps = per_block * blocks
    total = {False: 0.0, True: 0.0}
    for b in range(blocks):
        for learned in ((False, True) if b % 2 == 0 else (True, False)):
            total[learned] += timed(torch, st, per_block, lambda i: step(learned))
    ms = max_over_ranks(total[False])
    ms_mix = max_over_ranks(total[True])
    R = int(bufs["expert_offsets"][-1].item())
    flops = 4.0 * (R + wl.num_tokens) * wl.hidden_size * wl.ffn_size
    return {"workload": workload_desc(wl).replace("MoE layer forward", "PR-MoE forward (+ dense MLP)"),
            "value": job_tokens_per_s(world, wl.num_tokens, steps, ms), "unit": "tokens/s",
            "ms_per_step": ms / steps, "steps": steps,
            "expert_and_mlp_gemm_TFLOP/s": flops / (ms / steps * 1e-3) / 1e12,
            "learned_mix": {"value": job_tokens_per_s(world, wl.num_tokens, steps, ms_mix),
                            "unit": "tokens/s", "ms_per_step": ms_mix / steps}}


def decode_step(args, dev, max_over_ranks, world, peaks):
    """Inference shape: one decode step of 256 sequences through the 64-expert
    layer.  Each expert sees a handful of tokens, so the expert GEMMs stream
    the routed experts' weights: their roofline is HBM bandwidth."""
    import torch

    from mixture_experts_layer_86_b300.inputs import WORKLOADS

    wl = WORKLOADS["decode_e64"]
    run = LayerRun(wl, dev)
    st = torch.cuda.current_stream()
    steps = max(1, min(args.steps, 200))
    for _ in range(max(args.warmup, 3)):
        run.step(st)
    torch.cuda.synchronize()
    ev = _events(torch, steps, 2)
    ms = max_over_ranks(timed(torch, st, steps,
                              lambda i: run.step(st, ev[i], marks=("expert_ffn", "combine"))))
    ffn_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    rs = routing_stats(run)
    R, used = rs["rows_kept"], rs["experts_used"]
    dm, f = wl.hidden_size, wl.ffn_size
    # algorithmic bytes of the two expert GEMMs: the weights (and biases) of
    # every expert with a kept token, x_disp in, h out and back in, out_disp out
    ffn_bytes = used * (2 * f * dm + f + dm) * 2 + R * (2 * dm + 2 * f) * 2
    gbs = ffn_bytes / (ffn_ms * 1e-3) / 1e9
    return {"workload": workload_desc(wl), "value": job_tokens_per_s(world, wl.num_tokens, steps, ms),
            "unit": "tokens/s", "ms_per_step": ms / steps, "steps": steps, **rs,
            "expert_ffn": {"ms": ffn_ms, "bytes": ffn_bytes, "GB/s": gbs, "bound": "hbm",
                           "frac_hbm": gbs / peaks["hbm_gbs"]}}


# ------------------------------------------------------------------- CPU oracle
def _f32_numpy(t):
    import torch
    return t.to(torch.float32).numpy()


def _oracle_config(wl, n):
    from oracle import moe_oracle as O
    return O.LayerConfig(n, wl.hidden_size, wl.ffn_size, wl.num_experts, wl.k,
                         wl.capacity_factor, wl.min_capacity, wl.drop_tokens, wl.act,
                         wl.aux_loss_weight, wl.gate_temperature, wl.aux_loss_type)


def _oracle_step(wl, inp_cpu, n):
    """The oracle's forward (and, for a training workload, backward) on the
    first n tokens; the weights are passed as exact float32 copies of the
    bf16 values and the oracle widens each expert's slice to float64."""
    import numpy as np
    import torch

    from oracle import moe_oracle as O
    x = inp_cpu.x[:n].to(torch.float64).numpy()
    w = getattr(inp_cpu, "_f32", None)
    if w is None:
        w = [_f32_numpy(t) for t in (inp_cpu.w_gate, inp_cpu.w1, inp_cpu.b1, inp_cpu.w2,
                                     inp_cpu.b2)]
        inp_cpu._f32 = w
    wg, w1, b1, w2, b2 = w
    lb = inp_cpu.logit_bias
    if lb is not None:
        lb = lb.to(torch.float64).numpy()
        if lb.ndim == 2:
            lb = lb[:n]
    cfg = _oracle_config(wl, n)
    fwd = O.forward(cfg, x, wg, w1, b1, w2, b2, logit_bias=lb)
    if wl.backward:
        dy = inp_cpu.dy[:n].to(torch.float64).numpy()
        O.backward(cfg, fwd, x, wg, w1, w2, dy)
    return fwd, np.asarray(fwd["logits"])


def _blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else (os.cpu_count() or 1)
    except Exception:
        return os.cpu_count() or 1


def cpu_baseline(wl, inp_cpu, gpu_idx=None):
    """The oracle, as it stands, timed on the whole batch of the workload (a
    forward, or forward + backward for the training step).  Its own float64
    routing of that batch is compared with the GPU's: tokens routed
    differently are routing flips, reported with the largest top-k margin
    (float64 logits) among them."""
    import numpy as np
    S = wl.num_tokens
    t0 = time.perf_counter()
    fwd, logits = _oracle_step(wl, inp_cpu, S)
    dt = time.perf_counter() - t0
    out = {"value": S / dt, "unit": "tokens/s", "cores": _blas_threads(), "kind": "oracle",
           "sample": f"float64 oracle {'forward+backward' if wl.backward else 'forward'} on the "
                     f"whole batch of {S} tokens (one run, {dt:.1f} s, weight widening included)"}
    if gpu_idx is not None:
        own = fwd["routing"].idx
        flips = np.nonzero(np.any(own != gpu_idx, axis=1))[0]
        srt = -np.sort(-logits, axis=1)
        k = wl.k
        margin = srt[:, k - 1] - srt[:, k] if logits.shape[1] > k else np.full(S, np.inf)
        if k == 2:
            margin = np.minimum(margin, srt[:, 0] - srt[:, 1])
        out["routing_flips"] = int(len(flips))
        out["flip_max_margin"] = float(margin[flips].max()) if len(flips) else None
    return out


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from mixture_experts_layer_86_b300.inputs import WORKLOADS, make_inputs
    wl = WORKLOADS[args.workload]
    inp_cpu = make_inputs(wl)
    # the oracle's time grows as a + b n with the batch n (a: widening every
    # used expert's weights to float64 once per call); two batch sizes, both
    # large enough that every expert gets tokens, give a and b
    n1 = min(wl.num_tokens, 4 * wl.num_experts)
    n2 = min(wl.num_tokens, 3 * n1)
    t0 = time.perf_counter()
    _oracle_step(wl, inp_cpu, n1)
    t1 = time.perf_counter()
    _oracle_step(wl, inp_cpu, n2)
    t2 = time.perf_counter()
    per_tok = max((t2 - t1) - (t1 - t0), 1e-9) / max(n2 - n1, 1)
    fixed = max(0.0, (t1 - t0) - per_tok * n1)
    total_budget = 150.0
    per_step = total_budget / max(1, args.steps + args.warmup)
    n = int(min(wl.num_tokens, max(8, (per_step - fixed) / per_tok)))
    for _ in range(args.warmup):
        _oracle_step(wl, inp_cpu, n)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(wl, inp_cpu, n)
    dt = time.perf_counter() - t0
    v = n * args.steps / dt
    sample = (f"float64 oracle forward on the first {n} of {wl.num_tokens} tokens per step "
              f"(same layer, capacity recomputed for the sample); each call also pays a fixed "
              f"{fixed:.2f} s of weight widening, so the whole batch would take about "
              f"{fixed + per_tok * wl.num_tokens:.1f} s ({1.0 / per_tok:.0f} tokens/s after the "
              f"fixed cost)")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
            "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": {"workload": workload_desc(wl), "tokens_per_step": n},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": _blas_threads(),
                             "kind": "oracle", "sample": sample,
                             "tokens_per_s_after_fixed_cost": 1.0 / per_tok,
                             "fixed_cost_s_per_call": fixed},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="e64_bf16")
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-configs", action="store_true",
                    help="time only the headline workload, the decode and PR-MoE legs")
    ap.add_argument("--no-cpu", action="store_true", help="skip the oracle baselines")
    args = ap.parse_args()
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
