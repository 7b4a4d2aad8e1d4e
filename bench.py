#!/usr/bin/env python3
"""Benchmark of the hybrid Muon + AdamW optimizer step on one GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama7b|gpt124m|moe_mla|single|adamw_2p30]

A step is the whole hot path on one synthetic batch of gradients: the
batched Muon update of every routed matrix and view (momentum/Nesterov/norm
prologue, five quintic Newton-Schulz iterations as grouped tcgen05 GEMMs,
apply epilogue) followed by the fused AdamW step of the embedding, head and
norms. The default workload is the 7B-shape parameter set (d=4096, 32 layers,
GQA; 224 Muon views, 6.98 G Muon elements, 1.05 G AdamW elements), with all
inputs resident in HBM.

The JSON line reports the step time (value, ms/step, lower is better), the
Newton-Schulz throughput, a live roofline of the dominant kernel from CUDA
events recorded by the library on its launch stream, the end-to-end time with
host buffers (gradients copied in from pinned memory and updated parameters
copied back every step), the SM clocks sampled during the timed region, and
the fp64 CPU oracle timed on a bounded sample of the same workload.

Every call of the library uses one GPU. The Newton-Schulz GEMM loads its
operands with cluster-multicast TMA copies, which only one-GPU processes may
run, so --gpus N > 1 (or a torchrun launch with WORLD_SIZE > 1) prints one
"unavailable" line from rank 0 and exits 0 without touching a GPU.

--impl reference times the oracle (the plain fp64 CPU statement of the
method) on the host cores instead, each step a bounded sample of the same
workload extrapolated to the full step.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Muon+AdamW step ms at 7B-shape; Newton–Schulz TFLOP/s vs bf16 TC peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama7b",
                    help="llama7b (default), gpt124m, moe_mla, single, adamw_2p30, ns "
                         "(Newton-Schulz only, see --ns-n/--ns-aspect/--ns-batch), or ns_sweep "
                         "(every Newton-Schulz sweep point, one JSON line each)")
    ap.add_argument("--ns-n", type=int, default=4096)
    ap.add_argument("--ns-aspect", default="1:1", choices=["1:1", "1:4", "4:1"])
    ap.add_argument("--ns-batch", type=int, default=8)
    ap.add_argument("--max-grad-norm", type=float, default=None,
                    help="run the gradient control (global norm, clip to this value, overflow "
                         "skip) ahead of both halves; 0 observes the norm only")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-groups", action="store_true",
                    help="end to end: split the Muon tensors in two groups and copy the second "
                         "group's gradients in while the first computes (fast only where the "
                         "copy engines keep their rate beside the GEMMs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    return ap.parse_args()


# Kernel family -> the sources that define it. A DRAM-traffic record in
# profiles/ is used only while these files still hash to the digest it was
# taken on; once a kernel changes, its traffic is reported as null.
KERNEL_SOURCES = {
    "ns_gemm": ["ns_gemm.cu", "mh_ptx.cuh", "mh_internal.h", "mh_sr.cuh"],
    "muon_prologue": ["elementwise.cu", "mh_internal.h", "mh_sr.cuh"],
    "muon_apply": ["elementwise.cu", "mh_ptx.cuh", "mh_internal.h", "mh_sr.cuh"],
    "muon_colstats": ["elementwise.cu", "mh_ptx.cuh", "mh_internal.h"],
    "adamw": ["adamw.cu", "mh_internal.h", "mh_sr.cuh"],
    "grad_norm": ["grad_control.cu", "mh_internal.h"],
}


def sources_digest(family: str) -> str:
    import hashlib
    h = hashlib.sha256()
    for f in KERNEL_SOURCES.get(family, []):
        with open(os.path.join(ROOT, "muon_adamw_hybrid_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_records(workload: str) -> dict:
    """DRAM traffic of each kernel family from the `traffic-record:` lines of
    profiles/dram_*.md, kept only if the sources still match. A record gives
    either bytes_per_launch measured on this very workload, or the ratio of
    measured to algorithmic bytes on a slice of it (applies_to names the
    workloads it covers); the caller scales a ratio by its own algorithmic
    bytes per launch. Returns {family: ("bytes", value) or ("ratio", value)}."""
    import glob
    out = {}
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "dram_*.md"))):
        here = os.path.basename(path)[len("dram_"):-len(".md")]
        try:
            with open(path) as f:
                for line in f:
                    if not line.startswith("traffic-record:"):
                        continue
                    kv = dict(tok.split("=", 1) for tok in line.split()[1:])
                    fam = kv["kernel"]
                    applies = kv.get("applies_to", here).split(",")
                    if (workload not in applies or fam not in KERNEL_SOURCES
                            or kv.get("sources") != sources_digest(fam)):
                        continue
                    if "ratio" in kv:
                        out[fam] = ("ratio", float(kv["ratio"]))
                    else:
                        out[fam] = ("bytes", float(kv["bytes_per_launch"]))
        except (OSError, KeyError, ValueError):
            continue
    return out


def traffic_for(traffic: dict, fam: str, alg_bytes_per_launch: float):
    """DRAM bytes per launch of a family: measured, or the measured ratio on
    a slice times this run's algorithmic bytes per launch; None without a
    valid record."""
    rec = traffic.get(fam)
    if rec is None:
        return None
    kind, val = rec
    return round(val * alg_bytes_per_launch) if kind == "ratio" else val


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---- clocks ----------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.3)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return float("nan")
        sm = [num(r[1]) for r in rows]
        smax = max(num(r[2]) for r in rows)
        power = [num(r[3]) for r in rows]
        pmax = max(p for p in power if not math.isnan(p)) if any(not math.isnan(p) for p in power) else 0
        loaded = [i for i, p in enumerate(power) if p >= 0.5 * pmax] or list(range(len(rows)))
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = []
        for k, nm in enumerate(names):
            if any(rows[i][5 + k].lower() == "active" for i in loaded):
                reasons.append(nm)
        return {"sm_mhz": statistics.median(sm[i] for i in loaded), "sm_max_mhz": smax,
                "reasons": reasons, "samples": len(rows), "samples_under_load": len(loaded),
                "power_w_max": pmax}


# ---- one GPU only -------------------------------------------------------------------

SINGLE_GPU_REASON = "single-GPU build: the NS GEMM uses cluster-multicast TMA loads"


def multi_gpu_request(args) -> bool:
    """True when the run asks for more than one GPU: --gpus N > 1 or a launch
    with WORLD_SIZE > 1."""
    return args.gpus > 1 or int(os.environ.get("WORLD_SIZE", "1")) > 1


def refuse_multi_gpu(args) -> int:
    """Prints the one "unavailable" line (rank 0 only) and launches nothing."""
    if int(os.environ.get("RANK", "0")) == 0:
        print(json.dumps({"impl": args.impl, "metric": METRIC, "n_gpus": max(args.gpus, int(
            os.environ.get("WORLD_SIZE", "1"))), "unavailable": SINGLE_GPU_REASON}), flush=True)
    return 0


def gpu_setup():
    import torch
    torch.cuda.set_device(0)
    return torch.device("cuda", 0)


# ---- workload on the device -------------------------------------------------------------

class DeviceWorkload:
    def __init__(self, wl, device, max_grad_norm=None):
        import numpy as np
        import torch
        import muon_adamw_hybrid_gb300 as mh
        from synth import workloads as W
        self.wl, self.mh, self.torch = wl, mh, torch
        hp = wl.muon_hp
        self.hp = mh.make_hparams(lr=hp["lr"], momentum=hp["momentum"], nesterov=hp["nesterov"],
                                  eps=hp["eps"], ns_steps=hp["ns_steps"], coeffs=hp["coeffs"],
                                  normuon=hp.get("normuon", False), beta2=hp.get("beta2", 0.95),
                                  muon_plus=hp.get("muon_plus", False),
                                  plus_eps=hp.get("plus_eps", hp["eps"]),
                                  cautious=hp.get("cautious", 0))
        self.mW = [W.device_tensor(wl, W.KIND_W, i, device=device) for i in range(len(wl.muon))]
        self.mG = [W.device_tensor(wl, W.KIND_G, i, 0, device=device) for i in range(len(wl.muon))]
        sdt = torch.bfloat16 if wl.state_dtype == "bf16" else torch.float32
        self.mB = [torch.zeros(s.shape, dtype=sdt, device=device) for s in wl.muon]
        self.sm = [torch.zeros(s.views * s.rows, dtype=torch.float32, device=device)
                   if self.hp.normuon else None for s in wl.muon]
        self.aW = [W.device_tensor(wl, W.KIND_AW, j, device=device) for j in range(len(wl.adamw))]
        self.aG = [W.device_tensor(wl, W.KIND_AG, j, 0, device=device) for j in range(len(wl.adamw))]
        self.am = [torch.zeros(s.shape, dtype=sdt, device=device) for s in wl.adamw]
        self.av = [torch.zeros(s.shape, dtype=sdt, device=device) for s in wl.adamw]
        self.ts = [mh.muon_tensor(w, g, b, s.views, sm, s.lr_mult, s.wd,
                                  param_sr=wl.param_sr and w.dtype == torch.bfloat16)
                   for w, g, b, sm, s in zip(self.mW, self.mG, self.mB, self.sm, wl.muon)]
        self.at = [mh.adamw_tensor(w, g, m, v, s.lr_mult, s.wd,
                                   param_sr=wl.param_sr and w.dtype == torch.bfloat16)
                   for w, g, m, v, s in zip(self.aW, self.aG, self.am, self.av, wl.adamw)]
        need = mh.muon_workspace_bytes(self.ts, self.hp) if self.ts else 0
        self.ws = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
        self.step_count = 0
        self.ts_host = self.at_host = self.grefs_host = None
        # Optional gradient control (global norm over every gradient, clip,
        # overflow skip) ahead of both halves, as a trainer would run it.
        self.max_grad_norm = max_grad_norm
        self.control = None
        if max_grad_norm is not None:
            self.control = mh.GradientControl(device)
            self.grefs = [mh.grad_ref(g) for g in self.mG + self.aG]
            self.gws = torch.empty(mh.grad_prepare_workspace_bytes(self.grefs), dtype=torch.uint8,
                                   device=device)
            self.hp.grad_mult = self.control.grad_mult.data_ptr()
            self.hp.skip = self.control.skip.data_ptr()
            self.cstruct = self.control.struct()
        self.resident_bytes = sum(t.numel() * t.element_size() for t in
                                  self.mW + self.mG + self.mB + self.aW + self.aG + self.am + self.av)
        self.resident_bytes += self.ws.numel()

    def use_host_grads(self, muon_host, adam_host) -> None:
        """Point the step at page-locked host gradients, read in place by the
        kernels (the end-to-end path on a system whose GPU reads host memory)."""
        mh, wl = self.mh, self.wl
        self.ts_host = [mh.muon_tensor(w, g, b, s.views, sm, s.lr_mult, s.wd,
                                       param_sr=wl.param_sr and w.dtype == self.torch.bfloat16)
                        for w, g, b, sm, s in zip(self.mW, muon_host, self.mB, self.sm, wl.muon)]
        self.at_host = [mh.adamw_tensor(w, g, m, v, s.lr_mult, s.wd,
                                        param_sr=wl.param_sr and w.dtype == self.torch.bfloat16)
                        for w, g, m, v, s in zip(self.aW, adam_host, self.am, self.av, wl.adamw)]
        if self.control is not None:
            self.grefs_host = [mh.grad_ref(g) for g in list(muon_host) + list(adam_host)]

    def step(self, stream, host_grads: bool = False, param_fence=None, between=None,
             adam_grads=None) -> None:
        """One step on `stream`. `param_fence` (a torch.cuda.Event) holds back
        the step's first parameter write until the event has completed.
        `between`: the Muon step is split into its gradient phase and the rest,
        and between() is called in between; it may enqueue work that follows
        the last gradient read and return an event to use as the fence.
        `adam_grads`: called before AdamW; an event it returns means the AdamW
        gradients have been copied into the device buffers, which AdamW then
        reads (after waiting for the event) instead of the host ones."""
        s = stream.cuda_stream
        ts = self.ts_host if host_grads else self.ts
        at = self.at_host if host_grads else self.at
        self.step_count += 1
        self.hp.sr_seed = self.step_count
        if between is not None and ts:
            if self.control is not None:
                refs = self.grefs_host if host_grads else self.grefs
                self.mh._lib.grad_prepare(refs, 1.0, float(self.max_grad_norm), self.cstruct,
                                          self.gws.data_ptr(), self.gws.numel(), s)
            self.hp.param_fence = None
            self.hp.phase = self.mh.MH_STEP_GRADIENTS
            self.mh.muon_step_batched(ts, self.hp, self.ws.data_ptr(), self.ws.numel(), s)
            param_fence = between()
            self.hp.phase = self.mh.MH_STEP_FINISH
            self.hp.param_fence = param_fence.cuda_event if param_fence is not None else None
            self.mh.muon_step_batched(ts, self.hp, self.ws.data_ptr(), self.ws.numel(), s)
            self.hp.phase = self.mh.MH_STEP_ALL
            self.hp.param_fence = None
            self._adamw(self._adam_structs(at, stream, adam_grads), s)
            return
        if between is not None:            # no Muon tensors: the fence goes before AdamW
            param_fence = between()
        self.hp.param_fence = param_fence.cuda_event if (param_fence is not None and ts) else None
        if param_fence is not None and not ts:
            stream.wait_event(param_fence)
        if self.control is not None:
            refs = self.grefs_host if host_grads else self.grefs
            self.mh._lib.grad_prepare(refs, 1.0, float(self.max_grad_norm), self.cstruct,
                                      self.gws.data_ptr(), self.gws.numel(), s)
        if ts:
            self.mh.muon_step_batched(ts, self.hp, self.ws.data_ptr(), self.ws.numel(), s)
            self.hp.param_fence = None
        self._adamw(self._adam_structs(at, stream, adam_grads), s)

    def _adam_structs(self, at, stream, adam_grads):
        ready = adam_grads() if adam_grads is not None else None
        if ready is None:
            return at
        stream.wait_event(ready)
        return self.at

    def _adamw(self, at, s) -> None:
        if at:
            hp = self.wl.adam_hp
            if self.control is not None:
                self.mh.adamw_step_ctl(at, hp["lr"], hp["betas"][0], hp["betas"][1],
                                       hp["eps"], self.cstruct, s)
            else:
                self.mh.adamw_step(at, hp["lr"], hp["betas"][0], hp["betas"][1], hp["eps"],
                                   self.step_count, s)

    def check_status(self, stream) -> None:
        if self.ts:
            self.mh.workspace_status(self.ws.data_ptr(), stream.cuda_stream)


def family_stats(stats: dict) -> dict:
    """Merges the library's per-stage records ("ns_gemm.gram", ...) into
    kernel families ("ns_gemm")."""
    out = {}
    for name, v in stats.items():
        fam = name.split(".")[0]
        a = out.setdefault(fam, {"launches": 0, "total_ms": 0.0, "bytes": 0.0, "flops": 0.0,
                                 "flops_executed": 0.0})
        for k in a:
            a[k] += v[k]
    return out


def ns_flops(wl) -> float:
    steps = wl.muon_hp["ns_steps"]
    tot = 0.0
    for s in wl.muon:
        m, n = min(s.rows, s.cols), max(s.rows, s.cols)
        tot += s.views * steps * (4.0 * m * m * n + 2.0 * m ** 3)
    return tot


# Nominal dense bf16 tensor-core rate of one GB300 (NVIDIA datasheet, without
# sparsity): context beside the measured peaks the fractions are taken of.
DATASHEET_BF16_TFLOPS = 2250.0


def tensor_peak(peaks: dict, peak_src: str, clk: dict):
    """The measured bf16 peak that applies to a timed region: the sustained
    cuBLAS rate when the power cap was active while it ran (a long step), the
    burst rate otherwise."""
    capped = "sw_power_cap" in (clk or {}).get("reasons", [])
    key = "bf16_tflops_sustained" if capped else "bf16_tflops"
    return peaks[key], f"bf16 {'sustained' if capped else 'burst'} cuBLAS, of {peak_src}"


def gemm_roofline(v: dict, peaks: dict, peak_src: str, clk: dict, traffic=None) -> dict:
    """Roofline of the Newton-Schulz GEMM family from its event-timed stats:
    led by the executed FLOPs (the work the tensor cores do), with the
    contract's nominal count and the datasheet fraction beside it."""
    t = v["total_ms"] * 1e-3
    ex = v["flops_executed"] / t / 1e12
    nom = v["flops"] / t / 1e12
    peak, src = tensor_peak(peaks, peak_src, clk)
    return {"kernel": "ns_gemm", "bound": "tensor", "achieved": round(ex, 1), "peak": peak,
            "unit": "TFLOP/s", "frac": round(ex / peak, 4), "traffic": traffic,
            "achieved_basis": "executed FLOPs per launch (upper block triangle of XX^T and of "
                              "A A, every block of the apply) / CUDA-event time",
            "peak_source": src,
            "frac_of_datasheet": round(ex / DATASHEET_BF16_TFLOPS, 4),
            "datasheet_peak": DATASHEET_BF16_TFLOPS,
            "nominal_tflops": round(nom, 1), "nominal_frac": round(nom / peak, 4),
            "nominal_basis": "4m^2n + 2m^3 per view and iteration; counts the symmetric "
                             "products in full, so it exceeds the executed work",
            "launches": v["launches"],
            "algorithmic_bytes_per_launch": round(v["bytes"] / max(v["launches"], 1)),
            "traffic_unit": "DRAM bytes per launch (ncu record in profiles/, or null)"}


def hbm_roofline(name: str, v: dict, peaks: dict, peak_src: str, traffic=None) -> dict:
    ach = v["bytes"] / (v["total_ms"] * 1e-3) / 1e9
    return {"kernel": name, "bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"],
            "unit": "GB/s", "frac": round(ach / peaks["hbm_gbs"], 4), "traffic": traffic,
            "achieved_basis": "algorithmic bytes per launch (each operand read and each result "
                              "written once) / CUDA-event time",
            "algorithmic_bytes_per_launch": round(v["bytes"] / max(v["launches"], 1)),
            "launches": v["launches"], "peak_source": f"HBM copy, of {peak_src}"}


# ---- host buffers for the end-to-end measurement -------------------------------------

class PinnedMirror:
    """One page-locked host buffer (a single torch pinned allocation) mirroring
    a list of device tensors."""

    def __init__(self, tensors):
        import torch
        self.tensors = tensors
        self.nbytes = sum(t.numel() * t.element_size() for t in tensors)
        self.buf = torch.empty(max(self.nbytes, 1), dtype=torch.uint8, pin_memory=True)
        self.registered = bool(self.buf.is_pinned())
        self.host = []
        off = 0
        for t in tensors:
            nb = t.numel() * t.element_size()
            self.host.append(self.buf[off:off + nb].view(t.dtype).view(t.shape))
            off += nb

    def fill_from_device(self):
        for h, t in zip(self.host, self.tensors):
            h.copy_(t)

    def h2d(self):
        for h, t in zip(self.host, self.tensors):
            t.copy_(h, non_blocking=True)

    def d2h(self):
        for h, t in zip(self.host, self.tensors):
            h.copy_(t, non_blocking=True)

    def close(self):
        self.host = []
        self.buf = None


class HostPipeline:
    """The end-to-end step through pinned host buffers, as a user overlapping
    transfers with compute would run it.

    Each step reads this step's gradients from page-locked host memory: in
    place (on a GPU that maps that memory, the kernels read it over the host
    link) or through explicit copies otherwise. It also copies the previous
    step's parameters back to the host. The copy-out starts when this step's
    gradient phase has read the Muon gradients, so the two do not compete for
    host memory bandwidth. It runs on a second stream beside the
    Newton-Schulz stages, and this step's first parameter write waits for it
    (param_fence). With in-place reads the AdamW gradients are copied into
    the device buffers at the same point, on a third stream, and AdamW reads
    them there. finish() copies out the last step's parameters."""

    def __init__(self, dw):
        import torch
        self.dw, self.torch = dw, torch
        self.gin = PinnedMirror(dw.mG + dw.aG)
        self.pout = PinnedMirror(dw.mW + dw.aW)
        self.gin.fill_from_device()
        torch.cuda.synchronize()
        mh = dw.mh
        self.in_place = all(mh.pointer_device_accessible(h.data_ptr()) for h in self.gin.host)
        self.nm = len(dw.mG)
        if self.in_place:
            dw.use_host_grads(self.gin.host[:self.nm], self.gin.host[self.nm:])
        self.copy_stream = torch.cuda.Stream()
        self.h2d_stream = torch.cuda.Stream()
        self.pending = False
        self.timed = False
        self.copies = []       # (start, end) events of the timed copy-outs
        self.last_copy = None
        self._adam_ready = None

    def _after(self, stream, side):
        ready = self.torch.cuda.Event()
        ready.record(stream)
        side.wait_event(ready)

    def copy_out(self, stream):
        torch = self.torch
        self._after(stream, self.copy_stream)
        with torch.cuda.stream(self.copy_stream):
            c0 = torch.cuda.Event(enable_timing=True)
            c0.record(self.copy_stream)
            self.pout.d2h()
            landed = torch.cuda.Event(enable_timing=True)
            landed.record(self.copy_stream)
        if self.timed:
            self.copies.append((c0, landed))
        self.pending = False
        self.last_copy = landed
        return landed

    def _fetch_adam_grads(self, stream):
        torch, dw = self.torch, self.dw
        self._after(stream, self.h2d_stream)
        with torch.cuda.stream(self.h2d_stream):
            for h, t in zip(self.gin.host[self.nm:], dw.aG):
                t.copy_(h, non_blocking=True)
            ready = torch.cuda.Event()
            ready.record(self.h2d_stream)
        return ready

    def plan_groups(self, tflops: float = 2.0e3, link_gbs: float = 190.0):
        """Splits the Muon tensors in two for the grouped step: group A (most
        Newton-Schulz work per gradient byte first) reads its gradients in
        place; its Newton-Schulz stages must last long enough to cover the
        copy-in of every other gradient (group B and AdamW) at `link_gbs`."""
        wl, dw = self.dw.wl, self.dw
        items = []
        for i, spec in enumerate(wl.muon):
            m, n = min(spec.rows, spec.cols), max(spec.rows, spec.cols)
            flops = spec.views * wl.muon_hp["ns_steps"] * (4.0 * m * m * n + 2.0 * m ** 3)
            gbytes = dw.mG[i].numel() * dw.mG[i].element_size()
            items.append((gbytes / max(flops, 1.0), i, flops, gbytes))
        items.sort()
        rest = sum(g.numel() * g.element_size() for g in dw.mG + dw.aG)
        a, fa = [], 0.0
        for _, i, f, g in items:
            if fa / (tflops * 1e12) >= rest / (link_gbs * 1e9):
                break
            a.append(i)
            fa += f
            rest -= g
        b = [i for i in range(len(wl.muon)) if i not in set(a)]
        return sorted(a), b

    def _copy_tensors(self, idx, side):
        """D2H of the listed parameter tensors on the `side` stream (ordered
        after whatever that stream already waits for); returns the event
        recorded after them."""
        torch = self.torch
        with torch.cuda.stream(side):
            for i in idx:
                self.pout.host[i].copy_(self.pout.tensors[i], non_blocking=True)
            done = torch.cuda.Event(enable_timing=True)
            done.record(side)
        return done

    def step_grouped(self, stream, groups) -> None:
        """One step with the Muon tensors in two groups (plan_groups): group A
        runs its gradient phase on in-place host gradients; then the other
        gradients are copied into device memory (h2d stream) and the previous
        step's parameters out (copy stream, group A's first) while group A's
        Newton-Schulz stages run; group B and AdamW then run on device
        gradients. Each group's update is fenced on the copy-out of its own
        parameters."""
        torch, dw, mh = self.torch, self.dw, self.dw.mh
        a, b = groups
        s = stream.cuda_stream
        dw.step_count += 1
        dw.hp.sr_seed = dw.step_count
        if dw.control is not None:
            dw.mh._lib.grad_prepare(dw.grefs_host, 1.0, float(dw.max_grad_norm), dw.cstruct,
                                    dw.gws.data_ptr(), dw.gws.numel(), s)
        ts_a = [dw.ts_host[i] for i in a]
        dw.hp.param_fence = None
        dw.hp.phase = mh.MH_STEP_GRADIENTS
        dw.mh.muon_step_batched(ts_a, dw.hp, dw.ws.data_ptr(), dw.ws.numel(), s)
        ready = torch.cuda.Event()
        ready.record(stream)
        self.h2d_stream.wait_event(ready)
        with torch.cuda.stream(self.h2d_stream):
            for i in b:
                dw.mG[i].copy_(self.gin.host[i], non_blocking=True)
            for j, t in enumerate(dw.aG):
                t.copy_(self.gin.host[self.nm + j], non_blocking=True)
            grads_in = torch.cuda.Event()
            grads_in.record(self.h2d_stream)
        fence_a = fence_rest = None
        if self.pending:
            self.copy_stream.wait_event(ready)
            with torch.cuda.stream(self.copy_stream):
                c0 = torch.cuda.Event(enable_timing=True)
                c0.record(self.copy_stream)
            fence_a = self._copy_tensors(a, self.copy_stream)
            fence_rest = self._copy_tensors(b + [self.nm + j for j in range(len(dw.aW))],
                                            self.copy_stream)
            if self.timed:
                self.copies.append((c0, fence_rest))
            self.last_copy = fence_rest
            self.pending = False
        dw.hp.phase = mh.MH_STEP_FINISH
        dw.hp.param_fence = fence_a.cuda_event if fence_a is not None else None
        dw.mh.muon_step_batched(ts_a, dw.hp, dw.ws.data_ptr(), dw.ws.numel(), s)
        stream.wait_event(grads_in)
        dw.hp.phase = mh.MH_STEP_ALL
        if b:
            dw.hp.param_fence = fence_rest.cuda_event if fence_rest is not None else None
            dw.mh.muon_step_batched([dw.ts[i] for i in b], dw.hp, dw.ws.data_ptr(),
                                    dw.ws.numel(), s)
        elif fence_rest is not None:
            stream.wait_event(fence_rest)
        dw.hp.param_fence = None
        dw._adamw(dw.at, s)
        self.pending = True

    def step(self, stream) -> None:
        dw = self.dw
        if not self.in_place:
            self.gin.h2d()

        def between():
            fence = self.copy_out(stream) if self.pending else None
            self._adam_ready = (self._fetch_adam_grads(stream)
                                if self.in_place and dw.aG else None)
            return fence
        self._adam_ready = None
        dw.step(stream, host_grads=self.in_place, between=between,
                adam_grads=lambda: self._adam_ready)
        self.pending = True

    def finish(self, stream):
        landed = self.copy_out(stream)
        stream.wait_event(landed)
        return landed

    def close(self):
        if self.in_place:
            self.dw.ts_host = self.dw.at_host = None
        self.gin.close()
        self.pout.close()


# ---- oracle (CPU baseline / reference arm) ------------------------------------------------

def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        info = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return int(info[0]["num_threads"])
    except Exception:
        pass
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            return int(os.environ[var])
    return os.cpu_count() or 1


def oracle_sample_plan(wl, muon_flop_budget: float, adam_elems: int):
    """Whole Muon views taken in workload order, skipping any view that would
    overshoot the NS-FLOP budget, until the budget is half used or more; and
    the first ``adam_elems`` AdamW elements."""
    steps = wl.muon_hp["ns_steps"]
    cands = []
    for i, s in enumerate(wl.muon):
        m, n = min(s.rows, s.cols), max(s.rows, s.cols)
        f = steps * (4.0 * m * m * n + 2.0 * m ** 3)
        for v in range(s.views):
            cands.append((i, v, f))
    views, got = [], 0.0
    for c in cands:
        if got >= 0.5 * muon_flop_budget:
            break
        if got + c[2] <= muon_flop_budget:
            views.append(c)
            got += c[2]
    if not views and cands:
        views.append(min(cands, key=lambda c: c[2]))
    adam = []
    left = adam_elems
    for j, s in enumerate(wl.adamw):
        if left <= 0:
            break
        take = min(left, s.numel)
        adam.append((j, take))
        left -= take
    return views, adam


class OracleSample:
    """Inputs of a bounded sample, generated once; ``run()`` times the fp64
    oracle on them and returns (muon seconds, adamw seconds)."""

    def __init__(self, wl, views, adam, max_grad_norm=None):
        import numpy as np
        import oracle
        from synth import workloads as W
        self.wl, self.views, self.adam = wl, views, adam
        self.max_grad_norm = max_grad_norm
        hp = wl.muon_hp
        self.hp = oracle.MuonHparams(
            lr=hp["lr"], momentum=hp["momentum"], nesterov=hp["nesterov"], eps=hp["eps"],
            ns_steps=hp["ns_steps"], coeffs=tuple(hp["coeffs"]),
            normuon=hp.get("normuon", False), beta2=hp.get("beta2", 0.95),
            muon_plus=hp.get("muon_plus", False), plus_eps=hp.get("plus_eps", hp["eps"]),
            cautious=hp.get("cautious", 0))
        self.inputs = []
        for i, v, _ in views:
            s = wl.muon[i]
            off, cnt = v * s.rows * s.cols, s.rows * s.cols
            Wv = W.host_tensor(wl, W.KIND_W, i, offset=off, count=cnt).reshape(s.rows, s.cols)
            Gv = W.host_tensor(wl, W.KIND_G, i, offset=off, count=cnt).reshape(s.rows, s.cols)
            self.inputs.append((Wv, Gv, np.zeros_like(Wv), s))
        self.ainputs = [(W.host_tensor(wl, W.KIND_AW, j, count=cnt),
                         W.host_tensor(wl, W.KIND_AG, j, count=cnt), wl.adamw[j])
                        for j, cnt in adam]

    def run(self):
        """Seconds for (Muon views, AdamW chunks, gradient control of both)."""
        import numpy as np
        import oracle
        tc0 = time.perf_counter()
        if self.max_grad_norm is not None:
            oracle.grad_control([g for _, g, _, _ in self.inputs] + [g for _, g, _ in self.ainputs],
                                1.0, self.max_grad_norm)
        t0 = time.perf_counter()
        for Wv, Gv, Bv, s in self.inputs:
            res = oracle.muon_step_view(Wv, Gv, Bv, self.hp, s.lr_mult, s.wd,
                                        np.zeros(s.rows) if self.hp.normuon else None)
            if s.param_dtype == "bf16":
                oracle.round_bf16(res.W)
        t1 = time.perf_counter()
        ahp = self.wl.adam_hp
        for Wa, Ga, s in self.ainputs:
            n = Wa.size
            Wn, _, _ = oracle.adamw_step(Wa, Ga, np.zeros(n), np.zeros(n), ahp["lr"] * s.lr_mult,
                                         ahp["betas"][0], ahp["betas"][1], ahp["eps"], s.wd, 1)
            if s.param_dtype == "bf16":
                oracle.round_bf16(Wn)
        t2 = time.perf_counter()
        return t1 - t0, t2 - t1, t0 - tc0

    def grad_elems(self) -> int:
        return sum(g.size for _, g, _, _ in self.inputs) + sum(g.size for _, g, _ in self.ainputs)


def oracle_extrapolated_ms(wl, views, adam, muon_s, adam_s, ctl_s=0.0, ctl_elems=0):
    """Full-step ms: Muon time scaled by NS FLOPs, AdamW time by elements,
    gradient-control time by gradient elements."""
    ms = 0.0
    if ctl_elems > 0:
        ms += 1e3 * ctl_s * (wl.muon_elems + wl.adam_elems) / ctl_elems
    sample_flops = sum(f for _, _, f in views)
    if sample_flops > 0:
        ms += 1e3 * muon_s * ns_flops(wl) / sample_flops
    sample_adam = sum(c for _, c in adam)
    if sample_adam > 0:
        ms += 1e3 * adam_s * wl.adam_elems / sample_adam
    return ms


def sample_desc(wl, views, adam):
    parts = []
    for i, v, _ in views:
        s = wl.muon[i]
        parts.append(f"{s.name}[view {v}] {s.rows}x{s.cols}")
    for j, c in adam:
        parts.append(f"AdamW {wl.adamw[j].name}[:{c}]")
    return ("fp64 oracle on " + ", ".join(parts) +
            "; Muon time scaled to the full step by nominal NS FLOPs, AdamW time by elements")


# One bounded oracle sample per workload, shared by the CPU baseline of our
# arm and by every step of the reference arm, so the two time the same work:
# whole Muon views up to about 6 TFLOP of fp64 Newton-Schulz (a few seconds
# on the host cores) and up to 2^25 AdamW elements.
ORACLE_NS_FLOP_BUDGET = 6e12
ORACLE_ADAM_ELEMS = 1 << 25


def oracle_plan(wl):
    return oracle_sample_plan(wl, ORACLE_NS_FLOP_BUDGET, ORACLE_ADAM_ELEMS)


def blas_name() -> str:
    try:
        from threadpoolctl import threadpool_info
        info = [i for i in threadpool_info() if i.get("user_api") == "blas"]
        if info:
            return f"{info[0].get('internal_api', '?')} {info[0].get('version', '')}".strip()
    except Exception:
        pass
    return "numpy's BLAS"


def cpu_baseline_record(wl, views, adam, sample, seconds, ms: float) -> dict:
    """The oracle's time for the full step (extrapolated from the sample when
    the sample is not the whole step) with what it covered."""
    nsf = ns_flops(wl)
    f_ns = sum(f for _, _, f in views) / nsf if nsf else 1.0
    f_ad = sum(c for _, c in adam) / wl.adam_elems if wl.adam_elems else 1.0
    return {"value": round(ms, 3), "unit": "ms/step", "cores": blas_threads(),
            "host_cores": os.cpu_count(), "blas": blas_name(), "kind": "oracle",
            "sample": sample_desc(wl, views, adam),
            "extrapolated": bool(f_ns < 1.0 - 1e-12 or f_ad < 1.0 - 1e-12),
            "sample_fraction": {"ns_flops": round(f_ns, 6), "adamw_elems": round(f_ad, 6)},
            "sample_seconds": round(seconds, 3)}


def metric_for(wl) -> str:
    """The 7B-shape set carries the headline metric; the other sets are named
    by their workload in the same form."""
    if wl.name.startswith("llama7b_d4096_l32"):
        return METRIC
    return f"Muon+AdamW step ms ({wl.name}); Newton–Schulz TFLOP/s vs bf16 TC peak"


# ---- main ---------------------------------------------------------------------------------

def run_reference(args, wl):
    """The reference arm: the fp64 oracle timed on the host cores, each step
    the workload's bounded sample (oracle_plan), scaled to the full step."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    views, adam = oracle_plan(wl)
    sample = OracleSample(wl, views, adam, args.max_grad_norm)
    for _ in range(args.warmup):
        sample.run()
    per, secs = [], []
    for _ in range(args.steps):
        ms_muon, ms_adam, ms_ctl = sample.run()
        secs.append(ms_muon + ms_adam + ms_ctl)
        per.append(oracle_extrapolated_ms(wl, views, adam, ms_muon, ms_adam, ms_ctl,
                                          sample.grad_elems()))
    ms = statistics.mean(per)
    line = {
        "impl": "reference", "metric": metric_for(wl), "value": round(ms, 3), "unit": "ms/step",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": config_dict(wl, args.max_grad_norm),
        "cpu_baseline": cpu_baseline_record(wl, views, adam, sample, statistics.mean(secs), ms),
        "e2e": {"value": round(ms, 3), "unit": "ms/step", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 129e6               # GB300 L2
FLUSH_BELOW_BYTES = 4 * L2_BYTES   # resident sets smaller than this get an L2 flush per step


def config_dict(wl, max_grad_norm=None, l2=None):
    extra = {} if max_grad_norm is None else {
        "grad_control": {"max_grad_norm": max_grad_norm, "inv_loss_scale": 1.0}}
    pdt = sorted({s.param_dtype for s in wl.muon} | {s.param_dtype for s in wl.adamw})
    gdt = sorted({s.grad_dtype for s in wl.muon} | {s.grad_dtype for s in wl.adamw})
    state = ("fp32 optimizer state" if wl.state_dtype == "f32"
             else "bf16 optimizer state, stochastically rounded")
    return {**{"workload": wl.name,
            "muon_tensors": len(wl.muon), "muon_views": sum(s.views for s in wl.muon),
            "muon_elems": wl.muon_elems, "adamw_tensors": len(wl.adamw),
            "adamw_elems": wl.adam_elems, "ns_steps": wl.muon_hp["ns_steps"],
            "variants": {k: wl.muon_hp.get(k) for k in ("normuon", "muon_plus", "cautious")
                         if wl.muon_hp.get(k)},
            "precision": ("bf16 tensor-core NS operands, fp32 accumulate; fp32 elementwise math; "
                          f"{state}; params {'/'.join(pdt)}; grads {'/'.join(gdt)}"),
            "parallelism": "single GPU",
            "l2": l2 or "inputs larger than L2 (no flush needed)"}, **extra}


def run_ns_only(args):
    """Newton-Schulz alone on a batch of n x n, n x 4n or 4n x n matrices
    (entries N(0,1), bf16 in and out), timed like the full step; the oracle
    baseline runs the fp64 iteration on one view of the batch."""
    import numpy as np
    import torch
    import muon_adamw_hybrid_gb300 as mh
    import oracle
    import synth
    from synth.gpu import fill_normal
    device = gpu_setup()
    stream = torch.cuda.current_stream(device)
    peaks, peak_src = load_peaks()
    n = args.ns_n
    r, c = {"1:1": (n, n), "1:4": (n, 4 * n), "4:1": (4 * n, n)}[args.ns_aspect]
    b = args.ns_batch
    x = torch.empty(b * r, c, dtype=torch.bfloat16, device=device)
    fill_normal(x, 0, 5000 + n, 1.0)
    out = torch.empty_like(x)
    probs = [mh.ns_problem(x, out, b)]
    need = mh.ns_workspace_bytes(probs)
    ws = torch.empty(need, dtype=torch.uint8, device=device)
    a_, b_, c_ = 3.4445, -4.7750, 2.0315

    def call():
        mh.newton_schulz_batched(probs, 5, a_, b_, c_, 1e-7, ws.data_ptr(), need, stream.cuda_stream)
    for _ in range(max(args.warmup, 0)):
        call()
    torch.cuda.synchronize()
    def timed_calls(instrumented: bool) -> float:
        """ms per call over K calls; with `instrumented`, the library records
        CUDA events around each of its launches."""
        if instrumented:
            mh.profiler_reset()
        mh.profiler_enable(instrumented)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        e0.record(stream)
        for _ in range(args.steps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        mh.profiler_enable(False)
        return e0.elapsed_time(e1) / args.steps

    # K calls as a user makes them for the headline, then K instrumented
    # ones for the per-kernel statistics (see main()).
    clocks = ClockSampler(0)
    clocks.start()
    ms = timed_calls(False)
    ms_instr = timed_calls(True)
    clk = clocks.stop()
    ks = family_stats(mh.profiler_read())
    m_, n_ = min(r, c), max(r, c)
    flops = b * 5 * (4.0 * m_ * m_ * n_ + 2.0 * m_ ** 3)
    ns_workload = f"ns_{args.ns_aspect}_n{n}_batch{b}"
    traffic = traffic_records(ns_workload)
    roofline = None
    if "ns_gemm" in ks:
        v = ks["ns_gemm"]
        roofline = gemm_roofline(v, peaks, peak_src, clk,
                                 traffic_for(traffic, "ns_gemm", v["bytes"] / max(v["launches"], 1)))

    # End to end: the batch copied in from page-locked host memory, the call,
    # and the result copied back, every call.
    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    xh.copy_(x)
    oh = torch.empty_like(xh, pin_memory=True)
    torch.cuda.synchronize()
    e2, e3 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2.record(stream)
    for _ in range(args.steps):
        x.copy_(xh, non_blocking=True)
        call()
        oh.copy_(out, non_blocking=True)
    e3.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e2.elapsed_time(e3) / args.steps

    cpu = None
    if not args.no_cpu_baseline:
        q = synth.normal(0, 5000 + n, (r, c), dtype="bf16").astype(np.float64)
        t0 = time.perf_counter()
        oracle.newton_schulz(q)
        sec = time.perf_counter() - t0
        cpu = {"value": round(1e3 * sec * b, 3), "unit": "ms/call", "cores": blas_threads(),
               "host_cores": os.cpu_count(), "blas": blas_name(), "kind": "oracle",
               "sample": f"fp64 oracle on view 0 ({r}x{c}) of the batch, scaled by the batch "
                         f"count {b}",
               "extrapolated": b > 1, "sample_fraction": {"ns_flops": round(1.0 / b, 6)},
               "sample_seconds": round(sec, 3)}
    print(json.dumps({
        "metric": "Newton-Schulz call ms (5 quintic iterations, bf16 operands)",
        "value": round(ms, 4), "unit": "ms/call", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"ns_{args.ns_aspect}_n{n}_batch{b}", "rows": r, "cols": c,
                   "batch": b, "l2": "X operand " + ("larger" if b * r * c * 2 > 129e6
                                                     else "smaller") + " than L2 (no flush)"},
        "ns_tflops_nominal": round(flops / (ms * 1e-3) / 1e12, 1),
        "roofline": roofline, "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_ms, 4), "unit": "ms/call",
                "h2d_bytes_per_step": x.numel() * x.element_size(),
                "d2h_bytes_per_step": out.numel() * out.element_size()},
        "kernels": {k: {"launches": v["launches"], "total_ms": round(v["total_ms"], 3)}
                    for k, v in ks.items()},
        "kernel_stats_basis": ("the library's CUDA events around each of its launches, over K "
                               "further calls after the timed ones; value and ms_per_step come "
                               "from the K uninstrumented calls"),
        "ms_per_step_instrumented": round(ms_instr, 4),
        "gpu_launches": sum(v["launches"] for v in ks.values()), "clocks": clk}), flush=True)
    return 0


def run_ns_sweep(args):
    """The Newton-Schulz-only sweep (n x n, n x 4n, 4n x n for n = 512..8192,
    batches 1..256) in one process: one JSON line per point with the call time,
    nominal and executed TFLOP/s and each stage's time. X is capped at 16 GiB
    per point: with its output and the workspace (two X buffers, A and P) a
    point holds about 4x X on the device. Not the driver's one-line contract."""
    import torch
    import muon_adamw_hybrid_gb300 as mh
    from synth import workloads as W
    from synth.gpu import fill_normal
    device = torch.device("cuda", 0)
    stream = torch.cuda.current_stream(device)
    peaks, peak_src = load_peaks()
    a_, b_, c_ = 3.4445, -4.7750, 2.0315
    for aspect, n, batch, r, c in W.ns_sweep_shapes(16 * 2 ** 30):
        x = torch.empty(batch * r, c, dtype=torch.bfloat16, device=device)
        fill_normal(x, 0, 5000 + n, 1.0)
        out = torch.empty_like(x)
        probs = [mh.ns_problem(x, out, batch)]
        need = mh.ns_workspace_bytes(probs)
        ws = torch.empty(need, dtype=torch.uint8, device=device)

        def call():
            mh.newton_schulz_batched(probs, 5, a_, b_, c_, 1e-7, ws.data_ptr(), need,
                                     stream.cuda_stream)
        call()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        torch.cuda.synchronize()
        once = e0.elapsed_time(e1)
        reps = max(3, min(args.steps * 20, int(200.0 / max(once, 1e-3))))
        # Call time uninstrumented; stage times from as many calls again with
        # the library's per-launch events.
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / reps
        mh.profiler_reset()
        mh.profiler_enable(True)
        e0.record(stream)
        for _ in range(reps):
            call()
        e1.record(stream)
        torch.cuda.synchronize()
        mh.profiler_enable(False)
        ms_instr = e0.elapsed_time(e1) / reps
        st = mh.profiler_read()
        m_, n_ = min(r, c), max(r, c)
        flops = batch * 5 * (4.0 * m_ * m_ * n_ + 2.0 * m_ ** 3)
        fexec = sum(v["flops_executed"] for k, v in st.items() if k.startswith("ns_gemm"))
        print(json.dumps({
            "point": f"ns_{aspect}_n{n}_batch{batch}", "rows": r, "cols": c, "batch": batch,
            "x_gb": round(batch * r * c * 2 / 1e9, 3), "reps": reps, "ms_per_call": round(ms, 4),
            "ms_per_call_instrumented": round(ms_instr, 4),
            "tflops_nominal": round(flops / (ms * 1e-3) / 1e12, 1),
            "tflops_executed": round(fexec / reps / (ms * 1e-3) / 1e12, 1),
            "frac_executed_of_burst": round(fexec / reps / (ms * 1e-3) / 1e12 / peaks["bf16_tflops"], 4),
            "peak_source": f"bf16 burst, of {peak_src}",
            "stage_ms": {k: round(v["total_ms"] / reps, 4) for k, v in st.items()},
            "launches_per_call": sum(v["launches"] for v in st.values()) // reps}), flush=True)
        del x, out, ws
        torch.cuda.empty_cache()
    return 0


def launch_floor_us(stream, n: int = 2000) -> float:
    """Device time per launch of n back-to-back minimal kernels on `stream`: the
    floor a chain of dependent launches cannot go below."""
    import torch
    for _ in range(100):
        torch.cuda._sleep(0)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(n):
        torch.cuda._sleep(0)
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) * 1e3 / n


def main():
    args = parse_args()
    from synth import workloads as W
    if args.impl == "ours" and multi_gpu_request(args):
        return refuse_multi_gpu(args)
    if args.workload == "ns":
        return run_ns_only(args)
    if args.workload == "ns_sweep":
        return run_ns_sweep(args)
    if args.workload not in W.WORKLOADS:
        raise SystemExit(f"unknown workload {args.workload}; choose from {sorted(W.WORKLOADS)}")
    wl = W.WORKLOADS[args.workload]()
    if args.impl == "reference":
        return run_reference(args, wl)

    import torch
    import muon_adamw_hybrid_gb300 as mh

    device = gpu_setup()
    stream = torch.cuda.current_stream(device)
    peaks, peak_src = load_peaks()

    dw = DeviceWorkload(wl, device, args.max_grad_norm)
    torch.cuda.synchronize()
    for _ in range(max(args.warmup, 0)):
        dw.step(stream)
    torch.cuda.synchronize()
    dw.check_status(stream)

    # ---- timed region: K device-resident steps --------------------------------------
    # Sets far larger than L2 are timed as one span; smaller ones get an L2
    # flush (a write of twice L2) between steps, each step timed on its own.
    flush = None
    l2_note = None
    if dw.resident_bytes < FLUSH_BELOW_BYTES:
        flush = torch.empty(int(2 * L2_BYTES), dtype=torch.uint8, device=device)
        l2_note = (f"L2 flushed between timed steps (a {flush.numel() >> 20} MiB write, outside "
                   f"the timed spans); resident set {dw.resident_bytes / 1e6:.1f} MB")
    def timed_steps(instrumented: bool) -> float:
        """ms over K steps; with `instrumented`, the library records CUDA
        events around each of its launches (per-kernel statistics)."""
        if instrumented:
            mh.profiler_reset()
        torch.cuda.synchronize()
        if flush is None:
            mh.profiler_enable(instrumented)
            ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            ev0.record(stream)
            for _ in range(args.steps):
                dw.step(stream)
            ev1.record(stream)
            torch.cuda.synchronize()
            total = ev0.elapsed_time(ev1)
        else:
            spans = []
            for _ in range(args.steps):
                mh.profiler_enable(False)
                flush.fill_(1)
                mh.profiler_enable(instrumented)
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                dw.step(stream)
                e1.record(stream)
                spans.append((e0, e1))
            torch.cuda.synchronize()
            total = sum(a.elapsed_time(b) for a, b in spans)
        mh.profiler_enable(False)
        return total

    # The headline: K steps as a user runs them. Then K more with the
    # library's per-launch events for the per-kernel statistics and the
    # rooflines: an event recorded between two launches keeps the second from
    # starting early as a programmatic dependent, so those steps run longer
    # where launch latency matters (small sets); the kernels' own durations
    # are the same.
    clocks = ClockSampler(0)
    clocks.start()
    ms_total = timed_steps(False)
    dw.check_status(stream)
    ms_total_instr = timed_steps(True)
    clk = clocks.stop()
    ms_step = ms_total / args.steps
    stage_stats = mh.profiler_read()
    dw.check_status(stream)
    kstats = family_stats(stage_stats)
    launches = sum(v["launches"] for v in kstats.values())
    # Small sets are bound by launch latency: the chain of this step's launches
    # cannot run faster than launches x the device's per-launch floor.
    floor_us = launch_floor_us(stream)
    per_step = launches / max(args.steps, 1)
    launch_floor = {"us_per_launch": round(floor_us, 3), "launches_per_step": per_step,
                    "floor_ms_per_step": round(per_step * floor_us * 1e-3, 4),
                    "frac_of_step": round(per_step * floor_us * 1e-3 / ms_step, 4),
                    "kernel": "torch.cuda._sleep(0), 2000 back to back"}

    # ---- roofline of the dominant kernel and of the top HBM-bound kernel -------------
    kernels = {}
    for name, v in sorted(kstats.items(), key=lambda kv: -kv[1]["total_ms"]):
        avg = v["total_ms"] / max(v["launches"], 1)
        kernels[name] = {"launches": v["launches"], "total_ms": round(v["total_ms"], 3),
                         "avg_ms": round(avg, 4),
                         "share": round(v["total_ms"] / max(sum(x["total_ms"] for x in kstats.values()), 1e-9), 4)}
        if v["flops"] > 0:
            kernels[name]["tflops_nominal"] = round(v["flops"] / (v["total_ms"] * 1e-3) / 1e12, 1)
            kernels[name]["tflops_executed"] = round(v["flops_executed"] / (v["total_ms"] * 1e-3) / 1e12, 1)
        if v["bytes"] > 0:
            kernels[name]["gbs"] = round(v["bytes"] / (v["total_ms"] * 1e-3) / 1e9, 1)
            kernels[name]["algorithmic_bytes_per_launch"] = round(v["bytes"] / max(v["launches"], 1))
    traffic = traffic_records(args.workload)
    hbm = {k: v for k, v in kstats.items() if v["flops"] == 0 and v["bytes"] > 0}
    top_hbm = max(hbm, key=lambda k: hbm[k]["total_ms"]) if hbm else None
    def alg(fam):
        v = kstats[fam]
        return v["bytes"] / max(v["launches"], 1)
    roofline_hbm = (hbm_roofline(top_hbm, hbm[top_hbm], peaks, peak_src,
                                 traffic_for(traffic, top_hbm, alg(top_hbm)))
                    if top_hbm else None)
    # The dominant kernel: the Newton-Schulz GEMMs wherever the set has Muon
    # tensors, AdamW for the AdamW-only set.
    if "ns_gemm" in kstats:
        roofline = gemm_roofline(kstats["ns_gemm"], peaks, peak_src, clk,
                                 traffic_for(traffic, "ns_gemm", alg("ns_gemm")))
        if traffic.get("ns_gemm", ("", 0))[0] == "ratio":
            roofline["traffic_basis"] = ("measured DRAM bytes / algorithmic bytes on a slice of "
                                         "this workload (profiles/), times this run's "
                                         "algorithmic bytes per launch")
    else:
        roofline = roofline_hbm
    stages = {k: {"launches": v["launches"], "total_ms": round(v["total_ms"], 3),
                  "tflops_executed": round(v["flops_executed"] / (v["total_ms"] * 1e-3) / 1e12, 1)}
              for k, v in stage_stats.items() if "." in k and v["total_ms"] > 0}
    nsf = ns_flops(wl)
    ns_ms = kstats.get("ns_gemm", {}).get("total_ms", 0.0) / max(args.steps, 1)

    # ---- end to end with host buffers --------------------------------------------------
    e2e = None
    if not args.no_e2e:
        pipe = HostPipeline(dw)
        in_place = pipe.in_place
        gin, pout = pipe.gin, pipe.pout
        # The grouped step (--e2e-groups) copies most gradients in on the copy
        # engines while group A computes. On some hosts those copies keep
        # ~200 GB/s beside the GEMMs (7B end to end 359 ms against 385 ms
        # read in place); on others they fall to ~40 GB/s under load
        # (675-740 ms), so the in-place path is the default.
        groups = pipe.plan_groups() if args.e2e_groups and in_place and dw.ts else None
        grouped = groups is not None and bool(groups[0]) and bool(groups[1])

        def run_step():
            if grouped:
                pipe.step_grouped(stream, groups)
            else:
                pipe.step(stream)
        run_step()                          # warm-up step and its copy-out
        pipe.finish(stream)
        torch.cuda.synchronize()
        pipe.timed = True
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for k in range(args.steps):
            ev[k][0].record(stream)
            run_step()
            ev[k][1].record(stream)
        end = torch.cuda.Event(enable_timing=True)
        pipe.finish(stream)
        end.record(stream)
        torch.cuda.synchronize()
        e2e_ms = ev[0][0].elapsed_time(end) / args.steps
        step_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
        d2h_ms = statistics.mean(c[0].elapsed_time(c[1]) for c in pipe.copies)
        e2e = {"value": round(e2e_ms, 3), "unit": "ms/step", "h2d_bytes_per_step": gin.nbytes,
               "d2h_bytes_per_step": pout.nbytes,
               "step_ms": round(step_ms, 2), "d2h_ms": round(d2h_ms, 2),
               "path": ("C ABI calls whose kernels read this step's Muon gradients in place "
                        "from page-locked host memory over the host link; the AdamW gradients "
                        "copied in and the previous step's parameters copied out on two more "
                        "streams from the end of the gradient phase, beside the Newton-Schulz "
                        "stages (MH_STEP_GRADIENTS / MH_STEP_FINISH, param_fence)") if in_place else
                       ("C ABI calls with gradients copied in from pinned host memory and "
                        "updated parameters copied back each step on a second stream, from the "
                        "end of the next step's gradient phase up to its first parameter write "
                        "(MH_STEP_GRADIENTS / MH_STEP_FINISH, param_fence)"),
               "h2d_in_kernel": in_place,
               "muon_groups": [len(groups[0]), len(groups[1])] if grouped else None,
               "pinned": bool(gin.registered and pout.registered)}
        pipe.close()

    # ---- CPU oracle baseline: the same sample the reference arm times ----------------------
    cpu = None
    if not args.no_cpu_baseline:
        views, adam = oracle_plan(wl)
        osample = OracleSample(wl, views, adam, args.max_grad_norm)
        ms_muon, ms_adam, ms_ctl = osample.run()
        cpu_ms = oracle_extrapolated_ms(wl, views, adam, ms_muon, ms_adam, ms_ctl,
                                        osample.grad_elems())
        cpu = cpu_baseline_record(wl, views, adam, osample, ms_muon + ms_adam + ms_ctl, cpu_ms)

    line = {
        "metric": metric_for(wl), "value": round(ms_step, 3), "unit": "ms/step", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_step, 3),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config_dict(wl, args.max_grad_norm, l2_note),
        "ns_tflops": round(nsf / (ns_ms * 1e-3) / 1e12, 1) if ns_ms > 0 else None,
        "ns_ms_per_step": round(ns_ms, 3),
        "roofline": roofline, "roofline_hbm": roofline_hbm, "kernels": kernels,
        "kernel_stats_basis": ("the library's CUDA events around each of its launches, over K "
                               "further steps after the timed ones (same stream, same flush "
                               "policy); value and ms_per_step come from the K uninstrumented "
                               "steps"),
        "ms_per_step_instrumented": round(ms_total_instr / args.steps, 3),
        "ns_stages": stages,
        "launch_floor": launch_floor,
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches, "clocks": clk,
        "resident_gb": round(dw.resident_bytes / 1e9, 1),
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
