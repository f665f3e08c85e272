"""Benchmark of the MaxSim hot path on GB300.

Default workload: the in-batch contrastive all-pairs training step, bf16 in /
fp32 scores, Q[128,32,128] x D[128,1030,128], document lengths U[700,1030],
the loss the cross-entropy over the score rows with the diagonal as target.
One step = one liblik call (lik_maxsim_allpairs_ce_step: forward with the
saved argmax, the loss and its score gradient, backward to fp32 grad_Q and
grad_D) through the C ABI, inputs resident in HBM; --step fwd+bwd times the
forward and backward calls with the score gradient computed once outside the
steps instead.  The headline metric counts 2*Nq*Nd*Lq*Ld*dim FLOPs (padded Ld)
per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the fp64 CPU oracle, as it stands

The line also carries "roofline_bwd" (the backward timed through its plain
entry point, both gradients in the one launch the step runs and each gradient
alone, with the bytes each must move) and, in a single-GPU run of the default step,
"configs": one record per other workload (per-query candidates fwd+bwd,
long-document reranking fwd, large all-pairs inference fwd, and the in-batch
workload with fp32 inputs fwd+bwd), each measured
the same way, with its own roofline, clocks and CPU-oracle sample.

Under torchrun (N > 1) every rank runs an independent replica of the
workload (weak scaling, no collective on the data path); timings are
max-reduced over ranks and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from late_interaction_retrieval_gb300 import workloads as W  # noqa: E402

METRIC = "MaxSim fwd+bwd TFLOP/s (% dense bf16 peak); pairwise GB/s (% HBM peak)"
L2_FLUSH_BYTES = 256 << 20  # > 129 MB L2
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "ncu_traffic.json")
_CSRC = "late_interaction_retrieval_gb300/csrc/"
# every source file a kernel's code comes from: its DRAM counters stay valid
# only while all of them are unchanged
KERNEL_SOURCES = {
    "allpairs_fwd_tc_kernel": (_CSRC + "fwd_tc_allpairs.cu", _CSRC + "sm100_ptx.cuh", _CSRC + "lik_internal.h"),
    "stream_fwd_tc_kernel": (_CSRC + "fwd_tc_stream.cu", _CSRC + "sm100_ptx.cuh", _CSRC + "lik_internal.h"),
    "allpairs_fwd_tf32_kernel": (_CSRC + "fwd_tc_f32.cu", _CSRC + "sm100_ptx.cuh", _CSRC + "lik_internal.h"),
}


# ------------------------------------------------------------ utilities --

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(x: float, device) -> float:
    """Max of a per-rank float over the default process group (identity at N=1)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(world: int, steps: int, units_per_step: float, max_ms: float, scale: float) -> float:
    """Units all ranks processed divided by the slowest rank's time (weak scaling)."""
    return world * steps * units_per_step / (max_ms * 1e-3) / scale


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


def kernel_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if the kernel's
    source is unchanged since the capture (else None)."""
    if not os.path.exists(PROFILE_TRAFFIC):
        return None
    with open(PROFILE_TRAFFIC) as f:
        table = json.load(f)
    ent = table.get(kernel, {}).get(workload)
    if not ent:
        return None
    if ent.get("source_sha256") != source_digest(kernel):
        return None
    return ent.get("dram_bytes_per_launch")


def source_digest(kernel: str) -> str:
    """sha256 over the kernel's source files, in the listed order."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: torch.device):
        self.gpu = self._smi_id(device)
        self.proc = None
        self.path = None

    @staticmethod
    def _smi_id(device) -> str:
        """nvidia-smi id of a torch device (its UUID; CUDA_VISIBLE_DEVICES may renumber)."""
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES")
            idx = device.index or 0
            if vis:
                return vis.split(",")[idx].strip()
            return str(idx)

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        return self

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# --------------------------------------------------------------- workload --

class Step:
    """Device buffers and the liblik calls of one step of a workload."""

    def __init__(self, name: str, device: torch.device, grad_dtype: str = "f32", ce: bool = False,
                 recompute: bool = False):
        from late_interaction_retrieval_gb300 import binding
        self.binding = binding
        self.w = W.WORKLOADS[name]
        self.inp = W.generate(name, device=device)
        self.device = device
        w, i = self.w, self.inp
        self.layout = w.layout
        self.scores = torch.empty(w.score_shape, dtype=torch.float32, device=device)
        self.argmax = (torch.empty((*w.score_shape, w.lq), dtype=torch.int32, device=device)
                       if w.backward else None)
        # recompute: the forward saves no argmax; the backward re-runs the forward
        # into self.argmax (its workspace) through lik_maxsim_*_bwd_recompute
        self.recompute = recompute and w.backward
        if self.recompute and grad_dtype != "f32":
            raise SystemExit("--step recompute writes fp32 gradients")
        # gradients in fp32 (the default entry points) or in the inputs' dtype
        self.same_dtype = grad_dtype == "input"
        gdt = i.Q.dtype if self.same_dtype else torch.float32
        self.gQ = torch.empty(i.Q.shape, dtype=gdt, device=device) if w.backward else None
        self.gD = torch.empty(i.D.shape, dtype=gdt, device=device) if w.backward else None
        # ce: the workload's cross-entropy head (loss and score gradient) runs
        # inside every step, through lik_ce_rows, instead of once outside
        self.ce = ce and w.backward and i.ce_target is not None
        if ce and not self.ce:
            raise SystemExit(f"--step ce: workload {name} has no cross-entropy head")
        if self.ce:
            self.target = i.ce_target.to(device=device, dtype=torch.int32).contiguous()
            self.loss = torch.empty(1, dtype=torch.float32, device=device)
            self.row_loss = torch.empty(w.nq, dtype=torch.float32, device=device)
        self.fwd()
        torch.cuda.synchronize()
        if self.ce:
            self.g = torch.empty(w.score_shape, dtype=torch.float32, device=device)
        elif w.backward:
            if i.grad_out is not None:
                self.g = i.grad_out.to(device).float().contiguous()
            else:  # cross-entropy head of the workload: computed once, outside the timed steps
                self.g = W.ce_grad_rows(self.scores, i.ce_target).float().contiguous()
        binding.lik_check_device_error()

    def fwd(self, Q=None, D=None, qm=None, dm=None):
        i = self.inp
        Q = i.Q if Q is None else Q
        D = i.D if D is None else D
        qm = i.qmask if qm is None else qm
        dm = i.dmask if dm is None else dm
        getattr(self.binding, f"lik_maxsim_{self.layout}_fwd")(Q, D, qm, dm, self.scores,
                                                               None if self.recompute else self.argmax)

    def ce_step(self, Q=None, D=None, qm=None, dm=None, target=None):
        """The workload's loss head in one call: forward, loss, backward (the
        loss head runs inside the backward launch)."""
        i = self.inp
        getattr(self.binding, f"lik_maxsim_{self.layout}_ce_step")(
            i.Q if Q is None else Q, i.D if D is None else D, i.qmask if qm is None else qm,
            i.dmask if dm is None else dm, self.target if target is None else target, self.scores, self.argmax,
            self.loss, self.row_loss, self.g, self.gQ, self.gD)

    def bwd(self, Q=None, D=None, g=None, qm=None, dm=None):
        i = self.inp
        if self.recompute:
            getattr(self.binding, f"lik_maxsim_{self.layout}_bwd_recompute")(
                i.Q if Q is None else Q, i.D if D is None else D, i.qmask if qm is None else qm,
                i.dmask if dm is None else dm, self.g if g is None else g, self.argmax, self.gQ, self.gD)
            return
        if self.ce:
            self.binding.lik_ce_rows(self.scores.view(self.w.nq, -1), self.target, self.loss, self.row_loss,
                                     self.g.view(self.w.nq, -1))
        getattr(self.binding, f"lik_maxsim_{self.layout}_bwd" + ("_same_dtype" if self.same_dtype else ""))(
            i.Q if Q is None else Q, i.D if D is None else D, self.g if g is None else g,
            self.argmax, self.gQ, self.gD)

    @property
    def fused_bwd(self) -> bool:
        """Whether the backward is one launch for both gradients: fp32
        gradients, dim % 8 == 0, dim <= 256 and, with the loss head inside,
        at most 4096 score rows (else one launch for each gradient)."""
        w = self.w
        rows = w.nq
        cols = self.scores.numel() // rows
        return (not self.same_dtype and w.dim % 8 == 0 and w.dim <= 256
                and (not self.ce or (rows <= 4096 and rows * cols <= 1 << 20)))

    # launches of liblik kernels per step (cudaMemsetAsync of grad_D is not ours;
    # the streaming forward of the pairwise and kd layouts is a plan kernel and
    # the forward kernel; the cross-entropy head runs inside the backward's
    # launch; the recompute backward adds one forward)
    @property
    def launches_per_step(self) -> int:
        fwd = 1 if self.layout == "allpairs" else 2
        bwd = (1 if self.fused_bwd else 2) if self.w.backward else 0
        return fwd + bwd + (fwd if self.recompute else 0)

    def valid_flops(self) -> int:
        i, w = self.inp, self.w
        qv = i.qmask.sum(dim=1).double()  # [nq]
        dv = i.dmask.reshape(-1, w.ld).sum(dim=1).double()  # [n_doc]
        if w.layout == "allpairs":
            tot = float(qv.sum() * dv.sum())
        elif w.layout == "pairwise":
            tot = float((qv * dv).sum())
        else:
            tot = float((qv[:, None] * dv.view(w.nq, w.nd)).sum())
        return int(2 * w.dim * tot)

    def algorithmic_bytes(self) -> int:
        """Bytes a forward must move at least: valid D rows, Q, masks, scores,
        and the saved argmax when the step keeps one for its backward."""
        i, w = self.inp, self.w
        el = i.Q.element_size()
        dv = int(i.dmask.sum())
        qbytes = i.Q.numel() * el
        saved = self.argmax.numel() * 4 if self.argmax is not None else 0
        return (dv * w.dim * el + i.dmask.numel() + qbytes + i.qmask.numel() + self.scores.numel() * 4
                + saved)


# ---------------------------------------------------------------- our arm --

# Workloads measured after the headline one in a default single-GPU run, each
# as one record of the line's "configs" object.
EXTRA_WORKLOADS = ("kd_b256_n17_bf16", "rerank_b512_ld8192_f16", "allpairs_q128_d4096_bf16", "inbatch_b128_f32")
# nominal dense TF32 / BF16 tensor rates (1.1 / 2.25 PFLOP/s): the fp32 forward
# runs on TF32 tensor cores, three products per similarity
TF32_PER_BF16 = 1.1 / 2.25


def timed_steps(st: Step, args, stream, flush, world):
    """Warm-up steps, then `args.steps` device-timed steps (CUDA events on the
    launching stream, L2 flushed between steps), with the SM clocks sampled
    while they run (identical untimed steps extend the load to >= 1 s)."""
    w = st.w

    def one_step():
        if st.ce:
            st.ce_step()
            return
        st.fwd()
        if w.backward:
            st.bwd()

    for _ in range(max(args.warmup, 3)):
        flush.zero_()
        one_step()
    torch.cuda.synchronize()
    st.binding.lik_check_device_error()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(st.device).start()
    time.sleep(0.15)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_wall0 = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        e0, e1, e2 = ev[k]
        e0.record(stream)
        if st.ce:  # one call: the forward inside it is timed on its own below
            st.ce_step()
        else:
            st.fwd()
            e1.record(stream)
            if w.backward:
                st.bwd()
        e2.record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    while time.perf_counter() - t_wall0 < 1.0:
        for _ in range(20):
            flush.zero_()
            one_step()
        torch.cuda.synchronize()
    clocks = sampler.stop()
    st.binding.lik_check_device_error()
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    if st.ce:  # the forward kernel alone, for its roofline
        fwd_ms = []
        for a, b, _ in ev:
            flush.zero_()
            a.record(stream)
            st.fwd()
            b.record(stream)
        torch.cuda.synchronize()
        fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    else:
        fwd_ms = [a.elapsed_time(b) for a, b, _ in ev]
    return {"step_ms": step_ms, "fwd_ms": fwd_ms, "clocks": clocks, "wall_s": t_wall}


def forward_roofline(st: Step, name: str, fwd_avg_ms: float, peaks) -> dict:
    """Roofline of the step's forward kernel(s), from their CUDA-event time."""
    w = st.w
    if w.layout in ("pairwise", "kd"):
        kernel = "stream_fwd_tc_kernel"
        units = st.algorithmic_bytes()
        roof = {"bound": "hbm", "achieved": units / (fwd_avg_ms * 1e-3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "algorithmic_bytes": units}
    elif w.dtype == "f32":
        kernel = "allpairs_fwd_tf32_kernel"
        achieved = w.counted_flops / (fwd_avg_ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": peaks["bf16_tflops"] * TF32_PER_BF16,
                "unit": "TFLOP/s", "peak_dtype": "tf32 (measured bf16 burst x nominal tf32/bf16 ratio)",
                "tensor_flops_per_counted_flop": 3}
        roof["tensor_work_frac"] = 3 * achieved / roof["peak"]
    else:
        kernel = "allpairs_fwd_tc_kernel"
        roof = {"bound": "tensor", "achieved": w.counted_flops / (fwd_avg_ms * 1e-3) / 1e12,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = kernel_traffic(kernel, name)
    roof["kernel"] = kernel
    roof["peak_source"] = f"{peaks['source']} (burst; kernel timed alone within a short step)"
    if roof["bound"] == "tensor" and w.dtype != "f32":
        roof["frac_of_sustained"] = roof["achieved"] / peaks["bf16_tflops_sustained"]
    roof["kernel_ms"] = fwd_avg_ms
    return roof


def backward_roofline(st: Step, args, stream, flush, peaks) -> dict:
    """The backward timed through the plain backward entry point, with the
    bytes it must move: both gradients in one call (with fp32 gradients the
    one launch the training step runs, "grad_qd"), and each gradient alone
    (the entry point called with only grad_Q, then only grad_D).

    grad_Q gathers one document row per (pair, query token) hit; grad_D
    zero-fills grad_D (fp32 gradients) and adds one Q row per hit into it.
    `dram_bytes` is what the kernel must move to or from DRAM at least
    (argmax, upstream gradient, its output, the distinct rows it reads);
    `l2_bytes` is the row traffic it makes (gathers, or reductions into
    grad_D), served by L2 where the rows are resident.
    """
    w, i = st.w, st.inp
    el = i.Q.element_size()
    gel = st.gQ.element_size()
    hits = int((st.argmax >= 0).sum())
    pairs = st.argmax.numel() // w.lq
    am_bytes, g_bytes = st.argmax.numel() * 4, pairs * 4
    d_bytes = i.D.numel() * el
    fn = getattr(st.binding, f"lik_maxsim_{w.layout}_bwd" + ("_same_dtype" if st.same_dtype else ""))

    def time_it(gq, gd):
        for _ in range(3):
            flush.zero_()
            fn(i.Q, i.D, st.g, st.argmax, gq, gd)
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for a, b in ev:
            flush.zero_()
            a.record(stream)
            fn(i.Q, i.D, st.g, st.argmax, gq, gd)
            b.record(stream)
        torch.cuda.synchronize()
        st.binding.lik_check_device_error()
        return statistics.mean(a.elapsed_time(b) for a, b in ev)

    ms_q = time_it(st.gQ, None)
    ms_d = time_it(None, st.gD)
    gathered = hits * w.dim * el
    q_dram = am_bytes + g_bytes + st.gQ.numel() * gel + min(gathered, d_bytes)
    resident = d_bytes < (96 << 20)  # rows fit in L2 next to everything else
    gq = {"kernel": "grad_q_vec_kernel", "ms": ms_q, "hits": hits, "l2_bytes": gathered,
          "l2_gbs": gathered / (ms_q * 1e-3) / 1e9, "dram_bytes": q_dram,
          "achieved": q_dram / (ms_q * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
          "bound": "l2 (gathered document rows are L2-resident)" if resident else "hbm"}
    gq["frac"] = gq["achieved"] / gq["peak"]
    red_bytes = hits * w.dim * 4
    gd_out = st.gD.numel() * gel
    d_dram = am_bytes + g_bytes + i.Q.numel() * el + gd_out
    kernel_d = "grad_d_scatter_vec_kernel (after a zero-fill of grad_D)" if not st.same_dtype else \
        "grad_d (one write per row, inputs' dtype)"
    gd = {"kernel": kernel_d, "ms": ms_d, "hits": hits, "l2_bytes": red_bytes if not st.same_dtype else hits * w.dim * el,
          "reductions": hits * (w.dim // 4) if not st.same_dtype else 0,
          "dram_bytes": d_dram, "achieved": d_dram / (ms_d * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
          "bound": ("l2 (16-byte fp32 reductions into grad_D)" if resident else "hbm (grad_D write)")
          if not st.same_dtype else "hbm (grad_D write)"}
    gd["l2_gbs"] = gd["l2_bytes"] / (ms_d * 1e-3) / 1e9
    gd["frac"] = gd["achieved"] / gd["peak"]
    out = {"grad_q": gq, "grad_d": gd}
    if st.fused_bwd:
        ms_qd = time_it(st.gQ, st.gD)
        qd_dram = am_bytes + g_bytes + st.gQ.numel() * gel + min(gathered, d_bytes) + i.Q.numel() * el + gd_out
        out["grad_qd"] = {
            "kernel": "grad_qd_vec_kernel (after a zero-fill of grad_D: a memset here; the forward's side "
                      "work in the one-call all-pairs step)",
            "ms": ms_qd, "hits": hits, "l2_bytes": gathered + red_bytes, "gathered_bytes": gathered,
            "reduction_bytes": red_bytes, "reductions": hits * (w.dim // 4), "dram_bytes": qd_dram,
            "l2_gbs": (gathered + red_bytes) / (ms_qd * 1e-3) / 1e9,
            "achieved": qd_dram / (ms_qd * 1e-3) / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "bound": "l2 (gathers and 16-byte fp32 reductions)" if resident else "hbm"}
        out["grad_qd"]["frac"] = out["grad_qd"]["achieved"] / out["grad_qd"]["peak"]
    return out


def has_ce_head(name: str) -> bool:
    """The workload's upstream gradient comes from a cross-entropy over its score rows."""
    return name in ("inbatch_b128_bf16", "inbatch_b128_f32", "kd_b256_n17_bf16")


def config_record(name: str, device, args, stream, flush, peaks) -> dict:
    """One extra workload measured like the headline one (same steps, L2
    flush and clock sampling; its training step in one call when it has a
    cross-entropy head), as a record of the line's "configs"."""
    st = Step(name, device, "f32", ce=has_ce_head(name))
    w = st.w
    t = timed_steps(st, args, stream, flush, 1)
    ms = statistics.mean(t["step_ms"])
    fwd_ms = statistics.mean(t["fwd_ms"])
    if w.layout == "pairwise" and not w.backward:
        value, unit = st.algorithmic_bytes() / (ms * 1e-3) / 1e9, "GB/s"
    else:
        value, unit = w.counted_flops / (ms * 1e-3) / 1e12, "TFLOP/s"
    rec = {"workload": name, "layout": w.layout, "Q": list(w.q_shape), "D": list(w.d_shape), "dtype": w.dtype,
           "passes": "fwd+bwd" if w.backward else "fwd", "value": value, "unit": unit, "ms_per_step": ms,
           "fwd_ms": fwd_ms, "steps": args.steps, "counted_flops_per_step": w.counted_flops,
           "valid_token_flops_per_step": st.valid_flops(), "algorithmic_fwd_bytes": st.algorithmic_bytes(),
           "roofline": forward_roofline(st, name, fwd_ms, peaks), "clocks": t["clocks"],
           "gpu_launches": st.launches_per_step * args.steps}
    if w.backward:
        rec["grad_dtype"] = "f32"
        rec["loss_head"] = "cross-entropy inside the step (one call)" if st.ce else "score gradient precomputed"
        rec["roofline_bwd"] = backward_roofline(st, args, stream, flush, peaks)
    del st
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline:
        rec["cpu_baseline"] = cpu_baseline(name, unit, budget_s=4.0)
    return rec


def run_ours(args):
    world, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    name = args.workload
    st = Step(name, device, args.grad_dtype, ce=args.step == "ce", recompute=args.step == "recompute")
    w = st.w
    stream = torch.cuda.current_stream(device)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
    peaks = measured_peaks()

    # ---- device-timed steps, inputs resident in HBM, L2 flushed in between
    t = timed_steps(st, args, stream, flush, world)
    total_ms = max_over_ranks(sum(t["step_ms"]), device)
    fwd_avg_ms = statistics.mean(t["fwd_ms"])

    # ---- end to end through the public API: pinned host inputs in, results out
    e2e = run_e2e(st, args, stream, world)

    # ---- each backward kernel on its own (the plain backward entry point)
    bwd_roof = None
    if w.backward and not st.recompute:
        bwd_roof = backward_roofline(st, args, stream, flush, peaks)

    fwd_bytes_step = st.algorithmic_bytes()
    roof = forward_roofline(st, name, fwd_avg_ms, peaks)
    config = {
        "workload": name, "layout": w.layout,
        "Q": list(w.q_shape), "D": list(w.d_shape), "passes": "fwd+bwd" if w.backward else "fwd",
        "grad_dtype": ("input" if st.same_dtype else "f32") if w.backward else None,
        "loss_head": ("cross-entropy inside the step (one call; the head runs inside the backward "
                      "launch)") if st.ce else "score gradient precomputed",
        "argmax": ("recomputed in the backward" if st.recompute else "saved by the forward")
                  if w.backward else None,
        "counted_flops_per_step": w.counted_flops, "valid_token_flops_per_step": st.valid_flops(),
        "algorithmic_fwd_bytes": fwd_bytes_step,
        "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)",
        "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        "fwd_ms": fwd_avg_ms, "wall_s": t["wall_s"],
    }
    launches = st.launches_per_step * args.steps

    # ---- the other workloads, one record each (single GPU, default step only)
    configs = None
    if world == 1 and not args.no_extra_configs and args.step in ("fwd+bwd", "ce") and args.grad_dtype == "f32":
        del st
        torch.cuda.empty_cache()
        configs = {n: config_record(n, device, args, stream, flush, peaks) for n in EXTRA_WORKLOADS if n != name}

    if rank == 0:
        ms_per_step = total_ms / args.steps
        if w.layout == "pairwise" and not w.backward:
            value = whole_job_rate(world, args.steps, fwd_bytes_step, total_ms, 1e9)
            unit = "GB/s"
        else:
            value = whole_job_rate(world, args.steps, w.counted_flops, total_ms, 1e12)
            unit = "TFLOP/s"
        cpu = cpu_baseline(name, unit) if not args.no_cpu_baseline else None
        line = {
            "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic (seeded, L2-normalised Gaussian tokens)",
            "config": config,
            "roofline": roof,
            "cpu_baseline": cpu,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": t["clocks"],
        }
        if bwd_roof is not None:
            line["roofline_bwd"] = bwd_roof
        if configs:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


def _twin(st: Step) -> Step:
    """The same step with its own output buffers (inputs and masks shared):
    the second slot of the double-buffered end-to-end pipeline."""
    import copy
    t = copy.copy(st)
    for name in ("scores", "argmax", "gQ", "gD", "loss", "row_loss"):
        v = getattr(st, name, None)
        if v is not None:
            setattr(t, name, torch.empty_like(v))
    if st.ce:  # the score gradient is an output of the one-call step
        t.g = torch.empty_like(st.g)
    return t


def run_e2e(st: Step, args, stream, world, nslots: int = 2):
    """Same metric through the public API with host buffers: every step copies
    its inputs from pinned host memory and reads back its loss (or scores) and
    both gradients.  Two slots of device buffers on three streams, as a
    training loop would run it: step k's inputs go up (copy stream) while step
    k-1 computes and step k-2's results come down (second copy stream); every
    step's copies and compute lie inside the timed region."""
    i, w = st.inp, st.w
    host = {k: v.cpu().pin_memory() for k, v in
            (("Q", i.Q), ("D", i.D), ("qm", i.qmask), ("dm", i.dmask))}
    if st.ce:
        host["target"] = st.target.cpu().pin_memory()
    elif w.backward:
        host["g"] = st.g.cpu().pin_memory()
    slots = [st] + [_twin(st) for _ in range(nslots - 1)]
    dev = [{k: torch.empty_like(v, device=st.device) for k, v in host.items()} for _ in slots]

    def outs_of(x: Step):
        if st.ce:  # the loss head in one call; the loss and both gradients come back
            return [x.loss, x.gQ, x.gD]
        return [x.scores] + ([x.gQ, x.gD] if w.backward else [])

    back = [[torch.empty(o.shape, dtype=o.dtype).pin_memory() for o in outs_of(x)] for x in slots]
    h2d = sum(v.numel() * v.element_size() for v in host.values())
    d2h = sum(o.numel() * o.element_size() for o in outs_of(st))
    s_in, s_out = torch.cuda.Stream(st.device), torch.cuda.Stream(st.device)
    ev_in = [torch.cuda.Event() for _ in slots]
    ev_comp = [torch.cuda.Event() for _ in slots]
    ev_out = [torch.cuda.Event() for _ in slots]
    used = [False] * nslots

    def step_k(k):
        j = k % nslots
        x, d = slots[j], dev[j]
        if used[j]:
            s_in.wait_event(ev_comp[j])   # the slot's previous step has read its inputs
        with torch.cuda.stream(s_in):
            for key in host:
                d[key].copy_(host[key], non_blocking=True)
        ev_in[j].record(s_in)
        stream.wait_event(ev_in[j])
        if used[j]:
            stream.wait_event(ev_out[j])  # and its results have been copied out
        with torch.cuda.stream(stream):
            if st.ce:
                x.ce_step(d["Q"], d["D"], d["qm"], d["dm"], d["target"])
            else:
                x.fwd(d["Q"], d["D"], d["qm"], d["dm"])
                if w.backward:
                    x.bwd(d["Q"], d["D"], d["g"], d["qm"], d["dm"])
        ev_comp[j].record(stream)
        s_out.wait_event(ev_comp[j])
        with torch.cuda.stream(s_out):
            for o, b in zip(outs_of(x), back[j]):
                b.copy_(o, non_blocking=True)
        ev_out[j].record(s_out)
        used[j] = True

    k_next = [0]

    def step():
        step_k(k_next[0])
        k_next[0] += 1

    n = max(3, min(args.steps, 20))
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)  # before the first step's input copies
    for _ in range(n):
        step()
    e1.record(s_out)  # after the last step's result copies (which follow all its work)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), st.device)
    # the pipelined steps computed what a plain step computes: the last step's
    # loss (or scores), copied to the host, equals a plain step's bit for bit
    # (both are summed in a fixed order; the inputs are the same)
    last = back[(k_next[0] - 1) % nslots][0]
    if st.ce:
        st.ce_step()
    else:
        st.fwd()
    plain = outs_of(st)[0].cpu()
    if not torch.equal(last, plain):
        raise RuntimeError("end-to-end pipeline: the last step's result differs from a plain step's")
    if w.layout == "pairwise" and not w.backward:
        val, unit = whole_job_rate(world, n, st.algorithmic_bytes(), ms, 1e9), "GB/s"
    else:
        val, unit = whole_job_rate(world, n, w.counted_flops, ms, 1e12), "TFLOP/s"
    return {"value": val, "unit": unit, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n, "ms_per_step": ms / n,
            "pipeline": f"{nslots} buffer slots, inputs up / compute / results down on 3 streams"}


# ------------------------------------------------------------- oracle arm --

def oracle_sample(name: str, budget_s: float, max_steps: int | None = None):
    """Run the fp64 oracle on query subsets of the workload until `budget_s`
    seconds (or `max_steps` subsets) have passed.  Returns (list of per-subset
    (seconds, counted_flops, bytes)), threads, description."""
    import numpy as np

    import oracle
    orc = oracle.get()
    w = W.WORKLOADS[name]
    inp = W.generate(name, device="cpu") if w.layout != "kd" else None
    if inp is None:  # the kd workload is large to draw on the CPU: use the same recipe on fewer queries
        inp = W.generate(name, device="cuda" if torch.cuda.is_available() else "cpu")
    Qn, tag = W.to_numpy(inp.Q)
    Dn, _ = W.to_numpy(inp.D)
    qm = inp.qmask.cpu().numpy()
    dm = inp.dmask.cpu().numpy()
    per_q = w.counted_flops // w.nq
    sub = 1
    results = []
    t_start = time.perf_counter()
    q0 = 0
    while True:
        qs = slice(q0 % w.nq, q0 % w.nq + sub)
        t0 = time.perf_counter()
        if w.layout == "allpairs":
            s, am, _ = orc.allpairs_fwd(Qn[qs], Dn, qm[qs], dm, dtype=tag)
            if w.backward:
                g = np.random.default_rng(0).standard_normal(s.shape)
                orc.allpairs_bwd(Qn[qs], Dn, g, am, dtype=tag)
        elif w.layout == "pairwise":
            s, am, _ = orc.pairwise_fwd(Qn[qs], Dn[qs], qm[qs], dm[qs], dtype=tag)
        else:
            s, am, _ = orc.kd_fwd(Qn[qs], Dn[qs], qm[qs], dm[qs], dtype=tag)
            if w.backward:
                g = np.random.default_rng(0).standard_normal(s.shape)
                orc.kd_bwd(Qn[qs], Dn[qs], g, am, dtype=tag)
        dt = time.perf_counter() - t0
        results.append((dt, per_q * sub))
        q0 += sub
        if max_steps is not None and len(results) >= max_steps:
            break
        if max_steps is None and time.perf_counter() - t_start >= budget_s:
            break
    desc = (f"{name}: {sum(r[1] for r in results) // per_q} single-query passes (query q against "
            f"all of its documents, cycling over the {w.nq} queries), "
            f"{'fwd+bwd' if w.backward else 'fwd'}, fp64")
    return results, orc.num_threads(), desc


def cpu_baseline(name: str, unit: str, budget_s: float = 12.0):
    results, cores, desc = oracle_sample(name, budget_s=budget_s)
    secs = sum(r[0] for r in results)
    flops = sum(r[1] for r in results)
    w = W.WORKLOADS[name]
    if unit == "GB/s":
        frac = flops / w.counted_flops
        val = frac * fwd_bytes(name) / secs / 1e9
    else:
        val = flops / secs / 1e12
    return {"value": val, "unit": unit, "cores": cores, "kind": "oracle",
            "sample": desc + f", {secs:.1f} s"}


def fwd_bytes(name: str) -> int:
    """Algorithmic forward bytes of the full workload (CPU-side recount)."""
    w = W.WORKLOADS[name]
    inp = W.generate(name, device="cuda" if torch.cuda.is_available() else "cpu")
    el = inp.Q.element_size()
    return (int(inp.dmask.sum()) * w.dim * el + inp.dmask.numel() + inp.Q.numel() * el
            + inp.qmask.numel() + math.prod(w.score_shape) * 4)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    name = args.workload
    w = W.WORKLOADS[name]
    results, cores, desc = oracle_sample(name, budget_s=0, max_steps=args.warmup + args.steps)
    timed = results[args.warmup:]
    secs = sum(r[0] for r in timed)
    flops = sum(r[1] for r in timed)
    if w.layout == "pairwise" and not w.backward:
        unit = "GB/s"
        value = flops / w.counted_flops * fwd_bytes(name) / secs / 1e9
    else:
        unit = "TFLOP/s"
        value = flops / secs / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / max(len(timed), 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, L2-normalised Gaussian tokens)",
        "config": {"workload": name, "layout": w.layout, "Q": list(w.q_shape), "D": list(w.d_shape),
                   "passes": "fwd+bwd" if w.backward else "fwd",
                   "step": "one query of the workload against all its documents"},
        "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="inbatch_b128_bf16", choices=sorted(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra-configs", action="store_true",
                    help="measure only --workload (by default a single-GPU run of the default step also "
                         "measures the per-query-candidate, reranking and large all-pairs workloads)")
    ap.add_argument("--step", choices=["auto", "fwd+bwd", "ce", "recompute"], default="auto",
                    help="ce: the workload's training step in one call (forward, cross-entropy head, backward); "
                         "fwd+bwd: forward and backward with the score gradient computed once outside the steps; "
                         "recompute: the forward saves no argmax and the backward recomputes it; "
                         "auto (default): ce for workloads with a cross-entropy head, else fwd+bwd")
    ap.add_argument("--grad-dtype", choices=["f32", "input"], default="f32",
                    help="gradients in fp32 (default) or in the inputs' dtype (the _bwd_same_dtype entry points)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.step == "auto":
        args.step = "ce" if has_ce_head(args.workload) else "fwd+bwd"
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
