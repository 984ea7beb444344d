"""Benchmark of the MHLA forward hot path on one or more GPUs (one process per GPU).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload dit] [--impl ours|reference]

A step is one pass of the hot path over one batch of the workload: one
``mhla_forward`` (non-causal MHLA: summaries, mixing, output) for the default
DiT-S/2-like workload (B=8, H=6, N=4096, d=64, M=16 blocks of 256, bf16).
Inputs are generated on the device from the seeded streams of ``workloads``
and are resident in HBM before timing starts.  To keep L2 (129 MB on GB300)
from serving the inputs, the steps rotate over R copies of the inputs and
outputs whose total exceeds 3x L2.  The K timed steps are captured in CUDA
graphs and timed with CUDA events on the launching stream; per-step events
inside the graph give the average kernel duration used for the roofline.

The JSON line also carries ``e2e`` (the same metric through the C ABI with
the inputs copied from pinned host memory and the output read back every
step), ``roofline``, ``cpu_baseline`` (the float64 oracle on a bounded sample
on this host), ``clocks`` (nvidia-smi samples during the timed region) and
``gpu_launches``.

With ``--impl reference`` the float64 CPU oracle is the reference arm: each
step runs it on a bounded sample of the same workload (rank 0 only).

Under torchrun (N > 1) each rank runs its own copy of the workload on its own
GPU (independent problems, no data-path collective, weak scaling); the time
is the maximum over ranks and ``value`` counts the tokens of all ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MHLA fwd tokens/s (B*H*N) at N=4096,d=64 bf16; % of HBM roofline"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def workload_bytes(wl):
    """Algorithmic HBM bytes of one step: every input read once, every output written once."""
    eb = 2 if wl.dtype == "bf16" else 4
    t = wl.B * wl.H * wl.N * wl.d * eb
    if wl.kind in ("mhla", "causal"):
        mix = wl.H * wl.M * wl.M * 4 if wl.mixing != "none" else 0
        return 4 * t + mix
    if wl.kind == "decode":
        units = wl.B * wl.H
        return units * (2 * (wl.d * wl.d + wl.d) * 4 + 4 * wl.d * eb)
    if wl.kind == "decode_steps":  # the state once in and out, each step's q, k, v, out, den
        units = wl.B * wl.H
        return units * (2 * (wl.d * wl.d + wl.d) * 4 + wl.N * (4 * wl.d * eb + 4))
    if wl.kind == "stream":
        # each token's q, k, v, out, den; the summaries frozen before the call read once (and the
        # running summary of a block the call starts inside); each touched block's summary written once
        units, P, blk = wl.B * wl.H, wl.extra["prefix"], wl.block
        first, last = P // blk, (P + wl.N - 1) // blk
        slot = (wl.d * wl.d + wl.d) * 4
        reads = first * slot + (slot if P % blk else 0)
        return units * (wl.N * (4 * wl.d * eb + 4) + reads + (last - first + 1) * slot)
    if wl.kind == "rala":
        cx = wl.extra["cx"]
        return 4 * t + wl.B * wl.N * cx * eb + cx * wl.d * eb
    if wl.kind == "backward":  # Q, K, V, dY read once, dQ, dK, dV written once; the mixing in, dM out
        return 7 * t + 2 * wl.H * wl.M * wl.M * 4
    raise ValueError(wl.kind)


def tokens_per_step(wl):
    return wl.B * wl.H if wl.kind == "decode" else wl.B * wl.H * wl.N  # stream: N tokens a unit


def workload_flops(wl):
    """fp32 operations of one call (an FMA counts 2).
    Fused decode, per unit and step: the state update and the output read 2 d^2 FMAs, the
    denominator d FMAs, z d adds.
    MHLA backward: see the per-head-token count below.
    Causal MHLA inference, per unit and token: S_i += phi(k) v^T, R += m_ii phi(k) v^T and the
    output phi(q) R are 3 d^2 FMAs, z_i d adds, the mixed z and the denominator 2 d FMAs; per block
    that starts in the call, sum_{b<i} m_ib (S_b, z_b) is i (d^2 + d) FMAs."""
    d = wl.d
    if wl.kind == "decode_steps":
        return wl.B * wl.H * wl.N * (4 * d * d + 3 * d)
    if wl.kind == "backward":
        # per head-token: S_b, num, dphi(q), dS~, dphi(k), dv are 6 d^2 FMAs; z, den, dden, dnum,
        # dden z~, dz~, dq, dz, dk another 4 d FMAs and 5 d adds / multiplies; per unit the mixing,
        # its transpose and dM are 3 M^2 (d^2 + d) FMAs
        M = wl.M
        return wl.B * wl.H * (wl.N * (12 * d * d + 13 * d) + 6 * M * M * (d * d + d))
    assert wl.kind == "stream"
    P, blk = wl.extra["prefix"], wl.block
    starts = range(-(-P // blk), (P + wl.N - 1) // blk + 1)  # blocks starting inside the call
    mixed = sum(starts) + (P // blk if P % blk else 0)     # slots mixed at their starts
    return wl.B * wl.H * (wl.N * (6 * d * d + 5 * d) + mixed * 2 * (d * d + d))


def fp32_peak_tflops(sm_count, sm_mhz=2070.0):
    """FP32 FMA peak: 128 FP32 lanes per SM, 2 operations per FMA, at the given SM clock."""
    return sm_count * 128 * 2 * sm_mhz * 1e6 / 1e12


def max_over_ranks(ms, world, device=None):
    """The job's time: the largest of the ranks' times (an all-reduce MAX over
    the default process group when there is more than one rank)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(tokens_per_rank_step, steps, world, ms):
    """Whole-job throughput: every rank's units over the job's time (weak scaling)."""
    return world * tokens_per_rank_step * steps / (ms / 1e3)


VARIANT_KEYS = ("feature", "normalise", "gamma")


def variant_kwargs(wl):
    """The mhla_forward_ex options a workload asks for ({} = the plain forward)."""
    return {key: wl.extra[key] for key in VARIANT_KEYS if key in wl.extra}


def describe(wl):
    s = f"{wl.name}: B{wl.B} H{wl.H} N{wl.N} d{wl.d} {wl.dtype}"
    for key, val in variant_kwargs(wl).items():
        s += f" {key}={val}"
    if wl.kind == "mhla" and "grid" in wl.extra:
        gh, gw, th, tw = wl.extra["grid"]
        s += f" M{wl.M} (2-D blocks: {gh}x{gw} grid, {th}x{tw} tiles)"
    elif wl.kind == "mhla":
        s += f" M{wl.M} (blocks of {wl.block})"
    elif wl.kind == "causal":
        s += f" causal chunk {wl.block}"
    elif wl.kind == "decode":
        s = f"{wl.name}: {wl.B}x{wl.H} units d{wl.d} {wl.dtype}, one recurrent step, fp32 state"
    elif wl.kind == "decode_steps":
        s = (f"{wl.name}: {wl.B}x{wl.H} units d{wl.d} {wl.dtype}, {wl.N} recurrent steps in one call, "
             f"fp32 state")
    elif wl.kind == "stream":
        s = (f"{wl.name}: {wl.B}x{wl.H} units d{wl.d} {wl.dtype}, causal MHLA inference of {wl.N} tokens "
             f"after a {wl.extra['prefix']}-token prefix, blocks of {wl.block}, M{wl.M}")
    elif wl.kind == "rala":
        s += f" cx{wl.extra['cx']}"
    return s


# The sources whose code a kernel family's DRAM traffic depends on: a traffic
# record in profiles/ counts only while their digest is unchanged.
KERNEL_SOURCES = {
    "mhla_tcgen05": ["tc_mhla.cu"],
    "mhla_tcgen05_stream": ["tc_stream.cu", "stream_sched.h"],
    "causal_tcgen05": ["tc_causal.cu"],
    "causal_mhla_tcgen05": ["tc_causal.cu", "tc_mhla.cu"],
    "rala_tcgen05": ["tc_rala.cu"],
    "decode_steps_simt": ["decode_steps.cu"],
    "stream_simt": ["causal_stream.cu"],
    "backward_simt": ["mhla_backward.cu"],
    "backward_tcgen05": ["mhla_backward.cu", "tc_backward.cu"],
}
SHARED_SOURCES = ["tc_common.cuh", "common.cuh"]


def parse_traffic(kernel_name, workload_name):
    """DRAM bytes per call recorded from an ncu capture of this kernel family on this workload,
    if the family's sources are unchanged since (else None)."""
    import glob
    src = source_digest(kernel_name)
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path).read()
        m_k = re.search(r"^bench_kernel:\s*(\S+)", text, re.M)
        m_w = re.search(r"^workload:\s*(\S+)", text, re.M)
        m_t = re.search(r"^traffic_bytes_per_launch:\s*([0-9.eE+]+)", text, re.M)
        m_s = re.search(r"^source_sha256:\s*([0-9a-f]+)", text, re.M)
        if (m_k and m_w and m_t and m_s and m_k.group(1) == kernel_name and m_w.group(1) == workload_name
                and m_s.group(1) == src):
            return float(m_t.group(1))
    return None


def source_digest(kernel_name):
    """sha256 (16 hex digits) of the sources of one kernel family (unknown families: all of csrc)."""
    import glob
    csrc = os.path.join(ROOT, "token_level_head_gb300", "csrc")
    names = KERNEL_SOURCES.get(kernel_name)
    files = ([os.path.join(csrc, n) for n in names + SHARED_SOURCES] if names is not None
             else sorted(glob.glob(os.path.join(csrc, "*"))))
    h = hashlib.sha256()
    for path in files:
        with open(path, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.lines = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

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
        rows = []
        for ts, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        used = inside or [r for r in rows if t0 - 0.25 <= r[0] <= t1 + 0.25]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in used), "sm_max_mhz": max(r[2] for r in used),
                "reasons": reasons, "samples": len(used),
                "window": "timed region" if inside else "timed region +-0.25 s"}


# --------------------------------------------------------------- runners
class Runner:
    """Device buffers and the per-step call of one workload (R rotating sets)."""

    def __init__(self, wl, device, l2_bytes, sets=0):
        import torch
        from token_level_head_gb300 import binding
        import workloads

        self.wl, self.binding, self.torch = wl, binding, torch
        self.device = device
        step_bytes = workload_bytes(wl)
        self.R = sets if sets > 0 else max(1, min(16, math.ceil(3 * l2_bytes / step_bytes)))
        if wl.kind in ("decode", "decode_steps", "stream"):
            self.R = 1  # the recurrent state is carried from one step to the next
        self.sets = []
        if wl.kind in ("mhla", "causal"):
            base = workloads.mhla_device(wl, device)
            causal = wl.kind == "causal"
            self.ws = binding.new_workspace(binding.mhla_workspace_bytes(wl.B, wl.H, wl.N, wl.d, wl.block,
                                                                         int(causal)), device)
            for r in range(self.R):
                s = {k: (v if r == 0 else v.clone()) for k, v in base.items()}
                s["y"] = torch.empty_like(s["q"])
                self.sets.append(s)
        elif wl.kind == "backward":
            base = workloads.mhla_device(wl, device)
            self.ws = binding.new_workspace(binding.mhla_backward_workspace_bytes(wl.B, wl.H, wl.N, wl.d, wl.block),
                                            device)
            for r in range(self.R):
                s = {k: (v if r == 0 else v.clone()) for k, v in base.items()}
                for g in ("dq", "dk", "dv"):
                    s[g] = torch.empty_like(s["q"])
                s["dm"] = torch.empty_like(s["mixing"])
                self.sets.append(s)
        elif wl.kind == "rala":
            base = workloads.rala_device(wl, device)
            cx = wl.extra["cx"]
            self.ws = binding.new_workspace(binding.rala_workspace_bytes(wl.B, wl.H, wl.N, wl.d, cx), device)
            for r in range(self.R):
                s = {k: (v if r == 0 else v.clone()) for k, v in base.items()}
                s["y"] = torch.empty_like(s["q"])
                self.sets.append(s)
        elif wl.kind == "decode":
            dev = workloads.decode_device(wl, device, steps=64)
            kf = dev["prefix_k"].float()
            kf = torch.where(kf > 0, kf + 1, torch.exp(kf))
            S = torch.einsum("pbhc,pbhe->bhce", kf, dev["prefix_v"].float()).contiguous()
            z = kf.sum(dim=0).contiguous()
            self.sets.append({"steps": dev, "S": S, "z": z,
                              "out": torch.empty(wl.B, wl.H, wl.d, dtype=dev["step_q"].dtype, device=device)})
            self.ws = None
        elif wl.kind == "stream":
            dev = workloads.decode_device(wl, device)
            P, blk, M = wl.extra["prefix"], wl.block, wl.M
            kf = dev["prefix_k"].float()
            kf = torch.where(kf > 0, kf + 1, torch.exp(kf))
            S = torch.zeros(wl.B, wl.H, M, wl.d, wl.d, device=device)
            z = torch.zeros(wl.B, wl.H, M, wl.d, device=device)
            nb = P // blk
            kb = kf.view(nb, blk, wl.B, wl.H, wl.d)
            S[:, :, :nb] = torch.einsum("nsbhc,nsbhe->bhnce", kb, dev["prefix_v"].float().view(nb, blk, wl.B, wl.H, wl.d))
            z[:, :, :nb] = kb.sum(dim=1).permute(1, 2, 0, 3)
            del dev["prefix_k"], dev["prefix_v"], kf, kb
            mix = torch.from_numpy(workloads.make_mixing(wl).astype("float32")).to(device)
            self.sets.append({"steps": dev, "S": S, "z": z, "mixing": mix, "out": torch.empty_like(dev["step_q"]),
                              "den": torch.empty(dev["step_q"].shape[:-1], dtype=torch.float32, device=device)})
            self.ws = None
        elif wl.kind == "decode_steps":
            dev = workloads.decode_device(wl, device)
            kf = dev["prefix_k"].float()
            kf = torch.where(kf > 0, kf + 1, torch.exp(kf))
            S = torch.einsum("pbhc,pbhe->bhce", kf, dev["prefix_v"].float()).contiguous()
            z = kf.sum(dim=0).contiguous()
            del dev["prefix_k"], dev["prefix_v"], kf
            self.sets.append({"steps": dev, "S": S, "z": z, "out": torch.empty_like(dev["step_q"]),
                              "den": torch.empty(dev["step_q"].shape[:-1], dtype=torch.float32,
                                                 device=device)})
            self.ws = None
        self.step_index = 0

    def step(self, i):
        self._call(self.sets[i % self.R], i)

    def _call(self, s, i):
        wl, b = self.wl, self.binding
        if wl.kind == "mhla" and "grid" in wl.extra:
            gh, gw, th, tw = wl.extra["grid"]
            b.mhla_forward_grid(s["q"], s["k"], s["v"], s["mixing"], s["y"], (gh, gw), (th, tw), workspace=self.ws)
        elif variant_kwargs(wl):
            b.mhla_forward_ex(s["q"], s["k"], s["v"], s.get("mixing") if wl.kind == "mhla" else None, s["y"],
                              wl.block, causal=int(wl.kind == "causal"), workspace=self.ws, **variant_kwargs(wl))
        elif wl.kind == "mhla":
            b.mhla_forward(s["q"], s["k"], s["v"], s["mixing"], s["y"], wl.block, workspace=self.ws)
        elif wl.kind == "causal":
            b.mhla_forward_causal(s["q"], s["k"], s["v"], s.get("mixing"), s["y"], wl.block, workspace=self.ws)
        elif wl.kind == "rala":
            b.rala_forward(s["q"], s["k"], s["v"], s["x"], s["w"], s["y"], workspace=self.ws)
        elif wl.kind == "backward":
            b.mhla_backward(s["q"], s["k"], s["v"], s["mixing"], s["dy"], s["dq"], s["dk"], s["dv"], s["dm"],
                            wl.block, workspace=self.ws)
        elif wl.kind == "decode":
            st = s["steps"]
            t = i % st["step_q"].shape[0]
            b.linattn_decode_step(st["step_q"][t], st["step_k"][t], st["step_v"][t], s["S"], s["z"], s["out"])
        elif wl.kind == "decode_steps":
            st = s["steps"]
            b.linattn_decode_steps(st["step_q"], st["step_k"], st["step_v"], s["S"], s["z"], s["out"],
                                   den_out=s["den"])
        elif wl.kind == "stream":
            st = s["steps"]
            b.mhla_causal_stream(st["step_q"], st["step_k"], st["step_v"], s["mixing"], s["S"], s["z"], s["out"],
                                 wl.extra["prefix"], wl.block, den_out=s["den"])

    # ---- end to end: host inputs -> device -> forward -> host output
    def e2e_setup(self):
        torch = self.torch
        s = self.sets[0]
        if self.wl.kind == "decode":
            st = s["steps"]
            self.h_in = {k: st[k][:8].cpu().pin_memory() for k in ("step_q", "step_k", "step_v")}
            self.h_out = torch.empty_like(s["out"], device="cpu").pin_memory()
            return
        if self.wl.kind == "decode_steps":
            st = s["steps"]
            self.h_in = {k: st[k].cpu().pin_memory() for k in ("step_q", "step_k", "step_v")}
            self.h_out = torch.empty_like(s["out"], device="cpu").pin_memory()
            return
        names = ["q", "k", "v"] + (["x"] if self.wl.kind == "rala" else [])
        self.h_in = {n: s[n].cpu().pin_memory() for n in names}
        self.h_out = torch.empty_like(s["y"], device="cpu").pin_memory()
        # pipelined runs: two device sets, two pinned output buffers, copy streams
        self.nb = min(2, len(self.sets))
        self.h_outs = [self.h_out] + [torch.empty_like(self.h_out).pin_memory() for _ in range(self.nb - 1)]
        self.s_h2d = [torch.cuda.Stream() for _ in self.h_in]  # one per input: the copies run side by side
        self.s_d2h = torch.cuda.Stream()

    def e2e_step(self, i):
        s = self.sets[0]
        wl = self.wl
        if wl.kind == "decode":
            st = s["steps"]
            t = i % 8
            for n in ("step_q", "step_k", "step_v"):
                st[n][t].copy_(self.h_in[n][t], non_blocking=True)
            self.binding.linattn_decode_step(st["step_q"][t], st["step_k"][t], st["step_v"][t], s["S"], s["z"], s["out"])
            self.h_out.copy_(s["out"], non_blocking=True)
            return
        if wl.kind == "decode_steps":
            st = s["steps"]
            for n in ("step_q", "step_k", "step_v"):
                st[n].copy_(self.h_in[n], non_blocking=True)
            self._call(s, i)
            self.h_out.copy_(s["out"], non_blocking=True)
            return
        for n, h in self.h_in.items():
            s[n].copy_(h, non_blocking=True)
        self._call(s, i)
        self.h_out.copy_(s["y"], non_blocking=True)

    def e2e_run(self, k):
        """k steps from host buffers, copies and calls pipelined: the inputs of
        step i go up (copy stream) while step i - 1 computes and step i - 2's
        output comes down (second copy stream); every step still moves its own
        inputs and output.  Returns the elapsed ms (first copy to last copy)."""
        torch = self.torch
        if self.wl.kind in ("decode", "decode_steps"):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record()
            for i in range(k):
                self.e2e_step(i)
            e1.record()
            torch.cuda.synchronize()
            return e0.elapsed_time(e1)
        cs = torch.cuda.current_stream()
        h2d, d2h, nb = self.s_h2d, self.s_d2h, self.nb
        ev_in = [[torch.cuda.Event() for _ in h2d] for _ in range(k)]
        ev_done = [torch.cuda.Event() for _ in range(k)]
        ev_out = [torch.cuda.Event() for _ in range(k)]
        start = torch.cuda.Event(enable_timing=True)
        end = torch.cuda.Event(enable_timing=True)
        start.record(cs)
        for st in h2d:
            st.wait_stream(cs)
        for i in range(k):
            b = self.sets[i % nb]
            for j, (n, h) in enumerate(self.h_in.items()):
                with torch.cuda.stream(h2d[j]):
                    if i >= nb:
                        h2d[j].wait_event(ev_done[i - nb])  # the call that read this set's inputs is done
                    b[n].copy_(h, non_blocking=True)
                    ev_in[i][j].record(h2d[j])
            for ev in ev_in[i]:
                cs.wait_event(ev)
            if i >= nb:
                cs.wait_event(ev_out[i - nb])  # this set's previous output has been read back
            self._call(b, i)
            ev_done[i].record(cs)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev_done[i])
                self.h_outs[i % nb].copy_(b["y"], non_blocking=True)
                ev_out[i].record(d2h)
        end.record(d2h)
        torch.cuda.synchronize()
        return start.elapsed_time(end)

    def e2e_bytes(self):
        h2d = sum(t[:1].numel() * t.element_size() if self.wl.kind == "decode" else t.numel() * t.element_size()
                  for t in self.h_in.values())
        return h2d, self.h_out.numel() * self.h_out.element_size()


def capture(torch, runner, steps, first, with_events):
    """CUDA graph of `steps` consecutive steps starting at step index `first`; optional per-step events."""
    g = torch.cuda.CUDAGraph()
    events = None
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        if with_events:
            try:
                events = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(steps + 1)]
            except TypeError:
                events = None
        with torch.cuda.graph(g, stream=stream):
            if events:
                events[0].record()
            for i in range(steps):
                runner.step(first + i)
                if events:
                    events[i + 1].record()
    torch.cuda.current_stream().wait_stream(stream)
    return g, events


# ------------------------------------------------------------ our arm
def kernel_path(binding, wl):
    import torch
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    if wl.kind == "rala":
        return binding.rala_forward_path(wl.B, wl.H, wl.N, wl.d, wl.extra["cx"], tdt)
    if wl.kind == "decode":
        return "simt"
    if wl.kind in ("decode_steps", "stream"):
        return "simt"
    if wl.kind == "backward":
        return binding.mhla_backward_path(wl.B, wl.H, wl.N, wl.d, wl.block, tdt)
    if "grid" in wl.extra:
        return binding.mhla_forward_grid_path(wl.B, wl.H, *wl.extra["grid"], wl.d, tdt)
    if variant_kwargs(wl) or (wl.kind == "causal" and wl.mixing != "none"):
        causal = int(wl.kind == "causal")
        with_mixing = int(wl.mixing != "none")
        return binding.mhla_forward_ex_path(wl.B, wl.H, wl.N, wl.d, wl.block, causal, with_mixing, tdt,
                                            **variant_kwargs(wl))
    return binding.mhla_forward_path(wl.B, wl.H, wl.N, wl.d, wl.block or 1, int(wl.kind == "causal"), tdt)


def kernel_family(wl, path):
    """Name of the kernel family a workload runs (keys the traffic records in profiles/)."""
    if wl.kind == "causal" and wl.mixing != "none":
        return f"causal_mhla_{path}"
    return f"{wl.kind}_{path}"


def time_steps(torch, binding, runner, steps, warmup, world=1, sampler=None):
    """W eager + graph warm-up steps, then `steps` timed steps (CUDA graphs, events on the
    launching stream).  Returns (elapsed ms of the timed region, mean per-step ms from events
    inside the graph or None, kernels per step, wall-clock window)."""
    import torch.distributed as dist
    for i in range(max(1, warmup)):
        runner.step(i)
    torch.cuda.synchronize()
    launches0 = binding.mhla_launch_count()
    chunk = min(steps, 64 * runner.R)
    chunk -= chunk % runner.R if chunk >= runner.R else 0
    chunk = max(chunk, 1)
    g, events = capture(torch, runner, chunk, 0, True)
    per_step_kernels = (binding.mhla_launch_count() - launches0) / chunk
    rem = steps % chunk
    g_rem = capture(torch, runner, rem, 0, False)[0] if rem else None
    n_chunks = steps // chunk
    g_warm = capture(torch, runner, max(warmup, 1), 0, False)[0]
    torch.cuda.synchronize()
    g_warm.replay()
    torch.cuda.synchronize()
    if sampler is not None:
        sampler.start()
        time.sleep(0.3)
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    start.record()
    for _ in range(n_chunks):
        g.replay()
    if g_rem is not None:
        g_rem.replay()
    end.record()
    torch.cuda.synchronize()
    t1 = time.time()
    if world > 1:
        dist.barrier()
    if sampler is not None:
        time.sleep(0.2)
        sampler.stop()
    step_ms = None
    if events:
        durs = [events[i].elapsed_time(events[i + 1]) for i in range(chunk)]
        step_ms = sum(durs) / len(durs)
    return start.elapsed_time(end), step_ms, per_step_kernels, (t0, t1)


def parity_of_timed_output(runner, n_slices=4):
    """The timed output of one rotating set (after the graph replays: no den_out, the shared
    workspace) against the float64 oracle on sampled slices: max slice-relative error."""
    import numpy as np
    import oracle
    import workloads
    wl = runner.wl
    s = runner.sets[min(1, runner.R - 1)]
    if wl.kind in ("mhla", "causal"):
        units = wl.B * wl.H
        pick = sorted({0, units - 1} | {(units * i) // n_slices for i in range(n_slices)})[:n_slices]
        heads = [(u // wl.H, u % wl.H) for u in pick]
        x = workloads.mhla_host(wl, heads=heads)
        vk = variant_kwargs(wl)
        if wl.kind == "mhla" and "grid" in wl.extra:
            ids = oracle.grid_block_ids(*wl.extra["grid"])
            ref, _ = oracle.mhla_block_form_ids(x["q64"], x["k64"], x["v64"], x["mixing64"], ids)
        elif wl.kind == "mhla" and vk:
            ref, _ = oracle.mhla_block_form_feature(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block,
                                                    vk.get("feature", "elu1"), 1e-6, vk.get("normalise", True))
        elif wl.kind == "causal" and vk:
            ref, _ = oracle.causal_variant_recurrent(x["q64"], x["k64"], x["v64"], vk.get("feature", "elu1"),
                                                     vk.get("gamma", 1.0), 1e-6, vk.get("normalise", True))
        elif wl.kind == "mhla":
            ref, _ = oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block)
        elif wl.mixing != "none":
            ref, _ = oracle.causal_mhla_chunked(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block)
        else:
            ref, _ = oracle.causal_chunked(x["q64"], x["k64"], x["v64"], wl.block)
        got = np.stack([s["y"][b, h].float().cpu().numpy() for b, h in heads]).astype(np.float64)
        ref = ref[0]
        desc = f"{len(heads)} of {units} (batch, head) slices"
    elif wl.kind == "decode_steps":
        return parity_of_decode_steps(runner)
    elif wl.kind == "stream":
        return parity_of_stream(runner)
    elif wl.kind == "backward":
        return parity_of_backward(runner)
    elif wl.kind == "rala":
        batches = [0, wl.B - 1][:n_slices]
        host = workloads.rala_host(wl, batches)
        ref = oracle.rala_forward(host["q64"], host["k64"], host["v64"], host["x64"], host["w64"])
        got = s["y"][batches].float().cpu().numpy().astype(np.float64)
        ref = ref.reshape(len(batches) * wl.H, wl.N, wl.d)
        got = got.reshape(len(batches) * wl.H, wl.N, wl.d)
        desc = f"{len(batches)} of {wl.B} samples"
    else:
        return None
    err = np.abs(got - ref).reshape(len(got), -1).max(1) / np.abs(ref).reshape(len(ref), -1).max(1)
    tol = 2e-2 if wl.dtype == "bf16" else 1e-4
    return {"max_slice_rel_err": float(err.max()), "tol": tol, "ok": bool(err.max() <= tol),
            "sample": f"{desc}, timed output (no den_out, reused workspace, graph replay)"}


def parity_of_decode_steps(runner):
    """One more fused decode call in the timed configuration, with the state of two units (the
    first and the last) set to the oracle's prefix summary: those units' outputs and final state
    against the float64 oracle's recurrence."""
    import numpy as np
    import torch
    import oracle
    import workloads
    wl, s = runner.wl, runner.sets[0]
    U, d, T = wl.B * wl.H, wl.d, wl.N
    units = [0, U - 1]
    host = workloads.decode_host(wl, units)
    kf = oracle.phi(host["prefix_k64"])
    s0 = np.einsum("puc,pue->uce", kf, host["prefix_v64"]).astype(np.float32)
    z0 = kf.sum(axis=0).astype(np.float32)
    Sf, zf = s["S"].view(U, d, d), s["z"].view(U, d)
    for i, u in enumerate(units):
        Sf[u] = torch.from_numpy(s0[i]).to(Sf.device)
        zf[u] = torch.from_numpy(z0[i]).to(zf.device)
    runner.step(0)
    torch.cuda.synchronize()
    sel = torch.tensor(units, device=Sf.device)
    got = s["out"].view(T, U, d)[:, sel].float().cpu().numpy().astype(np.float64).transpose(1, 0, 2)
    s_got = Sf[sel].cpu().numpy().astype(np.float64)
    ref, _, s_t, _ = oracle.decode_steps(s0, z0, host["step_q64"], host["step_k64"], host["step_v64"])
    ref = ref.transpose(1, 0, 2)
    err = np.abs(got - ref).reshape(len(units), -1).max(1) / np.abs(ref).reshape(len(units), -1).max(1)
    s_err = float((np.abs(s_got - s_t).reshape(len(units), -1).max(1)
                   / np.abs(s_t).reshape(len(units), -1).max(1)).max())
    tol = 2e-2 if wl.dtype == "bf16" else 1e-4
    return {"max_slice_rel_err": float(err.max()), "state_rel_err": s_err, "tol": tol,
            "ok": bool(err.max() <= tol and s_err <= 1e-4),
            "sample": f"2 of {U} units, all {T} steps of one timed-configuration call, state set to the "
                      f"oracle's {wl.extra['prefix']}-token prefix summary"}


def parity_of_stream(runner):
    """Two units (the first and the last) of the timed stream call against the oracle's token-by-token
    causal MHLA over the prefix and the streamed tokens (the prefix's own outputs are not compared)."""
    import numpy as np
    import oracle
    import workloads
    wl, s = runner.wl, runner.sets[0]
    U, d, T, P = wl.B * wl.H, wl.d, wl.N, wl.extra["prefix"]
    units = [0, U - 1]
    host = workloads.decode_host(wl, units)
    k64 = np.concatenate([host["prefix_k64"], host["step_k64"]]).transpose(1, 0, 2)[None]
    v64 = np.concatenate([host["prefix_v64"], host["step_v64"]]).transpose(1, 0, 2)[None]
    q64 = np.concatenate([np.zeros_like(host["prefix_k64"]), host["step_q64"]]).transpose(1, 0, 2)[None]
    mix = workloads.make_mixing(wl)[[u % wl.H for u in units]]
    ref, _ = oracle.causal_mhla_stream(q64, k64, v64, mix, wl.block)
    ref = ref[0, :, P:]
    got = s["out"].view(T, U, d)[:, units].float().cpu().numpy().astype(np.float64).transpose(1, 0, 2)
    err = np.abs(got - ref).reshape(len(units), -1).max(1) / np.abs(ref).reshape(len(units), -1).max(1)
    tol = 2e-2 if wl.dtype == "bf16" else 1e-4
    return {"max_slice_rel_err": float(err.max()), "tol": tol, "ok": bool(err.max() <= tol),
            "sample": f"2 of {U} units, all {T} tokens of the timed call (graph replay)"}


def parity_of_backward(runner):
    """All eight samples of head 0 of the timed backward (dQ, dK, dV and the head's dM) against the
    oracle's backward."""
    import numpy as np
    import oracle
    import workloads
    wl, s = runner.wl, runner.sets[0]
    host = workloads.mhla_host(wl, heads=[(b, 0) for b in range(wl.B)])
    shp = (wl.B, 1, wl.N, wl.d)
    ref = oracle.mhla_block_form_backward(host["q64"].reshape(shp), host["k64"].reshape(shp), host["v64"].reshape(shp),
                                          host["mixing64"][:1], wl.block, host["dy64"].reshape(shp))
    got = [s[g][:, :1].float().cpu().numpy().astype(np.float64) for g in ("dq", "dk", "dv")]
    got.append(s["dm"][:1].cpu().numpy().astype(np.float64))
    errs = [float(np.max(np.abs(g - r)) / np.max(np.abs(r))) for g, r in zip(got, ref)]
    tol = 2e-2 if wl.dtype == "bf16" else 1e-4
    return {"max_rel_err": {"dq": errs[0], "dk": errs[1], "dv": errs[2], "dmixing": errs[3]}, "tol": tol,
            "ok": bool(max(errs) <= tol),
            "sample": f"head 0 of {wl.H}, all {wl.B} samples, of the timed call (graph replay)"}


def alu_roofline(torch, wl, device, launch_ms):
    """The roofline of the fp32 SIMT paths (fused decode, causal MHLA inference, the backward):
    fp32 FMA issue, which binds them (their minimal HBM time is well below their minimal FMA
    time), against the FP32 peak at the maximum SM clock (152 SMs x 128 lanes x 2 x 2070 MHz)."""
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    peak = fp32_peak_tflops(sms)
    achieved = workload_flops(wl) / (launch_ms / 1e3) / 1e12
    return {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "peak_source": f"derived: {sms} SMs x 128 FP32 lanes x 2 flops x 2070 MHz",
            "alg_flops_per_launch": workload_flops(wl)}


def workload_line(torch, binding, wl, device, l2, steps, warmup, sets=0):
    """value, launch time and roofline of one more workload (one GPU, no e2e or CPU baseline)."""
    runner = Runner(wl, device, l2, sets)
    elapsed_ms, step_ms, kernels, _ = time_steps(torch, binding, runner, steps, warmup)
    alg = workload_bytes(wl)
    peak, _ = hbm_peak()
    kernel_ms = step_ms if step_ms is not None else elapsed_ms / steps
    achieved = alg / (kernel_ms / 1e3) / 1e9
    path = kernel_path(binding, wl)
    kname = kernel_family(wl, path)
    out = {"workload": describe(wl), "value": tokens_per_step(wl) * steps / (elapsed_ms / 1e3),
           "unit": "tokens/s" if wl.kind != "decode" else "units/s", "steps": steps,
           "ms_per_step": elapsed_ms / steps, "launch_ms": kernel_ms, "kernels_per_step": kernels,
           "path": path, "alg_bytes": alg, "achieved_GBps": achieved, "roofline_frac": achieved / peak,
           "traffic": parse_traffic(kname, wl.name), "kernel": kname}
    if wl.kind == "decode":
        out["note"] = ("effective bandwidth: the 68 MB recurrent state may stay in L2 from one step to "
                       "the next, so this is not a DRAM figure")
    elif wl.kind == "decode_steps":
        out["unit"] = "unit-steps/s"
        out["roofline"] = alu_roofline(torch, wl, device, kernel_ms)
        out["parity"] = parity_of_timed_output(runner)
    elif wl.kind == "stream" or (wl.kind == "backward" and path == "simt"):
        out["roofline"] = alu_roofline(torch, wl, device, kernel_ms)
        out["parity"] = parity_of_timed_output(runner)
    elif wl.kind == "backward":  # tensor-core token passes: bound by HBM like the forward
        out["parity"] = parity_of_timed_output(runner)
    else:
        out["parity"] = parity_of_timed_output(runner, n_slices=2)
    del runner
    torch.cuda.empty_cache()
    return out


def run_ours(args, wl, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from token_level_head_gb300 import binding
    from token_level_head_gb300.build import build_library

    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    if rank == 0 or world == 1:
        build_library()
    if world > 1:
        dist.barrier()
    binding.load()
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 0) or (126 << 20)
    runner = Runner(wl, device, l2, args.sets)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    elapsed_ms, step_ms, per_step_kernels, (t_wall0, t_wall1) = time_steps(
        torch, binding, runner, args.steps, args.warmup, world, sampler)
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)
    parity = parity_of_timed_output(runner) if rank == 0 else None

    # end to end through host buffers
    e2e = None
    if not args.no_e2e and wl.kind != "backward":  # the end-to-end form covers the forward workloads
        runner.e2e_setup()
        k_e2e = max(3, min(args.steps, 50))
        runner.e2e_run(2)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        e_ms = runner.e2e_run(k_e2e)
        e_ms = max_over_ranks(e_ms, world, device)
        h2d, d2h = runner.e2e_bytes()
        e2e = {"value": job_value(tokens_per_step(wl), k_e2e, world, e_ms), "unit": "tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": k_e2e,
               "ms_per_step": e_ms / k_e2e,
               "pipelining": "host->device copies (one stream per input), calls and device->host "
                             "copies overlapped across steps, two device sets"}

    if rank != 0:
        return None
    alg = workload_bytes(wl)
    peak, peak_src = hbm_peak()
    kernel_ms = step_ms if step_ms is not None else elapsed_ms / args.steps
    achieved = alg / (kernel_ms / 1e3) / 1e9
    path = kernel_path(binding, wl)
    kernel_name = kernel_family(wl, path)
    value = job_value(tokens_per_step(wl), args.steps, world, elapsed_ms)
    line = {
        "metric": METRIC if wl.name == "dit" else f"{wl.name} tokens/s",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": elapsed_ms / args.steps,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if wl.dtype == "bf16" else "f32",
        "data": "synthetic (seeded SplitMix64 normal inputs, generated on the device)",
        "config": {"workload": describe(wl), "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d,
                   "block_size": wl.block, "M": wl.M, "parallelism": f"independent replicas x{world}",
                   "l2": f"inputs larger than L2: {runner.R} rotating input/output sets of "
                         f"{alg / 1e6:.1f} MB (L2 {l2 / 2**20:.0f} MiB)",
                   "timing": "CUDA graphs, CUDA events on the launching stream",
                   "path": path},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": parse_traffic(kernel_name, wl.name),
                     "kernel": kernel_name, "kernels_per_step": per_step_kernels,
                     "alg_bytes_per_launch": alg, "launch_ms": kernel_ms, "peak_source": peak_src,
                     "frac_of_nominal_8TBps": achieved / 8000.0},
        "gpu_launches": int(round(per_step_kernels * args.steps)),
        "clocks": sampler.summary(t_wall0, t_wall1),
        "parity": parity,
    }
    if wl.kind in ("decode_steps", "stream") or (wl.kind == "backward" and path == "simt"):  # fp32 FMA issue
        line["roofline"] = dict(alu_roofline(torch, wl, device, kernel_ms), kernel=kernel_name,
                                traffic=line["roofline"]["traffic"], kernels_per_step=per_step_kernels,
                                launch_ms=kernel_ms, effective_GBps=achieved)
    if e2e is not None:
        line["e2e"] = e2e
    # the other workloads of the pages (one GPU): rooflines and launch times beside the metric's
    if world == 1 and not args.no_workloads:
        del runner
        torch.cuda.empty_cache()
        extra = {}
        for name in ("dit_grid", "dit_unnormalised", "dit_relu", "hires", "hires_m1", "causal", "causal_mhla", "causal_decay",
                     "rala", "decode", "decode_fused", "stream", "dit_backward"):
            if name == wl.name:
                continue
            try:
                wl_x = workloads_mod().WORKLOADS[name]
                slow = wl_x.kind in ("decode_steps", "stream") or bench_path_is_simt(binding, wl_x)
                n_x = min(args.steps, 20 if slow else 200)
                extra[name] = workload_line(torch, binding, wl_x, device, l2, n_x, args.warmup)
            except Exception as e:  # report, do not lose the metric line
                extra[name] = {"error": f"{type(e).__name__}: {e}"[:300]}
        line["workloads"] = extra
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl, budget_s=args.cpu_seconds)
    return line


def bench_path_is_simt(binding, wl):
    return kernel_path(binding, wl) == "simt"


def workloads_mod():
    import workloads
    return workloads


# ------------------------------------------------------ oracle (CPU) arm
def _oracle_sample(wl, n_units):
    """Prepares one bounded sample of the workload for the oracle; returns (fn, tokens, description)."""
    import numpy as np
    import oracle
    import workloads

    if wl.kind in ("mhla", "causal"):
        heads = [(i // wl.H % wl.B, i % wl.H) for i in range(n_units)]
        x = workloads.mhla_host(wl, heads=heads)
        if wl.kind == "mhla" and "grid" in wl.extra:
            ids = oracle.grid_block_ids(*wl.extra["grid"])
            fn = lambda: oracle.mhla_block_form_ids(x["q64"], x["k64"], x["v64"], x["mixing64"], ids)  # noqa: E731
        elif wl.kind == "mhla":
            fn = lambda: oracle.mhla_block_form(x["q64"], x["k64"], x["v64"], x["mixing64"], wl.block)  # noqa: E731
        else:
            fn = lambda: oracle.causal_chunked(x["q64"], x["k64"], x["v64"], wl.block)  # noqa: E731
        return fn, n_units * wl.N, f"{n_units} of {wl.B * wl.H} (batch, head) slices, all {wl.N} tokens"
    if wl.kind == "decode":
        units = list(range(n_units))
        host = workloads.decode_host(wl, units, steps=1)
        s0 = np.zeros((n_units, wl.d, wl.d))
        z0 = np.zeros((n_units, wl.d))
        fn = lambda: oracle.decode_steps(s0, z0, host["step_q64"], host["step_k64"], host["step_v64"])  # noqa: E731
        return fn, n_units, f"{n_units} of {wl.B * wl.H} units, one step"
    if wl.kind == "decode_steps":
        units = list(range(n_units))
        host = workloads.decode_host(wl, units)
        s0 = np.zeros((n_units, wl.d, wl.d))
        z0 = np.zeros((n_units, wl.d))
        fn = lambda: oracle.decode_steps(s0, z0, host["step_q64"], host["step_k64"], host["step_v64"])  # noqa: E731
        return fn, n_units * wl.N, f"{n_units} of {wl.B * wl.H} units, all {wl.N} steps"
    if wl.kind == "rala":
        host = workloads.rala_host(wl, list(range(n_units)))
        fn = lambda: oracle.rala_forward(host["q64"], host["k64"], host["v64"], host["x64"], host["w64"])  # noqa: E731
        return fn, n_units * wl.H * wl.N, f"{n_units} of {wl.B} samples (all heads)"
    raise ValueError(wl.kind)


def _default_sample_units(wl):
    return {"mhla": max(1, min(wl.B * wl.H, 8)), "causal": 2, "decode": 256, "decode_steps": 4,
            "rala": 2}[wl.kind]


def _cpu_work(args):
    """One CPU-baseline worker: runs the oracle sample repeatedly for `seconds`."""
    name, n_units, seconds = args
    import workloads
    wl = workloads.WORKLOADS[name]
    fn, tokens, desc = _oracle_sample(wl, n_units)
    fn()
    t0 = time.perf_counter()
    n = 0
    while True:
        fn()
        n += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return n * tokens, dt, desc


_CPU_WORKER = r"""
import json, sys
sys.path.insert(0, %(root)r)
from bench import _cpu_work

if __name__ == "__main__":
    import multiprocessing as mp
    name, n_units, seconds, procs = sys.argv[1], int(sys.argv[2]), float(sys.argv[3]), int(sys.argv[4])
    if procs == 1:
        res = [_cpu_work((name, n_units, seconds))]
    else:
        with mp.get_context("spawn").Pool(procs) as pool:
            res = pool.map(_cpu_work, [(name, n_units, seconds)] * procs)
    tokens = sum(r[0] for r in res)
    wall = max(r[1] for r in res)
    print(json.dumps({"value": tokens / wall, "seconds": wall, "procs": procs, "desc": res[0][2]}))
"""


def cpu_baseline(wl, budget_s=10.0, n_units=None):
    """The oracle as it stands, on a bounded sample of the workload, timed on this host's cores:
    one spawned process per core (one BLAS thread each) running the sample side by side over
    independent slices, and one thread alone.  ``cores`` = the processes of the first figure."""
    cores = os.cpu_count() or 1
    n_units = n_units or _default_sample_units(wl)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    code = _CPU_WORKER % {"root": ROOT}
    out = {}
    for procs in (cores, 1):
        res = subprocess.run([sys.executable, "-c", code, wl.name, str(n_units), str(budget_s / 2), str(procs)],
                             capture_output=True, text=True, env=env, timeout=300)
        if res.returncode != 0:
            out[procs] = {"error": res.stderr.strip()[-300:]}
        else:
            out[procs] = json.loads(res.stdout.strip().splitlines()[-1])
    allc, one = out[cores], out[1]
    if "error" in allc:
        return {"value": None, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                "sample": f"failed: {allc['error']}"}
    return {"value": allc["value"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{allc['desc']}, per process; float64 numpy oracle, {cores} processes x 1 thread, "
                      f"{allc['seconds']:.1f} s",
            "host_cpus": cores,
            "single_thread": {"value": one.get("value"), "cores": 1}}


def run_reference(args, wl, rank):
    """Reference arm: the CPU oracle, each step a bounded sample of the workload (rank 0 only)."""
    if rank != 0:
        return None
    import multiprocessing  # noqa: F401  (no pool: the oracle runs in this process, single-threaded)
    n_units = _default_sample_units(wl)
    fn, tokens, desc = _oracle_sample(wl, n_units)
    t0 = time.perf_counter()
    fn()
    per = time.perf_counter() - t0
    budget = 150.0
    while n_units > 1 and per * (args.steps + args.warmup) > budget:
        n_units = max(1, n_units // 2)
        fn, tokens, desc = _oracle_sample(wl, n_units)
        t0 = time.perf_counter()
        fn()
        per = time.perf_counter() - t0
    for _ in range(args.warmup):
        fn()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        fn()
    dt = time.perf_counter() - t0
    value = tokens * args.steps / dt
    return {
        "impl": "reference",
        "metric": METRIC if wl.name == "dit" else f"{wl.name} tokens/s",
        "value": value, "unit": "tokens/s", "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded SplitMix64 normal inputs)",
        "config": {"workload": describe(wl), "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d,
                   "block_size": wl.block, "M": wl.M},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{desc} per step; float64 numpy oracle, 1 thread"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--workload", default="dit")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other workloads' roofline lines (the metric line only)")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--sets", type=int, default=0,
                   help="rotating input sets (default: enough to exceed 3x L2); 1 for small profiler captures")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    import workloads
    wl = workloads.WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        line = run_reference(args, wl, rank)
    else:
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("nccl")
        line = run_ours(args, wl, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
