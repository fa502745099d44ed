#!/usr/bin/env python3
"""Benchmark of the FP8 (e4m3) block-scaled linear layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload large_square]
                    [--impl ours|reference] [--no-cpu-baseline] [--no-configs]
                    [--profile-steps P]

One step = one pass of the whole path over one batch of synthetic input:
dense workloads run act_quant(X) and fp8_gemm with W quantised once before
timing (the large square adds weight_dequant(Wq); q_down_m<M>_fused runs the
GEMM with bias and FP8 output; <dense>_pow2 quantises both operands with
power-of-two scales and times the fp32-scale quantisers beside them);
moe runs act_quant over the expert-grouped token rows and the grouped
fp8_gemm, moe_swiglu the grouped w1|w3 stage with SwiGLU and FP8 h, and
moe_layer the whole routed layer with its router (expert weights quantised
once, before timing).  The default workload is the large square
(X [16384,7168] Student-t(3) x W [7168,7168]: act_quant + fp8_gemm +
weight_dequant), the largest configuration; the line also carries, under
"configs", each kernel's roofline row for all five configurations (tiny, the
KV down-projection, the Q down-projection sweep, the large square and the MoE
grouped GEMM).

Timing: W warm-up steps, then exactly K steps captured in CUDA graphs and
replayed between CUDA events, bracketed by a barrier and a synchronize; the
inputs rotate over enough buffer sets that the data touched between two uses
of a set exceeds the 126 MB L2.  Per-kernel times come from graphs holding K
launches of that kernel alone.  Under torchrun each rank runs its own
replica (the layer needs no exchange); rank 0 prints one JSON line with the
whole-job value (units of all ranks / max time over ranks).

--impl reference times the CPU oracle (plain C, test infrastructure) on a
bounded sample of the same workload instead -- the only arm that runs it,
besides the cpu_baseline leg of our own line.
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

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

L2_BYTES = 126 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
FP8_OVER_BF16 = 2.0  # nominal dense ratio: 4.5 PFLOP/s fp8 vs 2.25 PFLOP/s bf16
METRIC = "fp8_gemm TFLOP/s & % of dense FP8 peak; act_quant GB/s & % of HBM peak"


# ---------------------------------------------------------------- helpers

def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="large_square",
                    help="large_square | kv_down | tiny | q_down_m<M>[_fused] | <dense>_pow2 | moe | moe_e<G> | moe_swiglu | "
                         "moe_layer | moe_router | kv_down_wgrad | large_square_wgrad | q_down_m<M>_wgrad")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-kernel table of the five configurations")
    ap.add_argument("--profile-steps", type=int, default=0,
                    help="run this many eager steps of the workload and exit (for a profiler); nothing is timed")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="target CPU time of the oracle sample")
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of untimed steps before the warm-up, so the clock record sees sustained load")
    return ap.parse_args(argv)


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, local, world


def dist_init(world: int, backend: str):
    if world > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend)


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device: str = "cpu") -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x: float, world: int, device: str = "cpu") -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# the sources each kernel with a committed DRAM-traffic capture is built from
# (its own file, the shared PTX and codec headers, the launch declarations and
# the tensor-map encoder): a change to any of them voids the capture
KERNEL_SOURCES = {
    "fp8_gemm": ("gemm.cu", "ptx.cuh", "codec.cuh", "internal.h", "tmap.cu"),
}


def kernel_sources_sha(kernel: str = "fp8_gemm") -> str:
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "fp8_block_scaled_18_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since that capture."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    if kernel not in KERNEL_SOURCES:
        return None
    sha = kernel_sources_sha(kernel)
    for line in open(path):
        if line.startswith("#") or not line.strip():
            continue
        kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
        if kv.get("kernel") == kernel and kv.get("workload") == workload and kv.get("src_sha") == sha:
            return float(kv["dram_bytes_per_launch"])
    return None


class ClockSampler:
    """nvidia-smi clocks + throttle reasons every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()

    def summary(self) -> dict:
        rows = []
        self.file.seek(0)
        for line in self.file:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.file.name)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ---------------------------------------------------------------- workloads

class DenseWork:
    """act_quant(X) -> fp8_gemm (-> weight_dequant(Wq) for the large square),
    with W quantised once before timing (weight_quant is timed on its own as
    a table row).  fused: the GEMM is fp8bs_gemm_fused with a bias and the
    output re-quantised to FP8 (1x128 groups, ready for the next FP8 GEMM)
    instead of bf16.  pow2: both operands quantised with power-of-two
    (UE8M0-style) scales (fp8bs_act_quant_pow2 in the step, W by
    fp8bs_weight_quant_pow2), the fp32-scale quantisers timed beside them
    into buffers of their own."""

    def __init__(self, case, device, fused=False, min_sets=1, pow2=False):
        import torch
        from fp8_block_scaled_18_b300 import fp8bs as F
        self.F = F
        self.case = case
        self.device = device
        self.M, self.N, self.K = case.shape
        M, N, K = self.M, self.N, self.K
        self.x_host = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16)
        self.w_host = torch.from_numpy(case.w.view(np.int16)).view(torch.bfloat16)
        self.dequant = case.name == "large_square"  # the configuration's own extra step
        per_set = 2 * M * K + 2 * N * K + M * K + 4 * M * (K // 128) + N * K + 2 * M * N + 2 * N * K
        self.R = max(1, min(8, math.ceil(2 * L2_BYTES / per_set) + 1)) if per_set < 2 * L2_BYTES else 1
        self.R = max(self.R, min_sets)
        lds = max(4, (K // 128 + 3) // 4 * 4)
        ws_bytes = F.fp8bs_gemm_workspace_size(M, N, K)
        self.fused = fused
        self.pow2 = pow2
        if fused:
            self.bias = torch.from_numpy(
                np.random.default_rng(5).standard_normal(N).astype(np.float32)).to(torch.bfloat16).to(device)
        self.sets = []
        for _ in range(self.R):
            s = dict(x=self.x_host.to(device), w=self.w_host.to(device),
                     xq=torch.empty((M, K), dtype=torch.uint8, device=device),
                     sx=torch.empty((M, lds), dtype=torch.float32, device=device),
                     wq=torch.empty((N, K), dtype=torch.uint8, device=device),
                     sw=torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=device),
                     y=torch.empty((M, (N + 7) // 8 * 8), dtype=torch.bfloat16, device=device)[:, :N],
                     wd=torch.empty((N, K), dtype=torch.bfloat16, device=device),
                     ws=torch.empty(ws_bytes, dtype=torch.uint8, device=device) if ws_bytes else None)
            if fused:
                s["yq"] = torch.empty((M, N), dtype=torch.uint8, device=device)
                s["sy"] = torch.empty((M, max(4, (N // 128 + 3) // 4 * 4)), dtype=torch.float32, device=device)
                s["yq2"] = torch.empty((M, N), dtype=torch.uint8, device=device)
                s["sy2"] = torch.empty((M, max(4, (N // 128 + 3) // 4 * 4)), dtype=torch.float32, device=device)
            if pow2:  # outputs of the fp32-scale quantisers timed for comparison
                for k in ("xq", "sx", "wq", "sw"):
                    s[k + "_f32"] = torch.empty_like(s[k])
            self.sets.append(s)
        self.set_bytes = per_set
        self.gemm_launches = 2 if ws_bytes else 1
        self.flops = 2.0 * M * N * K
        nb, kb = (N + 127) // 128, K // 128
        # operand bytes of one GEMM: codes of X and W, scales, bf16 output
        gemm_bytes = 1.0 * M * K + 1.0 * N * K + 4.0 * M * kb + 4.0 * nb * kb + 2.0 * M * N
        self.kernels = {
            # name: (callable(set), launches, algorithmic units, bound[, bytes for a tensor-bound row])
            "weight_quant": (lambda s: F.fp8bs_weight_quant(s["w"], wq=s["wq"], sw=s["sw"]), 1,
                             3.0 * N * K + 4.0 * nb * kb, "hbm"),
            "act_quant": (lambda s: F.fp8bs_act_quant(s["x"], xq=s["xq"], sx=s["sx"]), 1,
                          3.0 * M * K + 4.0 * M * kb, "hbm"),
            "fp8_gemm": (lambda s: F.fp8bs_gemm(s["xq"], s["sx"], s["wq"], s["sw"], y=s["y"], workspace=s["ws"]),
                         self.gemm_launches, self.flops, "tensor", gemm_bytes),
            "weight_dequant": (lambda s: F.fp8bs_weight_dequant(s["wq"], s["sw"], w=s["wd"]), 1,
                               3.0 * N * K + 4.0 * nb * kb, "hbm"),
        }
        self.order = ["weight_quant", "act_quant", "fp8_gemm", "weight_dequant"]
        if pow2:
            self.kernels["weight_quant"] = (lambda s: F.fp8bs_weight_quant(s["w"], wq=s["wq_f32"], sw=s["sw_f32"]),
                                            1, 3.0 * N * K + 4.0 * nb * kb, "hbm")
            self.kernels["act_quant"] = (lambda s: F.fp8bs_act_quant(s["x"], xq=s["xq_f32"], sx=s["sx_f32"]), 1,
                                         3.0 * M * K + 4.0 * M * kb, "hbm")
            self.kernels["weight_quant_pow2"] = (
                lambda s: F.fp8bs_weight_quant_pow2(s["w"], wq=s["wq"], sw=s["sw"]), 1, 3.0 * N * K + 4.0 * nb * kb,
                "hbm")
            self.kernels["act_quant_pow2"] = (lambda s: F.fp8bs_act_quant_pow2(s["x"], xq=s["xq"], sx=s["sx"]), 1,
                                              3.0 * M * K + 4.0 * M * kb, "hbm")
            self.order = ["weight_quant", "weight_quant_pow2", "act_quant", "act_quant_pow2", "fp8_gemm",
                          "weight_dequant"]
        if fused:
            # the fused GEMM, and what it replaces: the plain GEMM plus act_quant over its output
            fused_bytes = gemm_bytes - 2.0 * M * N + 1.0 * M * N + 4.0 * M * (N // 128) + 2.0 * N
            self.kernels["fp8_gemm_fused"] = (
                lambda s: F.fp8bs_gemm_fused(s["xq"], s["sx"], s["wq"], s["sw"], bias=self.bias, want_y=False,
                                             want_fp8=True, yq=s["yq"], sy=s["sy"]), 1, self.flops, "tensor",
                fused_bytes)
            self.kernels["act_quant_of_y"] = (lambda s: F.fp8bs_act_quant(s["y"], xq=s["yq2"], sx=s["sy2"]), 1,
                                              3.0 * M * N + 4.0 * M * (N // 128), "hbm")
            self.order = ["weight_quant", "act_quant", "fp8_gemm_fused", "weight_dequant", "fp8_gemm",
                          "act_quant_of_y"]
        self.step_kernels = ["act_quant_pow2" if pow2 else "act_quant", "fp8_gemm_fused" if fused else "fp8_gemm"]
        if self.dequant:
            self.step_kernels.append("weight_dequant")

    def prepare(self):
        """The weight as a checkpoint holds it: quantised once, before timing."""
        quant = self.F.fp8bs_weight_quant_pow2 if self.pow2 else self.F.fp8bs_weight_quant
        for s in self.sets:
            quant(s["w"], wq=s["wq"], sw=s["sw"])

    def step(self, i):
        s = self.sets[i % self.R]
        F = self.F
        (F.fp8bs_act_quant_pow2 if self.pow2 else F.fp8bs_act_quant)(s["x"], xq=s["xq"], sx=s["sx"])
        if self.fused:
            F.fp8bs_gemm_fused(s["xq"], s["sx"], s["wq"], s["sw"], bias=self.bias, want_y=False, want_fp8=True,
                               yq=s["yq"], sy=s["sy"])
        else:
            F.fp8bs_gemm(s["xq"], s["sx"], s["wq"], s["sw"], y=s["y"], workspace=s["ws"])
        if self.dequant:
            F.fp8bs_weight_dequant(s["wq"], s["sw"], w=s["wd"])

    def launches_per_step(self):
        return sum(self.kernels[k][1] for k in self.step_kernels)

    # e2e: per step the bf16 X comes in from pinned host memory and the
    # result (bf16 Y, or FP8 Yq and its scales for the fused workload) goes
    # back; the weight stays resident in its quantised form
    def e2e_slots(self):
        import torch
        if len(self.sets) < 2:  # a second buffer set so copies overlap compute
            s0 = self.sets[0]
            s1 = {k: (torch.empty_like(v) if isinstance(v, torch.Tensor) else v) for k, v in s0.items()}
            s1["y"] = torch.empty((self.M, (self.N + 7) // 8 * 8), dtype=torch.bfloat16,
                                  device=self.device)[:, :self.N]
            s1["wq"], s1["sw"] = s0["wq"], s0["sw"]
            self.sets.append(s1)
        xp = self.x_host.pin_memory()
        slots = []
        for j in range(2):
            s = self.sets[j]
            if self.fused:
                outs = [(torch.empty(s["yq"].shape, dtype=torch.uint8).pin_memory(), s["yq"]),
                        (torch.empty(s["sy"].shape, dtype=torch.float32).pin_memory(), s["sy"])]
            else:
                outs = [(torch.empty((self.M, self.N), dtype=torch.bfloat16).pin_memory(), s["y"])]
            slots.append({"h2d": [(s["x"], xp)], "d2h": outs, "run": (lambda j=j: self.step(j))})
        self.R = max(self.R, 2) if len(self.sets) >= 2 else self.R
        return slots

    def config(self):
        step = ("act_quant_pow2+" if self.pow2 else "act_quant+") + (
            "fp8_gemm_fused(bias, fp8 out)" if self.fused else "fp8_gemm")
        if self.dequant:
            step += "+weight_dequant"
        wq = "W quantised once before timing, as a checkpoint stores it"
        if self.pow2:
            wq = "power-of-two (UE8M0-style) scales on both operands; " + wq
        return {"workload": self.case.name + ("_fused" if self.fused else "") + ("_pow2" if self.pow2 else ""),
                "M": self.M, "N": self.N, "K": self.K, "step": f"{step} ({wq})",
                "l2": f"inputs rotate over {self.R} buffer sets of {self.set_bytes / 1e6:.0f} MB (> 126 MB L2)"
                      if self.R > 1 else f"working set {self.set_bytes / 1e6:.0f} MB, larger than the 126 MB L2"}


class MoEWork:
    """act_quant over the expert-grouped rows -> grouped fp8_gemm.
    swiglu: the grouped GEMM is the expert first stage with w1 and w3 and the
    SwiGLU activation fused (h = silu(x w1^T) * (x w3^T))."""

    def __init__(self, device, swiglu=False, experts=None):
        import torch
        from fp8_block_scaled_18_b300 import fp8bs as F
        from fp8_block_scaled_18_b300 import synth
        self.F = F
        case = synth.moe() if experts is None else moe_small_case(experts)
        self.case = case
        G, N, K = case.n_experts, case.n, case.k
        self.G, self.N, self.K = G, N, K
        self.T = int(case.offsets[-1])
        x_rows = case.x_rows
        self.x_host = torch.from_numpy(x_rows.view(np.int16)).view(torch.bfloat16)
        self.x = self.x_host.to(device)
        self.wq = torch.empty((G, N, K), dtype=torch.uint8, device=device)
        self.sw = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device=device)
        for g in range(G):
            F.fp8bs_weight_quant(synth.expert_weight(case, g, device), wq=self.wq[g], sw=self.sw[g])
        self.swiglu = swiglu
        if swiglu:
            self.w3q = torch.empty((G, N, K), dtype=torch.uint8, device=device)
            self.sw3 = torch.empty((G, N // 128, K // 128), dtype=torch.float32, device=device)
            for g in range(G):
                F.fp8bs_weight_quant(synth.expert_weight(case, g, device, which=1), wq=self.w3q[g], sw=self.sw3[g])
        self.off = torch.from_numpy(case.offsets).to(device)
        lds = (K // 128 + 3) // 4 * 4
        self.xq = torch.empty((self.T, K), dtype=torch.uint8, device=device)
        self.sx = torch.empty((self.T, lds), dtype=torch.float32, device=device)
        self.y = torch.empty((self.T, N), dtype=torch.bfloat16, device=device)
        self.bufs = [{"x": self.x, "xq": self.xq, "sx": self.sx, "y": self.y}]
        self.R = 1
        counts = np.diff(case.offsets)
        self.flops = 2.0 * self.T * N * K
        gbytes = G * N * K + 4.0 * G * (N // 128) * (K // 128) + self.T * K + 4.0 * self.T * (K // 128) \
            + 2.0 * self.T * N
        self.kernels = {
            "act_quant": (lambda s: F.fp8bs_act_quant(self.x, xq=self.xq, sx=self.sx), 1,
                          3.0 * self.T * K + 4.0 * self.T * (K // 128), "hbm"),
            "grouped_gemm": (lambda s: F.fp8bs_grouped_gemm(self.xq, self.sx, self.wq, self.sw, self.off, y=self.y),
                             1, gbytes, "hbm"),
        }
        self.order = ["act_quant", "grouped_gemm"]
        if swiglu:
            self.flops = 4.0 * self.T * N * K
            gbytes3 = 2.0 * G * N * K + 8.0 * G * (N // 128) * (K // 128) + self.T * K + 4.0 * self.T * (K // 128) \
                + 2.0 * self.T * N
            # h leaves as FP8 (1x128 groups): the operand of the w2 GEMM
            self.hq = torch.empty((self.T, N), dtype=torch.uint8, device=device)
            self.sh = torch.empty((self.T, max(4, (N // 128 + 3) // 4 * 4)), dtype=torch.float32, device=device)
            self.bufs[0].update(hq=self.hq, sh=self.sh)
            del self.bufs[0]["y"]
            gbytes3 -= self.T * N  # one byte per h element instead of two
            self.kernels["grouped_gemm_swiglu"] = (
                lambda s: F.fp8bs_grouped_gemm_swiglu(self.xq, self.sx, self.wq, self.sw, self.w3q, self.sw3,
                                                      self.off, want_h=False, want_fp8=True, hq=self.hq,
                                                      sh=self.sh), 1, gbytes3, "hbm")
            del self.kernels["grouped_gemm"]
            self.order = ["act_quant", "grouped_gemm_swiglu"]
        self.grouped_flops = self.flops
        self.experts_nonempty = int((counts > 0).sum())
        self.step_kernels = list(self.order)

    def prepare(self):
        pass

    def step(self, i):
        b = self.bufs[i % len(self.bufs)]
        F = self.F
        F.fp8bs_act_quant(b["x"], xq=b["xq"], sx=b["sx"])
        if self.swiglu:
            F.fp8bs_grouped_gemm_swiglu(b["xq"], b["sx"], self.wq, self.sw, self.w3q, self.sw3, self.off,
                                        want_h=False, want_fp8=True, hq=b["hq"], sh=b["sh"])
        else:
            F.fp8bs_grouped_gemm(b["xq"], b["sx"], self.wq, self.sw, self.off, y=b["y"])

    def launches_per_step(self):
        return 2

    # e2e: per step the expert-grouped bf16 rows and the offsets come in, the
    # output (bf16 y, or FP8 h and its scales) goes back
    def e2e_slots(self):
        import torch
        if len(self.bufs) < 2:
            self.bufs.append({k: torch.empty_like(v) for k, v in self.bufs[0].items()})
        xp = self.x_host.pin_memory()
        offp = torch.from_numpy(self.case.offsets).pin_memory()
        slots = []
        for j in range(2):
            b = self.bufs[j]
            if self.swiglu:
                outs = [(torch.empty(b["hq"].shape, dtype=torch.uint8).pin_memory(), b["hq"]),
                        (torch.empty(b["sh"].shape, dtype=torch.float32).pin_memory(), b["sh"])]
            else:
                outs = [(torch.empty(b["y"].shape, dtype=torch.bfloat16).pin_memory(), b["y"])]
            # the offsets buffer is shared: every step carries the same routing
            slots.append({"h2d": [(b["x"], xp)] + ([(self.off, offp)] if j == 0 else []), "d2h": outs,
                          "run": (lambda j=j: self.step(j))})
        return slots

    def config(self):
        if self.swiglu:
            return {"workload": "moe_swiglu", "tokens": self.T // 8, "experts": self.G, "top_k": 8, "rows": self.T,
                    "I": self.N, "K": self.K,
                    "step": "act_quant+grouped w1|w3 fp8_gemm with SwiGLU, h out as FP8 (expert weights "
                            "pre-quantised)",
                    "l2": "working set (7.5 GB of expert weights) larger than the 126 MB L2"}
        wgb = self.G * self.N * self.K / 1e9
        return {"workload": "moe_grouped" if self.G == 256 else f"moe_e{self.G}", "tokens": self.T // 8,
                "experts": self.G, "top_k": 8, "rows": self.T,
                "N": self.N, "K": self.K, "step": "act_quant+grouped_fp8_gemm (expert weights pre-quantised)",
                "l2": f"working set ({wgb:.2f} GB of expert weights) larger than the 126 MB L2"}


class MoELayerWork:
    """The routed-expert layer end to end on the device: the router (gate
    logits, group-limited top-8, gate values) and its routing tables,
    act_quant of the tokens, dispatch into expert order, the w1|w3 SwiGLU
    stage with FP8 h, the w2 grouped GEMM, the shared expert (SwiGLU stage
    over all tokens, dense w2 GEMM) and the gated combine with the shared
    output added.  Expert, shared and gate weights are quantised (or, for the
    gate, stored in bf16) once, before timing."""

    def __init__(self, device):
        import torch
        from fp8_block_scaled_18_b300 import fp8bs as F
        from fp8_block_scaled_18_b300 import synth
        self.F = F
        case = synth.moe()
        self.case = case
        G, I, D = case.n_experts, case.n, case.k
        tokens = case.x_tokens.shape[0]
        self.G, self.I, self.D, self.tokens = G, I, D, tokens
        self.T = T = int(case.offsets[-1])
        self.topk = case.rows_of_token.shape[1]
        self.x_host = torch.from_numpy(case.x_tokens.view(np.int16)).view(torch.bfloat16)
        self.x = self.x_host.to(device)

        def quant(which, gs):
            n, k = (D, I) if which == 2 else (I, D)
            wq = torch.empty((len(gs), n, k), dtype=torch.uint8, device=device)
            sw = torch.empty((len(gs), n // 128, k // 128), dtype=torch.float32, device=device)
            for j, g in enumerate(gs):
                F.fp8bs_weight_quant(synth.expert_weight(case, g, device, which=which), wq=wq[j], sw=sw[j])
            return wq, sw

        routed, shared = list(range(G)), [G]
        self.w1q, self.sw1 = quant(0, routed)
        self.w3q, self.sw3 = quant(1, routed)
        self.w2q, self.sw2 = quant(2, routed)
        self.s1q, self.ss1 = quant(0, shared)
        self.s3q, self.ss3 = quant(1, shared)
        s2q, ss2 = quant(2, shared)
        self.s2q, self.ss2 = s2q[0], ss2[0]
        # the router runs on the device every step: gate weight and bias
        # resident, the routing tables written by fp8bs_moe_route
        self.gw = torch.from_numpy(case.gate_w.view(np.int16)).view(torch.bfloat16).to(device)
        self.gbias = torch.from_numpy(case.gate_bias).to(device)
        self.ids = torch.empty((tokens, self.topk), dtype=torch.int32, device=device)
        self.gates = torch.empty((tokens, self.topk), dtype=torch.float32, device=device)
        self.off = torch.empty(G + 1, dtype=torch.int32, device=device)
        self.off1 = torch.tensor([0, tokens], dtype=torch.int32, device=device)
        self.tor = torch.empty(T, dtype=torch.int32, device=device)
        self.rot = torch.empty((tokens, self.topk), dtype=torch.int32, device=device)
        self.wrow = torch.empty(T, dtype=torch.float32, device=device)
        ldk = (D // 128 + 3) // 4 * 4
        ldi = max(4, (I // 128 + 3) // 4 * 4)
        e = lambda *shape, dt=torch.uint8: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        self.xq, self.sx = e(tokens, D), e(tokens, ldk, dt=torch.float32)
        self.xr, self.sr = e(T, D), e(T, ldk, dt=torch.float32)
        self.hq, self.sh = e(T, I), e(T, ldi, dt=torch.float32)
        self.yk = e(T, D, dt=torch.bfloat16)
        self.hsq, self.shs = e(tokens, I), e(tokens, ldi, dt=torch.float32)
        self.z = e(tokens, D, dt=torch.bfloat16)
        self.y = e(tokens, D, dt=torch.bfloat16)
        self.R = 1
        KBd, KBi = D // 128, I // 128
        wsc = lambda n, k: 4.0 * (n // 128) * (k // 128)  # noqa: E731  (scales of one weight)
        self.kernels = {
            "moe_gate": (lambda s: F.fp8bs_moe_gate(self.x, self.gw, self.gbias, ids=self.ids, weights=self.gates), 1,
                         2.0 * tokens * G * D, "tensor_bf16"),
            "moe_route": (lambda s: F.fp8bs_moe_route(self.ids, self.gates, G, offsets=self.off, token_of_row=self.tor,
                                                      rows_of_token=self.rot, weight_of_row=self.wrow), 1,
                          8.0 * tokens * self.topk + 12.0 * T, "hbm"),
            "act_quant": (lambda s: F.fp8bs_act_quant(self.x, xq=self.xq, sx=self.sx), 1,
                          3.0 * tokens * D + 4.0 * tokens * KBd, "hbm"),
            # reads each token once (its repeats come from L2), writes every routed row
            "moe_dispatch": (lambda s: F.fp8bs_moe_dispatch(self.xq, self.sx, self.tor, xq_rows=self.xr,
                                                            sx_rows=self.sr), 1,
                             tokens * D + 4.0 * tokens * KBd + T * D + 4.0 * T * KBd, "hbm"),
            "grouped_gemm_swiglu": (
                lambda s: F.fp8bs_grouped_gemm_swiglu(self.xr, self.sr, self.w1q, self.sw1, self.w3q, self.sw3,
                                                      self.off, want_h=False, want_fp8=True, hq=self.hq,
                                                      sh=self.sh), 1,
                2.0 * G * I * D + 2 * G * wsc(I, D) + T * D + 4.0 * T * KBd + T * I + 4.0 * T * KBi, "hbm"),
            "grouped_gemm_w2": (
                lambda s: F.fp8bs_grouped_gemm(self.hq, self.sh, self.w2q, self.sw2, self.off, y=self.yk), 1,
                1.0 * G * D * I + G * wsc(D, I) + T * I + 4.0 * T * KBi + 2.0 * T * D, "hbm"),
            "shared_swiglu": (
                lambda s: F.fp8bs_grouped_gemm_swiglu(self.xq, self.sx, self.s1q, self.ss1, self.s3q, self.ss3,
                                                      self.off1, want_h=False, want_fp8=True, hq=self.hsq,
                                                      sh=self.shs), 1, 4.0 * tokens * I * D, "tensor"),
            "shared_w2": (lambda s: F.fp8bs_gemm(self.hsq, self.shs, self.s2q, self.ss2, y=self.z), 1,
                          2.0 * tokens * D * I, "tensor"),
            "moe_combine": (lambda s: F.fp8bs_moe_combine(self.yk, self.wrow, self.rot, z=self.z, y=self.y), 1,
                            2.0 * T * D + 4.0 * tokens * D + 4.0 * T + 4.0 * tokens * self.topk + 2.0 * tokens * D,
                            "hbm"),
        }
        self.order = ["moe_gate", "moe_route", "act_quant", "moe_dispatch", "grouped_gemm_swiglu", "grouped_gemm_w2",
                      "shared_swiglu", "shared_w2", "moe_combine"]
        self.flops = T * (4.0 * I * D + 2.0 * D * I) + tokens * (4.0 * I * D + 2.0 * D * I) + 2.0 * tokens * G * D
        self.grouped_flops = T * (4.0 * I * D + 2.0 * D * I)
        self.experts_nonempty = int((np.diff(case.offsets) > 0).sum())
        self.step_kernels = list(self.order)

    def prepare(self):
        pass

    def step(self, i):
        for k in self.order:
            self.kernels[k][0](None)

    def launches_per_step(self):
        return len(self.order)

    # e2e: per step the tokens come in (the router runs on the device) and the
    # layer output goes back; the kernels read self.x and write self.y, which
    # each slot points at its own pair of buffers before it runs
    def e2e_slots(self):
        import torch
        xs = [self.x, torch.empty_like(self.x)]
        ys = [self.y, torch.empty_like(self.y)]
        xp = self.x_host.pin_memory()

        def run(j):
            self.x, self.y = xs[j], ys[j]
            self.step(j)
        return [{"h2d": [(xs[j], xp)], "d2h": [(torch.empty(self.y.shape, dtype=torch.bfloat16).pin_memory(),
                                                ys[j])], "run": (lambda j=j: run(j))} for j in range(2)]

    def config(self):
        return {"workload": "moe_layer", "tokens": self.tokens, "experts": self.G, "top_k": self.topk,
                "rows": self.T, "dim": self.D, "I": self.I, "shared_experts": 1,
                "step": "router (bf16 gate GEMM, sigmoid, group-limited top-8) + routing tables, act_quant, "
                        "dispatch, grouped w1|w3 SwiGLU (FP8 h), grouped w2, shared expert (SwiGLU + dense w2), "
                        "gated combine (expert and shared weights pre-quantised)",
                "l2": "working set (11.3 GB of expert weights) larger than the 126 MB L2"}


class WgradWork:
    """The weight gradient of a dense layer of the given shape: dW = dY^T X
    over the M tokens, with dY [M, N] (a synthetic gradient: N(0,1) with 1 %
    of its channels x10) and X [M, K] the configuration's activations:
    act_quant_cols(dY) + act_quant_cols(X) (128x1 groups along the tokens,
    codes transposed) + gemm_wgrad (fp32 dW [N, K])."""

    def __init__(self, case, device):
        import torch
        from fp8_block_scaled_18_b300 import fp8bs as F
        from fp8_block_scaled_18_b300 import synth
        self.F = F
        self.case = case
        self.device = device
        M, N, K = case.shape
        self.M, self.N, self.K = M, N, K
        dy = synth.activations(np.random.default_rng(77), M, N, n_outlier=max(1, N // 100), outlier_scale=10.0)
        self.dy_host = torch.from_numpy(dy.view(np.int16)).view(torch.bfloat16)
        self.x_host = torch.from_numpy(case.x.view(np.int16)).view(torch.bfloat16)
        ldt = (M + 15) // 16 * 16
        TB = (M + 127) // 128
        e = lambda *shape, dt=torch.uint8: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        self.dy, self.x = self.dy_host.to(device), self.x_host.to(device)
        self.dyqt, self.sdy = e(N, ldt), e(TB, N, dt=torch.float32)
        self.xqt, self.sx = e(K, ldt), e(TB, K, dt=torch.float32)
        self.dw = e(N, (K + 3) // 4 * 4, dt=torch.float32)[:, :K]
        self.bufs = [{"dy": self.dy, "x": self.x, "dw": self.dw}]
        self.R = 1
        self.flops = 2.0 * M * N * K
        wbytes = 1.0 * N * M + 1.0 * K * M + 4.0 * TB * (N + K) + 4.0 * N * K
        self.kernels = {
            "act_quant_cols_dy": (lambda s: F.fp8bs_act_quant_cols(self.dy, xqt=self.dyqt, sc=self.sdy), 1,
                                  3.0 * M * N + 4.0 * TB * N, "hbm"),
            "act_quant_cols_x": (lambda s: F.fp8bs_act_quant_cols(self.x, xqt=self.xqt, sc=self.sx), 1,
                                 3.0 * M * K + 4.0 * TB * K, "hbm"),
            "gemm_wgrad": (lambda s: F.fp8bs_gemm_wgrad(self.dyqt, self.sdy, self.xqt, self.sx, M, dw=self.dw), 1,
                           self.flops, "tensor", wbytes),
        }
        self.order = ["act_quant_cols_dy", "act_quant_cols_x", "gemm_wgrad"]
        self.step_kernels = list(self.order)

    def prepare(self):
        pass

    def step(self, i):
        for k in self.order:
            self.kernels[k][0](None)

    def launches_per_step(self):
        return 3

    # e2e: per step dY and X come in (bf16), dW goes back (fp32)
    def e2e_slots(self):
        import torch
        b0 = self.bufs[0]
        b1 = {k: torch.empty_like(v) for k, v in b0.items()}
        dyp, xp = self.dy_host.pin_memory(), self.x_host.pin_memory()

        def run(b):
            self.dy, self.x, self.dw = b["dy"], b["x"], b["dw"]
            self.step(0)
        return [{"h2d": [(b["dy"], dyp), (b["x"], xp)],
                 "d2h": [(torch.empty(b["dw"].shape, dtype=torch.float32).pin_memory(), b["dw"])],
                 "run": (lambda b=b: run(b))} for b in (b0, b1)]

    def config(self):
        return {"workload": self.case.name + "_wgrad", "T": self.M, "N": self.N, "K": self.K,
                "step": "act_quant_cols(dY) + act_quant_cols(X) + gemm_wgrad (dW = dY^T X, fp32)",
                "l2": f"working set {(3.0 * self.M * (self.N + self.K) + 4.0 * self.N * self.K) / 1e6:.0f} MB"}


class RouterWork:
    """The MoE router alone on 4096 tokens: the gate (bf16 gate logits,
    sigmoid, group-limited top-8, gate values) and its routing tables."""

    def __init__(self, device):
        import torch
        from fp8_block_scaled_18_b300 import fp8bs as F
        from fp8_block_scaled_18_b300 import synth
        self.F = F
        case = synth.moe()
        self.case = case
        G, D = case.n_experts, case.k
        tokens = case.x_tokens.shape[0]
        self.G, self.D, self.tokens = G, D, tokens
        self.topk = case.rows_of_token.shape[1]
        T = tokens * self.topk
        self.x_host = torch.from_numpy(case.x_tokens.view(np.int16)).view(torch.bfloat16)
        self.x = self.x_host.to(device)
        self.gw = torch.from_numpy(case.gate_w.view(np.int16)).view(torch.bfloat16).to(device)
        self.gbias = torch.from_numpy(case.gate_bias).to(device)
        e = lambda *shape, dt=torch.int32: torch.empty(shape, dtype=dt, device=device)  # noqa: E731
        self.ids, self.gates = e(tokens, self.topk), e(tokens, self.topk, dt=torch.float32)
        self.off, self.tor, self.rot, self.wrow = e(G + 1), e(T), e(tokens, self.topk), e(T, dt=torch.float32)
        self.R = 1
        self.kernels = {
            "moe_gate": (lambda s: F.fp8bs_moe_gate(self.x, self.gw, self.gbias, ids=self.ids, weights=self.gates), 1,
                         2.0 * tokens * G * D, "tensor_bf16"),
            "moe_route": (lambda s: F.fp8bs_moe_route(self.ids, self.gates, G, offsets=self.off, token_of_row=self.tor,
                                                      rows_of_token=self.rot, weight_of_row=self.wrow), 1,
                          8.0 * tokens * self.topk + 12.0 * T, "hbm"),
        }
        self.order = ["moe_gate", "moe_route"]
        self.step_kernels = list(self.order)
        self.flops = 2.0 * tokens * G * D

    def prepare(self):
        pass

    def step(self, i):
        for k in self.order:
            self.kernels[k][0](None)

    def launches_per_step(self):
        return 2

    def e2e_slots(self):
        import torch
        xs = [self.x, torch.empty_like(self.x)]
        xp = self.x_host.pin_memory()

        def run(j):
            self.x = xs[j]
            self.step(j)
        return [{"h2d": [(xs[j], xp)],
                 "d2h": [(torch.empty(self.ids.shape, dtype=torch.int32).pin_memory(), self.ids),
                         (torch.empty(self.gates.shape, dtype=torch.float32).pin_memory(), self.gates)],
                 "run": (lambda j=j: run(j))} for j in range(2)]

    def config(self):
        return {"workload": "moe_router", "tokens": self.tokens, "experts": self.G, "top_k": self.topk,
                "dim": self.D, "step": "moe_gate (bf16 gate GEMM, sigmoid, group-limited top-8, gate values) + "
                                       "moe_route (routing tables)",
                "l2": "inputs (59 MB) re-read each step from L2: the router is latency-bound, not HBM-bound"}


def moe_small_case(experts: int):
    """The MoE grouped configuration over fewer experts with the same rows
    per expert (4096 tokens x top-8 over 256 experts: about 128 each)."""
    from fp8_block_scaled_18_b300 import synth
    return synth.moe(tokens=max(64, 4096 * experts // 256), n_experts=experts)


def make_work(name: str, device):
    from fp8_block_scaled_18_b300 import synth
    if name == "moe":
        return MoEWork(device)
    if name == "moe_swiglu":
        return MoEWork(device, swiglu=True)
    if name.startswith("moe_e"):  # the grouped GEMM over fewer experts (a capture-sized case)
        return MoEWork(device, experts=int(name[len("moe_e"):]))
    if name == "moe_layer":
        return MoELayerWork(device)
    if name == "moe_router":
        return RouterWork(device)
    if name.endswith("_wgrad"):
        base = name[:-len("_wgrad")]
        return WgradWork(synth.kv_down() if base == "kv_down" else synth.large_square() if base == "large_square"
                         else synth.q_down(int(base[len("q_down_m"):])), device)
    if name == "kv_down":
        return DenseWork(synth.kv_down(), device)
    if name == "tiny":
        return DenseWork(synth.tiny(), device)
    if name == "large_square":
        return DenseWork(synth.large_square(), device)
    if name.startswith("q_down_m") and name.endswith("_fused"):
        return DenseWork(synth.q_down(int(name[len("q_down_m"):-len("_fused")])), device, fused=True)
    if name.endswith("_pow2"):
        return DenseWork(make_case(name), device, pow2=True)
    if name.startswith("q_down_m"):
        return DenseWork(synth.q_down(int(name[len("q_down_m"):])), device)
    raise SystemExit(f"unknown workload {name}")


# ---------------------------------------------------------------- timing

def capture(fn, count: int, start: int = 0):
    """CUDA graph of `count` consecutive calls fn(start), fn(start+1), ..."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(count):
            fn(start + i)
    return g


def replay_timed(graphs, world, device):
    """Replay graphs between events, bracketed by barrier + synchronize.
    Returns milliseconds (max over ranks)."""
    import torch
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for g in graphs:
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1), world, device)


def chunked_graphs(fn, total: int, chunk: int = 200):
    graphs = []
    done = 0
    while done < total:
        n = min(chunk, total - done)
        graphs.append(capture(fn, n, done))
        done += n
    return graphs


def kernel_row(work, k, per_call_s, peaks):
    """Per-kernel roofline row.  A tensor-bound kernel's roofline time is
    max(FLOP / FP8 peak, bytes / HBM peak) (a GEMM's roofline is whichever is slower), so
    small-M GEMMs are held to the weight read; HBM-bound kernels to their
    algorithmic bytes.  frac = roofline time / measured time, against the
    burst peaks; frac_sustained against the sustained tensor peak."""
    entry = work.kernels[k]
    _, launches, units, bound = entry[:4]
    nbytes = entry[4] if len(entry) > 4 else None
    hbm = float(peaks["hbm_gbs"])
    row = {"us_per_call": round(per_call_s * 1e6, 3), "launches_per_call": launches, "bound": bound}
    if bound in ("tensor", "tensor_bf16"):
        peak = float(peaks["bf16_tflops"]) * (FP8_OVER_BF16 if bound == "tensor" else 1.0)
        peak_s = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * (
            FP8_OVER_BF16 if bound == "tensor" else 1.0)
        t_tensor = units / (peak * 1e12)
        t_hbm = nbytes / (hbm * 1e9) if nbytes else 0.0
        row.update(achieved=round(units / per_call_s / 1e12, 2), unit="TFLOP/s")
        row["roof_bound"] = "tensor" if t_tensor >= t_hbm else "hbm"
        row["frac"] = round(max(t_tensor, t_hbm) / per_call_s, 4)
        row["frac_sustained"] = round(max(units / (peak_s * 1e12), t_hbm) / per_call_s, 4)
        if nbytes:
            row["gbs"] = round(nbytes / per_call_s / 1e9, 1)
    else:
        row.update(achieved=round(units / per_call_s / 1e9, 2), unit="GB/s", roof_bound="hbm",
                   frac=round(units / per_call_s / 1e9 / hbm, 4))
    return row


def time_kernels(work, K, world, device):
    """ms for K launches of each kernel of work.order, alone, from graphs."""
    kernel_graphs = {k: chunked_graphs(lambda i, k=k: work.kernels[k][0](work.sets[i % work.R]
                                                                         if hasattr(work, "sets") else None), K)
                     for k in work.order}
    return {k: replay_timed(kernel_graphs[k], world, device) for k in work.order}


CONFIG_TABLE = ["tiny", "kv_down"] + [f"q_down_m{m}" for m in (1, 16, 64, 512, 4096, 16384)] + \
    ["large_square", "moe"]


def config_table(args, world, device, peaks, done=None):
    """The five configurations (tiny, KV down-projection, the Q sweep, the
    large square, the MoE grouped GEMM): each kernel timed alone (graphs of K
    launches) with its roofline row, and the configuration's step."""
    import gc
    import torch
    K = args.steps
    out = {}
    for name in CONFIG_TABLE:
        if done is not None and name == done[0]:
            out[name] = done[1]
            continue
        work = make_work(name, device)
        work.prepare()
        for i in range(max(3, work.R)):
            work.step(i)
        kernel_ms = time_kernels(work, K, world, device)
        step_ms = replay_timed(chunked_graphs(work.step, K), world, device)
        rows = {k: kernel_row(work, k, kernel_ms[k] / K * 1e-3, peaks) for k in work.order}
        out[name] = {"step": work.config()["step"], "us_per_step": round(step_ms / K * 1e3, 3),
                     "kernels": rows}
        del work
        gc.collect()
        torch.cuda.empty_cache()
    return out


def e2e_overlapped(work, K, W, world, device):
    """The same steps end to end through the public calls: each step's inputs
    copied in from pinned host memory and its result copied back, on two copy
    streams, double-buffered so that step i+1's upload and step i-1's
    download run while step i computes.  Returns (ms, h2d bytes, d2h bytes)
    per K steps."""
    import torch
    slots = work.e2e_slots()
    main = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(device=device), torch.cuda.Stream(device=device)
    h2d_done = [torch.cuda.Event() for _ in slots]
    computed = [torch.cuda.Event() for _ in slots]
    d2h_done = [torch.cuda.Event() for _ in slots]
    h2d_bytes = sum(src.numel() * src.element_size() for dst, src in slots[0]["h2d"])
    d2h_bytes = sum(dst.numel() * dst.element_size() for dst, src in slots[0]["d2h"])
    for ev in computed + d2h_done:
        ev.record(main)

    def upload(i):
        j = i % 2
        up.wait_event(computed[j])           # step i-2 no longer reads this slot's inputs
        with torch.cuda.stream(up):
            for dst, src in slots[j]["h2d"]:
                dst.copy_(src, non_blocking=True)
        h2d_done[j].record(up)

    def run(n):
        upload(0)
        for i in range(n):
            j = i % 2
            if i + 1 < n:
                upload(i + 1)
            main.wait_event(h2d_done[j])
            main.wait_event(d2h_done[j])     # step i-2's result has left this slot
            slots[j]["run"]()
            computed[j].record(main)
            down.wait_event(computed[j])
            with torch.cuda.stream(down):
                for dst, src in slots[j]["d2h"]:
                    dst.copy_(src, non_blocking=True)
            d2h_done[j].record(down)
        main.wait_stream(down)

    run(W)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(main)
    run(K)
    e1.record(main)
    torch.cuda.synchronize()
    barrier(world)
    return max_over_ranks(e0.elapsed_time(e1), world, device), h2d_bytes, d2h_bytes


def run_ours(args, rank, local, world):
    import torch
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    dist_init(world, "nccl")
    from fp8_block_scaled_18_b300 import fp8bs as F

    peaks, peaks_src = load_peaks()
    work = make_work(args.workload, device)
    work.prepare()
    # eager warm-up (also loads modules and sets kernel attributes before capture)
    for i in range(max(3, work.R)):
        work.step(i)
    st = F.fp8bs_sync_status()
    if st != 0:
        raise SystemExit(f"device status after warm-up: {F.fp8bs_status_string(st)}")
    if args.profile_steps:
        # a fixed number of eager steps for a profiler, nothing timed or printed
        for i in range(args.profile_steps):
            work.step(i)
        torch.cuda.synchronize()
        st = F.fp8bs_sync_status()
        if st != 0:
            raise SystemExit(f"device status: {F.fp8bs_status_string(st)}")
        return

    K, W = args.steps, max(3, args.warmup)
    step_graphs = chunked_graphs(work.step, K)
    warm_graphs = chunked_graphs(work.step, W)

    with ClockSampler(local) as clocks:
        # soak: ~1 s of steps so the clock record covers sustained load
        t_end = time.time() + args.soak
        while time.time() < t_end:
            for g in warm_graphs:
                g.replay()
            torch.cuda.synchronize()
        for g in warm_graphs:  # W untimed warm-up steps
            g.replay()
        step_ms = replay_timed(step_graphs, world, device)
        kernel_ms = time_kernels(work, K, world, device)
    clock = clocks.summary()
    st = F.fp8bs_sync_status()
    if st != 0:
        raise SystemExit(f"device status after timing: {F.fp8bs_status_string(st)}")

    ms_per_step = step_ms / K
    total_flops = sum_over_ranks(work.flops * K, world, device)
    value = total_flops / (step_ms * 1e-3) / 1e12

    # per-kernel roofline rows; shares and the roofline kernel over the
    # step's own kernels (other kernels are timed alone, without a share)
    step_kernels = work.step_kernels
    step_ms_sum = sum(kernel_ms[k] for k in step_kernels)
    kernels = {}
    for k in work.order:
        kernels[k] = kernel_row(work, k, kernel_ms[k] / K * 1e-3, peaks)
        kernels[k]["share"] = round(kernel_ms[k] / step_ms_sum, 4) if k in step_kernels else None
    dom = max(step_kernels, key=lambda k: kernel_ms[k])
    entry = work.kernels[dom]
    units, bound = entry[2], entry[3]
    dom_s = kernel_ms[dom] / K * 1e-3
    # A tensor-bound kernel timed while the power cap held the clock (the
    # clock record shows sw_power_cap, or a median SM clock under 90 % of the
    # maximum) is compared with the sustained peak, measured the same way (a
    # seconds-long back-to-back loop under the cap); otherwise with the burst
    # peak.  Both fractions are reported.
    capped = "sw_power_cap" in clock.get("reasons", []) or (
        clock.get("sm_mhz") and clock.get("sm_max_mhz") and clock["sm_mhz"] < 0.9 * clock["sm_max_mhz"])
    if bound == "tensor":
        burst = float(peaks["bf16_tflops"]) * FP8_OVER_BF16
        sustained = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"])) * FP8_OVER_BF16
        ach = units / dom_s / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": sustained if capped else burst, "unit": "TFLOP/s"}
        peak_note = (f"{peaks_src} {'sustained' if capped else 'burst'} bf16 x {FP8_OVER_BF16:g} (nominal fp8/bf16 "
                     f"dense ratio): the clock record {'shows the power cap (median SM ' + str(clock.get('sm_mhz')) + ' MHz)' if capped else 'shows no power cap'}")
        roof["frac_burst"] = round(ach / burst, 4)
        roof["frac_sustained"] = round(ach / sustained, 4)
    elif bound == "tensor_bf16":
        roof = {"bound": "tensor", "achieved": units / dom_s / 1e12, "peak": float(peaks["bf16_tflops"]),
                "unit": "TFLOP/s"}
        peak_note = f"{peaks_src} bf16 burst"
    else:
        roof = {"bound": "hbm", "achieved": units / dom_s / 1e9, "peak": float(peaks["hbm_gbs"]), "unit": "GB/s"}
        peak_note = f"{peaks_src} HBM copy bandwidth"
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(dom, work.config()["workload"])
    roof["kernel"] = dom
    roof["peak_source"] = peak_note
    roof["algorithmic_per_launch"] = units
    for key in ("achieved", "peak", "frac"):
        roof[key] = round(roof[key], 4)

    # end to end through the public calls with pinned host buffers
    e2e_ms, h2d, d2h = e2e_overlapped(work, K, W, world, device)
    e2e_value = total_flops / (e2e_ms * 1e-3) / 1e12
    main_row = {"step": work.config()["step"], "us_per_step": round(ms_per_step * 1e3, 3), "kernels": kernels}
    main_name = args.workload
    cfg = work.config()
    launches = work.launches_per_step()
    del work

    line = {
        "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": round(ms_per_step, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 MMA, fp32 promote, bf16 out", "data": "synthetic (seeded numpy / torch RNG)",
        "config": {**cfg, "parallelism": f"replicas{world}",
                   "timing": "CUDA graphs of K steps"},
        "roofline": roof, "kernels": kernels,
        "act_quant_gbs": kernels.get("act_quant", {}).get("achieved"),
        "act_quant_hbm_frac": kernels.get("act_quant", {}).get("frac"),
        "clocks": clock,
        "e2e": {"value": round(e2e_value, 4), "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h,
                "api": "fp8bs_* C ABI via the Python binding, eager, pinned host buffers, uploads and downloads "
                       "on two copy streams double-buffered against the compute"},
        "gpu_launches": K * launches,
    }
    if not args.no_configs:
        line["configs"] = config_table(args, world, device, peaks, done=(main_name, main_row))
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.workload, args.cpu_seconds)
    if rank == 0:
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- oracle legs

def oracle_sample_step(orc, case, rows, wq, sw, pow2=False):
    """One bounded oracle pass over a dense case's step: act_quant(rows) (with
    power-of-two scales for pow2) + gemm(rows) against the quantised W
    (+ weight_dequant of W for the large square); returns the GEMM flops
    done."""
    xq, sx = (orc.act_quant_pow2 if pow2 else orc.act_quant)(case.x[rows])
    orc.gemm(xq, sx, wq, sw)
    if case.name == "large_square":
        orc.weight_dequant(wq, sw)
    return 2.0 * len(rows) * case.w.shape[0] * case.x.shape[1]


def oracle_moe_step(orc, case, experts, x_rows, rows_per_expert, swiglu=False):
    """Per expert: weight_quant of its weight(s), act_quant and GEMM of up to
    rows_per_expert of its rows; with swiglu both w1 and w3 and silu(a) * b."""
    import torch
    from fp8_block_scaled_18_b300 import synth
    flops = 0.0
    for g in experts:
        r0, r1 = int(case.offsets[g]), int(case.offsets[g + 1])
        rows = np.arange(r0, min(r1, r0 + rows_per_expert))
        xq, sx = orc.act_quant(x_rows[rows])
        outs = []
        for which in ((0, 1) if swiglu else (0,)):
            wb = synth.expert_weight(case, g, "cpu", which=which).view(torch.int16).numpy().view(np.uint16)
            wq, sw = orc.weight_quant(wb)
            outs.append(orc.gemm(xq, sx, wq, sw)[0])
            flops += 2.0 * len(rows) * case.n * case.k
        if swiglu:
            orc.swiglu(outs[0], outs[1])
    return flops


def _expert_weights_q(orc, case, g, whichs):
    import torch
    from fp8_block_scaled_18_b300 import synth
    out = []
    for which in whichs:
        wb = synth.expert_weight(case, g, "cpu", which=which).view(torch.int16).numpy().view(np.uint16)
        out.append(orc.weight_quant(wb))
    return out


def oracle_layer_rows(orc, case, wts, rows):
    """The routed layer's oracle pass for some of one expert's rows: the router
    for their tokens, act_quant of the tokens, the w1 and w3 GEMMs, silu(a) * b, h rounded to bf16 and
    quantised, the w2 GEMM, and the gated combine of those rows (each taken
    alone).  wts = the expert's quantised (w1, w3, w2).  Returns flops."""
    from fp8_block_scaled_18_b300 import synth
    (w1q, sw1), (w3q, sw3), (w2q, sw2) = wts
    toks = case.token_of_row[rows]
    orc.moe_gate(case.x_tokens[toks], case.gate_w, case.gate_bias)  # the router for those tokens
    xq, sx = orc.act_quant(case.x_tokens[toks])
    a, _ = orc.gemm(xq, sx, w1q, sw1)
    b, _ = orc.gemm(xq, sx, w3q, sw3)
    h = orc.swiglu(a, b)
    hq, sh = orc.act_quant(synth.to_bf16_bits(h.astype(np.float32)))
    yk, _ = orc.gemm(hq, sh, w2q, sw2)
    orc.moe_combine(yk, case.weight_of_row[rows], np.arange(len(rows), dtype=np.int32).reshape(-1, 1))
    return len(rows) * (6.0 * case.n * case.k + 2.0 * case.n_experts * case.k)


def make_case(workload: str):
    """The dense case of a workload name (a _pow2 suffix names the same case)."""
    from fp8_block_scaled_18_b300 import synth
    if workload.endswith("_pow2"):
        workload = workload[:-len("_pow2")]
    if workload == "kv_down":
        return synth.kv_down()
    if workload == "tiny":
        return synth.tiny()
    if workload == "large_square":
        return synth.large_square()
    if workload.startswith("q_down_m"):
        return synth.q_down(int(workload[len("q_down_m"):]))
    raise SystemExit(f"unknown workload {workload}")


def oracle_rows_for(orc, case, seconds: float, wq, sw, pow2=False) -> int:
    """Rows of a dense case whose oracle pass takes about `seconds`
    (fixed weight-side cost + per-row GEMM cost, measured on 1 and 5 rows)."""
    M = case.x.shape[0]
    t0 = time.perf_counter()
    oracle_sample_step(orc, case, np.array([0]), wq, sw, pow2)
    t1 = time.perf_counter() - t0
    t0 = time.perf_counter()
    oracle_sample_step(orc, case, np.arange(5) % M, wq, sw, pow2)
    t5 = time.perf_counter() - t0
    per_row = max((t5 - t1) / 4, 1e-4)
    fixed = max(t1 - per_row, 0.0)
    return int(max(1, min(M, (seconds - fixed) / per_row)))


def wgrad_case(workload: str):
    from fp8_block_scaled_18_b300 import synth
    base = workload[:-len("_wgrad")]
    case = (synth.kv_down() if base == "kv_down" else synth.large_square() if base == "large_square"
            else synth.q_down(int(base[len("q_down_m"):])))
    M, N, K = case.shape
    dy = synth.activations(np.random.default_rng(77), M, N, n_outlier=max(1, N // 100), outlier_scale=10.0)
    return case, dy


def wgrad_oracle_sample(orc, workload: str, seconds: float) -> dict:
    """The oracle's weight-gradient pass on a bounded sample: the column
    quantisation of dY and X, then rows of dW until about `seconds`."""
    case, dy = wgrad_case(workload)
    M, N, K = case.shape
    t0 = time.perf_counter()
    dyq, sdy = orc.act_quant_cols(dy)
    xq, sx = orc.act_quant_cols(case.x)
    n = 0
    while n < N and (n == 0 or time.perf_counter() - t0 < seconds):
        orc.gemm_wgrad(dyq, sdy, xq, sx, rows=np.array([n], dtype=np.int64))
        n += 1
    dt = time.perf_counter() - t0
    return {"value": 2.0 * n * M * K / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "host_cores_available": cpu_cores(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"act_quant_cols of dY [{M},{N}] and X [{M},{K}], then {n} of {N} rows of dW; TFLOP/s over "
                      f"the sampled GEMM work (the quantisation time included)"}


def cpu_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_baseline(workload: str, seconds: float) -> dict:
    """The oracle as it stands, single-threaded C, on a bounded sample."""
    from fp8_block_scaled_18_b300 import synth
    from oracle import Oracle
    orc = Oracle()
    if workload.endswith("_wgrad"):
        return wgrad_oracle_sample(orc, workload, seconds)
    if workload == "moe_router":
        case = synth.moe()
        t0 = time.perf_counter()
        n = 0
        while time.perf_counter() - t0 < seconds and n < case.x_tokens.shape[0]:
            ids, w = orc.moe_gate(case.x_tokens[n:n + 16], case.gate_w, case.gate_bias)
            orc.moe_route(ids, w, case.n_experts)
            n += 16
        dt = time.perf_counter() - t0
        flops = 2.0 * n * case.n_experts * case.k
        sample = f"{n} of {case.x_tokens.shape[0]} tokens: router (gate GEMM, sigmoid, top-k) + routing tables"
        return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "host_cores_available": cpu_cores(),
                "kind": "oracle", "sample": sample, "seconds": round(dt, 2)}
    if workload == "moe_layer":
        case = synth.moe()
        counts = np.diff(case.offsets)
        experts = np.nonzero(counts)[0]
        t0 = time.perf_counter()
        flops, n = 0.0, 0
        while time.perf_counter() - t0 < seconds and n < len(experts):
            g = int(experts[n])
            wts = _expert_weights_q(orc, case, g, (0, 1, 2))
            r0, r1 = int(case.offsets[g]), int(case.offsets[g + 1])
            flops += oracle_layer_rows(orc, case, wts, np.arange(r0, min(r1, r0 + 32)))
            n += 1
        dt = time.perf_counter() - t0
        sample = (f"{n} experts x <=32 rows: weight_quant of the expert's w1, w3 and w2, router, act_quant, gemm x2, "
                  f"silu(a) * b, act_quant(h), gemm (w2), gated combine; TFLOP/s over the sampled GEMM work")
    elif workload in ("moe", "moe_swiglu") or workload.startswith("moe_e"):
        swiglu = workload == "moe_swiglu"
        case = moe_small_case(int(workload[len("moe_e"):])) if workload.startswith("moe_e") else synth.moe()
        counts = np.diff(case.offsets)
        x_rows = case.x_rows
        experts = np.nonzero(counts)[0]
        t0 = time.perf_counter()
        flops, n = 0.0, 0
        while time.perf_counter() - t0 < seconds and n < len(experts):
            flops += oracle_moe_step(orc, case, [experts[n]], x_rows, 32, swiglu=swiglu)
            n += 1
        dt = time.perf_counter() - t0
        sample = (f"{n} experts x <=32 rows: weight_quant of the expert's "
                  f"{'w1 and w3' if swiglu else 'weight'}, act_quant, gemm{' x2, silu(a) * b' if swiglu else ''}")
    else:
        case = make_case(workload)
        pow2 = workload.endswith("_pow2")
        M = case.x.shape[0]
        # untimed, as the GPU arm quantises W before timing
        wq, sw = (orc.weight_quant_pow2 if pow2 else orc.weight_quant)(case.w)
        rows = oracle_rows_for(orc, case, seconds, wq, sw, pow2)
        sel = np.linspace(0, M - 1, rows).astype(np.int64)
        t0 = time.perf_counter()
        flops = oracle_sample_step(orc, case, sel, wq, sw, pow2)
        dt = time.perf_counter() - t0
        sample = (f"{rows} of {M} rows: act_quant{'_pow2' if pow2 else ''}(rows) + gemm(rows)"
                  + (" + weight_dequant(W)" if case.name == "large_square" else "")
                  + ", W quantised before timing; TFLOP/s over the sampled GEMM work")
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": 1, "host_cores_available": cpu_cores(),
            "kind": "oracle", "sample": sample, "seconds": round(dt, 2)}


def run_reference(args, rank, local, world):
    """The base contract's reference arm for this build: the CPU oracle, timed
    as it stands on the host cores, rank 0 only."""
    if rank != 0:
        return
    from fp8_block_scaled_18_b300 import synth
    from oracle import Oracle
    orc = Oracle()
    K, W = args.steps, max(3, args.warmup)
    budget = 150.0  # seconds for the whole run
    if args.workload.endswith("_wgrad"):
        case, dy = wgrad_case(args.workload)
        M, N, Kd = case.shape
        dyq, sdy = orc.act_quant_cols(dy)   # set-up, untimed
        xq, sx = orc.act_quant_cols(case.x)
        t0 = time.perf_counter()
        orc.gemm_wgrad(dyq, sdy, xq, sx, rows=np.array([0], dtype=np.int64))
        per_row = max(time.perf_counter() - t0, 1e-4)
        rows = int(max(1, min(N, budget / (K + W) / per_row)))

        def step(i):
            # `rows` rows of dW (rotating), and the column quantisation of one
            # 128-token block of X
            b = i % ((M + 127) // 128)
            orc.act_quant_cols(case.x[128 * b:128 * (b + 1)])
            sel = (np.arange(rows) + i * rows) % N
            orc.gemm_wgrad(dyq, sdy, xq, sx, rows=sel.astype(np.int64))
            return 2.0 * rows * M * Kd
        sample = (f"{rows} of {N} rows of dW per step (rotating) and the column quantisation of one 128-token block "
                  f"of X; dY and X quantised before timing")
        cfg = {"workload": args.workload}
    elif args.workload == "moe_router":
        case = synth.moe()
        ntok = case.x_tokens.shape[0]
        t0 = time.perf_counter()
        orc.moe_gate(case.x_tokens[:8], case.gate_w, case.gate_bias)
        per_tok = max((time.perf_counter() - t0) / 8, 1e-5)
        rows = int(max(1, min(ntok, budget / (K + W) / per_tok)))

        def step(i):
            sel = (np.arange(rows) + i * rows) % ntok
            ids, w = orc.moe_gate(case.x_tokens[sel], case.gate_w, case.gate_bias)
            orc.moe_route(ids, w, case.n_experts)
            return 2.0 * rows * case.n_experts * case.k
        sample = f"{rows} of {ntok} tokens per step: router (gate GEMM, sigmoid, top-k) + routing tables"
        cfg = {"workload": "moe_router"}
    elif args.workload == "moe_layer":
        case = synth.moe()
        counts = np.diff(case.offsets)
        g = int(np.argmax(counts))  # the busiest expert
        r0, r1 = int(case.offsets[g]), int(case.offsets[g + 1])
        wts = _expert_weights_q(orc, case, g, (0, 1, 2))  # set-up, untimed
        import torch
        wg = synth.expert_weight(case, g, "cpu").view(torch.int16).numpy().view(np.uint16)
        nblk = (case.n + 127) // 128

        def layer_step(i, rows):
            # one 128-row block of the expert's w1 quantised (rotating), then
            # `rows` of its rows through the layer
            b = i % nblk
            orc.weight_quant(wg[128 * b:128 * (b + 1)])
            rs = r0 + (np.arange(rows) + i * rows) % (r1 - r0)
            return oracle_layer_rows(orc, case, wts, rs)

        t0 = time.perf_counter()
        layer_step(0, 1)
        t1 = time.perf_counter() - t0
        t0 = time.perf_counter()
        layer_step(0, 5)
        t5 = time.perf_counter() - t0
        per_row = max((t5 - t1) / 4, 1e-4)
        fixed = max(t1 - per_row, 0.0)
        rows = int(max(1, min(r1 - r0, (budget / (K + W) - fixed) / per_row)))
        step = lambda i: layer_step(i, rows)  # noqa: E731
        sample = (f"expert {g} ({r1 - r0} rows): per step one 128-row block of its w1 quantised, "
                  f"{rows} of its rows through the router, act_quant, w1/w3 gemm, silu * b, act_quant(h), w2 gemm, "
                  f"combine")
        cfg = {"workload": "moe_layer"}
    elif args.workload in ("moe", "moe_swiglu") or args.workload.startswith("moe_e"):
        import torch
        case = moe_small_case(int(args.workload[len("moe_e"):])) if args.workload.startswith("moe_e") else synth.moe()
        counts = np.diff(case.offsets)
        x_rows = case.x_rows
        g = int(np.argmax(counts))  # the busiest expert
        r0, r1 = int(case.offsets[g]), int(case.offsets[g + 1])
        swiglu = args.workload == "moe_swiglu"
        wg = synth.expert_weight(case, g, "cpu").view(torch.int16).numpy().view(np.uint16)
        # set-up, untimed: the expert's quantised weight(s)
        wts = _expert_weights_q(orc, case, g, (0, 1) if swiglu else (0,))
        nblk = (case.n + 127) // 128

        def moe_step(i, rows):
            # one 128-row block of the expert's weight quantised (rotating),
            # act_quant + gemm of `rows` of the expert's token rows (with
            # SwiGLU: the w1 and w3 GEMMs and silu(a) * b)
            b = i % nblk
            orc.weight_quant(wg[128 * b:128 * (b + 1)])
            rs = r0 + (np.arange(rows) + i * rows) % (r1 - r0)
            xq, sx = orc.act_quant(x_rows[rs])
            outs = [orc.gemm(xq, sx, wq, sw)[0] for wq, sw in wts]
            if swiglu:
                orc.swiglu(outs[0], outs[1])
            return 2.0 * rows * case.n * case.k * len(wts)

        t0 = time.perf_counter()
        moe_step(0, 1)
        t1 = time.perf_counter() - t0
        t0 = time.perf_counter()
        moe_step(0, 5)
        t5 = time.perf_counter() - t0
        per_row = max((t5 - t1) / 4, 1e-4)
        fixed = max(t1 - per_row, 0.0)
        rows = int(max(1, min(r1 - r0, (budget / (K + W) - fixed) / per_row)))
        step = lambda i: moe_step(i, rows)  # noqa: E731
        sample = (f"expert {g} ({r1 - r0} rows): per step one 128-row block of its weight quantised, "
                  f"act_quant + gemm of {rows} of its rows" + (" against w1 and w3, silu(a) * b" if swiglu else ""))
        cfg = {"workload": "moe_swiglu" if swiglu else "moe_grouped"}
    else:
        case = make_case(args.workload)
        pow2 = args.workload.endswith("_pow2")
        M, N, Kd = case.x.shape[0], case.w.shape[0], case.x.shape[1]
        nblk = (N + 127) // 128
        # set-up, untimed: the quantised weight the sampled GEMM rows use
        wq_all, sw_all = (orc.weight_quant_pow2 if pow2 else orc.weight_quant)(case.w)

        dequant = case.name == "large_square"

        def step(i, rows):
            # act_quant + gemm of `rows` activation rows against the whole
            # quantised W; for the large square also weight_dequant of one
            # 128-row block of W (rotating)
            if dequant:
                b = i % nblk
                orc.weight_dequant(wq_all[128 * b:128 * (b + 1)], sw_all[b:b + 1])
            rs = (np.arange(rows) + i * rows) % M
            xq, sx = (orc.act_quant_pow2 if pow2 else orc.act_quant)(case.x[rs])
            orc.gemm(xq, sx, wq_all, sw_all)
            return 2.0 * rows * N * Kd

        # size the step so that K + W steps take about `budget` seconds
        t0 = time.perf_counter()
        step(0, 1)
        t1 = time.perf_counter() - t0
        t0 = time.perf_counter()
        step(0, 5)
        t5 = time.perf_counter() - t0
        per_row = max((t5 - t1) / 4, 1e-4)
        fixed = max(t1 - per_row, 0.0)
        rows = int(max(1, min(M, (budget / (K + W) - fixed) / per_row)))
        step_fn = step
        step = lambda i: step_fn(i, rows)  # noqa: E731
        sample = (f"{rows} of {M} rows per step: act_quant{'_pow2' if pow2 else ''}(rows), gemm(rows) against "
                  f"the whole quantised W"
                  + (", weight_dequant of one 128-row block of W (rotating)" if dequant else ""))
        M_, N_, K_ = case.shape
        cfg = {"workload": case.name + ("_pow2" if pow2 else ""), "M": M_, "N": N_, "K": K_}
    for i in range(W):
        step(i)
    t0 = time.perf_counter()
    flops = 0.0
    for i in range(K):
        flops += step(i)
    dt = time.perf_counter() - t0
    value = flops / dt / 1e12
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": K, "warmup": W,
            "ms_per_step": dt / K * 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "fp64 oracle (fp32 quantisation)", "data": "synthetic", "impl": "reference",
            "config": {**cfg, "parallelism": "cpu oracle, rank 0"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle", "cores": 1,
                             "host_cores_available": cpu_cores(), "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    args = parse_args(argv)
    rank, local, world = dist_env()
    if world != args.gpus and world != 1:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)
    if args.impl == "reference":
        run_reference(args, rank, local, world)
    else:
        run_ours(args, rank, local, world)
    if world > 1:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
