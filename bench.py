#!/usr/bin/env python3
"""Benchmark of the video-DiT attention hot path on GB300 (one JSON line on rank 0).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Workloads (synthetic, seeded; the token grids of the Wan / LTX runs the pages describe):
  wan720  (default) Wan 720p 81-frame self-attention: B1 H40 D128, 21x45x80 = 75,600 tokens
          padded to 75,648, 3-D split-halves RoPE inside the attention launch, pad keys masked.
          The largest single-GPU workload (117 TFLOP of valid work per call).
  wan480  Wan 480x832x9 self-attention: 3x30x52 = 4680 tokens padded to 4736, same layout.
  cross   short-KV cross-attention: B2 H40 D128, 4680 (4736) queries x 512 text slots,
          per-batch valid lengths uniform on [1, 512].
  sharded 1024 queries over 37,800 keys in 4 shards (partials + LSE merge), B1 H32 D128.
  tiny    B1 H2 D64, 300 tokens padded to 384 (correctness-sized).

One step = one pass of the hot path over one batch held in HBM (padded layout, as the
sequence stays padded between blocks): the attention launch(es) of the workload (for
`sharded` the four partial launches and the merge). `value` is the algorithmic TFLOP/s on
valid tokens (4 * B * H * Lq * Lkv * D per attention) over all ranks. Three distinct input
sets rotate between steps, so every step reads inputs that are not L2-resident. `e2e` is the
same metric through the C-ABI with host buffers: every step copies the unpadded q/k/v from
pinned host memory into the padded layout (straight into the padded buffers when B = 1, else
through dit_pad_tokens), runs the attention, takes O and LSE back out (dit_unpad_tokens when
B > 1) and copies them to pinned host memory; consecutive steps overlap their copies with the
compute of their neighbours (two buffer sets, three streams). RoPE runs inside the attention launch: by default
(`--rope ws`) every q/k row is rotated once into a preallocated fp16 workspace before a grid
barrier, with `--rope fused` each loaded tile is rotated in shared memory instead.
`--impl reference` times the fp64 CPU oracle instead,
on the host cores, on a bounded sample of the same workload.

Peaks: the attention kernel's fraction is taken against the measured bf16 GEMM peak of
MEASURED_PEAKS.json, the sustained figure when the timed region runs longer than a second
of back-to-back launches (720p: 20 launches of ~78 ms), else the burst figure; the line also
carries the fraction of the nominal 2.25 PFLOP/s dense bf16 rate. All fractions come from
CUDA-event kernel time; `roofline.ncu_kernel_ms` repeats the committed ncu duration of the
same kernel sources where one exists. With the default workload the line also holds `also`,
timed kernel-only records of the other D = 128 workloads (Wan 480, short-KV cross,
sharded keys), each with its own clock record.

Multi-GPU: `python -m torch.distributed.run --nproc-per-node N bench.py --gpus N`; each rank
runs an independent replica (the problems are independent; no data-path collective), the
barrier and the max over ranks bracket the timed region, and units add up (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attention TFLOP/s (valid tokens) and % of GB300 BF16 peak; ms per call"
FALLBACK_PEAKS = {"bf16_tflops": 1900.0, "hbm_gbs": 6800.0}


# ----------------------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    except Exception:
        return dict(FALLBACK_PEAKS, bf16_tflops_sustained=1700.0, source="fallback")


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_over_ranks(elapsed_s: float, units: float, world: int):
    """(max elapsed over ranks, sum of units over ranks); identity for one rank."""
    if world <= 1:
        return elapsed_s, units
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([elapsed_s], dtype=torch.float64, device=dev)
    u = torch.tensor([units], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.all_reduce(u, op=dist.ReduceOp.SUM)
    return float(t.item()), float(u.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class ClockSampler:
    """nvidia-smi samples (100 ms) of SM clock, power and throttle reasons, host-timestamped."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]),
                                     parts[3:7]))
            except ValueError:
                pass

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1, busy_t0, busy_t1=None):
        """Median SM clock and the throttle reasons seen over the timed region [t0, t1]. When that
        region holds fewer than three samples (shorter than three sampling intervals), the
        summary covers the whole GPU-busy window [busy_t0, busy_t1] instead (warm-up, timed
        steps and the e2e leg), and `window` says so."""
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        where = "timed region"
        if len(win) < 3:
            hi = t1 if busy_t1 is None else busy_t1
            win = [s for s in self.samples if busy_t0 <= s[0] <= hi]
            where = ("GPU-busy window: warm-up, timed steps and e2e leg (the timed region is shorter "
                     "than three 100 ms sampling intervals)")
        if len(win) < 3:
            # still too short: the three samples nearest the timed region (at most 0.5 s away)
            mid = 0.5 * (t0 + t1)
            near = sorted((s for s in self.samples if abs(s[0] - mid) <= 0.5 + 0.5 * (t1 - t0)),
                          key=lambda s: abs(s[0] - mid))[:3]
            if len(near) > len(win):
                win = near
                where = "the 3 samples nearest the timed region (it is shorter than the sampling interval)"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": "none"}
        reasons = sorted({self.NAMES[i] for s in win for i, v in enumerate(s[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(s[1] for s in win), "sm_max_mhz": max(s[2] for s in win),
                "reasons": reasons, "samples": len(win), "window": where}


def gpu_id_for_smi(dev_index: int) -> str:
    import torch
    try:
        p = torch.cuda.get_device_properties(dev_index)
        return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
    except Exception:
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        return vis.split(",")[dev_index] if vis else str(dev_index)


# The sources of the kernel each workload's summary covers: a committed ncu summary applies
# while their hash matches (the cross workload runs cross_attn_kernel, the others
# attn_sp_kernel).
KERNEL_SOURCES = {"cross": ("cross_attn.cu", "ptx.cuh"), None: ("attn_fwd.cu", "attn_sp.cuh", "ptx.cuh")}


def profiled(name, variant=""):
    """Figures of the committed ncu summary of this workload (and kernel variant: "qknorm",
    "fixed_m"): {"traffic": DRAM bytes per launch of the dominant kernel (per step, the attention
    launch and the merge, for the sharded workload), "ncu_kernel_ms": its ncu duration per launch (per
    step for sharded) or None}, or None if there is no summary or the kernel sources changed
    since it was taken."""
    import hashlib
    base = {"wan480": "attn_sp_wan480x832x9", "wan720": "attn_sp_wan720p81f", "cross": "attn_sp_cross_shortkv",
            "sharded": "attn_sp_sharded_keys"}.get(name)
    if base is None:
        return None
    path = os.path.join(ROOT, "profiles", base + (f"_{variant}" if variant else "") + ".md")
    if not os.path.exists(path):
        return None
    srcs = [os.path.join(ROOT, "video_dit_attention_gb300", "csrc", f)
            for f in KERNEL_SOURCES.get(name, KERNEL_SOURCES[None])]
    h = hashlib.sha256(b"".join(open(f, "rb").read() for f in srcs)).hexdigest()[:16]
    sha = traffic = ncu_ms = None
    for line in open(path):
        if line.startswith("kernel sources sha256"):
            sha = line.split(":")[-1].strip()
        elif line.startswith(("traffic_bytes_per_launch:", "traffic_bytes_per_step:")):
            traffic = int(line.split(":")[1])   # per step for sharded (attention + merge), like achieved
        elif line.startswith(("ncu_ms_per_launch:", "ncu_ms_per_step:")):
            ncu_ms = float(line.split(":")[1])
    if sha != h:
        return None
    return {"traffic": traffic, "ncu_kernel_ms": ncu_ms}


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 0) for i in threadpool_info() if i.get("user_api") == "blas"]
        if n:
            return int(max(n))
    except Exception:
        pass
    return os.cpu_count() or 1


# ----------------------------------------------------------------------------- workloads
def workload_spec(name):
    from video_dit_attention_gb300 import inputs as I
    if name in ("wan480", "wan720", "tiny"):
        case = {"wan480": I.wan480_case, "wan720": I.wan720_case, "tiny": I.tiny_case}[name]()
        return case
    if name == "cross":
        return I.cross_case()
    if name == "sharded":
        return I.sharded_case()
    raise SystemExit(f"unknown workload {name}")


def config_dict(name, spec, rope_mode="ws"):
    if name == "sharded":
        return {"workload": "sharded-key attention + LSE merge", "B": spec.B, "H": spec.H, "D": spec.D,
                "queries": spec.Sq, "keys": sum(spec.shard_valid), "shards": list(spec.shard_valid),
                "rope": "1-D split halves, theta 10000, global key positions",
                "rope_path": "one dit_attn_fwd_sharded call: every shard's k rotated once into an fp16 "
                             "workspace, all key chunks attended in one launch, partials merged",
                "l2": "3 rotating input sets of 0.69 GB each (> 129 MB L2)"}
    d = {"workload": {"wan480": "Wan 480x832x9 self-attention", "wan720": "Wan 720p 81-frame self-attention",
                      "tiny": "tiny self-attention", "cross": "short-KV cross-attention"}[name],
         "B": spec.B, "H": spec.H, "D": spec.D, "q_valid": spec.q_valid, "q_padded": spec.Sq,
         "kv_valid": spec.kv_valid, "kv_padded": spec.Skv}
    if spec.rope == "3d":
        d["rope"] = f"3-D split halves, grid {'x'.join(map(str, spec.grid))}, 44/42/42, theta 10000"
    elif spec.rope == "1d":
        d["rope"] = "1-D split halves, theta 10000"
    else:
        d["rope"] = "none"
    if spec.rope in ("1d", "3d"):
        d["rope_path"] = _ROPE_PATH[rope_mode]
    d["l2"] = "3 rotating input sets, each larger than the 129 MB L2" if name != "tiny" else "tiny: L2-resident"
    return d


def spec_has_no_rope(spec):
    return getattr(spec, "rope", "1d") is None


def dominant_kernel(name, rope_mode):
    if name == "cross":
        return "cross_attn_kernel (K/V of a head resident in shared memory)"
    if name == "sharded":
        return "attn_sp_kernel (sharded keys: all key chunks in one launch) + lse_merge_fixed_kernel"
    if rope_mode == "fused":
        return "attn_fwd_kernel (RoPE per loaded tile)"
    return "attn_sp_kernel (workspace RoPE)"


_ROPE_PATH = {
    "ws": "in the attention launch: q/k rotated once into an fp16 workspace, grid barrier, attention",
    "fused": "in the attention launch: q/k tiles rotated in shared memory as they are loaded",
}


def step_flops(name, spec):
    if name == "sharded":
        return sum(4.0 * spec.B * spec.H * spec.q_valid * n * spec.D for n in spec.shard_valid)
    if name == "cross":
        return sum(4.0 * spec.H * spec.q_valid * L * spec.D for L in spec.kv_valid)
    return 4.0 * spec.B * spec.H * spec.q_valid * int(spec.kv_valid) * spec.D


class GpuWorkload:
    """Device buffers and the launch sequence of one step."""

    def __init__(self, name, spec, seed_offset=0, rope_mode="ws", qknorm=False, fixed_m=False, fp8=False):
        import torch

        from video_dit_attention_gb300 import dit_attn as lib
        from video_dit_attention_gb300 import inputs as I
        self.torch, self.lib, self.name, self.spec = torch, lib, name, spec
        self.rope_mode = rope_mode
        self.workspace = None
        self.norms = None
        self.fixed_m = fixed_m
        self.fp8 = fp8
        ws_bytes = (lib.dit_attn_fp8_workspace_bytes if fp8 else
                    lib.dit_attn_fixed_m_workspace_bytes if fixed_m else lib.dit_attn_workspace_bytes)
        dev = torch.device("cuda")
        if qknorm:
            self.norms = tuple(torch.from_numpy(I.make_norm_weights(spec.D, seed=spec.seed + 900 + i)).to(dev)
                               for i in range(2))
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).to(dev)
        self.sets = []
        if name == "sharded":
            spec.seed += seed_offset
            q, shards = I.make_sharded(spec)
            base = (bf(q), [(bf(k), bf(v)) for k, v in shards])
            self.host = (q, shards)
            cq, sq = lib.dit_rope_table_1d(spec.Sq, spec.q_valid, spec.D, spec.theta, 0)
            self.tq = (torch.from_numpy(cq).to(dev), torch.from_numpy(sq).to(dev))
            self.tk = []
            for off, n, npad in zip(spec.offsets, spec.shard_valid, spec.shard_pad):
                ck, sk = lib.dit_rope_table_1d(npad, n, spec.D, spec.theta, off)
                self.tk.append((torch.from_numpy(ck).to(dev), torch.from_numpy(sk).to(dev)))
            for r in range(3):
                qq = torch.roll(base[0], r, dims=2).contiguous()
                kv = [(torch.roll(k, r, dims=2).contiguous(), torch.roll(v, r, dims=2).contiguous())
                      for k, v in base[1]]
                entries = [(k, v, n, ck, sk) for (k, v), n, (ck, sk) in zip(kv, spec.shard_valid, self.tk)]
                out = torch.empty_like(qq)
                lse = torch.empty(tuple(qq.shape[:3]), dtype=torch.float32, device=dev)
                self.sets.append((qq, entries, out, lse))
            # one dit_attn_fwd_sharded call: the attention launch over all key chunks, the merge
            self.launches_per_step = 2
            nb = lib.dit_attn_sharded_workspace_bytes(spec.B, spec.Sq, spec.H, spec.D, spec.shard_pad,
                                                      spec.shard_valid)
            self.workspace = torch.empty(nb, dtype=torch.uint8, device=dev)
        else:
            spec.seed += seed_offset
            q, k, v = I.make_qkv(spec)
            self.host = (q, k, v)
            base = (bf(q), bf(k), bf(v))
            if spec.rope == "3d":
                cq, sq = lib.dit_rope_table_3d(spec.Sq, spec.grid, spec.D, spec.axis_dims, spec.theta)
                ck, sk = lib.dit_rope_table_3d(spec.Skv, spec.grid, spec.D, spec.axis_dims, spec.theta)
                self.tables = tuple(torch.from_numpy(t).to(dev) for t in (cq, sq, ck, sk))
            elif spec.rope == "1d":
                cq, sq = lib.dit_rope_table_1d(spec.Sq, spec.q_valid, spec.D, spec.theta, 0)
                ck, sk = lib.dit_rope_table_1d(spec.Skv, int(spec.kv_valid), spec.D, spec.theta, 0)
                self.tables = tuple(torch.from_numpy(t).to(dev) for t in (cq, sq, ck, sk))
            else:
                self.tables = (None, None, None, None)
            if name == "cross":
                self.kv_dev = torch.tensor(spec.kv_valid, dtype=torch.int32, device=dev)
            nsets = 1 if name == "tiny" else 3
            for r in range(nsets):
                qq, kk, vv = (torch.roll(t, r, dims=2).contiguous() for t in base)
                out = torch.empty_like(qq)
                lse = torch.empty(tuple(qq.shape[:3]), dtype=torch.float32, device=dev)
                self.sets.append((qq, kk, vv, out, lse))
            self.launches_per_step = 3 if fp8 else 1
            if fp8 or (rope_mode == "ws" and self.tables[0] is not None):
                nb = ws_bytes(spec.B, spec.Sq, spec.Skv, spec.H, spec.D)
                self.workspace = torch.empty(nb, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize()

    def attn(self, q, k, v, q_valid, kv_valid, tables, out, lse):
        """One self-attention launch: the two-phase RoPE path (rotation into the preallocated
        workspace) when a workspace is set, else the path with RoPE fused per tile."""
        if self.fp8:
            self.lib.dit_attn_fwd_fp8(q, k, v, q_valid, kv_valid, *tables, workspace=self.workspace,
                                      out=out, lse=lse)
        elif self.workspace is not None and self.fixed_m:
            self.lib.dit_attn_fwd_ws_fixed_m(q, k, v, q_valid, kv_valid, *tables, workspace=self.workspace,
                                             out=out, lse=lse)
        elif self.workspace is not None and self.norms is not None:
            self.lib.dit_attn_fwd_ws_qknorm(q, k, v, q_valid, kv_valid, *self.norms, *tables,
                                            workspace=self.workspace, out=out, lse=lse)
        elif self.workspace is not None:
            self.lib.dit_attn_fwd_ws(q, k, v, q_valid, kv_valid, *tables, workspace=self.workspace,
                                     out=out, lse=lse)
        else:
            self.lib.dit_attn_fwd(q, k, v, q_valid, kv_valid, *tables, out=out, lse=lse)

    def step(self, i, ev=None):
        """Launches one step on the current stream; ev = (start, end) events around the
        dominant kernel (the attention launch; for `sharded`, the one call: the attention launch
        over all key chunks and the merge of their partials)."""
        lib, spec = self.lib, self.spec
        s = self.sets[i % len(self.sets)]
        if ev is not None:
            ev[0].record()
        if self.name == "sharded":
            qq, entries, out, lse = s
            lib.dit_attn_fwd_sharded(qq, entries, spec.q_valid, *self.tq, workspace=self.workspace, out=out, lse=lse)
            if ev is not None:
                ev[1].record()
            return
        qq, kk, vv, out, lse = s
        if self.name == "cross":
            lib.dit_cross_attn_shortkv(qq, kk, vv, spec.q_valid, self.kv_dev, out=out, lse=lse)
        else:
            self.attn(qq, kk, vv, spec.q_valid, int(spec.kv_valid), self.tables, out, lse)
        if ev is not None:
            ev[1].record()

    def dominant_bytes(self):
        """Algorithmic HBM bytes of the dominant kernel per step (valid rows of q, k, v read;
        O and LSE written)."""
        sp = self.spec
        if self.name == "sharded":
            # q and k, v read once, O and LSE written once (the partials stay on the device)
            kv = sum(2 * sp.B * n * sp.H * sp.D * 2 for n in sp.shard_valid)
            return kv + sp.B * sp.q_valid * sp.H * (sp.D * 2 * 2 + 4)
        Lkv = sum(sp.kv_valid) if self.name == "cross" else sp.B * int(sp.kv_valid)
        return (sp.B * sp.q_valid * sp.H * sp.D * 2 + 2 * Lkv * sp.H * sp.D * 2
                + sp.B * sp.q_valid * sp.H * (sp.D * 2 + 4))


class E2E:
    """Host-buffer path through the C-ABI: pinned host q/k/v (unpadded) -> H2D -> pad ->
    attention -> unpad -> D2H of O and LSE (self-attention and cross workloads).

    Steps are pipelined over two buffer sets: step i's upload runs on a copy stream while
    step i-1 computes, and its download on another copy stream while step i+1 computes;
    events order each set's reuse. Every step still moves its own inputs and outputs, inside
    the timed region. With B = 1 the valid rows are a contiguous prefix of the padded
    buffers, so the upload writes straight into them and the download reads straight from
    the padded outputs (no pad / unpad launches); with B > 1 dit_pad_tokens and
    dit_unpad_tokens gather the rows on the device."""

    NBUF = 2

    def __init__(self, wl):
        torch = wl.torch
        self.wl, self.torch = wl, torch
        sp = wl.spec
        q, k, v = wl.host
        Lq = sp.q_valid
        Lk = int(sp.kv_valid) if wl.name != "cross" else sp.Skv
        pin = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).pin_memory()
        self.hq, self.hk, self.hv = pin(q[:, :Lq]), pin(k[:, :Lk]), pin(v[:, :Lk])
        dev = torch.device("cuda")
        self.direct = sp.B == 1
        self.sets = []
        for _ in range(self.NBUF):
            st = {}
            st["qp"] = torch.empty((sp.B, sp.Sq, sp.H, sp.D), dtype=torch.bfloat16, device=dev)
            st["kp"] = torch.empty((sp.B, sp.Skv, sp.H, sp.D), dtype=torch.bfloat16, device=dev)
            st["vp"] = torch.empty_like(st["kp"])
            st["out"] = torch.empty_like(st["qp"])
            st["lse"] = torch.empty((sp.B, sp.Sq, sp.H), dtype=torch.float32, device=dev)
            if not self.direct:
                st["dq"] = torch.empty(self.hq.shape, dtype=torch.bfloat16, device=dev)
                st["dk"] = torch.empty(self.hk.shape, dtype=torch.bfloat16, device=dev)
                st["dv"] = torch.empty(self.hv.shape, dtype=torch.bfloat16, device=dev)
                st["o_u"] = torch.empty((sp.B, Lq, sp.H, sp.D), dtype=torch.bfloat16, device=dev)
                st["l_u"] = torch.empty((sp.B, Lq, sp.H), dtype=torch.float32, device=dev)
            st["ho"] = torch.empty((sp.B, Lq, sp.H, sp.D), dtype=torch.bfloat16).pin_memory()
            st["hl"] = torch.empty((sp.B, Lq, sp.H), dtype=torch.float32).pin_memory()
            st["ev_in"], st["ev_done"], st["ev_out"] = (torch.cuda.Event() for _ in range(3))
            self.sets.append(st)
        # One upload stream: three (one per tensor) measured the same (about 190 GB/s in all).
        self.s_h2d, self.s_d2h = torch.cuda.Stream(), torch.cuda.Stream()
        self.Lq, self.Lk = Lq, Lk
        self.h2d = sum(t.numel() * t.element_size() for t in (self.hq, self.hk, self.hv))
        self.d2h = self.sets[0]["ho"].numel() * 2 + self.sets[0]["hl"].numel() * 4
        self.launches_per_step = 1 if self.direct else 6
        self.last = None

    def step(self, i):
        torch = self.torch
        lib, wl, sp = self.wl.lib, self.wl, self.wl.spec
        st = self.sets[i % self.NBUF]
        cs = torch.cuda.current_stream()
        Lq, Lk = self.Lq, self.Lk
        if self.direct:
            dsts = (st["qp"][:, :Lq], st["kp"][:, :Lk], st["vp"][:, :Lk])
        else:
            dsts = (st["dq"], st["dk"], st["dv"])
        with torch.cuda.stream(self.s_h2d):
            self.s_h2d.wait_event(st["ev_done"])        # the set's previous compute has read it
            for dst, src in zip(dsts, (self.hq, self.hk, self.hv)):
                dst.copy_(src, non_blocking=True)
            st["ev_in"].record(self.s_h2d)
        cs.wait_event(st["ev_in"])
        cs.wait_event(st["ev_out"])                      # the set's previous download is done
        if not self.direct:
            lib.dit_pad_tokens(st["dq"], sp.Sq, out=st["qp"])
            lib.dit_pad_tokens(st["dk"], sp.Skv, out=st["kp"])
            lib.dit_pad_tokens(st["dv"], sp.Skv, out=st["vp"])
        if wl.name == "cross":
            lib.dit_cross_attn_shortkv(st["qp"], st["kp"], st["vp"], sp.q_valid, wl.kv_dev, out=st["out"],
                                       lse=st["lse"])
        else:
            wl.attn(st["qp"], st["kp"], st["vp"], sp.q_valid, int(sp.kv_valid), wl.tables, st["out"], st["lse"])
        if self.direct:
            o_src, l_src = st["out"][:, :Lq], st["lse"][:, :Lq]
        else:
            lib.dit_unpad_tokens(st["out"], Lq, out=st["o_u"])
            lib.dit_unpad_tokens(st["lse"], Lq, out=st["l_u"])
            o_src, l_src = st["o_u"], st["l_u"]
        st["ev_done"].record(cs)
        with torch.cuda.stream(self.s_d2h):
            self.s_d2h.wait_event(st["ev_done"])
            st["ho"].copy_(o_src, non_blocking=True)
            st["hl"].copy_(l_src, non_blocking=True)
            st["ev_out"].record(self.s_d2h)
        self.last = st

    def finish(self):
        """Makes the current stream wait for the last step's download."""
        if self.last is not None:
            self.torch.cuda.current_stream().wait_event(self.last["ev_out"])


# ----------------------------------------------------------------------------- HBM-bound kernels
def measure_hbm_kernels(peaks):
    """The standalone RoPE and the LSE merge, each timed with CUDA events over back-to-back
    calls whose inputs rotate over sets larger than L2, and reported as algorithmic GB/s
    against the measured HBM copy bandwidth. Not part of the timed attention step."""
    import torch

    from video_dit_attention_gb300 import dit_attn as lib
    from video_dit_attention_gb300 import inputs as I
    dev = torch.device("cuda")
    gen = torch.Generator(device="cpu").manual_seed(5)
    out = {}

    def timed(fn, n, warm=5):
        for i in range(warm):
            fn(i)
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(n):
            fn(i)
        b.record()
        torch.cuda.synchronize()
        return a.elapsed_time(b) / 1e3 / n

    # RoPE on the Wan 480 q and k (stacked as B = 2 rows of the same positions), out of place.
    c = I.wan480_case()
    cs, sn = lib.dit_rope_table_3d(c.Sq, c.grid, c.D, c.axis_dims, c.theta)
    cs, sn = torch.from_numpy(cs).to(dev), torch.from_numpy(sn).to(dev)
    xs = [torch.randn((2, c.Sq, c.H, c.D), generator=gen).to(torch.bfloat16).to(dev) for _ in range(2)]
    ys = [torch.empty_like(x) for x in xs]
    t = timed(lambda i: lib.dit_rope_split_halves(xs[i % 2], cs, sn, out=ys[i % 2]), 40)
    nb = 2 * xs[0].numel() * 2
    out["rope_split_halves"] = {
        "workload": "Wan 480x832x9 q and k, [2, 4736, 40, 128] bf16, 3-D tables, out of place",
        "bytes_per_call": nb, "us": t * 1e6, "GB_s": nb / t / 1e9, "frac_of_hbm": nb / t / 1e9 / peaks["hbm_gbs"],
        "l2": "2 input sets of 97 MB, 194 MB moved per call (> 129 MB L2)"}
    w = torch.from_numpy(I.make_norm_weights(c.D, seed=7)).to(dev)
    t = timed(lambda i: lib.dit_qk_rmsnorm_rope(xs[i % 2], w, cs, sn, out=ys[i % 2]), 40)
    out["qk_rmsnorm_rope"] = {
        "workload": "Wan 480x832x9 q and k, [2, 4736, 40, 128] bf16, per-head RMSNorm then 3-D RoPE",
        "bytes_per_call": nb, "us": t * 1e6, "GB_s": nb / t / 1e9, "frac_of_hbm": nb / t / 1e9 / peaks["hbm_gbs"],
        "l2": "2 input sets of 97 MB, 194 MB moved per call (> 129 MB L2)"}
    del xs, ys
    # LSE merge of the sharded workload's 4 partials.
    sc = I.sharded_case()
    n = len(sc.shard_valid)
    sets = []
    for _ in range(4):
        po = torch.randn((n, sc.B, sc.Sq, sc.H, sc.D), generator=gen).to(torch.bfloat16).to(dev)
        pl = (torch.randn((n, sc.B, sc.Sq, sc.H), generator=gen) * 3).to(dev)
        sets.append((po, pl, torch.empty((sc.B, sc.Sq, sc.H, sc.D), dtype=torch.bfloat16, device=dev),
                     torch.empty((sc.B, sc.Sq, sc.H), dtype=torch.float32, device=dev)))
    t = timed(lambda i: lib.dit_attn_lse_merge(sets[i % 4][0], sets[i % 4][1], out=sets[i % 4][2],
                                               lse=sets[i % 4][3]), 200)
    rows = sc.B * sc.Sq * sc.H
    nb = rows * (n * (sc.D * 2 + 4) + sc.D * 2 + 4)
    out["lse_merge"] = {
        "workload": "4 partials of [1, 1024, 32, 128] bf16 + LSE -> merged O, LSE",
        "bytes_per_call": nb, "us": t * 1e6, "GB_s": nb / t / 1e9, "frac_of_hbm": nb / t / 1e9 / peaks["hbm_gbs"],
        "l2": "4 input sets of 43 MB rotate (170 MB > 129 MB L2)"}
    torch.cuda.synchronize()
    return out


# ----------------------------------------------------------------------------- oracle arm
def oracle_sample(name, spec, host, n_rows, n_heads, seed=0):
    """Runs the fp64 oracle once on (n_rows query rows) x (n_heads heads) of the workload;
    returns (seconds, algorithmic FLOPs of the sample)."""
    from oracle.attention import attention, lse_merge
    from oracle.rope import pad_angles, rope_angles_1d, rope_angles_3d
    rng = np.random.Generator(np.random.PCG64(seed))
    heads = sorted(rng.choice(spec.H, size=min(n_heads, spec.H), replace=False).tolist())
    rows = sorted(rng.choice(spec.q_valid, size=min(n_rows, spec.q_valid), replace=False).tolist())
    t0 = time.perf_counter()
    if name == "sharded":
        q, shards = host
        aq = pad_angles(rope_angles_1d(np.arange(spec.q_valid), spec.D, spec.theta), spec.Sq)
        po, pl = [], []
        for (k, v), off, n in zip(shards, spec.offsets, spec.shard_valid):
            ak = pad_angles(rope_angles_1d(np.arange(n) + off, spec.D, spec.theta), k.shape[1])
            O, L = attention(q, k, v, spec.q_valid, n, spec.scale, aq, ak, rows=rows, heads=heads)
            po.append(O)
            pl.append(L)
        lse_merge(np.stack(po), np.stack(pl))
        flops = sum(4.0 * len(rows) * len(heads) * n * spec.D for n in spec.shard_valid) * spec.B
    else:
        q, k, v = host
        aq = ak = None
        if spec.rope == "3d":
            a = rope_angles_3d(*spec.grid, spec.D, spec.axis_dims, spec.theta)
            aq, ak = pad_angles(a, spec.Sq), pad_angles(a, spec.Skv)
        elif spec.rope == "1d":
            aq = pad_angles(rope_angles_1d(np.arange(spec.q_valid), spec.D, spec.theta), spec.Sq)
            ak = pad_angles(rope_angles_1d(np.arange(int(spec.kv_valid)), spec.D, spec.theta), spec.Skv)
        attention(q, k, v, spec.q_valid, spec.kv_valid, spec.scale, aq, ak, rows=rows, heads=heads)
        Ls = spec.kv_valid if name == "cross" else [int(spec.kv_valid)] * spec.B
        flops = sum(4.0 * len(rows) * len(heads) * L * spec.D for L in Ls)
    return time.perf_counter() - t0, flops


def host_inputs(name, spec):
    from video_dit_attention_gb300 import inputs as I
    if name == "sharded":
        return I.make_sharded(spec)
    return I.make_qkv(spec)


def cpu_baseline(name, spec, host, budget_s=12.0):
    """Times the oracle, as it stands, on a bounded sample (about budget_s of CPU work)."""
    n_rows, n_heads = 32, min(8, spec.H)
    dt, fl = oracle_sample(name, spec, host, n_rows, n_heads, seed=1)
    reps = max(1, int(budget_s / max(dt, 1e-3)))
    tot_t, tot_f = dt, fl
    for r in range(reps - 1):
        d, f = oracle_sample(name, spec, host, n_rows, n_heads, seed=2 + r)
        tot_t += d
        tot_f += f
    return {"value": tot_f / tot_t / 1e12, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{reps} oracle calls of {n_rows} random valid query rows x {n_heads} heads "
                      f"(all valid keys), {tot_t:.1f} s of fp64 numpy on the host cores"}


def run_reference(args, name, spec, rank, world):
    if rank != 0:
        return
    host = host_inputs(name, spec)
    # size one step so that warm-up + timed steps end within about two minutes
    n_rows, n_heads = 16, min(4, spec.H)
    dt, _ = oracle_sample(name, spec, host, n_rows, n_heads, seed=0)
    budget = 120.0 / max(1, args.steps + args.warmup)
    while dt > budget and (n_rows > 1 or n_heads > 1):
        if n_rows > 1:
            n_rows //= 2
        else:
            n_heads = max(1, n_heads // 2)
        dt, _ = oracle_sample(name, spec, host, n_rows, n_heads, seed=0)
    for w in range(args.warmup):
        oracle_sample(name, spec, host, n_rows, n_heads, seed=100 + w)
    tt, tf = 0.0, 0.0
    for s in range(args.steps):
        d, f = oracle_sample(name, spec, host, n_rows, n_heads, seed=1000 + s)
        tt += d
        tf += f
    value = tf / tt / 1e12
    sample = (f"each step: the fp64 oracle on {n_rows} random valid query rows x {n_heads} heads "
              f"with all valid keys (algorithmic FLOPs of that sample)")
    line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "impl": "reference", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": tt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": config_dict(name, spec),
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- main
NOMINAL_BF16_TFLOPS = 2250.0   # GB300 dense bf16 tensor rate (vendor figure, no sparsity)
SUSTAINED_AFTER_S = 1.0        # a timed region longer than this is judged against the sustained peak
DEFAULT_STEPS = {"wan720": 20, "sharded": 200}


def time_steps(wl, steps, warmup, world, stream):
    """Warm-up, then `steps` timed steps bracketed by a barrier and a device synchronize on
    both sides, with events around the dominant kernel of each step. Returns (elapsed
    seconds of the timed region on the device, mean dominant-kernel seconds per step,
    host time at the start and end of the timed region, host time before the warm-up)."""
    import torch
    busy_t0 = time.time()
    for i in range(warmup):
        wl.step(i)
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(stream)
    for i in range(steps):
        wl.step(i, evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t1 = time.time()
    elapsed = start.elapsed_time(end) / 1e3
    kern_s = sum(a.elapsed_time(b) for a, b in evs) / 1e3 / steps
    status = wl.lib.dit_device_status()
    if status != 0:
        raise SystemExit(f"device status word {status:#x}: a kernel gave up on a bounded wait")
    return elapsed, kern_s, t0, t1, busy_t0


def pick_peak(peaks, elapsed_s, fp8=False):
    """(peak TFLOP/s, description): sustained for a timed region longer than SUSTAINED_AFTER_S
    of back-to-back launches, burst otherwise; fp8 takes twice the bf16 figure (the nominal
    fp8 / bf16 ratio, 4.5 / 2.25)."""
    key = "bf16_tflops_sustained" if elapsed_s > SUSTAINED_AFTER_S else "bf16_tflops"
    kind = "sustained" if key == "bf16_tflops_sustained" else "burst"
    peak, src = peaks[key], f"{key} ({kind}) of {peaks['source']} peaks"
    if fp8:
        return 2.0 * peak, f"2 x {src} (nominal fp8 / bf16 ratio)"
    return peak, src + f" (timed region {elapsed_s:.2f} s: {kind})"


def also_records(peaks, sampler, names, world, stream):
    """Kernel-only records of other workloads in the same run: value, kernel time and the
    fraction of the measured peak, each with the clocks seen over its own window."""
    import torch
    out = {}
    for name in names:
        spec = workload_spec(name)
        wl = GpuWorkload(name, spec)
        steps = 100 if name == "sharded" else 200
        elapsed, kern_s, t0, t1, busy_t0 = time_steps(wl, steps, 5, world, stream)
        flops = step_flops(name, spec)
        peak, peak_src = pick_peak(peaks, elapsed)
        achieved = flops / kern_s / 1e12
        prof = profiled(name) or {}
        out[name] = {"workload": config_dict(name, spec)["workload"], "steps": steps, "warmup": 5,
                     "value": flops * steps / elapsed / 1e12, "unit": "TFLOP/s",
                     "ms_per_step": elapsed / steps * 1e3, "kernel": dominant_kernel(name, "ws"),
                     "kernel_ms": kern_s * 1e3, "achieved": achieved, "peak": peak, "peak_source": peak_src,
                     "frac": achieved / peak, "frac_of_nominal_bf16": achieved / NOMINAL_BF16_TFLOPS,
                     "traffic": prof.get("traffic"), "ncu_kernel_ms": prof.get("ncu_kernel_ms"),
                     "algorithmic_bytes": wl.dominant_bytes(),
                     "clocks": sampler.summary(t0, t1, busy_t0, time.time())}
        del wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 20 for wan720, 200 for sharded, else 1000)")
    ap.add_argument("--warmup", type=int, default=None, help="warm-up steps (default: 3 for wan720, else 20)")
    ap.add_argument("--workload", default="wan720", choices=["wan480", "wan720", "cross", "sharded", "tiny"])
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--rope", default="ws", choices=["ws", "fused"],
                    help="ws: rotate q/k once per call into a workspace (default); fused: rotate per tile")
    ap.add_argument("--qknorm", action="store_true",
                    help="per-head q/k RMSNorm fused before the rotation (workspace path, RoPE workloads)")
    ap.add_argument("--fixed-m", action="store_true",
                    help="fixed-m softmax (32-row blocks whose norm bound allows it skip the running "
                         "maximum; workspace path, RoPE workloads)")
    ap.add_argument("--fp8", action="store_true",
                    help="FP8 (e4m3) attention: q/k/v rotated and quantised into a workspace, e4m3 "
                         "tensor-core products (D = 128 self-attention workloads)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-hbm-kernels", action="store_true", help="skip the RoPE / merge GB/s figures")
    ap.add_argument("--no-also", action="store_true",
                    help="skip the kernel-only records of the other workloads (default workload only)")
    ap.add_argument("--heads", type=int, default=None,
                    help="profiling only: run the workload with this many heads (a smaller ncu capture "
                         "whose per-head figures scale to the full workload); marks the line reduced")
    args = ap.parse_args()
    name = args.workload
    if args.steps is None:
        args.steps = DEFAULT_STEPS.get(name, 1000)
    if args.warmup is None:
        args.warmup = 3 if name == "wan720" else 20
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world, local = dist_env()
    spec = workload_spec(name)
    if args.heads is not None:
        if not 1 <= args.heads <= spec.H:
            raise SystemExit(f"--heads must be in [1, {spec.H}]")
        spec.H = args.heads

    if args.impl == "reference":
        run_reference(args, name, spec, rank, world)
        return

    import torch
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    peaks = load_peaks()
    if args.qknorm and (args.rope != "ws" or spec_has_no_rope(spec)):
        raise SystemExit("--qknorm needs a RoPE workload on the workspace path")
    if args.fixed_m and (args.rope != "ws" or spec_has_no_rope(spec) or args.qknorm):
        raise SystemExit("--fixed-m needs a RoPE workload on the workspace path, without --qknorm")
    if args.fp8 and (name in ("cross", "sharded") or spec.D != 128 or args.qknorm or args.fixed_m or args.rope != "ws"):
        raise SystemExit("--fp8 needs a D = 128 self-attention workload, without --qknorm / --fixed-m / --rope fused")
    wl = GpuWorkload(name, spec, seed_offset=rank, rope_mode=args.rope, qknorm=args.qknorm, fixed_m=args.fixed_m,
                     fp8=args.fp8)
    flops = step_flops(name, spec)
    stream = torch.cuda.current_stream()

    sampler = ClockSampler(gpu_id_for_smi(local))
    elapsed, kern_s, t0, t1, busy_t0 = time_steps(wl, args.steps, args.warmup, world, stream)

    # e2e through the C-ABI with host buffers (self / cross workloads)
    e2e = None
    if name != "sharded":
        ee = E2E(wl)
        for i in range(max(3, min(args.warmup, 10))):
            ee.step(i)
        ee.finish()
        torch.cuda.synchronize()
        n_e2e = max(3, min(args.steps, 200 if name != "wan720" else 10))
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize()
        a.record(stream)
        for i in range(n_e2e):
            ee.step(i)
        ee.finish()          # the last download is inside the timed region
        b.record(stream)
        torch.cuda.synchronize()
        barrier(world)
        e_el, e_units = reduce_over_ranks(a.elapsed_time(b) / 1e3, flops * n_e2e, world)
        e2e = {"value": e_units / e_el / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": ee.h2d,
               "d2h_bytes_per_step": ee.d2h, "steps": n_e2e,
               "path": ("pinned host q/k/v -> H2D -> " + ("(B = 1: into the padded buffers) " if ee.direct else
                                                          "dit_pad_tokens -> ")
                        + "attention -> " + ("" if ee.direct else "dit_unpad_tokens -> ")
                        + "D2H O, LSE; steps pipelined over two buffer sets (uploads, compute and "
                          "downloads on three streams)")}
        del ee
    busy_t1 = time.time()
    launches = wl.launches_per_step * args.steps
    host = wl.host
    dom_bytes = wl.dominant_bytes()
    del wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    max_el, units = reduce_over_ranks(elapsed, flops * args.steps, world)
    also = None
    if (rank == 0 and world == 1 and not args.no_also and name == "wan720" and args.rope == "ws"
            and not (args.qknorm or args.fixed_m or args.fp8)):
        also = also_records(peaks, sampler, ("wan480", "cross", "sharded"), world, stream)
    sampler.stop()
    if rank != 0:
        if world > 1:
            torch.distributed.destroy_process_group()
        return
    clocks = sampler.summary(t0, t1, busy_t0, busy_t1)
    achieved = flops / kern_s / 1e12
    peak, peak_source = pick_peak(peaks, elapsed, fp8=args.fp8)
    variant = "qknorm" if args.qknorm else ("fixed_m" if args.fixed_m else "")
    # FP8 is timed with its preparation kernels: no single-kernel traffic; the per-tile RoPE
    # kernel has no committed capture
    prof = None if (args.fp8 or (args.rope == "fused" and name != "cross")) else profiled(name, variant)
    prof = prof or {}
    value = units / max_el / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": max_el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8_e4m3" if args.fp8 else "bf16",
        "data": "synthetic", "config": dict(config_dict(name, spec, args.rope), **(
            {"reduced": f"{spec.H} heads instead of the workload's (profiling run; not a bench value)"}
            if args.heads is not None else {}), **(
            {"qk_norm": "per-head RMSNorm before the rotation, synthetic weights 1 + 0.1 N(0,1), eps 1e-6"}
            if args.qknorm else {}), **(
            {"softmax": "fixed-m: 32-row blocks whose bound scale*|q|*max|k| allows it skip the running maximum"}
            if args.fixed_m else {}), **(
            {"precision": "fp8 e4m3 operands (q per 128-row tile, k and v per head), P = e4m3(112 p), fp32 "
                          "accumulation; the step includes the two preparation kernels"} if args.fp8 else {})),
        "pct_of_bf16_peak": 100.0 * value / (peak * world),
        "pct_of_nominal_bf16_dense": 100.0 * value / ((2.0 if args.fp8 else 1.0) * NOMINAL_BF16_TFLOPS * world),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak,
                     "frac_of_burst": achieved / ((2.0 if args.fp8 else 1.0) * peaks["bf16_tflops"]),
                     "frac_of_nominal": achieved / ((2.0 if args.fp8 else 1.0) * NOMINAL_BF16_TFLOPS),
                     "traffic": prof.get("traffic"),
                     "ncu_kernel_ms": prof.get("ncu_kernel_ms"),
                     "kernel": dominant_kernel(name, args.rope) + (" + q/k RMSNorm" if args.qknorm else "")
                     + (" (fixed-m softmax)" if args.fixed_m else "")
                     + (" (fp8; timed with its two preparation kernels)" if args.fp8 else ""),
                     "kernel_ms": kern_s * 1e3, "algorithmic_bytes": dom_bytes,
                     "peak_source": peak_source,
                     "target": "attention >= 60 % of the measured dense bf16 peak (fractions from CUDA-event "
                               "kernel time)"},
        "gpu_launches": launches,
        "clocks": clocks,
    }
    if e2e is not None:
        line["e2e"] = e2e
    if also is not None:
        line["also"] = also
    if rank == 0 and not args.no_hbm_kernels:
        line["hbm_kernels"] = measure_hbm_kernels(peaks)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(name, spec, host)
    print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
