#!/usr/bin/env python
"""Throughput benchmark of the rotary position embedding hot path on GB300.

One step = one pass of RotaryEmbedding over one batch of the headline
workload, the largest published configuration: rank-4 float16 X
(8, 32, 4096, 128), interleaved pairs, rotary_embedding_dim 64 (the other 64
elements of every head copied through), position_ids uniform over a
(16384, 32) cos/sin cache; 541 MB of algorithmic traffic per pass. Launched
through the library's C ABI. Inputs are resident in HBM when the timed region
starts; X/Y rotate over enough buffer sets that no step finds its inputs in
L2. The other published configurations (the rank-3 gather, M-RoPE in both
layouts, the decode step, the float32 parity case) are timed after the timed
region and summarised under ``roofline.configs``.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gpu|reference]

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle (the
only comparison implementation available) on a bounded sample of the same
workload, on the host's cores. Under torchrun (N > 1) each rank runs the same
per-GPU workload on its own batch (weak scaling, no data-path collective);
the time is the maximum over ranks.
"""

import argparse
import ctypes
import hashlib
import json
import math
import os
import re
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rotary_position_embedding_gb300 import workloads as wl  # noqa: E402

L2_BYTES = 129 * 2 ** 20
FALLBACK_HBM_GBS = 6800.0
METRIC = "RoPE achieved HBM GB/s and Gelem/s, fp16, as % of GB300 HBM roofline"
# Sources of each kernel family -- its device code and the host code that plans
# its launches (rope_api.cu): a profiled DRAM figure is reported only while the
# code it was captured on is unchanged (comments and blank lines aside).
KERNEL_SOURCES = {
    "rope_rows_kernel": ["rope_api.cu", "rope_kernels.cuh", "k_rope.cu", "k_mrope.cu"],
    "rope_mrope_heads_kernel": ["rope_api.cu", "rope_kernels.cuh", "rope_mrope_heads.cuh", "k_mrope_heads.cu"],
    "rope_tma_kernel": ["rope_api.cu", "rope_kernels.cuh", "rope_packed.cuh", "rope_tma.cuh", "k_tma.cu"],
    "rope_fused_kernel": ["rope_api.cu", "rope_kernels.cuh", "rope_fused.cuh", "k_fused.cu"],
    "rope_qkv_kernel": ["rope_api.cu", "rope_kernels.cuh", "rope_qkv.cuh", "k_qkv.cu", "k_mrope_qkv.cu"],
    "rope_qkv_heads_kernel": ["rope_api.cu", "rope_kernels.cuh", "rope_qkv.cuh", "rope_packed.cuh",
                              "rope_qkv_heads.cuh", "k_qkv_heads.cu"],
    "rope_qkv_tma_kernel": ["rope_api.cu", "rope_kernels.cuh", "rope_tma.cuh", "rope_qkv.cuh", "rope_packed.cuh",
                            "rope_qkv_tma.cuh", "k_qkv_tma.cu", "k_mrope_qkv_tma.cu"],
}


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["gpu", "reference"], default="gpu")
    ap.add_argument("--workload", default=wl.HEADLINE, choices=list(wl.WORKLOADS))
    ap.add_argument("--no-rows", action="store_true",
                    help="time only the published configurations, not every workload")
    ap.add_argument("--row-steps", type=int, default=400)
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--variant", choices=["auto", "simt", "tma"], default="auto",
                    help="kernel variant for the timed region (the library's automatic choice by default)")
    ap.add_argument("--schedule", choices=["dynamic", "static"], default="dynamic",
                    help="tile schedule of the pipelined kernels: a 64-byte scratch counter per stream "
                         "(dynamic; measured 3-6 %% faster on M-RoPE, rank 4 and the Q/K prefill) or round "
                         "robin (no scratch)")
    ap.add_argument("--quick", action="store_true",
                    help="timed region only: no per-workload rows, end-to-end or CPU legs (profiling runs)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (host-side timing reduction only)
# ---------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), \
        int(os.environ.get("LOCAL_RANK", 0))


def max_over_ranks(x, device=None):
    """Largest value of x over all ranks (host-side timing reduction, not a data-path collective)."""
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(nbytes, numel, steps, total_ms, world):
    """Whole-job GB/s and Gelem/s: every rank moved `steps` passes of its own batch in <= total_ms."""
    sec = total_ms * 1e-3
    return world * nbytes * steps / sec / 1e9, world * numel * steps / sec / 1e9


def _code_only(text):
    """C/C++/CUDA source without comments, trailing blanks or blank lines."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash(family):
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[family]:
        with open(os.path.join(ROOT, "rotary_position_embedding_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: torch copy_, 1 Gi bf16)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback (no MEASURED_PEAKS.json)"


def profiled_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu capture, if taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[f"{kernel}:{workload}"]
        if e.get("source_hash") == kernel_source_hash(kernel):
            return e["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None
        time.sleep(0.4)

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.strip().split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 <= r[0] <= t1]
        note = "samples inside the timed region"
        if not inside and rows:  # region shorter than the sampling period: nearest samples
            rows.sort(key=lambda r: min(abs(r[0] - t0), abs(r[0] - t1)))
            inside = rows[:2]
            note = "timed region shorter than the 100 ms sampling period: nearest samples"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for r in inside:
            for name, v in zip(names[1:], r[3][1:]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median([r[1] for r in inside])), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": sorted(reasons), "samples": len(inside), "note": note}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

class QKVStep:
    """Q/K rotation with the cache append: one rope_apply_qkv call per step (packed
    [Q|K|V] in, Q out, rotated K and V into the caches at rows past[b] + s).

    With fused=False a step is what a caller does without that entry point:
    split Q and K out of the packed tensor (torch copies), rope_apply on each,
    and scatter K and V into the caches (torch indexing).
    """

    def __init__(self, rp, torch, w, device, n_sets, shard=0, dynamic=True):
        self.w, self.torch, self.rp = w, torch, rp
        self.lib = rp.load_library()
        self.dynamic = dynamic
        self.scratch = {}
        inp = wl.make_inputs(w, shard=shard)
        tdt = torch_dtype(torch, w.dtype)
        x0 = host_to_torch(torch, inp["x"]).to(device)
        self.xs = [x0] + [x0.clone() for _ in range(n_sets - 1)]
        B, S, H = w.batch, w.seq, w.head_size
        self.Nq, self.Nkv = w.num_heads, w.extra["kv_num_heads"]
        self.qo = [torch.empty((B, S, self.Nq * H), dtype=tdt, device=device) for _ in range(n_sets)]
        L = w.extra["max_len"]
        self.kc = torch.zeros((B, self.Nkv, L, H), dtype=tdt, device=device)
        self.vc = torch.zeros_like(self.kc)
        self.past = torch.from_numpy(inp["past_seq_lens"]).to(device)
        inv = torch.from_numpy(inp["inv_freq"]).to(device)
        self.cos, self.sin = rp.rope_cache_build(inv, w.cache_rows, tdt)
        self.code = DTYPE_CODES[w.dtype]
        self.H = H
        self.norm = bool(w.extra.get("rms_norm"))
        if self.norm:
            self.qw = host_to_torch(torch, inp["q_norm_weight"]).to(device)
            self.kw = host_to_torch(torch, inp["k_norm_weight"]).to(device)
            self.eps = float(w.extra["epsilon"])
        # M-RoPE: the three position streams and the section
        self.mrope = w.positions == "mrope"
        self.pos3 = torch.from_numpy(inp["position_ids"]).to(device) if self.mrope else None
        self.sec = (ctypes.c_int32 * 3)(*(w.mrope_section or (0, 0, 0)))
        # unfused path: positions past[b] + s and the (b, row) scatter indices
        s_idx = torch.arange(S, device=device, dtype=torch.int64)[None, :]
        self.pos = (self.past.to(torch.int64)[:, None] + s_idx).contiguous()
        self.bi = torch.arange(B, device=device)[:, None].expand(B, S)
        self.ri = self.pos
        torch.cuda.synchronize()

    def scratch_for(self, stream):
        return Step.scratch_for(self, stream)

    def launch(self, k, stream, fused=True):
        w, lib = self.w, self.lib
        vp = ctypes.c_void_p
        scr = self.scratch_for(stream)
        if fused and self.mrope:
            nw = (vp(self.qw.data_ptr()), vp(self.kw.data_ptr())) if self.norm else (None, None)
            return lib.mrope_apply_qkv(
                self.code, w.batch, w.seq, self.Nq, self.Nkv, self.H, vp(self.xs[k].data_ptr()), None, None,
                nw[0], nw[1], self.eps if self.norm else 0.0, vp(self.cos.data_ptr()), vp(self.sin.data_ptr()),
                w.cache_rows, vp(self.pos3.data_ptr()), self.sec, w.mrope_layout, w.scale,
                vp(self.past.data_ptr()), 0, 0, vp(self.qo[k].data_ptr()), None, vp(self.kc.data_ptr()),
                vp(self.vc.data_ptr()), w.extra["max_len"], None, scr, stream)
        if fused and self.norm:
            return lib.rope_apply_qkv_rmsnorm(
                self.code, w.batch, w.seq, self.Nq, self.Nkv, self.H, vp(self.xs[k].data_ptr()), None, None,
                vp(self.qw.data_ptr()), vp(self.kw.data_ptr()), self.eps, vp(self.cos.data_ptr()),
                vp(self.sin.data_ptr()), w.cache_rows, None, vp(self.past.data_ptr()), 0, 0,
                vp(self.qo[k].data_ptr()), None, vp(self.kc.data_ptr()), vp(self.vc.data_ptr()),
                w.extra["max_len"], None, scr, stream)
        if fused:
            return lib.rope_apply_qkv(self.code, w.batch, w.seq, self.Nq, self.Nkv, self.H,
                                      ctypes.c_void_p(self.xs[k].data_ptr()), None, None,
                                      ctypes.c_void_p(self.cos.data_ptr()), ctypes.c_void_p(self.sin.data_ptr()),
                                      w.cache_rows, None, ctypes.c_void_p(self.past.data_ptr()), 0, 0,
                                      ctypes.c_void_p(self.qo[k].data_ptr()), None,
                                      ctypes.c_void_p(self.kc.data_ptr()), ctypes.c_void_p(self.vc.data_ptr()),
                                      w.extra["max_len"], None, scr, stream)
        B, S, H, Nq, Nkv = w.batch, w.seq, self.H, self.Nq, self.Nkv
        x = self.xs[k].view(B, S, Nq + 2 * Nkv, H)
        if self.mrope:
            # torch RMSNorm, then M-RoPE on Q and on K (two library calls), then the cache scatter
            torch = self.torch
            xf = x[:, :, :Nq + Nkv].float()
            n = (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + self.eps)).to(x.dtype)
            q = (n[:, :, :Nq] * self.qw).reshape(B, S, Nq * H).contiguous()
            kk = (n[:, :, Nq:] * self.kw).reshape(B, S, Nkv * H).contiguous()
            sec = tuple(w.mrope_section)
            self.rp.mrope_apply(q, self.cos, self.sin, self.pos3, sec, mrope_layout=w.mrope_layout,
                                num_heads=Nq, out=self.qo[k])
            kr = self.rp.mrope_apply(kk, self.cos, self.sin, self.pos3, sec, mrope_layout=w.mrope_layout,
                                     num_heads=Nkv)
            self.kc[self.bi, :, self.ri] = kr.view(B, S, Nkv, H)
            self.vc[self.bi, :, self.ri] = x[:, :, Nq + Nkv:]
            return 0
        if self.norm:
            # QK-Norm as separate torch ops, then the fused rotation + append
            torch = self.torch
            xf = x[:, :, :Nq + Nkv].float()
            n = (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + self.eps)).to(x.dtype)
            wqk = torch.cat([self.qw.expand(Nq, H), self.kw.expand(Nkv, H)])
            xn = torch.cat([n * wqk, x[:, :, Nq + Nkv:]], dim=2).contiguous()
            return lib.rope_apply_qkv(self.code, B, S, Nq, Nkv, H, vp(xn.data_ptr()), None, None,
                                      vp(self.cos.data_ptr()), vp(self.sin.data_ptr()), w.cache_rows, None,
                                      vp(self.past.data_ptr()), 0, 0, vp(self.qo[k].data_ptr()), None,
                                      vp(self.kc.data_ptr()), vp(self.vc.data_ptr()), w.extra["max_len"], None,
                                      scr, stream)
        q = x[:, :, :Nq].reshape(B, S, Nq * H).contiguous()
        kk = x[:, :, Nq:Nq + Nkv].reshape(B, S, Nkv * H).contiguous()
        self.rp.rope_apply(q, self.cos, self.sin, self.pos, num_heads=Nq, out=self.qo[k])
        kr = self.rp.rope_apply(kk, self.cos, self.sin, self.pos, num_heads=Nkv)
        self.kc[self.bi, :, self.ri] = kr.view(B, S, Nkv, H)
        self.vc[self.bi, :, self.ri] = x[:, :, Nq + Nkv:]
        return 0


class Step:
    """One workload pass through the C ABI with pre-marshalled ctypes arguments."""

    def __init__(self, rp, torch, w, device, n_sets, shard=0, dynamic=True):
        self.w = w
        self.torch = torch
        # one zeroed scratch per stream this Step launches on (dynamic schedule)
        self.dynamic = dynamic
        self.scratch = {}
        lib = rp.load_library()
        self.lib = lib
        inp = wl.make_inputs(w, shard=shard)
        self.x_host = inp["x"]
        self.pos_host = inp["position_ids"]
        tdt = torch_dtype(torch, w.dtype)
        self.code = DTYPE_CODES[w.dtype]
        self.inv = torch.from_numpy(inp["inv_freq"]).to(device)
        x0 = host_to_torch(torch, self.x_host).to(device)
        self.xs = [x0] + [x0.clone() for _ in range(n_sets - 1)]
        self.ys = [torch.empty_like(x0) for _ in range(n_sets)]
        self.pos = None if self.pos_host is None else torch.from_numpy(self.pos_host).to(device)
        self.nh = w.num_heads if w.rank == 3 else 0
        self.xshape = (ctypes.c_int64 * w.rank)(*w.shape)
        if w.kind == "rope" and w.positions == "none":
            c, s = rp.rope_cache_build(self.inv, w.tokens, tdt)
            self.cos, self.sin = c.view(w.batch, w.seq, w.half), s.view(w.batch, w.seq, w.half)
        elif w.kind in ("rope", "mrope", "fused", "mrope_fused"):
            self.cos, self.sin = rp.rope_cache_build(self.inv, w.cache_rows, tdt,
                                                     attention_scaling=w.attention_scaling)
        self.cshape = (ctypes.c_int64 * self.cos.dim())(*self.cos.shape)
        self.sec = (ctypes.c_int32 * 3)(*(w.mrope_section or (0, 0, 0)))
        torch.cuda.synchronize()

    def launch(self, k, stream, fused=False):
        w = self.w
        x = ctypes.c_void_p(self.xs[k].data_ptr())
        y = ctypes.c_void_p(self.ys[k].data_ptr())
        return self.call(x, y, stream, fused)

    def scratch_for(self, stream):
        """The dynamic schedule's scratch for launches on `stream`: one zeroed buffer per
        stream, made on first use (outside any timed region or graph capture: every
        stream a timing loop uses gets its first launch in the warm-up)."""
        if not self.dynamic:
            return None
        key = stream.value if isinstance(stream, ctypes.c_void_p) else stream
        buf = self.scratch.get(key)
        if buf is None:
            buf = self.torch.zeros(8, dtype=self.torch.int64, device=self.xs[0].device)
            self.scratch[key] = buf
        return ctypes.c_void_p(buf.data_ptr())

    def call(self, x, y, stream, fused=False, pos=None):
        w = self.w
        lib = self.lib
        pt = self.pos if pos is None else pos
        pos = None if pt is None else ctypes.c_void_p(pt.data_ptr())
        scr = self.scratch_for(stream)
        cos = ctypes.c_void_p(self.cos.data_ptr())
        sin = ctypes.c_void_p(self.sin.data_ptr())
        if w.kind == "mrope_fused" and fused:
            st = lib.mrope_apply_fused(self.code, w.rank, self.xshape, x, y, ctypes.c_void_p(self.inv.data_ptr()),
                                       w.attention_scaling, pos, self.sec, w.mrope_layout, w.scale, w.interleaved,
                                       w.rotary_embedding_dim, self.nh, stream)
        elif w.kind in ("mrope", "mrope_fused"):
            st = lib.mrope_apply(self.code, w.rank, self.xshape, x, y, w.cache_rows, cos, sin, pos, self.sec,
                                 w.mrope_layout, w.scale, w.interleaved, w.rotary_embedding_dim, self.nh, 0,
                                 None, scr, stream)
        elif w.kind == "fused" and fused:
            st = lib.rope_apply_fused(self.code, w.rank, self.xshape, x, y, ctypes.c_void_p(self.inv.data_ptr()),
                                      w.attention_scaling, pos, w.interleaved, w.rotary_embedding_dim, self.nh,
                                      stream)
        else:
            st = lib.rope_apply(self.code, w.rank, self.xshape, x, y, self.cos.dim(), self.cshape, cos, sin, pos,
                                w.interleaved, w.rotary_embedding_dim, self.nh, None, scr, stream)
        if st != 0:
            raise RuntimeError(f"{w.name}: status {st}: {lib.rope_last_error().decode()}")


DTYPE_CODES = {"float32": 0, "float16": 1, "bfloat16": 2}
POSITION_RECIPES = {
    "none": "none: a (B, S, rd/2) table, row (b, s)",
    "offset": "s + U[0,4096) per batch",
    "uniform": "U[0, cache rows)",
    "mrope": "t/h/w: text spans equal, 32x32 image grids per frame, per-batch offset; 1 % of ids past the table",
    "past": "implicit: past[b] + s, past[b] ~ U[0, max past]",
}


def torch_dtype(torch, name):
    return {"float32": torch.float32, "float16": torch.float16, "bfloat16": torch.bfloat16}[name]


def host_to_torch(torch, a):
    """Host tensor over a numpy array (bfloat16 arrays are uint16 bit patterns)."""
    a = np.ascontiguousarray(a)
    if a.dtype == wl.BF16_BITS:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    return torch.from_numpy(a)


def make_step(rp, torch, w, device, n_sets, shard=0, dynamic=False):
    # the Q/K pipeline takes the same scratch counter: measured 35.9 -> 33.9 us per
    # launch on the RoPE Q/K prefill, unchanged (within 0.1 us) with QK-Norm and M-RoPE
    if w.kind == "qkv":
        return QKVStep(rp, torch, w, device, n_sets, shard=shard, dynamic=dynamic)
    return Step(rp, torch, w, device, n_sets, shard=shard, dynamic=dynamic)


def n_buffer_sets(w):
    per_set = 2 * w.numel * wl.itemsize(w.dtype)
    return max(2, math.ceil(4 * L2_BYTES / per_set))


def config_of(w, world):
    """The ``config`` object of the JSON line: the workload and how it is fed.
    Both arms print the same one."""
    n = n_buffer_sets(w)
    return {
        "workload": w.name, "shape": list(w.shape), "num_heads": w.num_heads,
        "head_size": w.head_size, "rotary_dim": w.rotary_dim, "interleaved": w.interleaved,
        "cache_rows": w.cache_rows, "positions": POSITION_RECIPES[w.positions],
        "algorithmic_bytes_per_step": wl.algorithmic_bytes(w),
        "l2": f"inputs rotate over {n} X/Y buffer sets "
              f"({n * 2 * w.numel * wl.itemsize(w.dtype) / 2**20:.0f} MiB) > 129 MiB L2; no flush kernel",
        "launch": "one C-ABI call per step on the current stream, queued ahead of the GPU; "
                  "timed region = one CUDA event pair around the K steps",
        "parallelism": f"{world} independent replicas (per-GPU batch)",
    }


def time_steps(torch, step, steps, stream_handle, fused=False):
    """Time `steps` back-to-back launches (rotating buffer sets) with one CUDA
    event pair on the launching stream around all of them."""
    n_sets = len(step.xs)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    torch.cuda._sleep(2_000_000)  # let the host queue launches ahead of the GPU
    t_start.record()
    for k in range(steps):
        step.launch(k % n_sets, stream_handle, fused)
    t_end.record()
    torch.cuda.synchronize()
    return t_start.elapsed_time(t_end)


def time_isolated(torch, step, samples, stream_handle, fused=False):
    """Durations of single launches, each alone between its own event pair.

    A short device-side sleep goes in front of every sample, so the start
    event, the launch and the end event are all queued before the GPU reaches
    them: the pair brackets the launch and nothing of the host. It still
    breaks the overlap that back-to-back launches get from programmatic
    dependent launch."""
    n_sets = len(step.xs)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(samples)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(samples)]
    torch.cuda.synchronize()
    for k in range(samples):
        torch.cuda._sleep(100_000)  # ~50 us at 2 GHz
        starts[k].record()
        step.launch(k % n_sets, stream_handle, fused)
        ends[k].record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in zip(starts, ends)]


def isolation_floor(torch, step, samples, stream_handle):
    """What an isolated launch costs beyond the kernel, measured the same way
    as time_isolated (device sleep, then an event pair around one launch):
      - an empty kernel (torch's device sleep of 0 cycles): the event pair and
        the launch of a one-block grid;
      - a device-to-device copy of X into Y (torch ``copy_``, a
        cudaMemcpyAsync, the operation the measured HBM peak was taken with):
        the same pair around a plain stream of 2 |X| bytes, whose own ramp
        and drain a bandwidth-bound kernel also pays.
    Medians in microseconds."""
    n_sets = len(step.xs)
    res = {}
    for label in ("empty_kernel", "copy_x_to_y"):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(samples)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(samples)]
        torch.cuda.synchronize()
        for k in range(samples):
            torch.cuda._sleep(100_000)
            starts[k].record()
            if label == "empty_kernel":
                torch.cuda._sleep(0)
            else:
                step.ys[k % n_sets].copy_(step.xs[k % n_sets])
            ends[k].record()
        torch.cuda.synchronize()
        res[label + "_us"] = round(float(np.median([a.elapsed_time(b) for a, b in zip(starts, ends)])) * 1e3, 3)
    return res


def time_graph(torch, step, launches, replays, fused=False):
    """Device time per launch with no host in the loop: `launches` calls
    (rotating buffer sets) captured once into a CUDA graph, replayed `replays`
    times between one event pair. For workloads whose kernels are shorter
    than the host's per-call cost, this is the GPU's own time per step."""
    n_sets = len(step.xs)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for k in range(3):
            step.launch(k % n_sets, ctypes.c_void_p(side.cuda_stream), fused)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        cap = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        for k in range(launches):
            step.launch(k % n_sets, cap, fused)
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / (replays * launches)
    del g
    return ms


def gpu_arm(args, rank, world, local_rank):
    import torch

    import rotary_position_embedding_gb300 as rp

    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=device)
    rp.load_library()
    rp.set_variant(args.variant)
    w = wl.WORKLOADS[args.workload]
    stream = torch.cuda.current_stream(device)
    sh = ctypes.c_void_p(stream.cuda_stream)
    # the on-the-fly workloads time their fused entry point; the Q/K workloads the fused op
    fused = w.kind in ("qkv", "fused", "mrope_fused")
    nbytes = wl.algorithmic_bytes(w, cached=not fused or w.kind == "qkv")
    step = make_step(rp, torch, w, device, n_buffer_sets(w), shard=rank, dynamic=args.schedule == "dynamic")
    for k in range(args.warmup):
        step.launch(k % len(step.xs), sh, fused)
    torch.cuda.synchronize()
    kernel_family = rp.last_kernel()  # what the variant chose for this workload

    sampler = ClockSampler(local_rank if "CUDA_VISIBLE_DEVICES" not in os.environ else
                           os.environ["CUDA_VISIBLE_DEVICES"].split(",")[local_rank])
    if rank == 0:
        sampler.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t0 = time.time()
    total_ms = time_steps(torch, step, args.steps, sh, fused=fused)
    t1 = time.time()
    total_ms_local = total_ms
    if world > 1:
        torch.distributed.barrier()
        total_ms = max_over_ranks(total_ms, device)
    clocks = sampler.stop(t0, t1) if rank == 0 else None

    ms_per_step = total_ms / args.steps
    value, gelem = aggregate_throughput(nbytes, w.numel, args.steps, total_ms, world)
    # A step is exactly one launch of one kernel, so that kernel's average
    # launch duration is this rank's timed region over K.
    kern_ms = total_ms_local / args.steps
    peak, peak_src = measured_peak()
    achieved = nbytes / (kern_ms * 1e-3) / 1e9
    # context, outside the timed region: the same launch bracketed alone by an event pair
    iso_ms = float(np.median(time_isolated(torch, step, 200, sh, fused=fused)))
    floor = isolation_floor(torch, step, 200, sh) if isinstance(step, Step) else None
    if kernel_family == "rope_rows_kernel":
        schedule = "n/a (SIMT kernel: fixed thread roles, no scratch)"
    elif args.schedule == "static":
        schedule = "static (tiles dealt round robin, no scratch)"
    else:
        schedule = "dynamic (tiles drawn from a 64-byte scratch counter per stream)"

    out = None
    if rank == 0:
        rows = {}
        if not args.quick:
            rows = measure_rows(args, torch, rp, device, peak,
                                names=wl.CONFIGS if args.no_rows else list(wl.WORKLOADS))
        e2e = None if (args.quick or fused) else measure_e2e(args, torch, step, sh, nbytes)
        cpu = cpu_baseline(args, w) if (world == 1 and not args.quick) else None
        out = {
            "metric": METRIC,
            "variant": args.variant,
            "value": round(value, 2),
            "unit": "GB/s",
            "gelem_per_s": round(gelem, 3),
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": {"float32": "f32", "float16": "f16", "bfloat16": "bf16"}[w.dtype],
            "data": "synthetic (seeded N(0,1) X, position ids per the workload recipe; caches from "
                    "rope_cache_build)",
            "config": config_of(w, world),
            "roofline": {
                "bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": profiled_traffic(kernel_family, w.name),
                "peak_source": peak_src,
                "kernel": f"{kernel_family} (variant {args.variant}: the one kernel of the step)",
                "schedule": schedule,
                "kernel_us": round(kern_ms * 1e3, 3),
                "kernel_us_how": "timed region / K on the launching stream (a step is one launch of this "
                                 "kernel, back to back as in a real stream)",
                "kernel_us_isolated": round(iso_ms * 1e3, 3),
                "frac_isolated": round(nbytes / (iso_ms * 1e-3) / 1e9 / peak, 4),
                "isolated_how": "median of 200 launches each bracketed alone by its own event pair behind a "
                                "short device sleep, outside the timed region (no overlap with a previous "
                                "launch)",
                "isolated_floor": floor,
                "frac_of_nominal_8tbs": round(achieved / 8000.0, 4),
                "configs": config_summary(rows, peak),
            },
            "clocks": clocks,
            "e2e": e2e,
            "gpu_launches": args.steps,
            "cpu_baseline": cpu,
            "rows": rows,
        }
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return out


def measure_rows(args, torch, rp, device, peak, names):
    """The workloads `names` (both M-RoPE layouts, fused and cached decode), timed three ways:
    each launch alone between its own event pair behind a device sleep
    (median), back to back from the host (includes the host's per-call cost
    where that exceeds the kernel), and replayed from a CUDA graph of 64
    launches (device time)."""
    stream = torch.cuda.current_stream(device)
    sh = ctypes.c_void_p(stream.cuda_stream)
    rows = {}
    prev = rp.get_variant()
    for name in names:
        w = wl.WORKLOADS[name]
        variants = [("cached", False, "auto"), ("cached", False, "simt")]
        if w.kind in ("fused", "mrope_fused"):
            variants = [("fused", True, "auto"), ("cached", False, "auto")]
        if w.kind == "qkv":
            variants = [("fused", True, "auto"), ("unfused", False, "auto")]
        step = make_step(rp, torch, w, device, n_buffer_sets(w), dynamic=args.schedule == "dynamic")
        for label, fused, variant in variants:
            rp.set_variant(variant)
            for k in range(20):
                step.launch(k % len(step.xs), sh, fused)
            torch.cuda.synchronize()
            kernel = rp.last_kernel() if not (w.kind == "qkv" and not fused) else "mixed (torch + library)"
            total_ms = time_steps(torch, step, args.row_steps, sh, fused)
            kern = time_isolated(torch, step, min(200, args.row_steps), sh, fused)
            graph_ms = None
            if not (w.kind == "qkv" and not fused):  # the unfused Q/K path is torch ops: not captured
                graph_ms = time_graph(torch, step, 64, max(2, args.row_steps // 64), fused)
            rp.set_variant(prev)
            nbytes = wl.algorithmic_bytes(w, cached=not fused or w.kind == "qkv")
            kern_ms = float(np.median(kern))
            gbs = nbytes / (kern_ms * 1e-3) / 1e9
            key = f"{name}:{label}:{variant}"
            rows[key] = {
                "kernel": kernel,
                "us_per_launch_median": round(kern_ms * 1e3, 3),
                "us_per_step_incl_gaps": round(total_ms / args.row_steps * 1e3, 3),
                "GB_s": round(gbs, 1), "Gelem_s": round(w.numel / (kern_ms * 1e-3) / 1e9, 2),
                "frac_of_measured_peak": round(gbs / peak, 4), "frac_of_nominal_8tbs": round(gbs / 8000, 4),
                "bytes": nbytes,
            }
            if graph_ms is not None:
                ggbs = nbytes / (graph_ms * 1e-3) / 1e9
                rows[key].update({"us_per_step_graph": round(graph_ms * 1e3, 3), "GB_s_graph": round(ggbs, 1),
                                  "frac_graph": round(ggbs / peak, 4)})
        if name in wl.CONFIGS and hasattr(step, "ys"):
            # what a plain device copy of the same X into Y costs alone, measured the same way:
            # the isolated launch's floor for this configuration's bytes
            floor = isolation_floor(torch, step, min(200, args.row_steps), sh)
            for key in rows:
                if key.startswith(name + ":"):
                    rows[key]["copy_x_to_y_us_isolated"] = floor["copy_x_to_y_us"]
        del step
        torch.cuda.empty_cache()
    # one-time setup row: cache build of the largest table
    inv = torch.from_numpy(wl.inv_freq(1e6, 128, 64)).to(device)
    c, s = rp.rope_cache_build(inv, 32768, torch.float16)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(10):
        rp.rope_cache_build(inv, 32768, torch.float16, cos_out=c, sin_out=s)
    ev1.record()
    torch.cuda.synchronize()
    rows["rope_cache_build(32768x64,f16)"] = {"us_per_launch": round(ev0.elapsed_time(ev1) / 10 * 1e3, 2)}
    return rows


def config_summary(rows, peak):
    """Compact figures of every published configuration: kernel, microseconds
    back to back (timed region / launches), from a CUDA graph and alone (median
    of event-bracketed single launches), the fractions of the measured peak they
    give with the configuration's algorithmic bytes, and (X-to-Y kernels) the
    time of a lone device copy of X into Y over the lone launch's time."""
    out = {}
    for name in wl.CONFIGS:
        w = wl.WORKLOADS[name]
        label = "fused" if w.kind in ("fused", "mrope_fused") else "cached"
        r = rows.get(f"{name}:{label}:auto")
        if r is None:
            continue
        nb = r["bytes"]
        d = {"kernel": r["kernel"], "bytes": nb, "us_b2b": r["us_per_step_incl_gaps"],
             "us_graph": r.get("us_per_step_graph"), "us_isolated": r["us_per_launch_median"]}
        for k in ("b2b", "graph", "isolated"):
            us = d["us_" + k]
            d["frac_" + k] = None if not us else round(nb / (us * 1e-6) / 1e9 / peak, 4)
        copy_us = r.get("copy_x_to_y_us_isolated")
        if copy_us:
            # a lone launch against a lone device copy of X into Y: 1.0 = as fast as the copy
            d["us_copy_x_to_y_isolated"] = copy_us
            d["isolated_copy_over_kernel"] = round(copy_us / d["us_isolated"], 4)
        out[name] = d
    return out


def measure_e2e(args, torch, step, sh, nbytes):
    """Same metric through the C ABI with host buffers, every step: H2D of that
    step's X and positions from pinned memory, the launch, D2H of Y into pinned
    memory. Two streams alternate steps, so one step's D2H overlaps the next
    step's H2D (the copy engines run both directions at once)."""
    x_host = [host_to_torch(torch, step.x_host).pin_memory() for _ in range(2)]
    y_host = [torch.empty_like(x_host[0]).pin_memory() for _ in range(2)]
    pos_host = None if step.pos_host is None else torch.from_numpy(step.pos_host).pin_memory()
    streams = [torch.cuda.Stream() for _ in range(2)]
    xd = [step.xs[0], step.xs[1 % len(step.xs)]]
    yd = [step.ys[0], step.ys[1 % len(step.ys)]]
    pd = [step.pos, None if step.pos is None else step.pos.clone()]

    def one(k, kernel=True):
        i = k % 2
        with torch.cuda.stream(streams[i]):
            xd[i].copy_(x_host[i], non_blocking=True)
            if pos_host is not None:
                pd[i].copy_(pos_host, non_blocking=True)
            if kernel:
                step.call(ctypes.c_void_p(xd[i].data_ptr()), ctypes.c_void_p(yd[i].data_ptr()),
                          ctypes.c_void_p(streams[i].cuda_stream), pos=pd[i])
            y_host[i].copy_(yd[i], non_blocking=True)

    def timed(kernel):
        for k in range(4):
            one(k, kernel)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for s_ in streams:
            s_.wait_event(e0)
        for k in range(args.e2e_steps):
            one(k, kernel)
        for s_ in streams:
            torch.cuda.current_stream().wait_stream(s_)
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / args.e2e_steps

    ms = timed(True)
    # the same loop with the copies only: the host link's own ceiling for this step
    ms_copies = timed(False)
    h2d = x_host[0].numel() * x_host[0].element_size() + (0 if pos_host is None else pos_host.numel() * 8)
    d2h = y_host[0].numel() * y_host[0].element_size()
    return {"value": round(nbytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "ms_per_step": round(ms, 4),
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "copies_only": {"value": round(nbytes / (ms_copies * 1e-3) / 1e9, 2), "unit": "GB/s",
                            "ms_per_step": round(ms_copies, 4),
                            "link_GB_s": round((h2d + d2h) / (ms_copies * 1e-3) / 1e9, 1)},
            "note": "transfer-bound: per step pinned host X/positions -> device, rope_apply, device Y -> "
                    "pinned host, two streams alternating; copies_only = the same loop without the kernel"}


# ---------------------------------------------------------------------------
# CPU oracle (baseline leg and the reference arm)
# ---------------------------------------------------------------------------

class OracleStep:
    """The oracle on the first `tokens` tokens of the workload (a bounded sample)."""

    def __init__(self, w, tokens=None):
        import oracle

        self.oracle = oracle
        self.w = w
        inp = wl.make_inputs(w)
        x, pos = inp["x"], inp["position_ids"]
        dtype = wl.storage_dtype(w.dtype)
        T = w.tokens if tokens is None else max(1, min(tokens, w.tokens))
        S = w.seq
        nb = max(1, math.ceil(T / S))
        s_keep = S if T >= S else T
        # rank 3 (B, S, N*H): whole batches, or a prefix of one sequence
        if w.rank == 3:
            self.x = np.ascontiguousarray(x[:nb, :s_keep])
        else:
            self.x = np.ascontiguousarray(x[:nb, :, :s_keep])
        if pos is None:
            self.pos = None
        elif w.positions == "mrope":
            self.pos = np.ascontiguousarray(pos[:, :nb, :s_keep])
        else:
            self.pos = np.ascontiguousarray(pos[:nb, :s_keep])
        self.tokens = nb * s_keep
        self.nh = w.num_heads if w.rank == 3 else 0
        self.cos, self.sin = oracle.cache_build(inp["inv_freq"], w.cache_rows if w.positions != "none"
                                                else w.tokens, dtype, w.attention_scaling)
        if w.positions == "none":
            self.cos = self.cos.reshape(w.batch, w.seq, w.half)[:nb, :s_keep]
            self.sin = self.sin.reshape(w.batch, w.seq, w.half)[:nb, :s_keep]
        self.inv = inp["inv_freq"]
        self.bytes = wl.algorithmic_bytes(w) * self.tokens / w.tokens
        if w.kind == "qkv":
            self.past = inp["past_seq_lens"][:nb]
            self.qw, self.kw = inp.get("q_norm_weight"), inp.get("k_norm_weight")
            shape = (nb, w.extra["kv_num_heads"], w.extra["max_len"], w.head_size)
            self.kc, self.vc = np.zeros(shape, dtype), np.zeros(shape, dtype)

    def run(self):
        w, o = self.w, self.oracle
        if w.kind == "qkv" and w.positions == "mrope":
            nkw = {}
            if w.extra.get("rms_norm"):
                nkw = dict(q_norm_weight=self.qw, k_norm_weight=self.kw, epsilon=w.extra["epsilon"])
            o.mrope_qkv(self.x, self.cos, self.sin, self.pos, w.mrope_section, w.mrope_layout, w.scale,
                        num_heads=w.num_heads, kv_num_heads=w.extra["kv_num_heads"], k_cache=self.kc,
                        v_cache=self.vc, past_seq_lens=self.past, **nkw)
        elif w.kind == "qkv":
            nkw = {}
            if w.extra.get("rms_norm"):
                nkw = dict(q_norm_weight=self.qw, k_norm_weight=self.kw, epsilon=w.extra["epsilon"])
            o.rope_qkv(self.x, self.cos, self.sin, None, num_heads=w.num_heads,
                       kv_num_heads=w.extra["kv_num_heads"], k_cache=self.kc, v_cache=self.vc,
                       past_seq_lens=self.past, **nkw)
        elif w.kind == "mrope":
            o.mrope(self.x, self.cos, self.sin, self.pos, w.mrope_section, w.mrope_layout, w.scale,
                    w.interleaved, w.rotary_embedding_dim, self.nh)
        elif w.kind == "mrope_fused":
            o.mrope_fused(self.x, self.inv, self.pos, w.mrope_section, w.mrope_layout, w.scale,
                          w.attention_scaling, w.interleaved, w.rotary_embedding_dim, self.nh)
        else:
            o.rope(self.x, self.cos, self.sin, self.pos, w.interleaved, w.rotary_embedding_dim, self.nh)


def cpu_baseline(args, w):
    st = OracleStep(w)
    st.run()  # warm
    reps, t0 = 0, time.perf_counter()
    while True:
        st.run()
        reps += 1
        el = time.perf_counter() - t0
        if el >= args.cpu_seconds or reps >= 1000:
            break
    gbs = st.bytes * reps / el / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{reps} full passes of {w.name} ({st.tokens} tokens each) in {el:.1f} s, "
                      f"single-threaded C oracle (binary64 arithmetic)",
            "host_cpus": os.cpu_count()}


def reference_arm(args, rank, world):
    if rank != 0:
        return None
    w = wl.WORKLOADS[args.workload]
    # size each step so warmup + steps take about two minutes at the oracle's rate
    probe = OracleStep(w, tokens=64)
    t0 = time.perf_counter()
    probe.run()
    per_token = (time.perf_counter() - t0) / probe.tokens
    budget = 120.0 / max(1, args.steps + args.warmup)
    tokens = int(max(1, min(w.tokens, budget / max(per_token, 1e-9))))
    st = OracleStep(w, tokens=tokens)
    for _ in range(args.warmup):
        st.run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        st.run()
    el = time.perf_counter() - t0
    gbs = st.bytes * args.steps / el / 1e9
    gelem = (w.numel * st.tokens / w.tokens) * args.steps / el / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 5), "unit": "GB/s",
        "gelem_per_s": round(gelem, 6), "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": {"float32": "f32", "float16": "f16", "bfloat16": "bf16"}[w.dtype],
        "data": "synthetic (same generator as the GPU arm)",
        "config": config_of(w, world),
        "cpu_baseline": {"value": round(gbs, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{st.tokens} of {w.tokens} tokens per step (bytes scaled to the sample); "
                                   "the pages publish no implementation to run, so this arm is the CPU oracle"},
        "e2e": {"value": round(gbs, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if args.impl == "reference":
        out = reference_arm(args, rank, world)
    else:
        out = gpu_arm(args, rank, world, local_rank)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
