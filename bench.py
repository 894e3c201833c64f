#!/usr/bin/env python3
"""Throughput benchmark of the depth-wise softmax read on GB300.

Default workload (the headline): Block AttnRes two-phase forward of one block,
bf16, d=4096, N=8 cached block representations, S=4 layers per block,
T=32768 tokens.  One step = phase 1 (4 queries x 8 sources, one pass over the
cache) + 3 phase-2 merges (layers 2..4 fold in their partial sums; layer 1
reads no partial).  Inputs are synthetic, seeded, resident in HBM and larger
than L2 (5.6 GB touched per step), so no explicit L2 flush is needed.

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle on the
same workload instead.  Other workloads (--workload mhar|mhar_block|msar|
msar_block|msar_chunked|msar_ps|msar_ws|msar_block_ws|msar_bwd|msar_bwd_ps|msar_block_bwd|
full_depth|block_d2048|block_fused|block_bwd|read_bwd|mhar_bwd|decode) are
for profiling and the design notes.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Block AttnRes fwd tokens/s (d=4096,N=8,S=4); achieved HBM GB/s vs GB300 peak"
PROFILE_DIR = os.path.join(ROOT, "profiles")
# Source files that define each profiled kernel; a committed ncu summary is
# only used while these files are unchanged.
CSRC = "depth_wise_attention_gb300/csrc/"
KERNEL_SOURCES = {
    "depth_read_mma": [CSRC + "depth_read_mma.cuh", CSRC + "common.cuh", CSRC + "kernels_mma.cu"],
    "depth_read_mma_multi": [CSRC + "depth_read_mma.cuh", CSRC + "common.cuh", CSRC + "kernels_mma_multi.cu"],
    "depth_read": [CSRC + "depth_read.cuh", CSRC + "common.cuh", CSRC + "dr_inst.cuh", CSRC + "kernels_bf16_multi.cu"],
    "phase2": [CSRC + "phase2.cuh", CSRC + "common.cuh", CSRC + "kernels_phase2.cu"],
    "msar": [CSRC + "msar.cu", CSRC + "msar.h", CSRC + "common.cuh"],
    "msar_tile": [CSRC + "msar_tile.cu", CSRC + "msar.h", CSRC + "common.cuh"],
    "read_bwd": [CSRC + "read_bwd.cuh", CSRC + "common.cuh", CSRC + "kernels_bwd.cu"],
    "read_bwd_split": [CSRC + "read_bwd_split.cuh", CSRC + "depth_read_mma.cuh", CSRC + "common.cuh",
                       CSRC + "kernels_bwd_split.cu", CSRC + "kernels_bwd.cu"],
    "read_bwd_many": [CSRC + "read_bwd_many.cuh", CSRC + "read_bwd_split.cuh", CSRC + "depth_read_mma.cuh",
                      CSRC + "common.cuh", CSRC + "kernels_bwd_split.cu", CSRC + "kernels_bwd.cu"],
    "msar_phase1": [CSRC + "msar_phase1.cu", CSRC + "msar.h", CSRC + "common.cuh"],
    "msar_phase2": [CSRC + "msar_phase2.cu", CSRC + "msar.h", CSRC + "common.cuh"],
    "merge_bwd": [CSRC + "merge_bwd.cuh", CSRC + "common.cuh", CSRC + "kernels_merge_bwd.cu"],
    "read_bwd_mh": [CSRC + "read_bwd.cuh", CSRC + "common.cuh", CSRC + "kernels_bwd.cu", CSRC + "kernels_bwd_mh.cu"],
    "depth_read_decode": [CSRC + "depth_read_decode.cuh", CSRC + "common.cuh", CSRC + "kernels_decode.cu"],
    "msar_bwd": [CSRC + "msar_bwd.cu", CSRC + "msar_bwd.h", CSRC + "msar.h", CSRC + "common.cuh",
                 CSRC + "read_bwd.cuh", CSRC + "kernels_bwd.cu", CSRC + "depth_read_mma.cuh", CSRC + "kernels_mma.cu",
                 CSRC + "read_bwd_one.cuh", CSRC + "read_bwd_many.cuh", CSRC + "read_bwd_split.cuh",
                 CSRC + "kernels_bwd_one.cu"],
    "read_bwd_one": [CSRC + "read_bwd_one.cuh", CSRC + "read_bwd_many.cuh", CSRC + "read_bwd_split.cuh",
                     CSRC + "depth_read_mma.cuh", CSRC + "read_bwd.cuh", CSRC + "common.cuh",
                     CSRC + "kernels_bwd_one.cu", CSRC + "kernels_bwd.cu"],
}


def kernel_sources_sha(kernel: str) -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}, "fallback"


def profile_traffic(kernel_tag: str, kernel: str):
    """dram bytes per launch of `kernel_tag` from the committed ncu summary, if
    it was taken on the current kernel sources (else None)."""
    path = os.path.join(PROFILE_DIR, f"{kernel_tag}.txt")
    if not os.path.exists(path):
        return None
    vals = {}
    with open(path) as f:
        for line in f:
            if "=" in line and not line.startswith("#"):
                k, v = line.split("=", 1)
                vals[k.strip()] = v.strip()
    if vals.get("kernel_sources_sha") != kernel_sources_sha(kernel):
        return None
    try:
        return float(vals["traffic_bytes_per_launch_full_size"])
    except (KeyError, ValueError):
        return None


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------

class BlockWorkload:
    """Block AttnRes two-phase forward of one block: phase 1 + (S-1) merges."""

    def __init__(self, T=32768, d=4096, N=8, S=4, seed=0, name="block_attnres_two_phase"):
        self.T, self.d, self.N, self.S, self.seed, self.name = T, d, N, S, seed, name
        b = 2
        self.phase1_bytes_per_token = N * d * b + S * d * b + S * 4
        self.merge_bytes_per_token = 3 * d * b + 4
        self.bytes_per_token = self.phase1_bytes_per_token + (S - 1) * self.merge_bytes_per_token
        self.launches_per_step = 1 + (S - 1)
        self.dominant = "depth_read_mma_kernel (phase 1)"
        self.dominant_src = "depth_read_mma"
        self.profile_tag = f"ncu_phase1_block_d{d}"

    def config(self):
        return {"workload": f"{self.name} bf16 d={self.d} N={self.N} S={self.S} T={self.T}",
                "T": self.T, "d": self.d, "N": self.N, "S": self.S, "dtype_sources": "bf16",
                "queries": "fp32", "l2": "inputs larger than L2 (no flush)",
                "bytes_per_token": self.bytes_per_token}

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        T, d, N, S = self.T, self.d, self.N, self.S
        self.cache, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=self.seed,
                                              device=device)
        self.cache = self.cache.view(N, T, d)
        self.queries = inputs.device_normal((S, d), (16.0 / d) ** 0.5, g, device=device)
        self.partials = torch.empty((S, T, d), dtype=torch.bfloat16, device=device)
        for i in range(S):
            self.partials[i].copy_(torch.randn((T, d), generator=g, device=device))
        self.o = torch.empty((S, T, d), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((S, T), dtype=torch.float32, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.attnres_block_phase1(self.cache, self.queries, None, 1e-6, o=self.o, lse=self.lse,
                                     stream=stream)
        if ev is not None:
            ev[1].record(stream)
        for i in range(1, self.S):
            attnres.attnres_block_phase2_merge(self.o[i], self.lse[i], self.partials[i],
                                               self.queries[i], None, 1e-6, out=self.o[i],
                                               stream=stream)

    def dominant_bytes_per_launch(self):
        return self.T * self.phase1_bytes_per_token

    # ---- end to end through the C ABI with host buffers
    def setup_host(self):
        import torch
        self.h_cache = torch.empty(self.cache.shape, dtype=self.cache.dtype, pin_memory=True)
        self.h_cache.copy_(self.cache)
        self.h_parts = torch.empty((self.S - 1,) + tuple(self.partials.shape[1:]),
                                   dtype=self.partials.dtype, pin_memory=True)
        self.h_parts.copy_(self.partials[1:])
        self.h_q = self.queries.cpu().pin_memory()
        self.h_out = torch.empty(self.o.shape, dtype=self.o.dtype, pin_memory=True)
        self.h2d = (self.h_cache.numel() + self.h_parts.numel()) * 2 + self.h_q.numel() * 4
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.partials[1:].copy_(self.h_parts, non_blocking=True)
        self.queries.copy_(self.h_q, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.o, non_blocking=True)

    def run_e2e_pipelined(self, stream, steps):
        """End to end with the steps overlapped the way a streaming caller would
        run them: two device buffer sets, a copy-in, a compute and a copy-out
        stream.  Step k copies its inputs into set k%2 while step k-1 computes
        and step k-2's outputs copy out; every step's copies stay inside the
        timed region.  Returns the elapsed milliseconds."""
        import torch
        from depth_wise_attention_gb300 import attnres
        if not hasattr(self, "e2e_sets"):
            self.e2e_sets = [(self.cache, self.partials, self.queries, self.o, self.lse),
                             tuple(torch.empty_like(x) for x in (self.cache, self.partials, self.queries, self.o,
                                                                 self.lse))]
            dev = self.cache.device
            self.s_in, self.s_comp, self.s_out = (torch.cuda.Stream(dev) for _ in range(3))
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_comp = [torch.cuda.Event() for _ in range(2)]
        ev_out = [torch.cuda.Event() for _ in range(2)]
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for st in (self.s_in, self.s_comp, self.s_out):
            st.wait_event(start)
        for k in range(steps):
            b = k % 2
            cache, parts, q, o, lse = self.e2e_sets[b]
            with torch.cuda.stream(self.s_in):
                if k >= 2:
                    self.s_in.wait_event(ev_comp[b])        # step k-2 has read set b's inputs
                cache.copy_(self.h_cache, non_blocking=True)
                parts[1:].copy_(self.h_parts, non_blocking=True)
                q.copy_(self.h_q, non_blocking=True)
                ev_in[b].record(self.s_in)
            self.s_comp.wait_event(ev_in[b])
            if k >= 2:
                self.s_comp.wait_event(ev_out[b])           # step k-2's outputs have left set b
            attnres.attnres_block_phase1(cache, q, None, 1e-6, o=o, lse=lse, stream=self.s_comp)
            for i in range(1, self.S):
                attnres.attnres_block_phase2_merge(o[i], lse[i], parts[i], q[i], None, 1e-6, out=o[i],
                                                   stream=self.s_comp)
            ev_comp[b].record(self.s_comp)
            self.s_out.wait_event(ev_comp[b])
            with torch.cuda.stream(self.s_out):
                self.h_out.copy_(o, non_blocking=True)
                ev_out[b].record(self.s_out)
        for st in (self.s_in, self.s_comp, self.s_out):
            stream.wait_stream(st)
        end.record(stream)
        torch.cuda.synchronize(self.cache.device)
        return start.elapsed_time(end)

    # ---- oracle on a sample of tokens
    def oracle_sample(self, n_tokens, seed=1):
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        import torch
        it = torch.from_numpy(idx).to(self.cache.device)
        cache = self.cache[:, it, :].float().cpu().numpy().astype(np.float64)
        parts = self.partials[:, it, :].float().cpu().numpy().astype(np.float64)
        q = self.queries.cpu().numpy().astype(np.float64)
        return cache, parts, q

    def run_oracle(self, sample):
        from oracle import oracle
        cache, parts, q = sample
        oracle.block_twophase(cache, parts, q, None, 1e-6)
        return cache.shape[1]


class BlockFusedWorkload(BlockWorkload):
    """Block AttnRes two-phase forward of one block with the intra-block
    partial sum maintained on the way: phase 1, then each layer i >= 2 adds the
    previous layer's output f_{i-1} to the partial and merges it in one fused
    call (the first call starts the partial from f_1).  The layer outputs are
    synthetic inputs [S, T, d] ~ N(0, 1)."""

    def __init__(self, T=32768, d=4096, N=8, S=4, seed=0):
        super().__init__(T, d, N, S, seed, name="block_attnres_two_phase_fused_update")
        b = 2
        first = 4 * d * b + 4          # read f, o, lse; write partial, out
        later = 5 * d * b + 4          # read partial, f, o, lse; write partial, out
        self.merge_bytes_per_token = later
        self.bytes_per_token = self.phase1_bytes_per_token + first + (S - 2) * later

    def setup(self, device):
        import torch
        super().setup(device)
        self.f = self.partials                       # f_1..f_S, one per layer
        self.p = torch.empty((self.T, self.d), dtype=torch.bfloat16, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.attnres_block_phase1(self.cache, self.queries, None, 1e-6, o=self.o, lse=self.lse,
                                     stream=stream)
        if ev is not None:
            ev[1].record(stream)
        for i in range(1, self.S):
            attnres.attnres_block_phase2_update_merge(self.p if i > 1 else None, self.f[i - 1], self.o[i],
                                                      self.lse[i], self.queries[i], None, 1e-6,
                                                      partial_out=self.p, out=self.o[i], stream=stream)

    def setup_host(self):
        super().setup_host()
        self.h_parts = torch_pinned_like(self.f[:self.S - 1])
        self.h2d = (self.h_cache.numel() + self.h_parts.numel()) * 2 + self.h_q.numel() * 4

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.f[:self.S - 1].copy_(self.h_parts, non_blocking=True)
        self.queries.copy_(self.h_q, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.o, non_blocking=True)

    def run_oracle(self, sample):
        from oracle import oracle
        cache, f, q = sample
        o, lse = oracle.block_phase1(cache, q, None, 1e-6)
        p = None
        for i in range(1, self.S):
            p, _ = oracle.block_phase2_update(p, f[i - 1], o[i], lse[i], q[i], None, 1e-6)
        return cache.shape[1]


def torch_pinned_like(t):
    import torch
    h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
    h.copy_(t)
    return h


class ReadBwdWorkload(BlockWorkload):
    """Backward of one Block layer's read in training: the layer's query over
    its 9 sources (the N=8 block reps and the partial sum), bf16, d=4096: the
    sources', the query's and the gain's gradients for a given output
    gradient, in one kernel through a ring of half-row stages.  Sources as the
    Block workload; output gradient ~ N(0, 1)."""

    def __init__(self, T=32768, d=4096, N=8, seed=0):
        super().__init__(T, d, N, 4, seed, name="attnres_read_backward")
        b = 2
        n_src = N + 1
        # read the sources and the output gradient, write the sources' gradients
        self.bytes_per_token = (2 * n_src + 1) * d * b
        self.phase1_bytes_per_token = self.bytes_per_token
        self.launches_per_step = 2            # streaming kernel + the workspace reduction
        self.dominant = "read_bwd_one16_kernel (one query through a ring of half-row stages)"
        self.dominant_src = "read_bwd_one"
        self.profile_tag = f"ncu_read_bwd_d{d}"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} n_src={self.N + 1} n_q=1 T={self.T}"
        c.pop("S", None)
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres, inputs
        T, d, N = self.T, self.d, self.N
        self.src, g = inputs.device_sources(N + 1, T, d, lambda n: 1.0 + n / 2.0 if n < N else 1.0,
                                            seed=self.seed, device=device)
        self.src = self.src.view(N + 1, T, d)
        self.queries = inputs.device_normal((1, d), (16.0 / d) ** 0.5, g, device=device)
        self.gain = torch.ones((d,), dtype=torch.float32, device=device)
        self.dout = torch.randn((1, T, d), generator=g, device=device).to(torch.bfloat16)
        self.dsrc = torch.empty_like(self.src)
        self.dq = torch.empty((1, d), dtype=torch.float32, device=device)
        self.dg = torch.empty((d,), dtype=torch.float32, device=device)
        nb = attnres.attnres_read_bwd_workspace_size(N + 1, T, d, 1, torch.bfloat16)
        self.ws = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)
        self.cache = self.src                   # for oracle_sample

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.attnres_read_bwd(self.src, self.queries, self.dout, self.gain, 1e-6, dsrc=self.dsrc,
                                 dqueries=self.dq, dgain=self.dg, workspace=self.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def setup_host(self):
        self.h_src = torch_pinned_like(self.src)
        self.h_dout = torch_pinned_like(self.dout)
        self.h_out = torch_pinned_like(self.dsrc)
        self.h2d = (self.h_src.numel() + self.h_dout.numel()) * 2
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.src.copy_(self.h_src, non_blocking=True)
        self.dout.copy_(self.h_dout, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.dsrc, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        import torch
        it = torch.from_numpy(idx).to(self.src.device)
        src = self.src[:, it, :].float().cpu().numpy().astype(np.float64)
        dout = self.dout[:, it, :].float().cpu().numpy().astype(np.float64)
        return src, self.queries.cpu().numpy().astype(np.float64), dout

    def run_oracle(self, sample):
        from oracle import oracle
        src, q, dout = sample
        oracle.read_bwd(src, q, dout, None, 1e-6)
        return src.shape[1]


class DeepReadBwdWorkload(ReadBwdWorkload):
    """Backward of the deepest layer of Full AttnRes at depth: one query over
    L = 64 sources ~ N(0, (1 + i/16)^2), bf16, d = 4096, T = 16384, output
    gradient ~ N(0, 1), in the two-kernel form (coefficients over all the
    sources, then channel slices).  Algorithmic bytes per token: the sources
    and the output gradient read, the sources' gradients written."""

    def __init__(self, T=16384, d=4096, L=64, seed=0):
        super().__init__(T, d, L - 1, seed)
        self.name = "attnres_read_backward_depth"
        self.L = L
        self.bytes_per_token = (2 * L + 1) * d * 2
        self.phase1_bytes_per_token = self.bytes_per_token
        self.launches_per_step = 3                      # coefficient kernel, apply kernel, reduction
        self.dominant = "read backward over 64 sources (read_bwd_coef_many_kernel + read_bwd_apply_many_kernel + reduction)"
        self.dominant_src = "read_bwd_many"
        self.profile_tag = f"ncu_read_bwd_depth_d{d}_L{L}"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} n_src={self.L} n_q=1 T={self.T}"
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres, inputs
        T, d, L = self.T, self.d, self.L
        self.src, g = inputs.device_sources(L, T, d, lambda n: 1.0 + n / 16.0, seed=self.seed, device=device)
        self.src = self.src.view(L, T, d)
        self.queries = inputs.device_normal((1, d), (16.0 / d) ** 0.5, g, device=device)
        self.gain = torch.ones((d,), dtype=torch.float32, device=device)
        self.dout = torch.randn((1, T, d), generator=g, device=device).to(torch.bfloat16)
        self.dsrc = torch.empty_like(self.src)
        self.dq = torch.empty((1, d), dtype=torch.float32, device=device)
        self.dg = torch.empty((d,), dtype=torch.float32, device=device)
        nb = attnres.attnres_read_bwd_workspace_size(L, T, d, 1, torch.bfloat16)
        self.ws = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)
        self.cache = self.src


class BlockBwdWorkload(BlockWorkload):
    """Backward of the headline Block step (bf16, d=4096, N=8, S=4): the
    merge backward of each layer (layers 2..4 with their partials, layer 1
    without, which passes its gradient straight to o), then phase 1's backward
    for the four layers' o and lse gradients (one pass of four queries in the
    two-kernel form: row coefficients, then channel slices).
    Algorithmic bytes per token: the merge backward reads o, p and dh and
    writes d_o and d_partial (3 layers), layer 1 copies dh to d_o, and phase
    1's backward reads the 8 sources and the 4 d_o rows and writes the 8
    source gradients once."""

    def __init__(self, T=32768, d=4096, N=8, S=4, seed=0):
        super().__init__(T, d, N, S, seed, name="block_attnres_two_phase_backward")
        b = 2
        self.phase1_bytes_per_token = (2 * N + S) * d * b + S * 4
        self.merge_bwd_bytes_per_token = 5 * d * b + 2 * 4
        self.bytes_per_token = self.phase1_bytes_per_token + (S - 1) * self.merge_bwd_bytes_per_token + 2 * d * b
        # merges (kernel + reduction each), layer 1's copy, phase 1's backward
        # (coefficient kernel, apply kernel, reduction)
        self.launches_per_step = (S - 1) * 2 + 1 + 3
        self.dominant = "phase-1 backward (read_bwd_coef_kernel + read_bwd_apply_kernel + reduction)"
        self.dominant_src = "read_bwd_split"
        self.profile_tag = f"ncu_block_bwd_phase1_d{d}"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} N={self.N} S={self.S} T={self.T}"
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres
        super().setup(device)
        T, d, N, S = self.T, self.d, self.N, self.S
        attnres.attnres_block_phase1(self.cache, self.queries, None, 1e-6, o=self.o, lse=self.lse)
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 7)
        self.dh = torch.randn((S, T, d), generator=g, device=device).to(torch.bfloat16)
        self.d_o = torch.empty_like(self.o)
        self.d_lse = torch.empty_like(self.lse)
        self.d_parts = torch.empty_like(self.partials)
        self.dsrc = torch.empty_like(self.cache)
        self.dq2 = torch.empty((S, d), dtype=torch.float32, device=device)
        self.dg2 = torch.empty((S, d), dtype=torch.float32, device=device)
        self.dq1 = torch.empty((S, d), dtype=torch.float32, device=device)
        self.dg1 = torch.empty((d,), dtype=torch.float32, device=device)
        nb = attnres.attnres_block_phase2_bwd_workspace_size(T, d, torch.bfloat16)
        self.ws2 = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)
        nb = attnres.attnres_read_bwd_workspace_size(N, T, d, S, torch.bfloat16)
        self.ws1 = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        for s_ in range(self.S):
            attnres.attnres_block_phase2_bwd(self.o[s_], self.lse[s_], self.partials[s_] if s_ > 0 else None,
                                             self.queries[s_], self.dh[s_], None, 1e-6, d_o=self.d_o[s_],
                                             d_lse=self.d_lse[s_], d_partial=self.d_parts[s_],
                                             dquery=self.dq2[s_], dgain=self.dg2[s_], workspace=self.ws2,
                                             stream=stream)
        if ev is not None:
            ev[0].record(stream)
        attnres.attnres_block_phase1_bwd(self.cache, self.queries, self.d_o, self.d_lse, None, 1e-6,
                                         dsrc=self.dsrc, dqueries=self.dq1, dgain=self.dg1, workspace=self.ws1,
                                         stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def setup_host(self):
        import torch
        self.h_cache = torch_pinned_like(self.cache)
        self.h_parts = torch_pinned_like(self.partials)
        self.h_dh = torch_pinned_like(self.dh)
        self.h_out = torch_pinned_like(self.dsrc)
        self.h2d = (self.h_cache.numel() + self.h_parts.numel() + self.h_dh.numel()) * 2
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.partials.copy_(self.h_parts, non_blocking=True)
        self.dh.copy_(self.h_dh, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.dsrc, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        import torch
        it = torch.from_numpy(idx).to(self.cache.device)
        c = self.cache[:, it, :].float().cpu().numpy().astype(np.float64)
        p = self.partials[:, it, :].float().cpu().numpy().astype(np.float64)
        h = self.dh[:, it, :].float().cpu().numpy().astype(np.float64)
        return c, p, h, self.queries.cpu().numpy().astype(np.float64)

    def run_oracle(self, sample):
        from oracle import oracle
        c, p, h, q = sample
        o, lse = oracle.block_phase1(c, q, None, 1e-6)
        d_o, d_lse = np.empty_like(o), np.empty_like(lse)
        for s_ in range(self.S):
            r = oracle.block_phase2_bwd(o[s_], lse[s_], p[s_] if s_ > 0 else None, q[s_], h[s_], None, 1e-6)
            d_o[s_], d_lse[s_] = r[0], r[1]
        oracle.block_phase1_bwd(c, q, d_o, d_lse, None, 1e-6)
        return c.shape[1]


class MharBwdWorkload(ReadBwdWorkload):
    """Backward of the MHAR read at the MHAR workload's sizes: 4 queries of
    H=8 heads over N=8 sources, bf16, d=4096: the sources', the queries' and
    the gain's gradients for a given output gradient, in the two-kernel form
    (per-head row coefficients, then channel slices).  The algorithmic bytes
    are one pass's: read the sources and the 4 output gradients, write the
    sources' gradients."""

    def __init__(self, T=131072, d=4096, N=8, H=8, n_q=4, seed=0):
        BlockWorkload.__init__(self, T, d, N, 4, seed, name="mhar_read_backward")
        b = 2
        self.H, self.n_q = H, n_q
        self.bytes_per_token = (2 * N + n_q) * d * b
        self.phase1_bytes_per_token = self.bytes_per_token
        self.launches_per_step = 3                      # coefficient kernel, apply kernel, reduction
        self.dominant = "mhar read backward (read_bwd_coef_kernel per head + read_bwd_apply_kernel + reduction)"
        self.dominant_src = "read_bwd_split"
        self.profile_tag = f"ncu_mhar_bwd_d{d}_H{H}"

    def config(self):
        c = BlockWorkload.config(self)
        c["workload"] = f"{self.name} bf16 d={self.d} H={self.H} n_src={self.N} n_q={self.n_q} T={self.T}"
        c.pop("S", None)
        c["H"], c["n_q"] = self.H, self.n_q
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres, inputs
        T, d, N, H, n_q = self.T, self.d, self.N, self.H, self.n_q
        self.src, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=self.seed, device=device)
        self.src = self.src.view(N, T, d)
        self.queries = inputs.device_normal((n_q, H, d // H), (16.0 / (d // H)) ** 0.5, g, device=device)
        self.gain = torch.ones((d,), dtype=torch.float32, device=device)
        self.dout = torch.randn((n_q, T, d), generator=g, device=device).to(torch.bfloat16)
        self.dsrc = torch.empty_like(self.src)
        self.dq = torch.empty((n_q, H, d // H), dtype=torch.float32, device=device)
        self.dg = torch.empty((d,), dtype=torch.float32, device=device)
        nb = attnres.mhar_read_bwd_workspace_size(N, T, d, H, n_q, torch.bfloat16)
        self.ws = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)
        self.cache = self.src

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.mhar_read_bwd(self.src, self.queries, self.dout, self.gain, 1e-6, dsrc=self.dsrc,
                              dqueries=self.dq, dgain=self.dg, workspace=self.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def run_oracle(self, sample):
        from oracle import oracle
        src, q, dout = sample
        oracle.mhar_bwd(src, q, dout, None, 1e-6)
        return src.shape[1]


class DecodeWorkload(BlockWorkload):
    """Decode-shaped Block AttnRes two-phase forward: a block (phase 1 + 3
    merges) over T=16 tokens, bf16, d=4096, N=8, S=4.  Each step reads its own
    set of inputs; the sets rotate through more than L2 holds, so every step
    starts from HBM.  A step's four launches are captured once per input set in
    a CUDA graph and replayed (decode latency is launch-bound otherwise).  The
    metric is tokens/s; ms_per_step is the latency of one block."""

    def __init__(self, T=16, d=4096, N=8, S=4, seed=0, sets=160):
        super().__init__(T, d, N, S, seed, name="block_attnres_two_phase_decode")
        self.sets = sets
        self.k = 0
        self.dominant = "decode step (graph: depth_read_decode_kernel + 3 merges)"
        self.dominant_src = "depth_read_decode"
        self.profile_tag = f"ncu_decode_d{d}_T{T}"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} N={self.N} S={self.S} T={self.T}"
        c["l2"] = f"{self.sets} rotating input sets ({self.sets * self.bytes_per_token * self.T / 1e6:.0f} MB > L2)"
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        T, d, N, S = self.T, self.d, self.N, self.S
        caches, g = inputs.device_sources(N * self.sets, T, d, lambda n: 1.0 + (n % N) / 2.0, seed=self.seed,
                                          device=device)
        self.caches = caches.view(self.sets, N, T, d)
        self.queries = inputs.device_normal((S, d), (16.0 / d) ** 0.5, g, device=device)
        self.parts = torch.randn((self.sets, S, T, d), generator=g, device=device).to(torch.bfloat16)
        self.os = torch.empty((self.sets, S, T, d), dtype=torch.bfloat16, device=device)
        self.lses = torch.empty((self.sets, S, T), dtype=torch.float32, device=device)
        self.cache, self.partials, self.o, self.lse = self.caches[0], self.parts[0], self.os[0], self.lses[0]
        # one graph per input set, captured after a warm-up run of each path
        cap = torch.cuda.Stream(device)
        with torch.cuda.stream(cap):
            self._launch(0, cap)
        torch.cuda.synchronize(device)
        self.graphs = []
        for j in range(self.sets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cap):
                self._launch(j, cap)
            self.graphs.append(g)
        torch.cuda.synchronize(device)

    def _launch(self, j, stream):
        from depth_wise_attention_gb300 import attnres
        cache, parts, o, lse = self.caches[j], self.parts[j], self.os[j], self.lses[j]
        attnres.attnres_block_phase1(cache, self.queries, None, 1e-6, o=o, lse=lse, stream=stream)
        for i in range(1, self.S):
            attnres.attnres_block_phase2_merge(o[i], lse[i], parts[i], self.queries[i], None, 1e-6, out=o[i],
                                               stream=stream)

    def dominant_bytes_per_launch(self):
        return self.T * self.bytes_per_token

    def step(self, stream, ev=None):
        j = self.k % self.sets
        self.k += 1
        if ev is not None:
            ev[0].record(stream)
        self.graphs[j].replay()
        if ev is not None:
            ev[1].record(stream)

    def step_e2e(self, stream):
        self.k = 0
        super().step_e2e(stream)


class MharWorkload(BlockWorkload):
    """MHAR read: S=4 queries x H=8 heads over N=8 block reps (no phase 2)."""

    def __init__(self, T=131072, d=4096, N=8, S=4, H=8, seed=0):
        super().__init__(T, d, N, S, seed, name="mhar_block_diagonal_read")
        self.H = H
        self.bytes_per_token = N * d * 2 + S * d * 2
        self.phase1_bytes_per_token = self.bytes_per_token
        self.launches_per_step = 1
        self.dominant = "depth_read_mma_kernel (MHAR)"
        self.dominant_src = "depth_read_mma"
        self.profile_tag = f"ncu_mhar_d{d}_H{H}"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} H={self.H} N={self.N} S={self.S} T={self.T}"
        c["H"] = self.H
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        T, d, N, S, H = self.T, self.d, self.N, self.S, self.H
        self.cache, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=self.seed,
                                              device=device)
        self.cache = self.cache.view(N, T, d)
        self.queries = inputs.device_normal((S, H, d // H), (16.0 / (d // H)) ** 0.5, g, device=device)
        self.o = torch.empty((S, T, d), dtype=torch.bfloat16, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.mhar_fwd(self.cache, self.queries, None, 1e-6, out=self.o, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def setup_host(self):
        import torch
        self.h_cache = torch.empty(self.cache.shape, dtype=self.cache.dtype, pin_memory=True)
        self.h_cache.copy_(self.cache)
        self.h_q = self.queries.cpu().pin_memory()
        self.h_out = torch.empty(self.o.shape, dtype=self.o.dtype, pin_memory=True)
        self.h2d = self.h_cache.numel() * 2 + self.h_q.numel() * 4
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.queries.copy_(self.h_q, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.o, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        import torch
        it = torch.from_numpy(idx).to(self.cache.device)
        return (self.cache[:, it, :].float().cpu().numpy().astype(np.float64),
                self.queries.cpu().numpy().astype(np.float64))

    def run_oracle(self, sample):
        from oracle import oracle
        src, q = sample
        oracle.mhar(src, q, None, 1e-6)
        return src.shape[1]


class MharBlockWorkload(MharWorkload):
    """MHAR inside the two-phase Block schedule at the MHAR size: phase 1 is
    the MHAR read of the S=4 queries x H=8 heads over the N=8 cached reps
    with each head's lse; layers 2..4 then merge their partial sums head by
    head (mhar_phase2_merge, in place)."""

    def __init__(self, T=131072, d=4096, N=8, S=4, H=8, seed=0):
        super().__init__(T, d, N, S, H, seed)
        self.name = "mhar_two_phase_block"
        b = 2
        self.phase1_bytes_per_token = N * d * b + S * d * b + S * H * 4
        self.bytes_per_token = self.phase1_bytes_per_token + (S - 1) * (3 * d * b + H * 4)
        self.launches_per_step = 1 + (S - 1)
        self.dominant = "depth_read_mma_kernel (MHAR phase 1 with per-head lse)"
        self.profile_tag = f"ncu_mhar_two_phase_d{d}_H{H}"

    def setup(self, device):
        import torch
        super().setup(device)
        T, d, S, H = self.T, self.d, self.S, self.H
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 11)
        self.lse = torch.empty((S, H, T), dtype=torch.float32, device=device)
        self.partials = torch.randn((S, T, d), generator=g, device=device).to(torch.bfloat16)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.mhar_fwd(self.cache, self.queries, None, 1e-6, out=self.o, lse=self.lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        for i in range(1, self.S):
            attnres.mhar_phase2_merge(self.o[i], self.lse[i], self.partials[i], self.queries[i], None, 1e-6,
                                      out=self.o[i], stream=stream)

    def setup_host(self):
        super().setup_host()
        self.h_parts = torch_pinned_like(self.partials[1:])
        self.h2d += self.h_parts.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.partials[1:].copy_(self.h_parts, non_blocking=True)
        self.queries.copy_(self.h_q, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.o, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        import torch
        it = torch.from_numpy(idx).to(self.cache.device)
        return (self.cache[:, it, :].float().cpu().numpy().astype(np.float64),
                self.partials[:, it, :].float().cpu().numpy().astype(np.float64),
                self.queries.cpu().numpy().astype(np.float64))

    def run_oracle(self, sample):
        from oracle import oracle
        src, parts, q = sample
        o, lse = oracle.mhar(src, q, None, 1e-6, want_lse=True)
        for i in range(1, self.S):
            oracle.mhar_phase2(o[i], lse[i], parts[i], q[i], None, 1e-6)
        return src.shape[1]


class MsarWorkload(BlockWorkload):
    """MSAR fused stream expansion + per-stream read + H^pre mixer."""

    def __init__(self, T=32768, d=4096, N=8, seed=0):
        super().__init__(T, d, N, 4, seed, name="msar_fused_read")
        self.ks = (4, 8, 12)
        self.bytes_per_token = N * d * 2 + d * 2
        self.phase1_bytes_per_token = self.bytes_per_token
        self.launches_per_step = 1
        # bf16 with kernel sizes 4/8/12 and d a multiple of 256 runs the
        # tile-batched kernel (one cluster exchange per tile of tokens)
        self.dominant = "msar_tile_kernel"
        self.dominant_src = "msar_tile"
        self.profile_tag = f"ncu_msar_tile_d{d}"
        # The read is bound by fp32 arithmetic, not HBM: its roofline is the
        # CUDA-core FMA rate.  Multiply-adds per token: the causal convolutions
        # (N sources x d channels x (4+8+12) taps), per (source, stream) the
        # sum of squares and the query dot (N x 4 x 2 x d), the weighted sums
        # (4 x N x d), the mixer's sum of squares (4d), projection (4d x 4) and
        # the output sum (4 x d).
        self.fma_per_token = N * d * sum(self.ks) + N * 4 * 2 * d + 4 * N * d + 4 * d + 4 * d * 4 + 4 * d

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} N={self.N} m=4 k=4/8/12 T={self.T}"
        c.pop("S", None)
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        T, d, N = self.T, self.d, self.N
        self.cache, g = inputs.device_sources(N, T, d, lambda n: 1.0 + n / 2.0, seed=self.seed,
                                              device=device)
        self.cache = self.cache.view(N, T, d)
        self.queries = inputs.device_normal((4, d), (16.0 / d) ** 0.5, g, device=device)
        self.conv_w = torch.cat([inputs.device_normal((d * k,), (1.0 / k) ** 0.5, g, device=device)
                                 for k in self.ks])
        self.mix_w = inputs.device_normal((4 * d, 4), (1.0 / (4 * d)) ** 0.5, g, device=device)
        self.out = torch.empty((T, d), dtype=torch.bfloat16, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.msar_expand_fwd(self.cache, self.ks, self.conv_w, self.queries, None, 1e-6, None,
                                self.mix_w, 1e-6, out=self.out, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def setup_host(self):
        import torch
        self.h_cache = torch.empty(self.cache.shape, dtype=self.cache.dtype, pin_memory=True)
        self.h_cache.copy_(self.cache)
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        self.h2d = self.h_cache.numel() * 2
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.out, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        # windows of 12 rows ending at each sampled token (the causal receptive field)
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        wins = []
        for t in idx:
            lo = max(0, int(t) - 11)
            wins.append(self.cache[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64))
        return (wins, self.conv_w.cpu().numpy().astype(np.float64),
                self.queries.cpu().numpy().astype(np.float64),
                self.mix_w.cpu().numpy().astype(np.float64))

    def run_oracle(self, sample):
        from oracle import oracle
        wins, cw, q, mw = sample
        for w in wins:
            oracle.msar(w, self.ks, cw, q, None, 1e-6, None, mw, 1e-6)
        return len(wins)


class MsarBwdWorkload(MsarWorkload):
    """Backward of the MSAR read at the MSAR workload's sizes (N=8 sources,
    bf16, d=4096, k=4/8/12, T=32768) for a dense output gradient dh ~ N(0, 1):
    the sources', conv kernels', stream queries', gain's and mixer's
    gradients.  One step is the whole chain (streams, 4 stream reads, mixer
    backward and its sums, 4 read backwards, the convolutions' transpose and
    the fixed-order sums).  Its roofline is the CUDA-core FMA rate of the
    arithmetic the backward cannot avoid, per token: the convolutions once
    forward and twice back (N d k_tot x 3), the 4 stream reads (N d x 3 each:
    sum of squares, query dot, weighted sum), their backward (N d x 7 each:
    the read again, dh . v, U, dsrc), and the mixer (4d x 16)."""

    def __init__(self, T=32768, d=4096, N=8, seed=0):
        super().__init__(T, d, N, seed)
        self.name = "msar_read_backward"
        b = 2
        # read the sources and dh, write the sources' gradients
        self.bytes_per_token = (2 * N + 1) * d * b
        self.phase1_bytes_per_token = self.bytes_per_token
        self.launches_per_step = 1 + 4 + 3 + 2 + 4 * 2 + 1 + 2
        self.dominant = "msar backward (whole chain)"
        self.dominant_src = "msar_bwd"
        self.profile_tag = f"ncu_msar_bwd_d{d}"
        self.fma_per_token = N * d * sum(self.ks) * 3 + 4 * N * d * 3 + 4 * N * d * 7 + 4 * d * 16

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres
        super().setup(device)
        T, d, N = self.T, self.d, self.N
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 7)
        self.dh = torch.randn((T, d), generator=g, device=device).to(torch.bfloat16)
        self.dsrc = torch.empty_like(self.cache)
        f32 = dict(dtype=torch.float32, device=device)
        self.grads = (torch.empty_like(self.conv_w), torch.empty((4, d), **f32), torch.empty((d,), **f32),
                      torch.empty((4 * d,), **f32), torch.empty((4 * d, 4), **f32))
        nb = attnres.msar_expand_bwd_workspace_size(N, T, d, torch.bfloat16, self.ks)
        self.ws = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.msar_expand_bwd(self.cache, self.ks, self.conv_w, self.queries, self.dh, None, 1e-6, None,
                                self.mix_w, 1e-6, dsrc=self.dsrc, grads=self.grads, workspace=self.ws,
                                stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def setup_host(self):
        self.h_cache = torch_pinned_like(self.cache)
        self.h_dh = torch_pinned_like(self.dh)
        self.h_out = torch_pinned_like(self.dsrc)
        self.h2d = (self.h_cache.numel() + self.h_dh.numel()) * 2
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.dh.copy_(self.h_dh, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.dsrc, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        # per sampled token t: the 12-row causal window ending at t and dh on row t alone
        wins, cw, q, mw = super().oracle_sample(n_tokens, seed)
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        dhs = []
        for w, t in zip(wins, idx):
            dw = np.zeros(w.shape[1:])
            dw[-1] = self.dh[int(t)].float().cpu().numpy()
            dhs.append(dw)
        return wins, dhs, cw, q, mw

    def run_oracle(self, sample):
        from oracle import oracle
        wins, dhs, cw, q, mw = sample
        for w, dw in zip(wins, dhs):
            oracle.msar_bwd(w, self.ks, cw, q, dw, None, 1e-6, None, mw, 1e-6)
        return len(wins)


class MsarBwdChunkedWorkload(MsarBwdWorkload):
    """The MSAR backward in chunks of 4096 tokens (msar_expand_bwd_chunk), each
    given the 11 source rows before it, in order: the first chunk writes the
    parameter gradients and the later ones add into them, and each chunk adds
    its share of the history rows' gradient.  The workspace is sized for one
    chunk (about an eighth of the one-call backward's)."""

    def __init__(self, T=32768, d=4096, N=8, seed=0, chunk=4096):
        super().__init__(T, d, N, seed)
        self.name = "msar_read_backward_chunked"
        self.chunk = chunk
        self.launches_per_step *= (T + chunk - 1) // chunk
        self.dominant = "msar backward, chunked (whole chain per chunk)"
        self.profile_tag = f"ncu_msar_bwd_chunked_d{d}"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} N={self.N} m=4 k=4/8/12 T={self.T} chunk={self.chunk}"
        c["chunk"] = self.chunk
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres
        super().setup(device)
        del self.ws
        nb = attnres.msar_expand_bwd_workspace_size(self.N, self.chunk, self.d, torch.bfloat16, self.ks)
        self.ws = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)
        self.workspace_bytes = nb

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        hist = max(self.ks) - 1
        if ev is not None:
            ev[0].record(stream)
        for c0 in range(0, self.T, self.chunk):
            c1 = min(self.T, c0 + self.chunk)
            h = min(hist, c0)
            attnres.msar_expand_bwd_chunk(self.cache[:, c0 - h:c1], h, self.ks, self.conv_w, self.queries,
                                          self.dh[c0:c1], self.dsrc[:, c0 - h:c1], self.grads, c0 > 0, None, 1e-6,
                                          None, self.mix_w, 1e-6, workspace=self.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)


class MsarBwdPerSourceWorkload(MsarBwdWorkload):
    """The MSAR backward with each of the N=8 sources' own conv kernels
    (msar_expand_bwd_ps): kernels ~ N(0, 1/k) per source, each source's
    kernel gradient on its own."""

    def __init__(self, T=32768, d=4096, N=8, seed=0):
        super().__init__(T, d, N, seed)
        self.name = "msar_read_backward_per_source_kernels"
        self.profile_tag = f"ncu_msar_bwd_per_source_d{d}"

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        super().setup(device)
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 5)
        self.conv_w = torch.stack([torch.cat([inputs.device_normal((self.d * k,), (1.0 / k) ** 0.5, g, device=device)
                                              for k in self.ks]) for _ in range(self.N)])
        self.grads = (torch.empty_like(self.conv_w),) + self.grads[1:]

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.msar_expand_bwd_ps(self.cache, self.ks, self.conv_w, self.queries, self.dh, None, 1e-6, None,
                                   self.mix_w, 1e-6, dsrc=self.dsrc, grads=self.grads, workspace=self.ws,
                                   stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def oracle_sample(self, n_tokens, seed=1):
        wins, dhs, _, q, mw = super().oracle_sample(n_tokens, seed)
        return wins, dhs, self.conv_w.cpu().numpy().astype(np.float64), q, mw

    def run_oracle(self, sample):
        from oracle import oracle
        wins, dhs, cw, q, mw = sample
        for w, dw in zip(wins, dhs):
            oracle.msar_ps_bwd(w, self.ks, cw, q, dw, None, 1e-6, None, mw, 1e-6)
        return len(wins)


class MsarWsWorkload(MsarWorkload):
    """The MSAR read through the workspace chain (msar_expand_fwd_ws): the
    conv streams written once, one read per stream, the sliced mixer; same
    inputs and outputs as the fused read."""

    def __init__(self, T=32768, d=4096, N=8, seed=0):
        super().__init__(T, d, N, seed)
        self.name = "msar_read_workspace_chain"
        self.launches_per_step = 1 + 4 + 2
        self.dominant = "msar read, workspace chain (streams + 4 reads + mixer)"
        self.dominant_src = "msar_bwd"
        self.profile_tag = f"ncu_msar_ws_d{d}"

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres
        super().setup(device)
        nb = attnres.msar_expand_fwd_ws_workspace_size(self.N, self.T, self.d, torch.bfloat16)
        self.ws = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.msar_expand_fwd_ws(self.cache, self.ks, self.conv_w, self.queries, None, 1e-6, None, self.mix_w,
                                   1e-6, out=self.out, workspace=self.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)


class MsarBlockWorkload(MsarWorkload):
    """MSAR inside the two-phase Block schedule: one block of S=4 layers over
    N=8 cached sources, bf16, d=4096.  One step = phase 1 (every source
    expanded once, read by the 4 x 4 stream queries of the block's layers)
    + 4 phase-2 calls (layers 2..4 merge their partial sums; layer 1 mixes
    the phase-1 state alone).  The dominant kernel is phase 1; its roofline is
    the CUDA-core FMA rate."""

    def __init__(self, T=32768, d=4096, N=8, S=4, seed=0):
        MsarWorkload.__init__(self, T, d, N, seed)
        self.name = "msar_two_phase_block"
        self.S = S
        b = 2
        # phase 1: read the cached sources, write o (S x 4 streams) and lse
        self.phase1_bytes_per_token = N * d * b + S * 4 * d * b + S * 4 * 4
        # phase 2 per layer: read o and lse (and the partial for layers 2..S), write h
        self.bytes_per_token = (self.phase1_bytes_per_token + S * (4 * d * b + 4 * 4 + d * b)
                                + (S - 1) * d * b)
        self.launches_per_step = 1 + S
        self.dominant = "msar_phase1_kernel"
        self.dominant_src = "msar_phase1"
        self.profile_tag = f"ncu_msar_phase1_d{d}"
        # phase 1 multiply-adds per token: the convolutions of the N sources,
        # per (source, stream) the sum of squares and one query dot per layer,
        # and per (layer, stream) the weighted sum over the sources
        self.fma_per_token = N * d * sum(self.ks) + N * 4 * d + S * N * 4 * d + S * 4 * N * d

    def config(self):
        c = MsarWorkload.config(self)
        c["workload"] = f"{self.name} bf16 d={self.d} N={self.N} S={self.S} m=4 k=4/8/12 T={self.T}"
        c["S"] = self.S
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        MsarWorkload.setup(self, device)
        T, d, S = self.T, self.d, self.S
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 1)
        self.queries = inputs.device_normal((S, 4, d), (16.0 / d) ** 0.5, g, device=device)
        self.parts = torch.randn((S, T, d), generator=g, device=device).to(torch.bfloat16)
        self.o = torch.empty((S, 4, T, d), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((S, 4, T), dtype=torch.float32, device=device)
        self.outs = torch.empty((S, T, d), dtype=torch.bfloat16, device=device)
        self.out = self.outs

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.msar_block_phase1(self.cache, self.ks, self.conv_w, self.queries, None, 1e-6, o=self.o,
                                  lse=self.lse, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        for s_ in range(self.S):
            attnres.msar_block_phase2(self.o[s_], self.lse[s_], self.parts[s_] if s_ > 0 else None, self.ks,
                                      self.conv_w, self.queries[s_], None, 1e-6, None, self.mix_w, 1e-6,
                                      out=self.outs[s_], stream=stream)

    def setup_host(self):
        import torch
        MsarWorkload.setup_host(self)
        self.h_parts = torch.empty((self.S - 1,) + tuple(self.parts.shape[1:]), dtype=self.parts.dtype,
                                   pin_memory=True)
        self.h_parts.copy_(self.parts[1:])
        self.h2d += self.h_parts.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.parts[1:].copy_(self.h_parts, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.outs, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        wins = []
        for t in idx:
            lo = max(0, int(t) - 11)
            wins.append((self.cache[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64),
                         self.parts[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)))
        return (wins, self.conv_w.cpu().numpy().astype(np.float64),
                self.queries.cpu().numpy().astype(np.float64),
                self.mix_w.cpu().numpy().astype(np.float64))

    def run_oracle(self, sample):
        from oracle import oracle
        wins, cw, q, mw = sample
        for cached, parts in wins:
            o, lse = oracle.msar_phase1(cached, self.ks, cw, q, None, 1e-6)
            for s_ in range(self.S):
                oracle.msar_phase2(o[s_], lse[s_], parts[s_] if s_ > 0 else None, self.ks, cw, q[s_], None,
                                   1e-6, None, mw, 1e-6)
        return len(wins)


class MsarPerSourceWorkload(MsarWorkload):
    """The MSAR read with each of the N=8 sources' own conv kernels
    (msar_expand_fwd_ps): kernels ~ N(0, 1/k) per source, read through L2."""

    def __init__(self, T=32768, d=4096, N=8, seed=0):
        super().__init__(T, d, N, seed)
        self.name = "msar_per_source_kernels"
        self.dominant = "msar_kernel (per-source kernels)"
        self.dominant_src = "msar"
        self.profile_tag = f"ncu_msar_per_source_d{d}"

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        super().setup(device)
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 5)
        self.conv_w = torch.stack([torch.cat([inputs.device_normal((self.d * k,), (1.0 / k) ** 0.5, g, device=device)
                                              for k in self.ks]) for _ in range(self.N)])

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.msar_expand_fwd_ps(self.cache, self.ks, self.conv_w, self.queries, None, 1e-6, None, self.mix_w,
                                   1e-6, out=self.out, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def run_oracle(self, sample):
        from oracle import oracle
        wins, cw, q, mw = sample
        for w in wins:
            oracle.msar_ps(w, self.ks, cw, q, None, 1e-6, None, mw, 1e-6)
        return len(wins)


class MsarChunkedWorkload(MsarWorkload):
    """Chunked prefill of the MSAR read: the T=32768 tokens in chunks of
    4096, each call given the 11 rows before its chunk as the causal history
    (msar_expand_fwd_chunk on strided views of the sources, nothing copied).
    Same outputs as the one-call read, bit for bit."""

    def __init__(self, T=32768, d=4096, N=8, seed=0, chunk=4096):
        super().__init__(T, d, N, seed)
        self.name = "msar_chunked_prefill"
        self.chunk = chunk
        self.launches_per_step = (T + chunk - 1) // chunk
        self.dominant = "msar_tile_kernel (all chunks)"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} N={self.N} m=4 k=4/8/12 T={self.T} chunk={self.chunk}"
        c["chunk"] = self.chunk
        return c

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        hist = max(self.ks) - 1
        if ev is not None:
            ev[0].record(stream)
        for c0 in range(0, self.T, self.chunk):
            c1 = min(self.T, c0 + self.chunk)
            h = min(hist, c0)
            attnres.msar_expand_fwd_chunk(self.cache[:, c0 - h:c1], h, self.ks, self.conv_w, self.queries, None,
                                          1e-6, None, self.mix_w, 1e-6, out=self.out[c0:c1], stream=stream)
        if ev is not None:
            ev[1].record(stream)


class FullDepthWorkload(BlockWorkload):
    """Full AttnRes at depth: 64 layers, layer l reads sources 0..l-1."""

    def __init__(self, T=16384, d=4096, L=64, seed=0):
        super().__init__(T, d, 8, 4, seed, name="full_attnres_depth")
        self.L = L
        self.bytes_per_token = sum((l + 1) * d * 2 for l in range(1, L + 1))
        self.phase1_bytes_per_token = (L + 1) * d * 2           # the deepest layer's read
        self.launches_per_step = L
        self.dominant = "depth_read_kernel (Full, layer 64: the general kernel, 6-source chunks)"
        self.dominant_src = "depth_read"
        self.profile_tag = f"ncu_full_depth_d{d}"

    def config(self):
        c = super().config()
        c["workload"] = f"{self.name} bf16 d={self.d} L={self.L} T={self.T}"
        c.pop("S", None)
        c.pop("N", None)
        c["L"] = self.L
        return c

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import inputs
        T, d, L = self.T, self.d, self.L
        self.cache, g = inputs.device_sources(L, T, d, lambda i: 1.0 + i / 16.0, seed=self.seed,
                                              device=device)
        self.cache = self.cache.view(L, T, d)
        self.queries = inputs.device_normal((L, d), (16.0 / d) ** 0.5, g, device=device)
        self.out = torch.empty((T, d), dtype=torch.bfloat16, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        for l in range(1, self.L + 1):
            if ev is not None and l == self.L:
                ev[0].record(stream)
            attnres.attnres_full_fwd(self.cache[:l], self.queries[l - 1], None, 1e-6, out=self.out,
                                     stream=stream)
            if ev is not None and l == self.L:
                ev[1].record(stream)

    def setup_host(self):
        import torch
        self.h_cache = torch.empty(self.cache.shape, dtype=self.cache.dtype, pin_memory=True)
        self.h_cache.copy_(self.cache)
        self.h_out = torch.empty(self.out.shape, dtype=self.out.dtype, pin_memory=True)
        self.h2d = self.h_cache.numel() * 2
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.out, non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        import torch
        it = torch.from_numpy(idx).to(self.cache.device)
        return (self.cache[:, it, :].float().cpu().numpy().astype(np.float64),
                self.queries.cpu().numpy().astype(np.float64))

    def run_oracle(self, sample):
        from oracle import oracle
        src, q = sample
        for l in range(1, self.L + 1):
            oracle.full(src[:l], q[l - 1], None, 1e-6)
        return src.shape[1]


class MsarBlockWsWorkload(MsarBlockWorkload):
    """The MSAR two-phase block through the workspace chains: phase 1
    (msar_block_phase1_ws: the cached sources' streams written once, each
    stream read by its 4 layers' queries with the tensor-core read) and
    phase 2 per layer (msar_block_phase2_ws: the partial's streams, one Block
    merge per stream, the sliced mixer).  Same inputs and outputs as the
    fused schedule."""

    def __init__(self, T=32768, d=4096, N=8, S=4, seed=0):
        super().__init__(T, d, N, S, seed)
        self.name = "msar_two_phase_block_workspace_chain"
        self.launches_per_step = 1 + 4 + 2 + (S - 1) * (1 + 4 + 2)
        self.dominant = "msar phase 1, workspace chain (streams + 4 reads of 4 queries)"
        self.dominant_src = "msar_bwd"
        self.profile_tag = f"ncu_msar_phase1_ws_d{d}"

    def setup(self, device):
        import torch
        from depth_wise_attention_gb300 import attnres
        super().setup(device)
        nb = attnres.msar_block_phase1_ws_workspace_size(self.N, self.T, self.d, torch.bfloat16, self.S)
        self.ws = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)
        nb = attnres.msar_block_phase2_ws_workspace_size(self.T, self.d, torch.bfloat16)
        self.ws2 = torch.empty(((nb + 3) // 4,), dtype=torch.float32, device=device)

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if ev is not None:
            ev[0].record(stream)
        attnres.msar_block_phase1_ws(self.cache, self.ks, self.conv_w, self.queries, None, 1e-6, o=self.o,
                                     lse=self.lse, workspace=self.ws, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        for s_ in range(self.S):
            attnres.msar_block_phase2_ws(self.o[s_], self.lse[s_], self.parts[s_] if s_ > 0 else None, self.ks,
                                         self.conv_w, self.queries[s_], None, 1e-6, None, self.mix_w, 1e-6,
                                         out=self.outs[s_], workspace=self.ws2, stream=stream)


class MsarBlockBwdWorkload(MsarBlockWorkload):
    """Backward of one MSAR two-phase block (N=8 cached sources, S=4 layers,
    bf16, d=4096, T=32768) for dense output gradients dh ~ N(0, 1) of every
    layer: phase 2's backward per layer (layers 2..4 with their partials,
    layer 1 without), then phase 1's backward with the layers' state
    gradients, as a training step would run it.  The phase-1 state is
    computed once, in the first warm-up step.  Algorithmic bytes per token: the cached sources,
    the partials, the state (o, lse), dh read; the sources' and the partials'
    gradients written."""

    def __init__(self, T=32768, d=4096, N=8, S=4, seed=0):
        super().__init__(T, d, N, S, seed)
        self.name = "msar_two_phase_block_backward"
        b = 2
        self.bytes_per_token = ((N + (S - 1) + S * 4 + S) * d * b + S * 4 * 4 + (N + (S - 1)) * d * b)
        self.phase1_bytes_per_token = self.bytes_per_token
        self.fma_per_token = None
        # phase 2 with a partial: streams 1, merges 4, mixer 3 + 2 sums, merge backwards 4 x 2, conv 1 + 2 sums;
        # without: mixer 3 + 2; phase 1: streams 1, 4 read backwards x 2, conv 1 + 2 sums
        self.launches_per_step = (S - 1) * 21 + 5 + 12
        self.dominant = "msar two-phase block backward (4 x phase 2 backward + phase 1 backward)"
        self.dominant_src = "msar_bwd"
        self.profile_tag = f"ncu_msar_block_bwd_d{d}"

    def setup(self, device):
        import torch
        super().setup(device)
        T, d, S = self.T, self.d, self.S
        g = torch.Generator(device=device)
        g.manual_seed(self.seed + 9)
        self.dh = torch.randn((S, T, d), generator=g, device=device).to(torch.bfloat16)
        self.device = device
        self.ready = False

    def _prepare(self):
        # the CUDA arm's state: the block's phase-1 state and the output and
        # workspace buffers (made in the first, untimed warm-up step)
        import torch
        from depth_wise_attention_gb300 import attnres
        T, d, S, N, device = self.T, self.d, self.S, self.N, self.device
        attnres.msar_block_phase1(self.cache, self.ks, self.conv_w, self.queries, None, 1e-6, o=self.o, lse=self.lse)
        f32 = dict(dtype=torch.float32, device=device)
        self.d_o = torch.empty_like(self.o)
        self.d_lse = torch.empty((S, 4, T), **f32)
        self.d_p = torch.empty((S, T, d), dtype=torch.bfloat16, device=device)
        self.p2g = [(torch.empty_like(self.conv_w), torch.empty((4, d), **f32), torch.empty((d,), **f32),
                     torch.empty((4 * d,), **f32), torch.empty((4 * d, 4), **f32)) for _ in range(S)]
        self.p1g = (torch.empty_like(self.cache), torch.empty_like(self.conv_w), torch.empty((S, 4, d), **f32),
                    torch.empty((d,), **f32))
        ks = (ctypes.c_int32 * 3)(*self.ks)
        n = ctypes.c_size_t(0)
        attnres._check("ws", attnres.load().msar_block_phase2_bwd_workspace_size(
            T, d, 1, 4, ctypes.cast(ks, ctypes.c_void_p), ctypes.byref(n)))
        self.ws2 = torch.empty(((n.value + 3) // 4,), **f32)
        attnres._check("ws", attnres.load().msar_block_phase1_bwd_workspace_size(
            N, T, d, 1, 4, ctypes.cast(ks, ctypes.c_void_p), S, ctypes.byref(n)))
        self.ws1 = torch.empty(((n.value + 3) // 4,), **f32)
        self.out = self.p1g[0]
        self.ready = True

    def step(self, stream, ev=None):
        from depth_wise_attention_gb300 import attnres
        if not self.ready:
            self._prepare()
        if ev is not None:
            ev[0].record(stream)
        for s_ in range(self.S):
            p = self.parts[s_] if s_ > 0 else None
            outs = (self.d_o[s_], self.d_lse[s_], self.d_p[s_] if s_ > 0 else None) + self.p2g[s_]
            attnres.msar_block_phase2_bwd(self.o[s_], self.lse[s_], p, self.ks, self.conv_w, self.queries[s_],
                                          self.dh[s_], None, 1e-6, None, self.mix_w, 1e-6, outs=outs,
                                          workspace=self.ws2, stream=stream)
        attnres.msar_block_phase1_bwd(self.cache, self.ks, self.conv_w, self.queries, self.d_o, self.d_lse, None,
                                      1e-6, outs=self.p1g, workspace=self.ws1, stream=stream)
        if ev is not None:
            ev[1].record(stream)

    def setup_host(self):
        if not self.ready:
            self._prepare()
        self.h_cache = torch_pinned_like(self.cache)
        self.h_dh = torch_pinned_like(self.dh)
        self.h_out = torch_pinned_like(self.p1g[0])
        self.h2d = (self.h_cache.numel() + self.h_dh.numel()) * 2
        self.d2h = self.h_out.numel() * 2

    def step_e2e(self, stream):
        self.cache.copy_(self.h_cache, non_blocking=True)
        self.dh.copy_(self.h_dh, non_blocking=True)
        self.step(stream)
        self.h_out.copy_(self.p1g[0], non_blocking=True)

    def oracle_sample(self, n_tokens, seed=1):
        # per sampled token t: the 12-row causal windows and dh of every layer on row t alone
        rng = np.random.default_rng(seed)
        idx = np.sort(rng.choice(self.T, size=min(n_tokens, self.T), replace=False))
        out = []
        for t in idx:
            lo = max(0, int(t) - 11)
            win = self.cache[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
            pw = self.parts[:, lo:int(t) + 1, :].float().cpu().numpy().astype(np.float64)
            dw = np.zeros((self.S,) + win.shape[1:])
            dw[:, -1] = self.dh[:, int(t)].float().cpu().numpy()
            out.append((win, pw, dw))
        return (out, self.conv_w.cpu().numpy().astype(np.float64), self.queries.cpu().numpy().astype(np.float64),
                self.mix_w.cpu().numpy().astype(np.float64))

    def run_oracle(self, sample):
        from oracle import oracle
        wins, cw, q, mw = sample
        for win, pw, dw in wins:
            o, lse = oracle.msar_phase1(win, self.ks, cw, q, None, 1e-6)
            d_o, d_l = np.zeros_like(o), np.zeros_like(lse)
            for s_ in range(self.S):
                r = oracle.msar_phase2_bwd(o[s_], lse[s_], pw[s_] if s_ > 0 else None, self.ks, cw, q[s_], dw[s_],
                                           None, 1e-6, None, mw, 1e-6)
                d_o[s_], d_l[s_] = r[0], r[1]
            oracle.msar_phase1_bwd(win, self.ks, cw, q, d_o, d_l, None, 1e-6)
        return len(wins)


WORKLOADS = ["block", "block_d2048", "block_fused", "block_bwd", "read_bwd", "mhar_bwd", "mhar_block",
             "msar_chunked", "msar_ps", "decode", "mhar", "msar", "msar_block", "msar_bwd", "msar_bwd_ps", "msar_ws",
             "msar_block_ws", "msar_block_bwd", "full_depth", "msar_bwd_chunked", "depth_bwd"]


def make_workload(name, T=None):
    if name == "block":
        return BlockWorkload(T=T or 32768)
    if name == "block_d2048":
        return BlockWorkload(T=T or 8192, d=2048)
    if name == "mhar":
        return MharWorkload(T=T or 131072)
    if name == "msar":
        return MsarWorkload(T=T or 32768)
    if name == "decode":
        return DecodeWorkload(T=T or 16)
    if name == "read_bwd":
        return ReadBwdWorkload(T=T or 32768)
    if name == "block_bwd":
        return BlockBwdWorkload(T=T or 32768)
    if name == "mhar_block":
        return MharBlockWorkload(T=T or 131072)
    if name == "msar_ps":
        return MsarPerSourceWorkload(T=T or 32768)
    if name == "msar_chunked":
        return MsarChunkedWorkload(T=T or 32768)
    if name == "mhar_bwd":
        return MharBwdWorkload(T=T or 131072)
    if name == "msar_block":
        return MsarBlockWorkload(T=T or 32768)
    if name == "msar_ws":
        return MsarWsWorkload(T=T or 32768)
    if name == "msar_block_ws":
        return MsarBlockWsWorkload(T=T or 32768)
    if name == "msar_bwd":
        return MsarBwdWorkload(T=T or 32768)
    if name == "msar_bwd_chunked":
        return MsarBwdChunkedWorkload(T=T or 32768)
    if name == "depth_bwd":
        return DeepReadBwdWorkload(T=T or 16384)
    if name == "msar_block_bwd":
        return MsarBlockBwdWorkload(T=T or 32768)
    if name == "msar_bwd_ps":
        return MsarBwdPerSourceWorkload(T=T or 32768)
    if name == "block_fused":
        return BlockFusedWorkload(T=T or 32768)
    if name == "full_depth":
        return FullDepthWorkload(T=T or 16384)
    raise SystemExit(f"unknown workload {name}")


# --------------------------------------------------------------------------
# distributed plumbing (one process per GPU; no data-path collective)
# --------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int, device) -> float:
    """Max of a scalar over all ranks (timing only)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# --------------------------------------------------------------------------
# arms
# --------------------------------------------------------------------------

def aggregate(tokens_per_rank: int, steps: int, world: int, elapsed_ms_max: float):
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    return tokens_per_rank * steps * world / (elapsed_ms_max / 1e3)


def run_cuda(args):
    import torch
    from depth_wise_attention_gb300 import attnres
    from depth_wise_attention_gb300.build import build

    world, rank, local = dist_env()
    if world != args.gpus:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    dist_init(world, "nccl")
    if rank == 0:
        build()
    barrier(world)
    attnres.load()

    wl = make_workload(args.workload, args.T)
    wl.setup(device)
    stream = torch.cuda.current_stream(device)
    torch.cuda.synchronize(device)

    for _ in range(args.warmup):
        wl.step(stream)
    attnres.attnres_sync_status(stream)

    # ---------------- timed region: K steps, events around the dominant kernel
    K = args.steps
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(K)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(device)
        start.record(stream)
        for k in range(K):
            wl.step(stream, evs[k])
        end.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
    attnres.attnres_sync_status(stream)
    elapsed_ms = start.elapsed_time(end)
    dom_ms = statistics.mean(a.elapsed_time(b) for a, b in evs)
    elapsed_ms = max_over_ranks(elapsed_ms, world, device)

    value = aggregate(wl.T, K, world, elapsed_ms)
    ms_per_step = elapsed_ms / K
    peaks, peaks_kind = measured_peaks()
    hbm_peak = float(peaks["hbm_gbs"])
    dom_bytes = wl.dominant_bytes_per_launch()
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    step_gbs = wl.bytes_per_token * wl.T / (ms_per_step / 1e3) / 1e9
    traffic = profile_traffic(wl.profile_tag, wl.dominant_src)

    # ---------------- end to end: host buffers, copies inside the timed region
    wl.setup_host()
    E = max(3, min(K, args.e2e_steps))
    pipelined = type(wl).step is BlockWorkload.step    # the overlapped schedule runs the Block step
    if pipelined:
        wl.run_e2e_pipelined(stream, 2)    # warm-up
        barrier(world)
        torch.cuda.synchronize(device)
        e2e_ms = wl.run_e2e_pipelined(stream, E)
        torch.cuda.synchronize(device)
        barrier(world)
    else:
        for _ in range(2):
            wl.step_e2e(stream)
        barrier(world)
        torch.cuda.synchronize(device)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(E):
            wl.step_e2e(stream)
        e1.record(stream)
        torch.cuda.synchronize(device)
        barrier(world)
        e2e_ms = e0.elapsed_time(e1)
    attnres.attnres_sync_status(stream)
    e2e_ms = max_over_ranks(e2e_ms, world, device)
    e2e_value = wl.T * E * world / (e2e_ms / 1e3)

    # ---------------- CPU oracle baseline (rank 0, N=1 only)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.cpu_seconds)

    if rank != 0:
        return
    roofline = {"kernel": wl.dominant, "bound": "hbm", "achieved": achieved,
                "peak": hbm_peak, "peak_kind": peaks_kind, "unit": "GB/s",
                "frac": achieved / hbm_peak,
                "bytes_per_launch": dom_bytes, "ms_per_launch": dom_ms,
                "traffic": traffic}
    fma = getattr(wl, "fma_per_token", None)
    if fma:
        # fp32 CUDA-core peak from the unit counts and the clock: 152 SMs x
        # 128 fp32 lanes x 2 flops per FMA x the maximum SM clock (2070 MHz)
        alu_peak = 152 * 128 * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12
        tflops = 2.0 * fma * wl.T / (dom_ms / 1e3) / 1e12
        roofline = {"kernel": wl.dominant, "bound": "alu", "achieved": tflops, "peak": alu_peak,
                    "peak_kind": "derived: 152 SMs x 128 fp32 lanes x 2 flops x 2070 MHz",
                    "unit": "TFLOP/s", "frac": tflops / alu_peak,
                    "flops_per_launch": 2.0 * fma * wl.T, "ms_per_launch": dom_ms,
                    "hbm_gbs": achieved, "traffic": traffic}
    line = {
        "metric": METRIC if args.workload == "block" else f"{wl.name} tokens/s",
        "value": value,
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms_per_step,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded, shapes and distributions of the workload)",
        "config": dict(wl.config(), parallelism=f"replicas x{world} (no collective)"),
        "hbm_gbs_step": step_gbs,
        "hbm_frac_step": step_gbs / hbm_peak,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "steps": E,
                "schedule": ("pipelined: copy-in, compute and copy-out streams over two device buffer sets"
                             if pipelined else "serial on one stream"),
                "h2d_bytes_per_step": wl.h2d, "d2h_bytes_per_step": wl.d2h},
        "gpu_launches": wl.launches_per_step * K,
        "clocks": clk.summary(),
        "library": attnres.version(),
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(wl, seconds):
    """Time the oracle, as it stands, on a bounded sample of the workload."""
    probe = wl.oracle_sample(4, seed=2)
    t0 = time.perf_counter()
    wl.run_oracle(probe)
    per_tok = (time.perf_counter() - t0) / 4
    n = int(max(8, min(wl.T, seconds / max(per_tok, 1e-6))))
    sample = wl.oracle_sample(n, seed=1)
    t0 = time.perf_counter()
    done = wl.run_oracle(sample)
    dt = time.perf_counter() - t0
    return {"value": done / dt, "unit": "tokens/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} tokens drawn with seed 1 from the same inputs "
                      f"({dt:.1f} s, single-threaded C oracle, float64)"}


def run_reference(args):
    """The reference arm: the CPU oracle on the same workload, metric and unit."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import torch
    torch.cuda.set_device(0)
    wl = make_workload(args.workload, args.T)
    wl.setup(torch.device("cuda", 0))
    probe = wl.oracle_sample(4, seed=2)
    t0 = time.perf_counter()
    wl.run_oracle(probe)
    per_tok = (time.perf_counter() - t0) / 4
    budget = args.cpu_seconds * 4
    per_step = int(max(1, min(wl.T, budget / max(per_tok, 1e-6) / max(1, args.steps + args.warmup))))
    samples = [wl.oracle_sample(per_step, seed=10 + k) for k in range(args.steps + args.warmup)]
    for k in range(args.warmup):
        wl.run_oracle(samples[k])
    t0 = time.perf_counter()
    done = 0
    for k in range(args.steps):
        done += wl.run_oracle(samples[args.warmup + k])
    dt = time.perf_counter() - t0
    value = done / dt
    line = {
        "impl": "reference",
        "metric": METRIC if args.workload == "block" else f"{wl.name} tokens/s",
        "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded, same inputs as the CUDA arm)",
        "config": dict(wl.config(), parallelism="CPU oracle, rank 0 only"),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"{per_step} tokens per step, seeds 10.., single-threaded"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["cuda", "reference"], default="cuda")
    ap.add_argument("--workload", default="block", choices=WORKLOADS)
    ap.add_argument("--T", type=int, default=None, help="override the token count")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_cuda(args)


if __name__ == "__main__":
    main()
