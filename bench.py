#!/usr/bin/env python
"""Throughput of CP-chunk attention on one GB300 (or N replicas under torchrun).

Default workload (the headline): dense causal CP chunk, bf16 in / fp32
accumulate, rank 2 of 4 of an 8192-token sequence -> 2048 queries at
causal_offset 4096 against 8192 keys, 16 query heads over 4 KV heads, d = 128,
scale 1/sqrt(128), N(0,1) * 0.5 inputs (seed 0).  One step = one
cpattn_chunk_fwd call over the whole problem (all KV chunks folded and
merged in the kernel).  The metric is algorithmic TFLOP/s: 4 * d FLOPs per
permitted (query, key) pair per head (QK^T and PV), masked work not counted.

Other workloads (--workload zigzag | dsa | moba) are measurement aids.

Timing: W untimed warm-up steps, then exactly K timed steps; before each
timed step a 256 MiB buffer is written to flush the 129 MB L2; each step is
bracketed by CUDA events on the launching stream; barrier + synchronize
around the timed region; max over ranks.  `e2e` times the same call with
host (pinned) inputs copied in and outputs copied out inside each step.
`--impl reference` times the float64 CPU oracle instead (bounded samples).
"""

from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from context_attention_softmax_gb300 import inputs  # noqa: E402

L2_FLUSH_BYTES = 256 << 20
METRIC = "CP-chunk attention fwd TFLOP/s (dense) & GB/s (top-k sparse) vs GB300 peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0}


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

# DRAM bytes per launch of the dominant kernel (dram__bytes_read.sum +
# dram__bytes_write.sum from one ncu capture, summarised under profiles/),
# valid only while the kernel's sources hash to the value they had then.
TRAFFIC = {
    "dense_gqa": {"bytes": 21_066_496 + 0, "kernel": "dense_tc_kernel",
                  "sources": ["dense_tc.cu", "dense_tc_common.cuh", "sm100.cuh", "common.cuh"],
                  "sha": "710df07de8adbb71"},
    "dsa": {"bytes": 662_182_656 + 505_942_016, "kernel": "dsa_attn_kernel",
            "sources": ["dsa_tc.cu", "sm100.cuh", "common.cuh"], "sha": "1a2d63f8b3cc8586"},
}


def measured_traffic(name):
    """(bytes, kernel) if the recorded counters still describe the kernel, else (None, why)."""
    import hashlib
    t = TRAFFIC.get(name)
    if t is None:
        return None, "no ncu capture recorded for this workload"
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "context_attention_softmax_gb300",
                        "csrc")
    m = hashlib.sha256()
    for f in t["sources"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            m.update(fh.read())
    if m.hexdigest()[:16] != t["sha"]:
        return None, "kernel changed since the recorded ncu capture"
    return t["bytes"], t["kernel"]


class DenseRunner:
    """The headline workload: one dense GQA CP-chunk call."""

    name = "dense_gqa"

    def __init__(self, device=None):
        self.w = w = inputs.dense_gqa()
        Tq, Hq, D = w.q.shape
        qpos = w.causal_offset + np.arange(Tq)
        pairs = int(np.minimum(qpos + 1, w.Tk).sum())          # causal, one sequence
        self.pairs_per_head = pairs
        self.flops = 4.0 * D * pairs * Hq
        self.launches_per_step = 1
        self.bound = "tensor"
        self.config = {
            "workload": "dense causal CP chunk, bf16 in / fp32 acc: 2048 queries (rank 2 of 4, "
                        "causal_offset 4096) x 8192 keys, 16 q heads / 4 kv heads, d=128, "
                        "KV folded in-kernel (4 chunks of 2048, chunk 3 fully masked)",
            "Tq": Tq, "Tk": w.Tk, "Hq": Hq, "Hkv": w.k.shape[1], "D": D,
            "causal_offset": w.causal_offset, "permitted_pairs_per_head": pairs,
            "l2": "flushed by a 256 MiB write before every timed step",
            "seed": 0,
        }
        if device is not None:
            self.dev = device
            self.q, self.k, self.v = (t.to(device) for t in (w.q, w.k, w.v))
            self.o = torch.empty((Tq, Hq, w.v.shape[2]), dtype=torch.bfloat16, device=device)
            self.lse = torch.empty((Tq, Hq), dtype=torch.float32, device=device)
            self.ws = torch.empty(64 << 20, dtype=torch.uint8, device=device)   # per-piece summaries

    def step(self, q=None, k=None, v=None):
        from context_attention_softmax_gb300 import cpattn_chunk_fwd
        w = self.w
        cpattn_chunk_fwd(q if q is not None else self.q, k if k is not None else self.k,
                         v if v is not None else self.v, scale=w.scale, causal=True,
                         causal_offset=w.causal_offset, out=self.o, lse=self.lse,
                         workspace=self.ws)

    # host buffers for the end-to-end measurement
    def host_inputs(self):
        return [self.w.q.pin_memory(), self.w.k.pin_memory(), self.w.v.pin_memory()]

    def host_outputs(self):
        return [torch.empty_like(self.o, device="cpu").pin_memory(),
                torch.empty_like(self.lse, device="cpu").pin_memory()]

    def outputs(self):
        return [self.o, self.lse]

    # the oracle on a bounded sample of query rows
    def oracle_sample(self, rows):
        import oracle as orc
        w = self.w
        if not hasattr(self, "_f64"):
            self._f64 = (inputs.as_f64(w.q), inputs.as_f64(w.k), inputs.as_f64(w.v))
            self._lay = orc.make_layout(w.Tq, w.Tk, True, w.causal_offset)
        q, k, v = self._f64
        orc.dense_attention(q, k, v, w.scale, self._lay, rows=rows)
        qpos = w.causal_offset + rows
        return 4.0 * w.q.shape[2] * float(np.minimum(qpos + 1, w.Tk).sum()) * w.q.shape[1]


class ZigzagRunner:
    """All 8 zigzag ranks of the packed THD varlen workload (8 calls per step)."""

    name = "zigzag"

    def __init__(self, device):
        from context_attention_softmax_gb300 import _lib  # noqa: F401
        self.z = z = inputs.zigzag_varlen()
        self.dev = device
        self.k, self.v = z.k_gathered.to(device), z.v_gathered.to(device)
        self.qs = [z.rank_q(r).to(device) for r in range(z.cp_size)]
        self.maps = [torch.as_tensor(z.rank_chunks(r), dtype=torch.int32, device=device)
                     for r in range(z.cp_size)]
        self.kvmap = torch.as_tensor(z.kv_chunk_map, dtype=torch.int32, device=device)
        self.cu = torch.as_tensor(z.cu_seqlens, dtype=torch.int32, device=device)
        self.o = [torch.empty_like(q) for q in self.qs]
        self.lse = [torch.empty(q.shape[:2], dtype=torch.float32, device=device) for q in self.qs]
        self.ws = torch.empty(64 << 20, dtype=torch.uint8, device=device)   # per-piece summaries
        lens = np.diff(z.cu_seqlens.astype(np.int64))
        pairs = int((lens * (lens + 1) // 2).sum())
        H, D = z.q_global.shape[1], z.q_global.shape[2]
        self.flops = 4.0 * D * pairs * H
        self.launches_per_step = z.cp_size
        self.bound = "tensor"
        self.config = {"workload": "packed THD varlen, zigzag cp=8, 16384 tokens / 8 seqs, "
                                   "32 heads, d=128, causal; all 8 rank calls",
                       "lengths": lens.tolist(), "permitted_pairs_per_head": pairs,
                       "l2": "flushed by a 256 MiB write before every timed step"}

    def step(self):
        from context_attention_softmax_gb300 import cpattn_chunk_fwd
        z = self.z
        for r in range(z.cp_size):
            cpattn_chunk_fwd(self.qs[r], self.k, self.v, scale=z.scale, causal=True,
                             cu_seqlens=self.cu, q_chunk_map=self.maps[r], kv_chunk_map=self.kvmap,
                             chunk_len=z.chunk_len, out=self.o[r], lse=self.lse[r],
                             workspace=self.ws)


class DsaRunner:
    """DSA top-2048 sparse attention on absorbed-MLA shapes."""

    name = "dsa"

    def __init__(self, device):
        self.w = w = inputs.dsa_absorbed(device=device)
        self.q, self.kv = w.q.to(device), w.k.to(device)
        self.v = self.kv[:, :, :512]
        self.idx = w.indices.to(device)
        Tq, Hq, Dqk = w.q.shape
        self.o = torch.empty((Tq, Hq, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((Tq, Hq), dtype=torch.float32, device=device)
        self.flops = 2.0 * Tq * Hq * w.topk * (Dqk + 512)
        self.gathered_bytes = Tq * w.topk * Dqk * 2
        self.launches_per_step = 1
        self.bound = "tensor"
        self.config = {"workload": "DSA top-2048 sparse, absorbed MLA: 4096 q x 32768 kv, "
                                   "128 heads / 1 kv head, dqk 576, dv 512",
                       "gathered_bytes": self.gathered_bytes}

    def step(self):
        from context_attention_softmax_gb300 import cpattn_topk_sparse_fwd
        w = self.w
        cpattn_topk_sparse_fwd(self.q, self.kv, self.v, self.idx, block_size=1, scale=w.scale,
                               causal_offset=w.causal_offset, out=self.o, lse=self.lse)


class MobaRunner:
    """MoBA gate + block-sparse attention (2+1 launches per step)."""

    name = "moba"

    def __init__(self, device):
        self.w = w = inputs.moba()
        self.q, self.k, self.v = (t.to(device) for t in (w.q, w.k, w.v))
        Tq, H, D = w.q.shape
        self.sel = torch.empty((Tq, H, w.topk + 1), dtype=torch.int32, device=device)
        self.o = torch.empty_like(self.q)
        self.lse = torch.empty((Tq, H), dtype=torch.float32, device=device)
        from context_attention_softmax_gb300 import _lib, cpattn_workspace_size
        nbytes = cpattn_workspace_size(_lib.OP_BLOCK_GATE, self.q, self.k, topk=w.topk,
                                       block_size=w.block_size)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        nsp = cpattn_workspace_size(_lib.OP_TOPK_SPARSE_FWD, self.q, self.k, self.v, topk=w.topk + 1,
                                    block_size=w.block_size)
        self.ws_sparse = torch.empty(max(nsp, 16), dtype=torch.uint8, device=device)
        B = w.block_size
        qpos = w.causal_offset + np.arange(Tq)
        keys = 3 * B + (qpos % B) + 1
        self.flops = 4.0 * D * H * float(keys.sum())
        self.hbm_bytes = (2 * w.k.numel() + 2 * w.q.numel() * 2 + w.v.numel() * 2 + self.o.numel() * 2)
        self.launches_per_step = 7   # gate: 2; attention: count, scan, scatter, attend, merge
        self.bound = "hbm"
        self.config = {"workload": "MoBA gate (top-3 + own of 512-key blocks) + block-sparse "
                                   "attention: 8192 q x 65536 kv, 32 heads, d=128",
                       "compulsory_bytes": self.hbm_bytes}

    def step(self):
        from context_attention_softmax_gb300 import cpattn_block_gate, cpattn_topk_sparse_fwd
        w = self.w
        cpattn_block_gate(self.q, self.k, w.block_size, w.topk, causal_offset=w.causal_offset,
                          sel=self.sel, workspace=self.ws)
        cpattn_topk_sparse_fwd(self.q, self.k, self.v, self.sel, block_size=w.block_size,
                               scale=w.scale, causal_offset=w.causal_offset, out=self.o,
                               lse=self.lse, workspace=self.ws_sparse)


class IndexerRunner:
    """The DSA indexer: top-2048 keys of 4096 queries at offset 16384 over 32768
    keys, 4 fp32 indexer heads of 128 (the indices the DSA workload attends to)."""

    name = "dsa_indexer"

    def __init__(self, device):
        self.w = w = inputs.dsa_absorbed(device=device)
        self.qI, self.kI, self.wt = (w.extra[k].to(device) for k in ("qI", "kI", "w"))
        Tq, H, D = self.qI.shape
        Tk = self.kI.shape[0]
        self.out = torch.empty((Tq, w.topk), dtype=torch.int32, device=device)
        from context_attention_softmax_gb300 import _lib, _args
        a = _args(self.qI, self.kI.unsqueeze(1), None, 1.0, True, w.causal_offset, None, None, None,
                  0, None, None)
        nbytes = _lib.load().cpattn_workspace_size(_lib.OP_DSA_INDEXER, ctypes.byref(a), w.topk, 1)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        n_keys = np.minimum(w.causal_offset + np.arange(Tq) + 1, Tk)     # causal, one sequence
        self.flops = 2.0 * float(n_keys.sum()) * H * D
        self.launches_per_step = 3   # norms, scores, selection
        self.bound = "alu"
        self.config = {"workload": "DSA indexer top-2048: 4096 q (offset 16384) x 32768 keys, "
                                   "4 fp32 indexer heads x 128, scores sum_h w_h relu(qI.kI)",
                       "permitted_pairs": int(n_keys.sum())}

    def step(self):
        from context_attention_softmax_gb300 import cpattn_dsa_indexer
        cpattn_dsa_indexer(self.qI, self.kI, self.wt, self.w.topk, causal_offset=self.w.causal_offset,
                           out=self.out, workspace=self.ws)

    def oracle_sample(self, rows):
        import oracle as orc
        w = self.w
        if not hasattr(self, "_np"):
            self._np = tuple(w.extra[k].numpy() for k in ("qI", "kI", "w"))
            self._lay = orc.make_layout(self._np[0].shape[0], self._np[1].shape[0], True, w.causal_offset)
        qI, kI, wt = self._np
        orc.dsa_indexer_topk(qI, kI, wt, self._lay, w.topk, rows=rows)
        n_keys = np.minimum(w.causal_offset + np.asarray(rows) + 1, kI.shape[0])
        return 2.0 * float(n_keys.sum()) * qI.shape[1] * qI.shape[2]


RUNNERS = {"dense_gqa": DenseRunner, "zigzag": ZigzagRunner, "dsa": DsaRunner, "moba": MobaRunner,
           "dsa_indexer": IndexerRunner}


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        self.gpu = gpu_index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.count(",") >= 8]
        os.unlink(self.f.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except ValueError:
                continue
            for n, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def time_steps(fn, steps, warmup, flush, world):
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    barrier(world)
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(world)
    for s in range(steps):
        flush.zero_()
        ev[s][0].record(stream)
        fn()
        ev[s][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    return [a.elapsed_time(b) for a, b in ev]


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def host_info():
    """CPU model and the BLAS numpy was built against, for the oracle timings."""
    model = platform.machine()
    try:
        with open("/proc/cpuinfo") as fh:
            for ln in fh:
                key = ln.split(":")[0].strip().lower()
                if key in ("model name", "cpu part"):
                    model = ln.split(":", 1)[1].strip() if key == "model name" else \
                        f"{platform.machine()} part {ln.split(':', 1)[1].strip()}"
                    break
    except OSError:
        pass
    blas = "unknown"
    try:
        blas = np.show_config(mode="dicts")["Build Dependencies"]["blas"]["name"]
    except Exception:
        pass
    return {"cpu_model": model, "blas": blas}


def cpu_baseline(runner, budget_s=12.0, batch=32):
    """Time the oracle as it stands on a bounded sample of query rows."""
    rng = np.random.default_rng(123)
    n = runner.w.Tq
    t0 = time.perf_counter()
    flops = 0.0
    rows_done = 0
    while time.perf_counter() - t0 < budget_s:
        rows = np.sort(rng.choice(n, size=batch, replace=False))
        flops += runner.oracle_sample(rows)
        rows_done += batch
    dt = time.perf_counter() - t0
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": len(os.sched_getaffinity(0)),
            "kind": "oracle", **host_info(),
            "sample": f"{rows_done} query rows drawn at random ({rows_done / n:.1f}x the "
                      f"{n}-row problem; all heads, all permitted keys), float64 numpy, "
                      f"{dt:.1f} s"}


def run_reference(args, world, rank):
    if rank != 0:
        return
    runner = DenseRunner(None)
    rng = np.random.default_rng(7)
    per_step_rows = 16
    for _ in range(args.warmup):
        runner.oracle_sample(np.sort(rng.choice(runner.w.Tq, per_step_rows, replace=False)))
    times, flops = [], []
    for _ in range(args.steps):
        rows = np.sort(rng.choice(runner.w.Tq, per_step_rows, replace=False))
        t0 = time.perf_counter()
        flops.append(runner.oracle_sample(rows))
        times.append(time.perf_counter() - t0)
    value = sum(flops) / sum(times) / 1e12
    ms_full = runner.flops / (value * 1e12) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "ms_full_problem_extrapolated": ms_full, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic (seeded N(0,1)*0.5, bf16-rounded)",
        "config": runner.config,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "kind": "oracle",
                         "cores": len(os.sched_getaffinity(0)), **host_info(),
                         "sample": f"each step: {per_step_rows} random query rows x all heads of "
                                   "the workload; ms_per_step extrapolated to the full problem "
                                   "by permitted pairs"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_ours(args, world, rank, local):
    from context_attention_softmax_gb300 import build as _build
    _build.build()
    dev = torch.device("cuda", local)
    runner = RUNNERS[args.workload](dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)

    clocks = ClockSampler(local)
    clocks.start()
    times = time_steps(runner.step, args.steps, args.warmup, flush, world)
    clk = clocks.stop()
    mean_ms = statistics.mean(times)
    mean_ms = max_over_ranks(mean_ms, world)
    value = world * runner.flops / (mean_ms * 1e-3) / 1e12

    # end to end through the public API with pinned host buffers
    e2e = None
    if hasattr(runner, "host_inputs"):
        hin, hout = runner.host_inputs(), runner.host_outputs()
        din = [torch.empty_like(t, device=dev) for t in hin]
        dout = runner.outputs()

        def e2e_step():
            for h, d in zip(hin, din):
                d.copy_(h, non_blocking=True)
            runner.step(*din)
            for d, h in zip(dout, hout):
                h.copy_(d, non_blocking=True)

        et = time_steps(e2e_step, args.steps, max(args.warmup, 3), flush, world)
        e_ms = max_over_ranks(statistics.mean(et), world)
        e2e = {"value": world * runner.flops / (e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
               "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hin)),
               "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hout))}

    peaks, src = load_peaks()
    if runner.bound == "tensor":
        achieved = runner.flops / (mean_ms * 1e-3) / 1e12
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None, "peak_source": f"{src} bf16 burst"}
    elif runner.bound == "alu":
        # fp32 FMA pipes: SMs x 128 lanes x 2 FLOP x the maximum SM clock
        achieved = runner.flops / (mean_ms * 1e-3) / 1e12
        sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = n_sm * 128 * 2 * sm_mhz * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None,
                "peak_source": f"fp32 FMA: {n_sm} SMs x 128 lanes x 2 x {sm_mhz:.0f} MHz"}
    else:
        achieved = runner.hbm_bytes / (mean_ms * 1e-3) / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": None, "peak_source": f"{src} copy"}
    roof["kernel"] = {"moba": "moba step", "dsa_indexer": "dsa indexer (scores + selection)"}.get(
        runner.name, "cpattn_chunk_fwd")
    traffic, what = measured_traffic(runner.name)
    if traffic is not None:
        roof["traffic"] = traffic
        roof["kernel"] = what
        roof["traffic_note"] = "ncu dram bytes read + written per launch, see profiles/"
    else:
        roof["traffic_note"] = what

    if rank != 0:
        return
    line = {
        "metric": METRIC,
        "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": mean_ms,
        "ms_min": min(times), "ms_median": statistics.median(times),
        "ms_p90": float(np.percentile(times, 90)),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded; no dataset)",
        "config": runner.config, "roofline": roof, "clocks": clk,
        "gpu_launches": runner.launches_per_step * args.steps,
        "e2e": e2e,
    }
    if world == 1 and not args.no_cpu_baseline and hasattr(runner, "oracle_sample"):
        line["cpu_baseline"] = cpu_baseline(runner)
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: 2000 for our arm, so the clock sampler sees the "
                         "timed region; 20 for the reference arm)")
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(RUNNERS), default="dense_gqa")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 2000
    world, rank, local = dist_setup()
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
