#!/usr/bin/env python
"""Throughput of CP-chunk attention on one GB300 (or N replicas under torchrun).

Headline (the top-level `value`): dense causal CP chunk, bf16 in / fp32
accumulate, rank 2 of 4 of an 8192-token sequence -> 2048 queries at
causal_offset 4096 against 8192 keys, 16 query heads over 4 KV heads, d = 128,
scale 1/sqrt(128), N(0,1) * 0.5 inputs (seed 0).  One step = one
cpattn_chunk_fwd call over the whole problem (all KV chunks folded and
merged in the kernel).  Metric: algorithmic TFLOP/s, 4 * d FLOPs per
permitted (query, key) pair per head (QK^T and PV), masked work not counted.

The same JSON line carries one record per other workload under "workloads",
each timed the same way with its own roofline, oracle baseline and
end-to-end figure:
  dense_gqa_4chunks  the headline problem as 4 KV-chunk summaries + merge
  dense_gqa_bwd      its backward (dq, dk, dv; TFLOP/s at 10 d per pair)
  zigzag             packed THD varlen, zigzag cp=8, all 8 rank calls (TFLOP/s)
  dsa                DSA top-2048 sparse attention, absorbed MLA (TFLOP/s and
                     gathered GB/s)
  moba               MoBA gate + block-sparse attention (compulsory GB/s)
  dsa_indexer        the DSA indexer's exact top-2048 (TFLOP/s of its fp32 scores)
  mla_v_up           absorbed-MLA value up-projection of the DSA output (GB/s)
  mla_kv             MLA K/V materialisation from gathered latents (TFLOP/s)
`--workload NAME` times one of them alone as the top-level record.

Timing: W untimed warm-up steps, then exactly K timed steps; before each
timed step a 256 MiB buffer is written to flush the 129 MB L2; each step is
bracketed by CUDA events on the launching stream; barrier + synchronize
around the timed region; max over ranks.  Before the first timed step the
GPU is given a short backlog of flush writes so that it never waits for the
host to enqueue a step.  `e2e` times the same public call with pinned host
inputs copied in and the outputs copied out inside each step.
`--impl reference` times the float64 CPU oracle instead (bounded samples).
"""

from __future__ import annotations

import argparse
import datetime
import json
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
L2_NOTE = "flushed by a 256 MiB write before every timed step"


# ---------------------------------------------------------------------------
# recorded DRAM traffic of the dominant kernels
# ---------------------------------------------------------------------------

# dram__bytes_read.sum + dram__bytes_write.sum per launch of a workload's
# dominant kernel from one ncu capture (summarised under profiles/), valid
# only while the kernel's sources hash to the value they had then.
TRAFFIC = {
    "dense_gqa": {"bytes": 21_190_912 + 0, "kernel": "dense_tc_kernel<0>",
                  "sources": ["dense_tc.cu", "dense_tc_common.cuh", "sm100.cuh", "common.cuh"],
                  "sha": "351887c4dbfdd44c"},
    "dense_gqa_4chunks": {"bytes": 21_075_200 + 12_354_048, "kernel": "dense_tc_kernel<1>",
                          "sources": ["dense_tc.cu", "dense_tc_common.cuh", "sm100.cuh",
                                      "common.cuh"],
                          "sha": "351887c4dbfdd44c"},
    "dsa": {"bytes": 661_886_208 + 507_494_400, "kernel": "dsa_attn_kernel",
            "sources": ["dsa_tc.cu", "sm100.cuh", "common.cuh"], "sha": "6fea0a102583429c"},
    "mla_kv": {"bytes": 577_171_712 + 2_627_442_176, "kernel": "mla_kv_kernel",
               "sources": ["mla_gemm.cu", "sm100.cuh", "common.cuh"], "sha": "083dccee2bdb63db"},
    "mla_v_up": {"bytes": 553_840_384 + 112_673_792, "kernel": "mla_gemm_kernel<1>",
                 "sources": ["mla_gemm.cu", "sm100.cuh", "common.cuh"], "sha": "083dccee2bdb63db"},
    "dense_gqa_bwd": {"bytes": 30_470_656 + 5_928_960, "kernel": "bwd_kernel",
                      "sources": ["dense_bwd.cu", "dense_tc_common.cuh", "sm100.cuh", "common.cuh"],
                      "sha": "5085abcec64ca82e"},
    "dsa_indexer": {"bytes": 331_365_632 + 28_990_208, "kernel": "idx_select_kernel",
                    "sources": ["dsa_indexer.cu", "dsa_indexer_tc.cu", "sm100.cuh", "common.cuh"],
                    "sha": "63fddb7a129a018f"},
    "moba": {"bytes": 1_150_921_984 + 257_916_160, "kernel": "moba_attn_kernel",
             "sources": ["moba_tc.cu", "sm100.cuh", "common.cuh"], "sha": "be1ba744dc70c6c4"},
}


def measured_traffic(name):
    """(bytes, kernel) if the recorded counters still describe the kernel, else (None, why)."""
    import hashlib
    t = TRAFFIC.get(name)
    if t is None:
        return None, "no ncu capture recorded for this workload"
    csrc = os.path.join(ROOT, "context_attention_softmax_gb300", "csrc")
    m = hashlib.sha256()
    for f in t["sources"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            m.update(fh.read())
    if m.hexdigest()[:16] != t["sha"]:
        return None, "kernel changed since the recorded ncu capture"
    return t["bytes"], t["kernel"]


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------

class Runner:
    """One workload: device inputs, one step through the public API, its
    algorithmic work per step, and the oracle on a sample of its query rows.

    work / seconds / scale = value in `unit`.
    """

    name = ""
    unit = "TFLOP/s"
    scale = 1e12
    bound = "tensor"
    kernel = "cpattn_chunk_fwd"
    launches_per_step = 1
    work = 0.0
    n_rows = 0
    extras: dict = {}

    def device_inputs(self):
        raise NotImplementedError

    def step(self, *ins):
        raise NotImplementedError

    def outputs(self):
        raise NotImplementedError

    def oracle_sample(self, rows):
        """Run the oracle on query rows `rows`; return the work units done."""
        raise NotImplementedError

    def extra_figures(self, seconds):
        return {}


class DenseRunner(Runner):
    """The headline workload: one dense GQA CP-chunk call (KV folded in-kernel)."""

    name = "dense_gqa"

    def __init__(self, device=None, kv_chunks=False):
        self.w = w = inputs.dense_gqa()
        self.kv_chunks = kv_chunks
        Tq, Hq, D = w.q.shape
        qpos = w.causal_offset + np.arange(Tq)
        pairs = int(np.minimum(qpos + 1, w.Tk).sum())          # causal, one sequence
        self.pairs_per_head = pairs
        self.work = 4.0 * D * pairs * Hq
        self.n_rows = Tq
        if kv_chunks:
            self.name = "dense_gqa_4chunks"
            self.launches_per_step = 2                        # chunk summaries, LSE merge
            how = ("KV as 4 chunks of 2048: per-chunk finalised summaries (O_c, LSE_c) only, "
                   "then cpattn_lse_merge (chunk 3 fully masked, neutral)")
        else:
            how = "KV folded in-kernel (4 chunks of 2048, chunk 3 fully masked)"
        self.config = {
            "workload": "dense causal CP chunk, bf16 in / fp32 acc: 2048 queries (rank 2 of 4, "
                        "causal_offset 4096) x 8192 keys, 16 q heads / 4 kv heads, d=128, " + how,
            "Tq": Tq, "Tk": w.Tk, "Hq": Hq, "Hkv": w.k.shape[1], "D": D,
            "causal_offset": w.causal_offset, "permitted_pairs_per_head": pairs,
            "l2": L2_NOTE, "seed": 0,
        }
        if device is not None:
            self.q, self.k, self.v = (t.to(device) for t in (w.q, w.k, w.v))
            self.o = torch.empty((Tq, Hq, w.v.shape[2]), dtype=torch.bfloat16, device=device)
            self.lse = torch.empty((Tq, Hq), dtype=torch.float32, device=device)
            self.ws = torch.empty(64 << 20, dtype=torch.uint8, device=device)   # per-piece summaries
            if kv_chunks:
                n = -(-w.Tk // w.kv_chunk_len)
                self.po = torch.empty((n, Tq, Hq, D), dtype=torch.float32, device=device)
                self.pl = torch.empty((n, Tq, Hq), dtype=torch.float32, device=device)

    def device_inputs(self):
        return [self.q, self.k, self.v]

    def step(self, q, k, v):
        from context_attention_softmax_gb300 import cpattn_chunk_fwd, cpattn_lse_merge
        w = self.w
        if self.kv_chunks:
            cpattn_chunk_fwd(q, k, v, scale=w.scale, causal=True, causal_offset=w.causal_offset,
                             kv_chunk_len=w.kv_chunk_len, partial_o=self.po, partial_lse=self.pl,
                             workspace=self.ws, merged=False)
            cpattn_lse_merge(self.po, self.pl, out=self.o, lse=self.lse)
        else:
            cpattn_chunk_fwd(q, k, v, scale=w.scale, causal=True, causal_offset=w.causal_offset,
                             out=self.o, lse=self.lse, workspace=self.ws)

    def outputs(self):
        return [self.o, self.lse]

    def oracle_sample(self, rows):
        import oracle as orc
        w = self.w
        if not hasattr(self, "_f64"):
            self._f64 = (inputs.as_f64(w.q), inputs.as_f64(w.k), inputs.as_f64(w.v))
            self._lay = orc.make_layout(w.Tq, w.Tk, True, w.causal_offset)
        q, k, v = self._f64
        if self.kv_chunks:
            orc.summarised_attention(q, k, v, w.scale, self._lay, w.kv_chunk_len, rows=rows)
        else:
            orc.dense_attention(q, k, v, w.scale, self._lay, rows=rows)
        qpos = w.causal_offset + rows
        return 4.0 * w.q.shape[2] * float(np.minimum(qpos + 1, w.Tk).sum()) * w.q.shape[1]


class DenseBwdRunner(Runner):
    """Backward of the headline workload: dq, dk, dv from the forward's O and
    LSE and a seeded d_out (prep, dk/dv kernel, dq kernel)."""

    name = "dense_gqa_bwd"
    kernel = "cpattn_chunk_bwd (bwd_prep_kernel, then bwd_kernel: dk/dv and dq CTAs in one launch)"
    launches_per_step = 3   # interval init, prep, bwd_kernel (dk/dv and dq CTAs)

    def __init__(self, device):
        from context_attention_softmax_gb300 import cpattn_chunk_fwd
        self.w = w = inputs.dense_gqa()
        Tq, Hq, D = w.q.shape
        qpos = w.causal_offset + np.arange(Tq)
        pairs = int(np.minimum(qpos + 1, w.Tk).sum())
        # the usual count: five 2*d products per permitted pair and head
        # (S recomputed, dP, dV, dQ, dK)
        self.work = 10.0 * D * pairs * Hq
        self.n_rows = Tq
        self.q, self.k, self.v = (t.to(device) for t in (w.q, w.k, w.v))
        self.o, self.lse = cpattn_chunk_fwd(self.q, self.k, self.v, scale=w.scale, causal=True,
                                            causal_offset=w.causal_offset)
        rng = np.random.default_rng(7)
        self.g_host = inputs.to_device_dtype(
            (rng.standard_normal(tuple(self.o.shape)) * 0.5).astype(np.float32), "bf16")
        self.g = self.g_host.to(device)
        self.dq = torch.empty(self.q.shape, dtype=torch.float32, device=device)
        self.dk = torch.empty(self.k.shape, dtype=torch.float32, device=device)
        self.dv = torch.empty(self.v.shape, dtype=torch.float32, device=device)
        self.ws = torch.empty(16 << 20, dtype=torch.uint8, device=device)
        self.config = {"workload": "backward of the dense causal CP chunk: 2048 queries (causal_offset "
                                   "4096) x 8192 keys, 16 q heads / 4 kv heads, d=128; bf16 q, k, v, "
                                   "o, d_out, fp32 dq, dk, dv",
                       "permitted_pairs_per_head": pairs,
                       "flops_note": "10 d per permitted pair and head (5 products of 2 d)",
                       "l2": L2_NOTE}

    def device_inputs(self):
        return [self.q, self.k, self.v, self.o, self.lse, self.g]

    def step(self, q, k, v, o, lse, g):
        from context_attention_softmax_gb300 import cpattn_chunk_bwd
        w = self.w
        cpattn_chunk_bwd(q, k, v, o, lse, g, scale=w.scale, causal=True,
                         causal_offset=w.causal_offset, dq=self.dq, dk=self.dk, dv=self.dv,
                         workspace=self.ws)

    def outputs(self):
        return [self.dq, self.dk, self.dv]

    def oracle_sample(self, rows):
        """The oracle backward of the query rows `rows` (their dq, and their
        contribution to dk, dv)."""
        import oracle as orc
        w = self.w
        if not hasattr(self, "_f64"):
            self._f64 = (inputs.as_f64(w.q), inputs.as_f64(w.k), inputs.as_f64(w.v),
                         inputs.as_f64(self.g_host))
        q, k, v, g = self._f64
        lay = orc.make_layout(len(rows), w.Tk, True, 0)
        lay.qpos = w.causal_offset + np.asarray(rows)
        lay.qseq = np.zeros(len(rows), dtype=np.int64)
        orc.dense_attention_backward(q[rows], k, v, w.scale, lay, g[rows])
        qpos = w.causal_offset + rows
        return 10.0 * w.q.shape[2] * float(np.minimum(qpos + 1, w.Tk).sum()) * w.q.shape[1]


class ZigzagRunner(Runner):
    """All 8 zigzag ranks of the packed THD varlen workload (8 calls per step)."""

    name = "zigzag"

    def __init__(self, device):
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
        # The 8 rank calls are independent (own queries and outputs, shared
        # read-only K/V), as on 8 GPUs: each gets its own stream, started
        # after everything already on the caller's stream and joined back
        # into it, so one call's last CTAs overlap the other calls' work
        # (0.623 -> 0.446 ms per step against one stream).  Each stream has
        # its own workspace.
        self.streams = [torch.cuda.Stream(device) for _ in range(z.cp_size)]
        self.ws = [torch.empty(64 << 20, dtype=torch.uint8, device=device)
                   for _ in range(z.cp_size)]   # per-piece summaries
        lens = np.diff(z.cu_seqlens.astype(np.int64))
        pairs = int((lens * (lens + 1) // 2).sum())
        H, D = z.q_global.shape[1], z.q_global.shape[2]
        self.work = 4.0 * D * pairs * H
        self.n_rows = z.q_global.shape[0]
        self.launches_per_step = z.cp_size
        self.config = {"workload": "packed THD varlen, zigzag cp=8, 16384 tokens / 8 seqs, "
                                   "32 heads, d=128, causal; all 8 rank calls, one stream each",
                       "lengths": lens.tolist(), "permitted_pairs_per_head": pairs, "l2": L2_NOTE}

    def device_inputs(self):
        return self.qs + [self.k, self.v]

    def step(self, *ins):
        from context_attention_softmax_gb300 import cpattn_chunk_fwd
        z = self.z
        qs, k, v = ins[:z.cp_size], ins[z.cp_size], ins[z.cp_size + 1]
        main = torch.cuda.current_stream()
        start = torch.cuda.Event()
        start.record(main)
        for s in self.streams:
            s.wait_event(start)
        for r in range(z.cp_size):
            cpattn_chunk_fwd(qs[r], k, v, scale=z.scale, causal=True, cu_seqlens=self.cu,
                             q_chunk_map=self.maps[r], kv_chunk_map=self.kvmap,
                             chunk_len=z.chunk_len, out=self.o[r], lse=self.lse[r],
                             workspace=self.ws[r], stream=self.streams[r])
        for s in self.streams:
            main.wait_stream(s)

    def outputs(self):
        return self.o + self.lse

    def oracle_sample(self, rows):
        """rows: logical positions of the packed stream (whatever rank owns them)."""
        import oracle as orc
        z = self.z
        if not hasattr(self, "_f64"):
            self._f64 = tuple(inputs.as_f64(t) for t in (z.q_global, z.k_global, z.v_global))
            T = z.q_global.shape[0]
            self._lay = orc.make_layout(T, T, True, 0, z.cu_seqlens)
        q, k, v = self._f64
        orc.dense_attention(q, k, v, z.scale, self._lay, rows=rows)
        cu = z.cu_seqlens.astype(np.int64)
        s = np.searchsorted(cu, rows, side="right") - 1
        keys = rows - cu[s] + 1
        return 4.0 * q.shape[2] * q.shape[1] * float(keys.sum())


_DSA_INPUTS = {}


def dsa_inputs(device):
    """The DSA workload's inputs, drawn once per process (the attention and
    the indexer workloads share them)."""
    if device not in _DSA_INPUTS:
        _DSA_INPUTS[device] = inputs.dsa_absorbed(device=device)
    return _DSA_INPUTS[device]


class DsaRunner(Runner):
    """DSA top-2048 sparse attention on absorbed-MLA shapes."""

    name = "dsa"

    def __init__(self, device):
        self.w = w = dsa_inputs(device)
        self.q, self.kv = w.q.to(device), w.k.to(device)
        self.idx = w.indices.to(device)
        Tq, Hq, Dqk = w.q.shape
        self.o = torch.empty((Tq, Hq, 512), dtype=torch.bfloat16, device=device)
        self.lse = torch.empty((Tq, Hq), dtype=torch.float32, device=device)
        self.work = 2.0 * Tq * Hq * w.topk * (Dqk + 512)
        self.gathered_bytes = Tq * w.topk * Dqk * 2
        self.n_rows = Tq
        self.kernel = "cpattn_topk_sparse_fwd"
        self.config = {"workload": "DSA top-2048 sparse, absorbed MLA: 4096 q (causal_offset 16384) "
                                   "x 32768 kv, 128 heads / 1 kv head, dqk 576, dv 512 (v = first "
                                   "512 channels of k), indices from the seeded indexer",
                       "gathered_bytes": self.gathered_bytes, "l2": L2_NOTE}

    def device_inputs(self):
        return [self.q, self.kv, self.idx]

    def step(self, q, kv, idx):
        from context_attention_softmax_gb300 import cpattn_topk_sparse_fwd
        w = self.w
        cpattn_topk_sparse_fwd(q, kv, kv[:, :, :512], idx, block_size=1, scale=w.scale,
                               causal_offset=w.causal_offset, out=self.o, lse=self.lse)

    def outputs(self):
        return [self.o, self.lse]

    def extra_figures(self, seconds):
        return {"gathered_gbs": self.gathered_bytes / seconds / 1e9,
                "gathered_frac_of_hbm": self.gathered_bytes / seconds / 1e9 / hbm_peak()[0]}

    def oracle_sample(self, rows):
        import oracle as orc
        w = self.w
        if not hasattr(self, "_f64"):
            self._f64 = (inputs.as_f64(w.q), inputs.as_f64(w.k))
            self._lay = orc.make_layout(w.Tq, w.Tk, True, w.causal_offset)
            self._idx = w.indices.numpy()
        q, kv = self._f64
        orc.sparse_attention(q, kv, kv[:, :, :512], w.scale, self._lay, self._idx, rows=rows)
        n_keys = (self._idx[rows, 0, :] >= 0).sum()
        return 2.0 * w.q.shape[1] * (w.q.shape[2] + 512) * float(n_keys)


class MobaRunner(Runner):
    """MoBA gate + block-sparse attention (gate, then the attention call)."""

    name = "moba"
    unit = "GB/s"
    scale = 1e9
    bound = "hbm"
    kernel = "moba step (cpattn_block_gate + cpattn_topk_sparse_fwd)"
    launches_per_step = 8   # gate: means, split, tensor-core gate; attention: count, scan,
    #                         scatter, attend, merge

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
        kb, qb, vb, ob = (t.numel() * t.element_size() for t in (self.k, self.q, self.v, self.o))
        selb, lseb = self.sel.numel() * 4, self.lse.numel() * 4
        # gate: K, Q read, sel written; attention: Q, K, V, sel read, O, LSE written
        self.work = float((kb + qb + selb) + (qb + kb + vb + selb + ob + lseb))
        self.n_rows = Tq
        self.config = {"workload": "MoBA gate (top-3 + own of 512-key blocks) + block-sparse "
                                   "attention: 8192 q (causal_offset 57344) x 65536 kv, 32 heads, "
                                   "d=128",
                       "compulsory_bytes": int(self.work),
                       "compulsory_bytes_note": "gate reads K and Q and writes sel; attention "
                                                "reads Q, K, V and sel and writes O and LSE "
                                                "(K counted twice)",
                       "attention_flops": self.flops, "l2": L2_NOTE}

    def device_inputs(self):
        return [self.q, self.k, self.v]

    def step(self, q, k, v):
        from context_attention_softmax_gb300 import cpattn_block_gate, cpattn_topk_sparse_fwd
        w = self.w
        cpattn_block_gate(q, k, w.block_size, w.topk, causal_offset=w.causal_offset,
                          sel=self.sel, workspace=self.ws)
        cpattn_topk_sparse_fwd(q, k, v, self.sel, block_size=w.block_size, scale=w.scale,
                               causal_offset=w.causal_offset, out=self.o, lse=self.lse,
                               workspace=self.ws_sparse)

    def outputs(self):
        return [self.o, self.lse, self.sel]

    def extra_figures(self, seconds):
        return {"attention_tflops": self.flops / seconds / 1e12}

    def oracle_sample(self, rows):
        import oracle as orc
        w = self.w
        if not hasattr(self, "_f64"):
            self._f64 = (inputs.as_f64(w.q), inputs.as_f64(w.k), inputs.as_f64(w.v))
            self._lay = orc.make_layout(w.Tq, w.Tk, True, w.causal_offset)
        q, k, v = self._f64
        sel = orc.moba_block_gate(q, k, self._lay.qpos, w.block_size, w.topk, rows=rows)
        full = np.full((w.Tq,) + sel.shape[1:], -1, dtype=np.int32)
        full[rows] = sel
        orc.moba_attention(q, k, v, w.scale, self._lay, full, w.block_size, rows=rows)
        return self.work * len(rows) / w.Tq


class IndexerRunner(Runner):
    """The DSA indexer: top-2048 keys of 4096 queries at offset 16384 over 32768
    keys, 4 fp32 indexer heads of 128 (the indices the DSA workload attends to)."""

    name = "dsa_indexer"
    bound = "alu"
    kernel = ("cpattn_dsa_indexer (norms, operand split, tile intervals, tensor-core scores, "
              "selection)")
    launches_per_step = 5   # norms, split, tile intervals, scores, selection

    def __init__(self, device):
        self.w = w = dsa_inputs(device)
        self.qI, self.kI, self.wt = (w.extra[k].to(device) for k in ("qI", "kI", "w"))
        Tq, H, D = self.qI.shape
        Tk = self.kI.shape[0]
        self.out = torch.empty((Tq, w.topk), dtype=torch.int32, device=device)
        import ctypes
        from context_attention_softmax_gb300 import _lib, _args
        a = _args(self.qI, self.kI.unsqueeze(1), None, 1.0, True, w.causal_offset, None, None, None,
                  0, None, None)
        nbytes = _lib.load().cpattn_workspace_size(_lib.OP_DSA_INDEXER, ctypes.byref(a), w.topk, 1)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)
        n_keys = np.minimum(w.causal_offset + np.arange(Tq) + 1, Tk)     # causal, one sequence
        self.work = 2.0 * float(n_keys.sum()) * H * D
        self.n_rows = Tq
        self.config = {"workload": "DSA indexer top-2048: 4096 q (offset 16384) x 32768 keys, "
                                   "4 fp32 indexer heads x 128, scores sum_h w_h relu(qI.kI), "
                                   "selection exact against float64",
                       "permitted_pairs": int(n_keys.sum()), "l2": L2_NOTE}

    def device_inputs(self):
        return [self.qI, self.kI, self.wt]

    def step(self, qI, kI, wt):
        from context_attention_softmax_gb300 import cpattn_dsa_indexer
        cpattn_dsa_indexer(qI, kI, wt, self.w.topk, causal_offset=self.w.causal_offset,
                           out=self.out, workspace=self.ws)

    def outputs(self):
        return [self.out]

    def oracle_sample(self, rows):
        import oracle as orc
        w = self.w
        if not hasattr(self, "_np"):
            self._np = tuple(w.extra[k].numpy() for k in ("qI", "kI", "w"))
            self._lay = orc.make_layout(self._np[0].shape[0], self._np[1].shape[0], True,
                                        w.causal_offset)
        qI, kI, wt = self._np
        orc.dsa_indexer_topk(qI, kI, wt, self._lay, w.topk, rows=rows)
        n_keys = np.minimum(w.causal_offset + np.asarray(rows) + 1, kI.shape[0])
        return 2.0 * float(n_keys.sum()) * qI.shape[1] * qI.shape[2]


class MlaVUpRunner(Runner):
    """Value up-projection after absorbed attention: [4096, 128, 512] latent
    outputs x up_v_weight [128, 512, 128] (the DSA workload's shapes)."""

    name = "mla_v_up"
    unit = "GB/s"
    scale = 1e9
    bound = "hbm"
    kernel = "mla_gemm_kernel (cpattn_mla_v_up)"

    def __init__(self, device):
        self.w = w = inputs.mla_v_up()
        self.o, self.wt = w.o_latent.to(device), w.up_v_weight.to(device)
        T, H, L = self.o.shape
        V = self.wt.shape[2]
        self.out = torch.empty((T, H, V), dtype=torch.bfloat16, device=device)
        self.flops = 2.0 * T * H * L * V
        self.work = float(self.o.numel() * 2 + self.wt.numel() * 2 + self.out.numel() * 2)
        self.n_rows = T
        self.config = {"workload": "absorbed-MLA value up-projection: o_latent [4096, 128, 512] "
                                   "x up_v_weight [128, 512, 128] -> [4096, 128, 128], bf16 in, "
                                   "fp32 accumulate",
                       "compulsory_bytes": int(self.work), "flops": self.flops, "l2": L2_NOTE}

    def device_inputs(self):
        return [self.o, self.wt]

    def step(self, o, wt):
        from context_attention_softmax_gb300 import cpattn_mla_v_up
        cpattn_mla_v_up(o, wt, out=self.out)

    def outputs(self):
        return [self.out]

    def extra_figures(self, seconds):
        return {"tflops": self.flops / seconds / 1e12}

    def oracle_sample(self, rows):
        from oracle import mla
        if not hasattr(self, "_f64"):
            self._f64 = (inputs.as_f64(self.w.o_latent), inputs.as_f64(self.w.up_v_weight))
        o, wt = self._f64
        mla.absorbed_v_up(o[rows], wt)
        return self.work * len(rows) / self.n_rows


class MlaKvRunner(Runner):
    """K/V materialisation from gathered latents: 32768 tokens, latent 512,
    128 heads x (128 key + 128 value) channels, shared rope key 64."""

    name = "mla_kv"
    kernel = "mla_gemm_kernel (cpattn_mla_kv_materialise)"

    def __init__(self, device):
        self.w = w = inputs.mla_kv()
        self.c, self.ks, self.wb = (t.to(device) for t in (w.kv_c, w.k_shared, w.wkv_b))
        T, L = self.c.shape
        R = self.ks.shape[1]
        self.k = torch.empty((T, w.H, w.N + R), dtype=torch.bfloat16, device=device)
        self.v = torch.empty((T, w.H, w.V), dtype=torch.bfloat16, device=device)
        self.work = 2.0 * T * L * w.H * (w.N + w.V)
        self.bytes = float(sum(t.numel() * 2 for t in (self.c, self.ks, self.wb, self.k, self.v)))
        self.n_rows = T
        self.config = {"workload": "MLA K/V materialisation from gathered latents: kv_c [32768, 512] "
                                   "x wkv_b^T [512, 128 x 256] -> K [32768, 128, 128 + 64] "
                                   "(shared rope key appended), V [32768, 128, 128], bf16 in, "
                                   "fp32 accumulate",
                       "compulsory_bytes": int(self.bytes), "l2": L2_NOTE}

    def device_inputs(self):
        return [self.c, self.ks, self.wb]

    def step(self, c, ks, wb):
        from context_attention_softmax_gb300 import cpattn_mla_kv_materialise
        w = self.w
        cpattn_mla_kv_materialise(c, ks, wb, w.H, w.N, w.V, k_out=self.k, v_out=self.v)

    def outputs(self):
        return [self.k, self.v]

    def extra_figures(self, seconds):
        return {"gbs": self.bytes / seconds / 1e9}

    def oracle_sample(self, rows):
        from oracle import mla
        w = self.w
        if not hasattr(self, "_f64"):
            self._f64 = tuple(inputs.as_f64(t) for t in (w.kv_c, w.k_shared, w.wkv_b))
        c, ks, wb = self._f64
        mla.materialise_kv(c[rows], ks[rows], wb, w.H, w.N, w.V)
        return self.work * len(rows) / self.n_rows


RUNNERS = {"dense_gqa": DenseRunner,
           "dense_gqa_4chunks": lambda dev: DenseRunner(dev, kv_chunks=True),
           "zigzag": ZigzagRunner, "dsa": DsaRunner, "moba": MobaRunner,
           "dsa_indexer": IndexerRunner, "mla_v_up": MlaVUpRunner, "mla_kv": MlaKvRunner,
           "dense_gqa_bwd": DenseBwdRunner}
ALL_ORDER = ["dense_gqa", "dense_gqa_4chunks", "dense_gqa_bwd", "zigzag", "dsa", "moba",
             "dsa_indexer", "mla_v_up", "mla_kv"]


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


def hbm_peak():
    p, src = load_peaks()
    return float(p.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])), src


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled in the background.

    start() returns once nvidia-smi has written its first sample, so the
    sampler is running before the timed steps begin; mark() records the host
    time at the start and at the end of the timed steps; stop() waits for
    one sample after the end and reports the samples inside that window,
    widened to the nearest sample on either side when the window is shorter
    than the sampling interval (a few-millisecond timed region)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    INTERVAL_MS = 50

    def __init__(self, gpu_index):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.proc = None
        self.gpu = gpu_index
        self.window = [None, None]

    def _rows(self):
        self.f.flush()
        with open(self.f.name) as fh:
            rows = [r.split(",") for r in fh.read().strip().splitlines() if r.count(",") >= 9]
        out = []
        for r in rows:
            try:
                sm, smax = float(r[2]), float(r[3])
            except ValueError:
                continue
            try:   # host time of the sample; None if the format is not the expected one
                t = datetime.datetime.strptime(r[0].strip(), "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                t = None
            out.append((t, sm, smax, [v.strip().lower() for v in r[6:10]]))
        return out

    def _wait_rows(self, pred, timeout_s):
        t_end = time.time() + timeout_s
        while time.time() < t_end:
            if pred(self._rows()):
                return True
            time.sleep(0.01)
        return False

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", str(self.INTERVAL_MS)],
                stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
            return
        self._wait_rows(lambda rows: len(rows) > 0, 5.0)

    def mark(self, which):
        self.window[which] = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        t0, t1 = self.window
        if t1 is not None:   # one sample after the timed steps
            self._wait_rows(lambda rows: any(t is not None and t > t1 for t, *_ in rows), 2.0)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = self._rows()
        os.unlink(self.f.name)
        timed = [r for r in rows if r[0] is not None]
        have_window = t0 is not None and t1 is not None
        inside = [r for r in timed if have_window and t0 <= r[0] <= t1]
        chosen = inside
        if not inside and have_window:
            before = [r for r in timed if r[0] < t0][-1:]
            after = [r for r in timed if r[0] > t1][:1]
            chosen = before + after
        if not chosen:
            chosen = rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        for _, _, _, flags in chosen:
            for n, val in zip(names, flags):
                if val == "active":
                    reasons.add(n)
        sm = [r[1] for r in chosen]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in chosen) if chosen else None,
                "reasons": sorted(reasons), "samples": len(chosen),
                "samples_in_timed_region": len(inside),
                "timed_region_ms": None if t0 is None or t1 is None else round(1e3 * (t1 - t0), 2)}


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


def time_steps(fn, steps, warmup, flush, world, marks=None):
    """Per-step device times (ms) of `steps` timed calls of fn, L2 flushed before each.

    marks(0) / marks(1), if given, are called on the host right before the
    first timed step is enqueued and right after the last one has finished."""
    for _ in range(warmup):
        fn()
    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    torch.cuda.synchronize()
    barrier(world)
    # a backlog of flush writes (~0.6 ms of GPU work) so that the host has
    # enqueued the first step before the GPU reaches it
    for _ in range(16):
        flush.zero_()
    if marks is not None:
        marks(0)
    for s in range(steps):
        flush.zero_()
        ev[s][0].record(stream)
        fn()
        ev[s][1].record(stream)
    torch.cuda.synchronize()
    if marks is not None:
        marks(1)
    barrier(world)
    return [a.elapsed_time(b) for a, b in ev]


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


def cpu_baseline(runner, budget_s=8.0, batch=16):
    """Time the oracle as it stands on a bounded sample of query rows."""
    rng = np.random.default_rng(123)
    n = runner.n_rows
    runner.oracle_sample(np.array([n - 1]))   # untimed: widens the inputs to float64 once
    t0 = time.perf_counter()
    work = 0.0
    rows_done = 0
    while time.perf_counter() - t0 < budget_s:
        rows = np.sort(rng.choice(n, size=min(batch, n), replace=False))
        work += runner.oracle_sample(rows)
        rows_done += len(rows)
    dt = time.perf_counter() - t0
    return {"value": work / dt / runner.scale, "unit": runner.unit,
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle", **host_info(),
            "sample": f"{rows_done} query rows drawn at random out of {n} (all heads, every "
                      f"permitted or selected key of each row), float64 numpy, {dt:.1f} s; "
                      "value = the rows' share of the workload's work / time"}


def roofline(runner, mean_ms, dev):
    peaks, src = load_peaks()
    sec = mean_ms * 1e-3
    if runner.bound == "tensor":
        achieved = runner.work / sec / 1e12
        peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None, "peak_source": f"{src} bf16 burst"}
    elif runner.bound == "alu":
        # fp32 FMA pipes: SMs x 128 lanes x 2 FLOP x the maximum SM clock
        achieved = runner.work / sec / 1e12
        sm_mhz = float(peaks.get("sm_max_mhz", 2070.0))
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        peak = n_sm * 128 * 2 * sm_mhz * 1e6 / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": None,
                "peak_source": f"fp32 FMA: {n_sm} SMs x 128 lanes x 2 x {sm_mhz:.0f} MHz "
                               "(the ceiling of these fp32 scores on the FMA pipes; the scores "
                               "run on the tensor cores and the selection dominates the step)"}
    else:
        achieved = runner.work / sec / 1e9
        peak = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": None, "peak_source": f"{src} copy"}
    roof["kernel"] = runner.kernel
    traffic, what = measured_traffic(runner.name)
    if traffic is not None:
        roof["traffic"] = traffic
        roof["kernel"] = what
        roof["traffic_note"] = "ncu dram bytes read + written per launch, see profiles/"
    else:
        roof["traffic_note"] = what
    return roof


def measure(runner, args, world, dev, flush, with_cpu):
    """Timed steps, e2e steps and the oracle baseline of one workload."""
    ins = runner.device_inputs()
    clocks = ClockSampler(dev.index or 0)
    clocks.start()
    times = time_steps(lambda: runner.step(*ins), args.steps, args.warmup, flush, world,
                       marks=clocks.mark)
    clk = clocks.stop()
    mean_ms = max_over_ranks(statistics.mean(times), world)
    rec = {
        "value": world * runner.work / (mean_ms * 1e-3) / runner.scale, "unit": runner.unit,
        "ms_per_step": mean_ms, "ms_min": min(times), "ms_median": statistics.median(times),
        "ms_p90": float(np.percentile(times, 90)),
        "config": runner.config, "roofline": roofline(runner, mean_ms, dev), "clocks": clk,
        "gpu_launches": runner.launches_per_step * args.steps,
    }
    rec.update(runner.extra_figures(mean_ms * 1e-3))

    # end to end through the public API: pinned host inputs in, outputs out
    hin = [t.detach().to("cpu").pin_memory() for t in ins]
    din = [torch.empty_like(t) for t in ins]
    outs = runner.outputs()
    hout = [torch.empty(t.shape, dtype=t.dtype, device="cpu").pin_memory() for t in outs]

    def e2e_step():
        for h, d in zip(hin, din):
            d.copy_(h, non_blocking=True)
        runner.step(*din)
        for d, h in zip(outs, hout):
            h.copy_(d, non_blocking=True)

    et = time_steps(e2e_step, args.steps, max(args.warmup, 3), flush, world)
    e_ms = max_over_ranks(statistics.mean(et), world)
    rec["e2e"] = {"value": world * runner.work / (e_ms * 1e-3) / runner.scale, "unit": runner.unit,
                  "ms_per_step": e_ms,
                  "h2d_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hin)),
                  "d2h_bytes_per_step": int(sum(t.numel() * t.element_size() for t in hout))}
    del hin, din, hout
    if with_cpu:
        rec["cpu_baseline"] = cpu_baseline(runner)
    return rec


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------

def run_reference(args, world, rank):
    if rank != 0:
        return
    runner = DenseRunner(None)
    rng = np.random.default_rng(7)
    per_step_rows = 16
    for _ in range(args.warmup):
        runner.oracle_sample(np.sort(rng.choice(runner.w.Tq, per_step_rows, replace=False)))
    times, work = [], []
    for _ in range(args.steps):
        rows = np.sort(rng.choice(runner.w.Tq, per_step_rows, replace=False))
        t0 = time.perf_counter()
        work.append(runner.oracle_sample(rows))
        times.append(time.perf_counter() - t0)
    value = sum(work) / sum(times) / 1e12
    ms_full = runner.work / (value * 1e12) * 1e3
    line = {
        "impl": "reference", "metric": METRIC, "value": value,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.mean(times), "ms_full_problem_extrapolated": ms_full,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
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
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    with_cpu = world == 1 and not args.no_cpu_baseline
    names = ALL_ORDER if args.workload == "all" else [args.workload]
    records = {}
    for name in names:
        runner = RUNNERS[name](dev)
        records[name] = measure(runner, args, world, dev, flush, with_cpu)
        del runner
        torch.cuda.empty_cache()
    if rank != 0:
        return
    head_name = names[0]
    head = records.pop(head_name)
    line = {
        "metric": METRIC,
        "value": head["value"], "unit": head["unit"], "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
        "ms_min": head["ms_min"], "ms_median": head["ms_median"], "ms_p90": head["ms_p90"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1), bf16-rounded; no dataset)",
        "config": head["config"], "roofline": head["roofline"], "clocks": head["clocks"],
        "gpu_launches": head["gpu_launches"] + sum(r["gpu_launches"] for r in records.values()),
        "e2e": head["e2e"],
    }
    if "cpu_baseline" in head:
        line["cpu_baseline"] = head["cpu_baseline"]
    if records:
        line["workloads"] = records
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawTextHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps per workload (default: 100 for our arm, 20 for the "
                         "reference arm)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["all"] + sorted(RUNNERS), default="all",
                    help="all (default): the headline plus one record per other workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.steps is None:
        args.steps = 20 if args.impl == "reference" else 100
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
