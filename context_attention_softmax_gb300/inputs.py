"""Seeded synthetic inputs for the five workloads (shared by tests, bench and smoke).

This module only draws and lays out input tensors; it computes no attention.
Every tensor comes from ``numpy.random.default_rng(seed)`` as standard-normal
float64, times a stated factor, cast to float32 and, for bf16 workloads,
rounded to bfloat16 (round-to-nearest-even, by torch).  Tensors are drawn in
the order Q, K, V, then the extras.  The float64 copies handed to the oracle
are the exact values handed to the GPU, widened.

The DSA workload's key indices are part of its input: per query, the 2048
keys with the largest indexer score sum_h w_h * relu(qI_h . kI_j) among keys at
or before the query's position (ties to the lower key), listed in ascending
order and padded with -1.  They are computed here with torch float32 ops on
the device given, so both sides of a comparison receive the same tensor.

Layouts: every tensor is token-major [T, H, D] with D contiguous.  For the
zigzag workload the gathered KV buffer is rank-major: slot 2r holds logical
chunk r and slot 2r+1 holds logical chunk 2*cp-1-r, and rank r's local query
rows are its two chunks in that order.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def _draw(rng, shape, factor=1.0):
    return (rng.standard_normal(shape) * factor).astype(np.float32)


def to_device_dtype(x32: np.ndarray, dtype: str) -> torch.Tensor:
    """float32 numpy -> torch CPU tensor of the workload dtype (bf16 by RNE)."""
    t = torch.from_numpy(np.ascontiguousarray(x32))
    return t.to(torch.bfloat16) if dtype == "bf16" else t.clone()


def as_f64(t: torch.Tensor) -> np.ndarray:
    """The exact values of a bf16/fp32 tensor, widened to float64 numpy."""
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


@dataclass
class Workload:
    name: str
    dtype: str                      # "bf16" or "fp32"
    q: torch.Tensor                 # [Tq, Hq, Dqk]
    k: torch.Tensor                 # [Tk, Hkv, Dqk]
    v: torch.Tensor                 # [Tk, Hkv, Dv]  (may alias k's storage)
    scale: float
    causal: bool = True
    causal_offset: int = 0
    cu_seqlens: np.ndarray | None = None
    q_chunk_map: np.ndarray | None = None
    kv_chunk_map: np.ndarray | None = None
    chunk_len: int = 0
    kv_chunk_len: int = 0
    indices: torch.Tensor | None = None   # int32 [Tq, index_heads, topk]
    block_size: int = 1
    topk: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def Tq(self):
        return self.q.shape[0]

    @property
    def Tk(self):
        return self.k.shape[0]


def tiny_fp32(seed=0, Tq=128, Tk=256, D=64, offset=128, kv_chunk_len=128):
    """Tiny dense causal CP chunk in fp32: chunk 1 of a 256-token sequence.

    Queries are global positions 128..255 against all 256 keys, computed as
    two KV-chunk summaries then merged.  Q, K, V iid N(0, 1), 1 head, D = 64.
    """
    rng = np.random.default_rng(seed)
    q = _draw(rng, (Tq, 1, D))
    k = _draw(rng, (Tk, 1, D))
    v = _draw(rng, (Tk, 1, D))
    return Workload("tiny_fp32_cp_chunk", "fp32", to_device_dtype(q, "fp32"),
                    to_device_dtype(k, "fp32"), to_device_dtype(v, "fp32"),
                    scale=1.0 / np.sqrt(D), causal=True, causal_offset=offset,
                    kv_chunk_len=kv_chunk_len)


def dense_gqa(seed=0, global_seq=8192, cp_size=4, rank=2, Hq=16, Hkv=4, D=128,
              factor=0.5, kv_chunks=4, Tk=None, v_factor=None):
    """Dense causal CP chunk, GQA, bf16: rank ``rank`` of ``cp_size``.

    Default: 2048 queries at causal_offset 4096 against 8192 keys, 16 query
    heads over 4 KV heads, D = 128, scale 1/sqrt(128), N(0,1) * 0.5, the KV
    processed in 4 chunks of 2048.
    """
    rng = np.random.default_rng(seed)
    local = global_seq // cp_size
    Tk = global_seq if Tk is None else Tk
    q = _draw(rng, (local, Hq, D), factor)
    k = _draw(rng, (Tk, Hkv, D), factor)
    v = _draw(rng, (Tk, Hkv, D), factor if v_factor is None else v_factor)
    return Workload(f"dense_causal_gqa_{local}x{Tk}_h{Hq}/{Hkv}_d{D}", "bf16",
                    to_device_dtype(q, "bf16"), to_device_dtype(k, "bf16"),
                    to_device_dtype(v, "bf16"), scale=1.0 / np.sqrt(D), causal=True,
                    causal_offset=rank * local,
                    kv_chunk_len=-(-Tk // kv_chunks) if kv_chunks else 0)


def seeded_lengths(rng, n_seqs, total, lo, hi):
    """n_seqs lengths drawn uniformly from [lo, hi], rescaled to sum to total.

    Each length is scaled by total / sum and floored; the remainder goes to the
    last sequence.
    """
    raw = rng.integers(lo, hi + 1, n_seqs)
    lens = np.floor(raw * (total / raw.sum())).astype(np.int64)
    lens[-1] += total - lens.sum()
    return lens


@dataclass
class ZigzagWorkload:
    """Packed THD varlen input split over cp_size ranks in the zigzag layout."""

    name: str
    q_global: torch.Tensor          # [T, H, D] logical order
    k_global: torch.Tensor
    v_global: torch.Tensor
    k_gathered: torch.Tensor        # [T, H, D] rank-major physical order
    v_gathered: torch.Tensor
    kv_chunk_map: np.ndarray        # physical slot -> logical chunk
    cu_seqlens: np.ndarray          # int32 [S+1] over logical positions
    chunk_len: int
    cp_size: int
    scale: float
    lengths: np.ndarray

    def rank_chunks(self, r):
        return np.array([r, 2 * self.cp_size - 1 - r], dtype=np.int32)

    def rank_q(self, r):
        """Rank r's local query rows: its two logical chunks, in that order."""
        L = self.chunk_len
        return torch.cat([self.q_global[c * L:(c + 1) * L] for c in self.rank_chunks(r)])

    def rank_workload(self, r) -> Workload:
        return Workload(f"{self.name}_rank{r}", "bf16", self.rank_q(r), self.k_gathered,
                        self.v_gathered, scale=self.scale, causal=True, causal_offset=0,
                        cu_seqlens=self.cu_seqlens, q_chunk_map=self.rank_chunks(r),
                        kv_chunk_map=self.kv_chunk_map, chunk_len=self.chunk_len)


def zigzag_varlen(seed=0, total=16384, n_seqs=8, len_lo=512, len_hi=4096, cp_size=8,
                  H=32, D=128):
    """Packed THD varlen workload, zigzag over ``cp_size`` ranks, bf16.

    Default: 16384 tokens in 8 sequences with lengths drawn from [512, 4096]
    and renormalised, 32 heads, D = 128, causal, 16 chunks of 1024; rank r
    owns logical chunks r and 15 - r.
    """
    rng = np.random.default_rng(seed)
    lens = seeded_lengths(rng, n_seqs, total, len_lo, len_hi)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    q = to_device_dtype(_draw(rng, (total, H, D)), "bf16")
    k = to_device_dtype(_draw(rng, (total, H, D)), "bf16")
    v = to_device_dtype(_draw(rng, (total, H, D)), "bf16")
    n_chunks = 2 * cp_size
    L = total // n_chunks
    kv_map = np.array([c for r in range(cp_size) for c in (r, n_chunks - 1 - r)], dtype=np.int32)
    perm = torch.from_numpy(np.concatenate([np.arange(c * L, (c + 1) * L) for c in kv_map]))
    return ZigzagWorkload(f"thd_zigzag_cp{cp_size}_{total}tok_{n_seqs}seq_h{H}", q, k, v,
                          k[perm].contiguous(), v[perm].contiguous(), kv_map, cu, L,
                          cp_size, 1.0 / np.sqrt(D), lens)


def indexer_topk(qI: torch.Tensor, kI: torch.Tensor, w: torch.Tensor, qpos: torch.Tensor,
                 topk: int, row_block: int = 256) -> torch.Tensor:
    """Key indices chosen by the seeded indexer (input synthesis for DSA).

    score(i, j) = sum_h w_h * relu(qI[i, h] . kI[j]) over keys j <= qpos_i;
    the top ``topk`` keys by score (ties to the lower j), then sorted
    ascending; -1 pads rows with fewer permitted keys.  float32 on the device
    of the inputs.  Returns int32 [Tq, 1, topk].
    """
    Tq = qI.shape[0]
    Tk = kI.shape[0]
    out = torch.full((Tq, 1, topk), -1, dtype=torch.int32, device=qI.device)
    j = torch.arange(Tk, device=qI.device)
    for r0 in range(0, Tq, row_block):
        r1 = min(r0 + row_block, Tq)
        s = torch.einsum("ihd,jd->ihj", qI[r0:r1], kI).clamp_min_(0)
        s = torch.einsum("ihj,h->ij", s, w)
        ok = j[None, :] <= qpos[r0:r1, None]
        s = torch.where(ok, s, torch.full_like(s, float("-inf")))
        order = torch.sort(s, dim=1, descending=True, stable=True).indices[:, :topk]
        n_ok = ok.sum(dim=1)
        chosen = torch.where(torch.arange(order.shape[1], device=qI.device)[None, :] < n_ok[:, None],
                             order, torch.full_like(order, Tk))
        chosen = torch.sort(chosen, dim=1).values
        chosen = torch.where(chosen == Tk, torch.full_like(chosen, -1), chosen)
        out[r0:r1, 0, :chosen.shape[1]] = chosen.to(torch.int32)
    return out


def dsa_absorbed(seed=0, Tq=4096, Tk=32768, offset=16384, Hq=128, d_latent=512,
                 d_rope=64, topk=2048, index_heads=4, index_dim=128, device="cpu"):
    """DSA-style top-k sparse attention on absorbed-MLA shapes, bf16.

    Default: 4096 queries at causal_offset 16384, 128 heads sharing one KV
    head, key rows of 576 = 512 latent + 64 rope, values = the latent (the
    first 512 channels of the same rows), top-2048 key indices from the seeded
    indexer (4 heads, dim 128, float32, w ~ U(0, 1)).  Q, KV ~ N(0, 1).
    """
    rng = np.random.default_rng(seed)
    Dqk = d_latent + d_rope
    q = to_device_dtype(_draw(rng, (Tq, Hq, Dqk)), "bf16")
    kv = to_device_dtype(_draw(rng, (Tk, 1, Dqk)), "bf16")
    qI = torch.from_numpy(_draw(rng, (Tq, index_heads, index_dim))).to(device)
    kI = torch.from_numpy(_draw(rng, (Tk, index_dim))).to(device)
    w = torch.from_numpy(rng.uniform(0.0, 1.0, index_heads).astype(np.float32)).to(device)
    qpos = torch.arange(Tq, device=device) + offset
    idx = indexer_topk(qI, kI, w, qpos, topk).cpu()
    return Workload(f"dsa_absorbed_{Tq}x{Tk}_h{Hq}_top{topk}", "bf16", q, kv, kv[:, :, :d_latent],
                    scale=1.0 / np.sqrt(Dqk), causal=True, causal_offset=offset,
                    indices=idx, block_size=1, topk=topk,
                    extra={"qI": qI.cpu(), "kI": kI.cpu(), "w": w.cpu()})


def moba(seed=0, Tq=8192, Tk=65536, offset=57344, H=32, D=128, block_size=512, topk=3):
    """MoBA-style block-gated sparse attention, bf16.

    Default: 8192 queries at causal_offset 57344 against 65536 keys, 32 heads,
    D = 128, blocks of 512, top-3 gated blocks plus the own block.
    """
    rng = np.random.default_rng(seed)
    q = to_device_dtype(_draw(rng, (Tq, H, D)), "bf16")
    k = to_device_dtype(_draw(rng, (Tk, H, D)), "bf16")
    v = to_device_dtype(_draw(rng, (Tk, H, D)), "bf16")
    return Workload(f"moba_{Tq}x{Tk}_h{H}_b{block_size}_top{topk}", "bf16", q, k, v,
                    scale=1.0 / np.sqrt(D), causal=True, causal_offset=offset,
                    block_size=block_size, topk=topk)


@dataclass
class MlaVUpWorkload:
    o_latent: torch.Tensor      # bf16 [T, H, L]
    up_v_weight: torch.Tensor   # bf16 [H, L, V]


def mla_v_up(seed=0, T=4096, H=128, L=512, V=128):
    """Value up-projection after absorbed attention, bf16: the DSA workload's
    latent output shape [4096, 128, 512] times up_v_weight [128, 512, 128].
    o_latent ~ N(0, 1); up_v_weight ~ N(0, 1) / sqrt(L) (unit-variance output)."""
    rng = np.random.default_rng(seed)
    o = to_device_dtype(_draw(rng, (T, H, L)), "bf16")
    w = to_device_dtype(_draw(rng, (H, L, V), 1.0 / np.sqrt(L)), "bf16")
    return MlaVUpWorkload(o, w)


@dataclass
class MlaKvWorkload:
    kv_c: torch.Tensor          # bf16 [T, L]   gathered compressed latents
    k_shared: torch.Tensor      # bf16 [T, R]   gathered head-shared key
    wkv_b: torch.Tensor         # bf16 [H * (N + V), L]
    H: int
    N: int
    V: int


def mla_kv(seed=0, T=32768, H=128, L=512, N=128, V=128, R=64):
    """K/V materialisation from gathered latents, bf16, on the DSA workload's
    absorbed-MLA dims (latent 512, shared rope key 64) over its 32768-token
    gathered sequence, 128 heads with 128 key and 128 value channels each.
    kv_c, k_shared ~ N(0, 1); wkv_b ~ N(0, 1) / sqrt(L)."""
    rng = np.random.default_rng(seed)
    c = to_device_dtype(_draw(rng, (T, L)), "bf16")
    ks = to_device_dtype(_draw(rng, (T, R)), "bf16")
    wb = to_device_dtype(_draw(rng, (H * (N + V), L), 1.0 / np.sqrt(L)), "bf16")
    return MlaKvWorkload(c, ks, wb, H, N, V)
