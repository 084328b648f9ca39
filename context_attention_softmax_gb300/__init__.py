"""GB300 context-parallel chunk attention: thin PyTorch binding of libcpattn.so.

Each function marshals torch CUDA tensors (pointers, strides, the current
stream) into one C-ABI call of the same name (include/cpattn.h); every step of
the computation runs in the library's CUDA kernels.  Outputs not supplied by
the caller are allocated with torch (device memory plumbing only).
"""

from __future__ import annotations

import ctypes
import functools
import inspect
import math

import torch

from . import _lib
from ._lib import CPATTN_BF16, CPATTN_FP32, CpattnError  # noqa: F401

__all__ = [
    "cpattn_chunk_fwd", "cpattn_chunk_bwd", "cpattn_lse_merge", "cpattn_topk_sparse_fwd", "cpattn_block_gate",
    "cpattn_dsa_indexer", "cpattn_mla_v_up", "cpattn_mla_kv_materialise",
    "cpattn_workspace_size", "cpattn_version", "CpattnError",
]


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CPATTN_BF16
    if t.dtype == torch.float32:
        return CPATTN_FP32
    raise TypeError(f"unsupported dtype {t.dtype} (bf16 or fp32)")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _on_call_stream(fn):
    """Runs the call with its `stream` as torch's current stream, so that the
    tensors the binding creates (host index arrays copied to the device,
    outputs and workspaces the caller left out) are copied and allocated on
    the stream the kernels run on: their copies land before the kernels, and
    the caching allocator reuses their memory only after them."""
    pos = list(inspect.signature(fn).parameters).index("stream")

    @functools.wraps(fn)
    def wrapper(*args, **kwargs):
        stream = args[pos] if len(args) > pos else kwargs.get("stream")
        if stream is None:
            return fn(*args, **kwargs)
        with torch.cuda.stream(stream):
            return fn(*args, **kwargs)

    return wrapper


def _device_i32(x, device):
    if x is None:
        return None
    if isinstance(x, torch.Tensor):
        if x.dtype != torch.int32 or x.device != device:
            x = x.to(device=device, dtype=torch.int32)
        return x.contiguous()
    return torch.as_tensor(x, dtype=torch.int32, device=device).contiguous()


def _thd(name, t):
    if t.dim() != 3 or t.stride(2) != 1:
        raise ValueError(f"{name} must be [T, H, D] with the last dimension contiguous")


def _args(q, k, v, scale, causal, causal_offset, cu_seqlens, q_chunk_map, kv_chunk_map,
          chunk_len, o, lse, kv_chunk_len=0, partial_o=None, partial_lse=None, dev_status=None):
    _thd("q", q)
    _thd("k", k)
    if v is not None:
        _thd("v", v)
    a = _lib.AttnArgs()
    a.dtype = _code(q)
    a.q, a.q_stride_t, a.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    a.Tq, a.Hq, a.Dqk = q.shape
    a.k, a.k_stride_t, a.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    a.Tk, a.Hkv = k.shape[0], k.shape[1]
    if v is not None:
        a.v, a.v_stride_t, a.v_stride_h = v.data_ptr(), v.stride(0), v.stride(1)
        a.Dv = v.shape[2]
    a.scale = float(1.0 / math.sqrt(q.shape[2]) if scale is None else scale)
    a.causal = int(bool(causal))
    a.causal_offset = int(causal_offset)
    if cu_seqlens is not None:
        a.cu_seqlens, a.num_seqs = cu_seqlens.data_ptr(), cu_seqlens.numel() - 1
    if q_chunk_map is not None:
        a.q_chunk_map, a.n_q_chunks = q_chunk_map.data_ptr(), q_chunk_map.numel()
    if kv_chunk_map is not None:
        a.kv_chunk_map, a.n_kv_chunks = kv_chunk_map.data_ptr(), kv_chunk_map.numel()
    a.chunk_len = int(chunk_len)
    if o is not None:
        _thd("out", o)
        a.o, a.o_stride_t, a.o_stride_h = o.data_ptr(), o.stride(0), o.stride(1)
    a.lse = _ptr(lse)
    a.kv_chunk_len = int(kv_chunk_len)
    a.partial_o, a.partial_lse = _ptr(partial_o), _ptr(partial_lse)
    a.dev_status = _ptr(dev_status)
    return a


@_on_call_stream
def cpattn_chunk_fwd(q, k, v, scale=None, causal=True, causal_offset=0, cu_seqlens=None,
                     q_chunk_map=None, kv_chunk_map=None, chunk_len=0, kv_chunk_len=0,
                     out=None, lse=None, partial_o=None, partial_lse=None, dev_status=None,
                     workspace=None, stream=None, merged=True):
    """Dense CP-chunk attention; returns (out, lse) or, with kv_chunk_len > 0,
    (out, lse, partial_o, partial_lse) - out and lse None when merged=False
    (partial summaries only).  `workspace` (uint8, device) enables the
    SM-balanced schedule; one is allocated when it is missing or short."""
    dev = q.device
    cu, qm, km = (_device_i32(x, dev) for x in (cu_seqlens, q_chunk_map, kv_chunk_map))
    Tq, Hq = q.shape[0], q.shape[1]
    if not merged and kv_chunk_len > 0:
        out, lse = None, None
    else:
        if out is None:
            out = torch.empty((Tq, Hq, v.shape[2]), dtype=q.dtype, device=dev)
        if lse is None:
            lse = torch.empty((Tq, Hq), dtype=torch.float32, device=dev)
    if kv_chunk_len > 0:
        n = -(-k.shape[0] // kv_chunk_len)
        if partial_o is None:
            partial_o = torch.empty((n, Tq, Hq, v.shape[2]), dtype=torch.float32, device=dev)
        if partial_lse is None:
            partial_lse = torch.empty((n, Tq, Hq), dtype=torch.float32, device=dev)
    a = _args(q, k, v, scale, causal, causal_offset, cu, qm, km, chunk_len, out, lse,
              kv_chunk_len, partial_o, partial_lse, dev_status)
    lib = _lib.load()
    ws_bytes = lib.cpattn_workspace_size(_lib.OP_CHUNK_FWD, ctypes.byref(a), 0, 1)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _lib.check(lib.cpattn_chunk_fwd(ctypes.byref(a), _ptr(workspace) if ws_bytes else None,
                                    ws_bytes, _stream(stream)))
    if kv_chunk_len > 0:
        return out, lse, partial_o, partial_lse
    return out, lse


@_on_call_stream
def cpattn_chunk_bwd(q, k, v, out, lse, d_out, scale=None, causal=True, causal_offset=0,
                     cu_seqlens=None, q_chunk_map=None, kv_chunk_map=None, chunk_len=0,
                     dq=None, dk=None, dv=None, dev_status=None, workspace=None, stream=None):
    """Gradients (dq, dk, dv), fp32, of cpattn_chunk_fwd given its outputs
    (out, lse) and d_out; dk, dv hold this chunk's contribution to every
    gathered KV row."""
    dev = q.device
    cu, qm, km = (_device_i32(x, dev) for x in (cu_seqlens, q_chunk_map, kv_chunk_map))
    _thd("d_out", d_out)
    if dq is None:
        dq = torch.empty(q.shape, dtype=torch.float32, device=dev)
    if dk is None:
        dk = torch.empty(k.shape, dtype=torch.float32, device=dev)
    if dv is None:
        dv = torch.empty(v.shape, dtype=torch.float32, device=dev)
    for n, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _thd(n, t)
    a = _args(q, k, v, scale, causal, causal_offset, cu, qm, km, chunk_len, out, lse,
              dev_status=dev_status)
    lib = _lib.load()
    ws_bytes = lib.cpattn_workspace_size(_lib.OP_CHUNK_BWD, ctypes.byref(a), 0, 1)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _lib.check(lib.cpattn_chunk_bwd(ctypes.byref(a), d_out.data_ptr(), d_out.stride(0),
                                    d_out.stride(1), dq.data_ptr(), dq.stride(0), dq.stride(1),
                                    dk.data_ptr(), dk.stride(0), dk.stride(1), dv.data_ptr(),
                                    dv.stride(0), dv.stride(1),
                                    _ptr(workspace) if ws_bytes else None, ws_bytes,
                                    _stream(stream)))
    return dq, dk, dv


@_on_call_stream
def cpattn_lse_merge(part_o, part_lse, out=None, lse=None, out_dtype=torch.bfloat16, stream=None):
    """Merge finalised per-chunk (O_c, LSE_c) [n, Tq, H, Dv] / [n, Tq, H]."""
    n, Tq, H, Dv = part_o.shape
    if out is None:
        out = torch.empty((Tq, H, Dv), dtype=out_dtype, device=part_o.device)
    if lse is None:
        lse = torch.empty((Tq, H), dtype=torch.float32, device=part_o.device)
    po, pl = part_o.contiguous(), part_lse.contiguous()
    _lib.check(_lib.load().cpattn_lse_merge(n, po.data_ptr(), pl.data_ptr(), Tq, H, Dv,
                                            out.data_ptr(), _code(out), out.stride(0),
                                            out.stride(1), _ptr(lse), _stream(stream)))
    return out, lse


@_on_call_stream
def cpattn_topk_sparse_fwd(q, k, v, indices, block_size=1, scale=None, causal=True,
                           causal_offset=0, cu_seqlens=None, q_chunk_map=None, kv_chunk_map=None,
                           chunk_len=0, out=None, lse=None, dev_status=None, workspace=None,
                           stream=None):
    """Top-k sparse attention over token indices (block_size 1) or key blocks."""
    dev = q.device
    cu, qm, km = (_device_i32(x, dev) for x in (cu_seqlens, q_chunk_map, kv_chunk_map))
    idx = _device_i32(indices, dev)
    Tq, Hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty((Tq, Hq, v.shape[2]), dtype=q.dtype, device=dev)
    if lse is None:
        lse = torch.empty((Tq, Hq), dtype=torch.float32, device=dev)
    a = _args(q, k, v, scale, causal, causal_offset, cu, qm, km, chunk_len, out, lse,
              dev_status=dev_status)
    lib = _lib.load()
    ws_bytes = lib.cpattn_workspace_size(_lib.OP_TOPK_SPARSE_FWD, ctypes.byref(a), idx.shape[2],
                                         block_size)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _lib.check(lib.cpattn_topk_sparse_fwd(ctypes.byref(a), idx.data_ptr(), idx.shape[2],
                                          idx.shape[1], int(block_size), _ptr(workspace),
                                          ws_bytes, _stream(stream)))
    return out, lse


@_on_call_stream
def cpattn_block_gate(q, k, block_size, topk, causal_offset=0, q_chunk_map=None, chunk_len=0,
                      sel=None, workspace=None, stream=None):
    """MoBA block selection: int32 [Tq, Hq, topk + 1], ascending, -1 padded."""
    dev = q.device
    qm = _device_i32(q_chunk_map, dev)
    if sel is None:
        sel = torch.empty((q.shape[0], q.shape[1], topk + 1), dtype=torch.int32, device=dev)
    a = _args(q, k, None, 1.0, True, causal_offset, None, qm, None, chunk_len, None, None)
    lib = _lib.load()
    ws_bytes = lib.cpattn_workspace_size(_lib.OP_BLOCK_GATE, ctypes.byref(a), topk, block_size)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _lib.check(lib.cpattn_block_gate(ctypes.byref(a), int(block_size), int(topk), sel.data_ptr(),
                                     _ptr(workspace), ws_bytes, _stream(stream)))
    return sel


@_on_call_stream
def cpattn_dsa_indexer(qI, kI, w, topk, causal=True, causal_offset=0, cu_seqlens=None,
                       q_chunk_map=None, chunk_len=0, out=None, workspace=None, stream=None):
    """DSA indexer top-k: int32 [Tq, topk] key indices, ascending, -1 padded.

    qI: fp32 [Tq, H, D], kI: fp32 [Tk, 1, D] (or [Tk, D]), w: fp32 [H].
    """
    dev = qI.device
    if kI.dim() == 2:
        kI = kI.unsqueeze(1)
    cu = _device_i32(cu_seqlens, dev)
    qm = _device_i32(q_chunk_map, dev)
    if out is None:
        out = torch.empty((qI.shape[0], topk), dtype=torch.int32, device=dev)
    a = _args(qI, kI, None, 1.0, causal, causal_offset, cu, qm, None, chunk_len, None, None)
    lib = _lib.load()
    ws_bytes = lib.cpattn_workspace_size(_lib.OP_DSA_INDEXER, ctypes.byref(a), topk, 1)
    if ws_bytes and (workspace is None or workspace.numel() < ws_bytes):
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    _lib.check(lib.cpattn_dsa_indexer(ctypes.byref(a), w.data_ptr(), int(topk), out.data_ptr(),
                                      _ptr(workspace), ws_bytes, _stream(stream)))
    return out


def cpattn_workspace_size(op, q, k, v=None, topk=0, block_size=1):
    a = _args(q, k, v, 1.0, True, 0, None, None, None, 0, None, None)
    return _lib.load().cpattn_workspace_size(op, ctypes.byref(a), topk, block_size)


def cpattn_version():
    return _lib.load().cpattn_version()


@_on_call_stream
def cpattn_mla_v_up(o_latent, up_v_weight, out=None, dev_status=None, stream=None):
    """Value up-projection after absorbed attention: out[t, h] = o_latent[t, h] @ W[h].

    o_latent: bf16 [T, H, L] (last dim contiguous), up_v_weight: bf16 [H, L, V]
    contiguous; returns bf16 [T, H, V].
    """
    _thd("o_latent", o_latent)
    T, H, L = o_latent.shape
    w = up_v_weight.contiguous()
    V = w.shape[2]
    if out is None:
        out = torch.empty((T, H, V), dtype=torch.bfloat16, device=o_latent.device)
    _thd("out", out)
    _lib.check(_lib.load().cpattn_mla_v_up(o_latent.data_ptr(), o_latent.stride(0),
                                           o_latent.stride(1), w.data_ptr(), T, H, L, V,
                                           out.data_ptr(), out.stride(0), out.stride(1),
                                           _ptr(dev_status), 0, _stream(stream)))
    return out


@_on_call_stream
def cpattn_mla_kv_materialise(kv_c, k_shared, wkv_b, H, N, V, k_out=None, v_out=None,
                              dev_status=None, stream=None):
    """Per-head K [T, H, N + R] and V [T, H, V] (bf16) from gathered latents.

    kv_c: bf16 [T, L], k_shared: bf16 [T, R], wkv_b: bf16 [H * (N + V), L]
    (a linear layer's weight, contiguous).
    """
    T, L = kv_c.shape
    R = k_shared.shape[1]
    wb = wkv_b.contiguous()
    dev = kv_c.device
    if k_out is None:
        k_out = torch.empty((T, H, N + R), dtype=torch.bfloat16, device=dev)
    if v_out is None:
        v_out = torch.empty((T, H, V), dtype=torch.bfloat16, device=dev)
    _thd("k_out", k_out)
    _thd("v_out", v_out)
    _lib.check(_lib.load().cpattn_mla_kv_materialise(
        kv_c.data_ptr(), kv_c.stride(0), k_shared.data_ptr(), k_shared.stride(0), wb.data_ptr(),
        T, L, H, N, R, V, k_out.data_ptr(), k_out.stride(0), k_out.stride(1), v_out.data_ptr(),
        v_out.stride(0), v_out.stride(1), _ptr(dev_status), 0, _stream(stream)))
    return k_out, v_out
