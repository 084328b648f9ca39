"""cpattn_block_gate_static: the MoBA block gate for callers that cannot
allocate device memory at the call (a plugin given only its input and output
buffers, code in a host callback, a runtime that owns every allocation).

It keeps its scratch (the per-block key means and their split terms) in a
fixed 16 MiB array inside the library.  These tests call it through the C ABI
on several calls in a row, largest shape first, so that a later, smaller call
finds the previous call's contents in the shared array: the MoBA workload's
gate shape (128 blocks x 32 KV heads x d 128, 9.4 MB of scratch, the
tensor-core gate), then a smaller bf16 shape, then an fp32 shape of head dim
64 (the SIMT gate).  Each result must equal the float64 oracle's selection and
the selection of the workspace-taking cpattn_block_gate given a fresh
workspace.  A shape needing more scratch than the array holds is refused
before any launch.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import numpy as np
import pytest
import torch

import oracle as orc
from context_attention_softmax_gb300 import _lib, cpattn_block_gate


@pytest.fixture(scope="module")
def lib():
    from context_attention_softmax_gb300 import build
    build.build()
    return _lib.load()


def _gate_args(q, k, causal_offset):
    a = _lib.AttnArgs()
    a.dtype = _lib.CPATTN_BF16 if q.dtype == torch.bfloat16 else _lib.CPATTN_FP32
    a.q, a.q_stride_t, a.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    a.Tq, a.Hq, a.Dqk = q.shape
    a.k, a.k_stride_t, a.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    a.Tk, a.Hkv = k.shape[0], k.shape[1]
    a.scale, a.causal, a.causal_offset = 1.0, 1, causal_offset
    return a


def _inputs(seed, Tq, Tk, H, D, dtype):
    rng = np.random.default_rng(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    q = torch.tensor(rng.standard_normal((Tq, H, D)), dtype=torch.float32).to(tdt)
    k = torch.tensor(rng.standard_normal((Tk, H, D)), dtype=torch.float32).to(tdt)
    return q, k


# (seed, Tq, Tk, H, D, dtype, block size, topk, causal offset): largest scratch first
CASES = [
    (31, 96, 65536, 32, 128, "bf16", 512, 3, 57344),   # MoBA gate shape, tensor-core gate
    (32, 300, 8192, 4, 128, "bf16", 512, 3, 7000),     # fewer blocks and heads
    (33, 40, 3072, 3, 64, "fp32", 256, 3, 3000),       # fp32, d 64: the SIMT gate
]


@pytest.mark.gpu
def test_static_gate_matches_oracle_and_workspace_gate_on_calls_in_a_row(lib):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed, Tq, Tk, H, D, dtype, B, topk, offset in CASES:
        q, k = _inputs(seed, Tq, Tk, H, D, dtype)
        qd, kd = q.cuda(), k.cuda()
        sel = torch.full((Tq, H, topk + 1), -7, dtype=torch.int32, device="cuda")
        a = _gate_args(qd, kd, offset)
        status = lib.cpattn_block_gate_static(ctypes.byref(a), B, topk, sel.data_ptr(), stream)
        assert status == 0, lib.cpattn_last_error().decode()
        ref = cpattn_block_gate(qd, kd, B, topk, causal_offset=offset)   # fresh workspace
        torch.cuda.synchronize()
        got = sel.cpu().numpy()
        qpos = offset + np.arange(Tq)
        exact = orc.moba_block_gate(q.double().numpy(), k.double().numpy(), qpos, B, topk)
        np.testing.assert_array_equal(got, exact, err_msg=f"seed {seed}: differs from the oracle")
        assert torch.equal(sel, ref), f"seed {seed}: differs from cpattn_block_gate"


def test_static_gate_rejects_scratch_beyond_its_array(lib):
    # 256 blocks x 64 KV heads x d 128 needs 25 MB of block means (> 16 MiB).
    a = _lib.AttnArgs()
    a.dtype = _lib.CPATTN_BF16
    a.q, a.q_stride_t, a.q_stride_h, a.Tq, a.Hq, a.Dqk = 0x10000, 64 * 128, 128, 16, 64, 128
    a.k, a.k_stride_t, a.k_stride_h, a.Tk, a.Hkv = 0x20000, 64 * 128, 128, 65536, 64
    status = lib.cpattn_block_gate_static(ctypes.byref(a), 256, 3, 0x30000, None)
    assert status == 2
    assert "scratch" in lib.cpattn_last_error().decode()
