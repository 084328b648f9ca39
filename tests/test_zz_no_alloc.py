"""cpattn_block_gate_static: the MoBA block gate for callers that cannot
allocate device memory at the call (a plugin given only its input and output
buffers, code in a host callback, a runtime that owns every allocation).

It keeps its scratch (the per-block key means) in a fixed array inside the
library.  These tests call it through the C ABI and check that it selects
exactly the blocks the workspace-taking cpattn_block_gate selects, on two
calls in a row with different inputs (the shared array keeps the previous
call's contents, which must not leak into the next result), and that a shape
needing more scratch than the array holds is refused before any launch.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""

import ctypes

import pytest
import torch

from context_attention_softmax_gb300 import _lib, cpattn_block_gate, inputs


@pytest.fixture(scope="module")
def lib():
    from context_attention_softmax_gb300 import build
    build.build()
    return _lib.load()


def _gate_args(q, k, causal_offset):
    a = _lib.AttnArgs()
    a.dtype = _lib.CPATTN_BF16
    a.q, a.q_stride_t, a.q_stride_h = q.data_ptr(), q.stride(0), q.stride(1)
    a.Tq, a.Hq, a.Dqk = q.shape
    a.k, a.k_stride_t, a.k_stride_h = k.data_ptr(), k.stride(0), k.stride(1)
    a.Tk, a.Hkv = k.shape[0], k.shape[1]
    a.scale, a.causal, a.causal_offset = 1.0, 1, causal_offset
    return a


@pytest.mark.gpu
def test_static_gate_matches_workspace_gate_on_two_calls(lib):
    B, topk, offset = 512, 3, 7000
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for seed in (21, 22):
        w = inputs.moba(seed=seed, Tq=600, Tk=8192, offset=offset, H=4, block_size=B, topk=topk)
        q, k = w.q.cuda(), w.k.cuda()
        ref = cpattn_block_gate(q, k, B, topk, causal_offset=offset)
        sel = torch.full((q.shape[0], q.shape[1], topk + 1), -7, dtype=torch.int32, device="cuda")
        a = _gate_args(q, k, offset)
        status = lib.cpattn_block_gate_static(ctypes.byref(a), B, topk, sel.data_ptr(), stream)
        assert status == 0, lib.cpattn_last_error().decode()
        torch.cuda.synchronize()
        assert torch.equal(sel, ref), f"seed {seed}: selections differ"
        assert (sel[:, :, -1] != -7).all()


def test_static_gate_rejects_scratch_beyond_its_array(lib):
    # 128 blocks x 64 KV heads x d 128 needs 12.6 MB of block means (> 8 MiB).
    a = _lib.AttnArgs()
    a.dtype = _lib.CPATTN_BF16
    a.q, a.q_stride_t, a.q_stride_h, a.Tq, a.Hq, a.Dqk = 0x10000, 64 * 128, 128, 16, 64, 128
    a.k, a.k_stride_t, a.k_stride_h, a.Tk, a.Hkv = 0x20000, 64 * 128, 128, 65536, 64
    status = lib.cpattn_block_gate_static(ctypes.byref(a), 512, 3, 0x30000, None)
    assert status == 2
    assert "scratch" in lib.cpattn_last_error().decode()
