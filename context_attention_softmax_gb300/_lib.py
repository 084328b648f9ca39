"""ctypes view of libcpattn.so (include/cpattn.h).

Loading fails loudly when the library has not been built: there is no
fallback implementation.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcpattn.so")

CPATTN_FP32 = 0
CPATTN_BF16 = 1
OP_CHUNK_FWD, OP_TOPK_SPARSE_FWD, OP_BLOCK_GATE, OP_DSA_INDEXER, OP_CHUNK_BWD = 0, 1, 2, 3, 4

STATUS = {
    0: "CPATTN_OK",
    1: "CPATTN_ERR_INVALID_ARG",
    2: "CPATTN_ERR_UNSUPPORTED",
    3: "CPATTN_ERR_CUDA",
    4: "CPATTN_ERR_WORKSPACE",
    5: "CPATTN_ERR_TIMEOUT",
    6: "CPATTN_ERR_BAD_INDEX",
}

# every symbol include/cpattn.h declares
EXPORTS = (
    "cpattn_chunk_fwd",
    "cpattn_chunk_bwd",
    "cpattn_lse_merge",
    "cpattn_topk_sparse_fwd",
    "cpattn_block_gate",
    "cpattn_block_gate_static",
    "cpattn_dsa_indexer",
    "cpattn_mla_v_up",
    "cpattn_mla_kv_materialise",
    "cpattn_workspace_size",
    "cpattn_last_error",
    "cpattn_version",
)

c_i32, c_i64, c_f32, c_p = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p


class AttnArgs(ctypes.Structure):
    """Mirror of ``cpattn_attn_args`` (same field order and C alignment)."""

    _fields_ = [
        ("dtype", c_i32),
        ("q", c_p), ("q_stride_t", c_i64), ("q_stride_h", c_i64),
        ("Tq", c_i32), ("Hq", c_i32), ("Dqk", c_i32),
        ("k", c_p), ("k_stride_t", c_i64), ("k_stride_h", c_i64),
        ("Tk", c_i32), ("Hkv", c_i32),
        ("v", c_p), ("v_stride_t", c_i64), ("v_stride_h", c_i64),
        ("Dv", c_i32),
        ("scale", c_f32),
        ("causal", c_i32),
        ("causal_offset", c_i64),
        ("cu_seqlens", c_p), ("num_seqs", c_i32),
        ("q_chunk_map", c_p), ("kv_chunk_map", c_p),
        ("chunk_len", c_i32), ("n_q_chunks", c_i32), ("n_kv_chunks", c_i32),
        ("o", c_p), ("o_stride_t", c_i64), ("o_stride_h", c_i64),
        ("lse", c_p),
        ("kv_chunk_len", c_i32),
        ("partial_o", c_p), ("partial_lse", c_p),
        ("dev_status", c_p),
        ("wait_limit_ns", c_i64),
    ]


_LIB = None


def load(path: str = LIB_PATH):
    """Load the library once and declare the argument types of every export."""
    global _LIB
    if _LIB is not None:
        return _LIB
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is not built: run `python -c 'import __graft_entry__ as g; g.build()'` "
            "(the CUDA library is required; there is no fallback)")
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(AttnArgs)
    lib.cpattn_chunk_fwd.argtypes = [P, c_p, ctypes.c_size_t, c_p]
    lib.cpattn_chunk_bwd.argtypes = [P, c_p, c_i64, c_i64, c_p, c_i64, c_i64, c_p, c_i64, c_i64,
                                     c_p, c_i64, c_i64, c_p, ctypes.c_size_t, c_p]
    lib.cpattn_lse_merge.argtypes = [c_i32, c_p, c_p, c_i32, c_i32, c_i32, c_p, c_i32, c_i64,
                                     c_i64, c_p, c_p]
    lib.cpattn_topk_sparse_fwd.argtypes = [P, c_p, c_i32, c_i32, c_i32, c_p, ctypes.c_size_t, c_p]
    lib.cpattn_block_gate.argtypes = [P, c_i32, c_i32, c_p, c_p, ctypes.c_size_t, c_p]
    lib.cpattn_block_gate_static.argtypes = [P, c_i32, c_i32, c_p, c_p]
    lib.cpattn_dsa_indexer.argtypes = [P, c_p, c_i32, c_p, c_p, ctypes.c_size_t, c_p]
    lib.cpattn_mla_v_up.argtypes = [c_p, c_i64, c_i64, c_p, c_i32, c_i32, c_i32, c_i32, c_p, c_i64,
                                    c_i64, c_p, c_i64, c_p]
    lib.cpattn_mla_kv_materialise.argtypes = [c_p, c_i64, c_p, c_i64, c_p, c_i32, c_i32, c_i32,
                                              c_i32, c_i32, c_i32, c_p, c_i64, c_i64, c_p, c_i64,
                                              c_i64, c_p, c_i64, c_p]
    lib.cpattn_workspace_size.argtypes = [c_i32, P, c_i32, c_i32]
    lib.cpattn_workspace_size.restype = ctypes.c_size_t
    for name in ("cpattn_chunk_fwd", "cpattn_chunk_bwd", "cpattn_lse_merge", "cpattn_topk_sparse_fwd",
                 "cpattn_block_gate", "cpattn_block_gate_static", "cpattn_dsa_indexer",
                 "cpattn_mla_v_up", "cpattn_mla_kv_materialise"):
        getattr(lib, name).restype = c_i32
    lib.cpattn_last_error.argtypes = []
    lib.cpattn_last_error.restype = ctypes.c_char_p
    lib.cpattn_version.argtypes = []
    lib.cpattn_version.restype = c_i32
    _LIB = lib
    return lib


class CpattnError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status


def check(status: int):
    if status != 0:
        raise CpattnError(status, load().cpattn_last_error().decode())
