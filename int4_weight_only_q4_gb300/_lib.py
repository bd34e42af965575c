"""ctypes binding of libq4.so (argument marshalling only; every step runs in the library).

The library must have been built in-tree (``python -m int4_weight_only_q4_gb300.build``
or ``__graft_entry__.build()``); importing this module without it raises.
"""
from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
# Q4_LIBRARY_PATH selects another build of the same library (e.g. to compare two builds side by
# side); by default the in-tree build next to this file.
LIB_PATH = os.environ.get("Q4_LIBRARY_PATH") or os.path.join(HERE, "libq4.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "q4.h")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"libq4.so is not built ({LIB_PATH} missing); run `python -m int4_weight_only_q4_gb300.build`")

lib = ctypes.CDLL(LIB_PATH)

c_i64 = ctypes.c_int64
c_vp = ctypes.c_void_p


class q4_matrix(ctypes.Structure):
    _fields_ = [("codes", c_vp), ("scales", c_vp), ("mins", c_vp), ("N", c_i64), ("K", c_i64), ("tiled", c_vp)]


class q8_matrix(ctypes.Structure):
    _fields_ = [("codes", c_vp), ("scales", c_vp), ("N", c_i64), ("K", c_i64), ("tiled", c_vp)]


class q4_plan_info(ctypes.Structure):
    _fields_ = [("row_blocks", ctypes.c_int32), ("k_splits", ctypes.c_int32),
                ("warps_per_cta", ctypes.c_int32), ("prefetch_depth", ctypes.c_int32),
                ("kernel", ctypes.c_int32), ("sm_count", ctypes.c_int32)]


STATUS = {0: "Q4_OK", 1: "Q4_ERR_INVALID_ARG", 2: "Q4_ERR_UNSUPPORTED_SHAPE", 3: "Q4_ERR_MISALIGNED",
          4: "Q4_ERR_WORKSPACE", 5: "Q4_ERR_CUDA", 6: "Q4_ERR_TIMEOUT"}
Q4_OK = 0
Q4_ERR_INVALID_ARG = 1
Q4_ERR_UNSUPPORTED_SHAPE = 2
Q4_ERR_MISALIGNED = 3
Q4_ERR_WORKSPACE = 4
Q4_ERR_CUDA = 5
Q4_ERR_TIMEOUT = 6
Q4_STEP_INDEPENDENT = 1

lib.q4_pack_host.argtypes = [c_vp, c_i64, c_i64, c_vp, c_vp, c_vp, ctypes.c_int]
lib.q4_pack_host.restype = ctypes.c_int
lib.q4_tiled_bytes.argtypes = [c_i64, c_i64]
lib.q4_tiled_bytes.restype = ctypes.c_size_t
lib.q4_tile.argtypes = [ctypes.POINTER(q4_matrix), c_vp, ctypes.c_size_t, c_vp]
lib.q4_tile.restype = ctypes.c_int
lib.q4_workspace_bytes.argtypes = [c_i64, c_i64, ctypes.c_int]
lib.q4_workspace_bytes.restype = ctypes.c_size_t
lib.q4_plan.argtypes = [c_i64, c_i64, ctypes.POINTER(q4_plan_info)]
lib.q4_plan.restype = ctypes.c_int
lib.q4_gemv.argtypes = [ctypes.POINTER(q4_matrix), c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]
lib.q4_gemv.restype = ctypes.c_int
lib.q4_gemm_skinny.argtypes = [ctypes.POINTER(q4_matrix), c_vp, ctypes.c_int, c_vp, c_vp, ctypes.c_size_t, c_vp]
lib.q4_gemm_skinny.restype = ctypes.c_int
lib.q4_decode_step.argtypes = [ctypes.POINTER(q4_matrix), ctypes.c_int, ctypes.POINTER(c_vp),
                               ctypes.POINTER(c_vp), ctypes.c_int, c_vp, ctypes.c_size_t, ctypes.c_uint, c_vp]
lib.q4_decode_step.restype = ctypes.c_int
lib.q4_decode_step_workspace_bytes.argtypes = [ctypes.POINTER(c_i64), ctypes.POINTER(c_i64), ctypes.c_int,
                                               ctypes.c_int, ctypes.c_uint]
lib.q4_decode_step_workspace_bytes.restype = ctypes.c_size_t
lib.q4_step_workspace_bytes.argtypes = [ctypes.POINTER(c_i64), ctypes.c_int, ctypes.c_int]
lib.q4_step_workspace_bytes.restype = ctypes.c_size_t
lib.q4_step_prepare.argtypes = [ctypes.POINTER(q4_matrix), ctypes.c_int, ctypes.POINTER(c_vp), ctypes.c_int, c_vp,
                                ctypes.c_size_t, c_vp]
lib.q4_step_prepare.restype = ctypes.c_int
lib.q4_step_stream.argtypes = [ctypes.POINTER(q4_matrix), ctypes.c_int, ctypes.POINTER(c_vp), ctypes.c_int, c_vp,
                               ctypes.c_size_t, c_vp]
lib.q4_step_stream.restype = ctypes.c_int
lib.q4_step_stream_readonly.argtypes = [ctypes.POINTER(q4_matrix), ctypes.c_int, ctypes.POINTER(c_vp), ctypes.c_int,
                                        c_vp, ctypes.c_size_t, c_vp]
lib.q4_step_stream_readonly.restype = ctypes.c_int
lib.q4_gemm_skinny_noalloc.argtypes = [ctypes.POINTER(q4_matrix), c_vp, ctypes.c_int, c_vp, c_vp]
lib.q4_gemm_skinny_noalloc.restype = ctypes.c_int
lib.q4_noalloc_scratch_bytes.argtypes = []
lib.q4_noalloc_scratch_bytes.restype = ctypes.c_size_t
lib.q4_device_status.argtypes = [c_vp]
lib.q4_device_status.restype = ctypes.c_int
lib.q4_argmax_f32.argtypes = [c_vp, ctypes.c_int, c_i64, c_vp, c_vp]
lib.q4_argmax_f32.restype = ctypes.c_int
lib.q4_argmax_key_f32.argtypes = [c_vp, ctypes.c_int, c_i64, c_i64, c_vp, c_vp]
lib.q4_argmax_key_f32.restype = ctypes.c_int
lib.q4_argmax_key_index.argtypes = [c_vp, ctypes.c_int, c_vp, c_vp]
lib.q4_argmax_key_index.restype = ctypes.c_int
lib.q8_pack_host.argtypes = [c_vp, c_i64, c_i64, c_vp, c_vp, ctypes.c_int]
lib.q8_pack_host.restype = ctypes.c_int
lib.q8_tiled_bytes.argtypes = [c_i64, c_i64]
lib.q8_tiled_bytes.restype = ctypes.c_size_t
lib.q8_tile.argtypes = [ctypes.POINTER(q8_matrix), c_vp, ctypes.c_size_t, c_vp]
lib.q8_tile.restype = ctypes.c_int
lib.q8_head_workspace_bytes.argtypes = [c_i64, c_i64, ctypes.c_int]
lib.q8_head_workspace_bytes.restype = ctypes.c_size_t
lib.q8_head.argtypes = [ctypes.POINTER(q8_matrix), c_vp, ctypes.c_int, c_vp, c_vp, c_vp, ctypes.c_size_t, c_vp]
lib.q8_head.restype = ctypes.c_int
lib.q4_sample_topk.argtypes = [c_vp, ctypes.c_int, c_i64, ctypes.c_int, ctypes.c_float, c_vp, c_vp, c_vp, c_vp]
lib.q4_sample_topk.restype = ctypes.c_int
lib.q4_prefill_workspace_bytes.argtypes = [c_i64, c_i64]
lib.q4_prefill_workspace_bytes.restype = ctypes.c_size_t
lib.q4_gemm_prefill.argtypes = [ctypes.POINTER(q4_matrix), c_vp, c_i64, c_vp, c_vp, ctypes.c_size_t, c_vp]
lib.q4_gemm_prefill.restype = ctypes.c_int
lib.q4_prefill_kernel.argtypes = [c_i64, c_i64]
lib.q4_prefill_kernel.restype = ctypes.c_int
lib.q4_flash_decode_chunks.argtypes = [ctypes.c_int, ctypes.c_int]
lib.q4_flash_decode_chunks.restype = ctypes.c_int
lib.q4_flash_decode_workspace_bytes.argtypes = [ctypes.c_int] * 5
lib.q4_flash_decode_workspace_bytes.restype = ctypes.c_size_t
lib.q4_flash_decode.argtypes = [c_vp, c_vp, c_vp, c_vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                c_i64, ctypes.c_float, ctypes.c_int, c_vp, c_vp, ctypes.c_size_t, c_vp]
lib.q4_flash_decode.restype = ctypes.c_int
lib.q4_status_string.argtypes = [ctypes.c_int]
lib.q4_status_string.restype = ctypes.c_char_p


class Q4Error(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = lib.q4_status_string(status).decode()
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})")


def check(status: int, where: str) -> None:
    if status != Q4_OK:
        raise Q4Error(status, where)


def header_functions() -> list[str]:
    """Names of every function declared in include/q4.h."""
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(q[48]_[a-z0-9_]+)\s*\(", src)))
