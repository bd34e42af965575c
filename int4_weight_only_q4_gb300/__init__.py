"""int4 group-128 weight-only GEMV / skinny GEMM for GB300 (sm_103a).

Python front end of libq4.so.  PyTorch is used for device memory and streams
only; every step of the computation runs in the library's CUDA kernels, and
the host packer runs in the library's C++ code.  There is no CPU fallback:
without the built library this package does not import.

Weight format (rumik-oss-1 int4 engine page, "Step 3"): groups of 128 columns,
an fp16 scale and an fp16 minimum per group, two 4-bit codes per byte (column
2j in the low nibble), w = code * scale + min.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from ._lib import (Q4_OK, Q4Error, check, c_vp, header_functions, lib, q4_matrix,  # noqa: F401
                   q4_plan_info)

GROUP = 128
MAX_B = 8

__all__ = ["GROUP", "MAX_B", "Q4Error", "QuantizedMatrix", "Workspace", "pack_host", "plan",
           "workspace_bytes", "gemv", "gemm_skinny", "decode_step", "argmax", "DecodeStepGraph",
           "header_functions", "lib"]


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t: torch.Tensor) -> int:
    return int(t.data_ptr())


# ---------------------------------------------------------------------------- host packer
def pack_host(w: np.ndarray, n_threads: int = 0):
    """fp32 [N, K] -> (codes uint8 [N, K/2], scales uint16 [N, K/128], mins uint16 [N, K/128]).

    Runs q4_pack_host (C++, multithreaded)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    codes = np.empty((N, K // 2), np.uint8)
    G = max(K // GROUP, 1)
    scales = np.empty((N, G), np.uint16)
    mins = np.empty((N, G), np.uint16)
    st = lib.q4_pack_host(w.ctypes.data, N, K, codes.ctypes.data, scales.ctypes.data, mins.ctypes.data,
                          int(n_threads))
    check(st, "q4_pack_host")
    return codes, scales, mins


def plan(N: int, K: int) -> dict:
    info = q4_plan_info()
    check(lib.q4_plan(N, K, ctypes.byref(info)), "q4_plan")
    return {f: getattr(info, f) for f, _ in info._fields_}


def workspace_bytes(N: int, K: int, B: int = 1) -> int:
    return int(lib.q4_workspace_bytes(N, K, B))


# ---------------------------------------------------------------------------- device data
@dataclass
class QuantizedMatrix:
    """One int4 matrix resident on the GPU in the canonical layout."""
    codes: torch.Tensor   # uint8 [N, K/2]
    scales: torch.Tensor  # float16 [N, K/128] (the fp16 bit patterns)
    mins: torch.Tensor    # float16 [N, K/128]
    N: int
    K: int

    @classmethod
    def from_packed(cls, codes: np.ndarray, scales: np.ndarray, mins: np.ndarray, device="cuda"):
        N, H = codes.shape
        c = torch.from_numpy(np.ascontiguousarray(codes)).to(device)
        s = torch.from_numpy(np.ascontiguousarray(scales).view(np.float16)).to(device)
        m = torch.from_numpy(np.ascontiguousarray(mins).view(np.float16)).to(device)
        return cls(c, s, m, N, 2 * H)

    @classmethod
    def from_float(cls, w: np.ndarray, device="cuda", n_threads: int = 0):
        return cls.from_packed(*pack_host(w, n_threads), device=device)

    def c_struct(self) -> q4_matrix:
        return q4_matrix(_ptr(self.codes), _ptr(self.scales), _ptr(self.mins), self.N, self.K)


class Workspace:
    """A zero-filled device buffer for the k-split partial sums and arrival counters."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = int(nbytes)
        self.buf = torch.zeros(max(self.nbytes, 16), dtype=torch.uint8, device=device) if self.nbytes else None

    @classmethod
    def for_shapes(cls, shapes, B: int = MAX_B, device="cuda"):
        need = max([workspace_bytes(N, K, B) for N, K in shapes] + [0])
        return cls(need, device)

    def ptr(self) -> int:
        return _ptr(self.buf) if self.buf is not None else 0


def _ws_args(ws):
    if ws is None:
        return None, 0
    return (ws.ptr() or None), ws.nbytes


def _as_bf16(x: torch.Tensor) -> torch.Tensor:
    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise TypeError("activations must be a contiguous torch.bfloat16 CUDA tensor")
    return x


# ---------------------------------------------------------------------------- calls
def gemm_skinny(W: QuantizedMatrix, X: torch.Tensor, Y: torch.Tensor | None = None,
                workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """Y[b] = W X[b] for X bf16 [B, K] (1 <= B <= 8); Y fp32 [B, N]."""
    X = _as_bf16(X)
    B = 1 if X.dim() == 1 else X.shape[0]
    if Y is None:
        Y = torch.empty((B, W.N), dtype=torch.float32, device=X.device)
    if workspace is None and workspace_bytes(W.N, W.K, B):
        workspace = Workspace(workspace_bytes(W.N, W.K, B), X.device)
    ws_p, ws_n = _ws_args(workspace)
    m = W.c_struct()
    st = lib.q4_gemm_skinny(ctypes.byref(m), _ptr(X), B, _ptr(Y), ws_p, ws_n, _stream_ptr(stream))
    check(st, "q4_gemm_skinny")
    return Y


def gemv(W: QuantizedMatrix, x: torch.Tensor, y: torch.Tensor | None = None,
         workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """y = W x for x bf16 [K]; y fp32 [N]."""
    x = _as_bf16(x)
    if y is None:
        y = torch.empty((W.N,), dtype=torch.float32, device=x.device)
    if workspace is None and workspace_bytes(W.N, W.K, 1):
        workspace = Workspace(workspace_bytes(W.N, W.K, 1), x.device)
    ws_p, ws_n = _ws_args(workspace)
    m = W.c_struct()
    check(lib.q4_gemv(ctypes.byref(m), _ptr(x), _ptr(y), ws_p, ws_n, _stream_ptr(stream)), "q4_gemv")
    return y


def decode_step(mats, Xs, Ys, workspace: Workspace | None = None, stream=None) -> None:
    """Enqueue one decode step: Ys[i] = mats[i] Xs[i] for every matrix, in list order."""
    n = len(mats)
    B = Xs[0].shape[0] if Xs[0].dim() == 2 else 1
    arr = (q4_matrix * n)(*[m.c_struct() for m in mats])
    xp = (c_vp * n)(*[_ptr(_as_bf16(x)) for x in Xs])
    yp = (c_vp * n)(*[_ptr(y) for y in Ys])
    ws_p, ws_n = _ws_args(workspace)
    check(lib.q4_decode_step(arr, n, xp, yp, B, ws_p, ws_n, _stream_ptr(stream)), "q4_decode_step")


def argmax(Y: torch.Tensor, idx: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per batch row of fp32 logits [B, N]: index of the max, lowest index on ties (int32 [B])."""
    if Y.dtype != torch.float32 or not Y.is_contiguous():
        raise TypeError("logits must be a contiguous float32 CUDA tensor")
    Y2 = Y if Y.dim() == 2 else Y.view(1, -1)
    B, N = Y2.shape
    if idx is None:
        idx = torch.empty((B,), dtype=torch.int32, device=Y.device)
    check(lib.q4_argmax_f32(_ptr(Y2), B, N, _ptr(idx), _stream_ptr(stream)), "q4_argmax_f32")
    return idx


class DecodeStepGraph:
    """One decode step (all matrices, in order) captured once into a CUDA graph and replayed.

    The activations and outputs are fixed device buffers: write new activations
    into ``self.X[i]`` and read ``self.Y[i]`` after ``replay()``.
    """

    def __init__(self, mats, B: int, X=None, Y=None, workspace: Workspace | None = None, device="cuda",
                 with_argmax_of: int | None = None):
        self.mats = list(mats)
        self.B = B
        self.X = X if X is not None else [torch.zeros((B, m.K), dtype=torch.bfloat16, device=device)
                                           for m in self.mats]
        self.Y = Y if Y is not None else [torch.empty((B, m.N), dtype=torch.float32, device=device)
                                           for m in self.mats]
        self.ws = workspace if workspace is not None else \
            Workspace.for_shapes([(m.N, m.K) for m in self.mats], B, device)
        self.idx = torch.zeros((B,), dtype=torch.int32, device=device) if with_argmax_of is not None else None
        self.argmax_of = with_argmax_of
        self.graph = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(device=device)
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            self._enqueue(side)           # warm-up outside capture: sets kernel attributes
        side.synchronize()
        with torch.cuda.graph(self.graph, stream=side):
            self._enqueue(side)
        torch.cuda.current_stream().wait_stream(side)

    def _enqueue(self, stream):
        decode_step(self.mats, self.X, self.Y, self.ws, stream=stream)
        if self.argmax_of is not None:
            argmax(self.Y[self.argmax_of], self.idx, stream=stream)

    def replay(self):
        self.graph.replay()

    def run_host(self, X_host, Y_host, idx_host=None):
        """One step end to end: copy activations from (pinned) host tensors, replay, copy the
        outputs (and the argmax indices) back, and wait for them."""
        for d, h in zip(self.X, X_host):
            d.copy_(h, non_blocking=True)
        self.graph.replay()
        for d, h in zip(self.Y, Y_host):
            h.copy_(d, non_blocking=True)
        if idx_host is not None and self.idx is not None:
            idx_host.copy_(self.idx, non_blocking=True)
        torch.cuda.current_stream().synchronize()
