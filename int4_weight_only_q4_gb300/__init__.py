"""int4 group-128 weight-only GEMV / skinny GEMM for GB300 (sm_103a).

Python front end of libq4.so.  PyTorch is used for device memory and streams
only; every step of the computation runs in the library's CUDA kernels, and
the host packer runs in the library's C++ code.  There is no CPU fallback:
without the built library this package does not import.

Weight format (rumik-oss-1 int4 engine page, "Step 3"): for every row, each run of
128 columns carries one fp16 scale and one fp16 minimum; codes are 4 bits, packed
in pairs (column 2j in the low nibble), w = code * scale + min.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from ._lib import (Q4_OK, Q4_STEP_INDEPENDENT, Q4Error, check, c_i64, c_vp, header_functions,  # noqa: F401
                   lib, q4_matrix, q4_plan_info, q8_matrix)

GROUP = 128
MAX_B = 8

__all__ = ["GROUP", "MAX_B", "Q4Error", "QuantizedMatrix", "Workspace", "pack_host", "plan",
           "workspace_bytes", "decode_step_workspace_bytes", "tiled_bytes", "gemv", "gemm_skinny", "decode_step",
           "argmax", "device_status", "DecodeStepGraph", "step_workspace_bytes", "step_prepare", "step_stream",
           "step_stream_readonly", "argmax_keys", "argmax_key_index",
           "gemm_skinny_noalloc", "pack_int8_host", "Int8Head", "sample_topk", "gemm_prefill",
           "flash_decode", "flash_decode_workspace", "header_functions", "lib"]


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t: torch.Tensor) -> int:
    """Device address of a tensor handed to the library, which reads and writes it from kernels on
    the current device: anything else is refused here (a host address would fault the GPU)."""
    if not t.is_cuda:
        raise TypeError(f"expected a CUDA tensor, got one on {t.device}")
    if t.device.index != torch.cuda.current_device():
        raise TypeError(f"tensor on {t.device}, but the current device is cuda:{torch.cuda.current_device()}")
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


def pack_int8_host(w: np.ndarray, n_threads: int = 0):
    """fp32 [N, K] -> (codes int8 [N, K], scales uint16 [N]) for the int8 output head
    (q8_pack_host: one symmetric fp16 scale per row)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    N, K = w.shape
    codes = np.empty((N, K), np.int8)
    scales = np.empty((N,), np.uint16)
    check(lib.q8_pack_host(w.ctypes.data, N, K, codes.ctypes.data, scales.ctypes.data, int(n_threads)),
          "q8_pack_host")
    return codes, scales


def plan(N: int, K: int) -> dict:
    info = q4_plan_info()
    check(lib.q4_plan(N, K, ctypes.byref(info)), "q4_plan")
    return {f: getattr(info, f) for f, _ in info._fields_}


def workspace_bytes(N: int, K: int, B: int = 1) -> int:
    return int(lib.q4_workspace_bytes(N, K, B))


def decode_step_workspace_bytes(shapes, B: int, independent: bool = True) -> int:
    n = len(shapes)
    Ns = (c_i64 * n)(*[int(N) for N, _ in shapes])
    Ks = (c_i64 * n)(*[int(K) for _, K in shapes])
    return int(lib.q4_decode_step_workspace_bytes(Ns, Ks, n, B, Q4_STEP_INDEPENDENT if independent else 0))


def device_status(stream=None) -> None:
    """Wait for the stream and raise Q4Error(Q4_ERR_TIMEOUT) if a bounded device-side wait gave up."""
    check(lib.q4_device_status(_stream_ptr(stream)), "q4_device_status")


# ---------------------------------------------------------------------------- device data
def tiled_bytes(N: int, K: int) -> int:
    return int(lib.q4_tiled_bytes(N, K))


@dataclass
class QuantizedMatrix:
    """One int4 matrix resident on the GPU: the canonical layout and/or its tiled copy."""
    codes: torch.Tensor | None   # uint8 [N, K/2]
    scales: torch.Tensor | None  # float16 [N, K/128] (the fp16 bit patterns)
    mins: torch.Tensor | None    # float16 [N, K/128]
    N: int
    K: int
    tiled: torch.Tensor | None = None  # uint8 [tiled_bytes(N, K)]

    @classmethod
    def from_packed(cls, codes: np.ndarray, scales: np.ndarray, mins: np.ndarray, device="cuda",
                    tiled: bool = True, keep_canonical: bool = True, stream=None):
        N, H = codes.shape
        c = torch.from_numpy(np.ascontiguousarray(codes)).to(device)
        s = torch.from_numpy(np.ascontiguousarray(scales).view(np.float16)).to(device)
        m = torch.from_numpy(np.ascontiguousarray(mins).view(np.float16)).to(device)
        W = cls(c, s, m, N, 2 * H)
        if tiled:
            W.build_tiled(stream)
            if not keep_canonical:
                torch.cuda.current_stream(c.device).synchronize()
                W.codes = W.scales = W.mins = None
        return W

    @classmethod
    def from_float(cls, w: np.ndarray, device="cuda", n_threads: int = 0, tiled: bool = True):
        return cls.from_packed(*pack_host(w, n_threads), device=device, tiled=tiled)

    def build_tiled(self, stream=None):
        """Build the tiled copy (q4_tile) from the canonical arrays."""
        nb = tiled_bytes(self.N, self.K)
        self.tiled = torch.empty(nb, dtype=torch.uint8, device=self.codes.device)
        m = self.c_struct()
        check(lib.q4_tile(ctypes.byref(m), _ptr(self.tiled), nb, _stream_ptr(stream)), "q4_tile")
        return self

    def c_struct(self) -> q4_matrix:
        p = lambda t: _ptr(t) if t is not None else None
        return q4_matrix(p(self.codes), p(self.scales), p(self.mins), self.N, self.K, p(self.tiled))


class Workspace:
    """A zero-filled device buffer for the k-split partial sums and arrival counters."""

    def __init__(self, nbytes: int, device="cuda"):
        self.nbytes = int(nbytes)
        self.buf = torch.zeros(max(self.nbytes, 16), dtype=torch.uint8, device=device) if self.nbytes else None

    @classmethod
    def for_shapes(cls, shapes, B: int = MAX_B, device="cuda", independent: bool = True):
        return cls(decode_step_workspace_bytes(shapes, B, independent), device)

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


def _check_x(X: torch.Tensor, K: int) -> int:
    """Batch size of activations X ([K] or [B, K], bf16, contiguous) for a matrix of K columns."""
    _as_bf16(X)
    if X.dim() not in (1, 2) or X.shape[-1] != K:
        raise ValueError(f"activations of shape {tuple(X.shape)} do not match a matrix of K = {K} columns")
    return 1 if X.dim() == 1 else X.shape[0]


def _check_y(Y: torch.Tensor, B: int, N: int) -> None:
    """The kernels write B * N fp32 values from Y's first element on: refuse anything smaller, of
    another dtype or not contiguous (a short buffer would be written past its end)."""
    if Y.dtype != torch.float32 or not Y.is_contiguous():
        raise TypeError("outputs must be a contiguous torch.float32 CUDA tensor")
    if Y.numel() < B * N:
        raise ValueError(f"output of {Y.numel()} elements is smaller than B * N = {B} * {N}")


# ---------------------------------------------------------------------------- calls
def gemm_skinny(W: QuantizedMatrix, X: torch.Tensor, Y: torch.Tensor | None = None,
                workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """Y[b] = W X[b] for X bf16 [B, K] (1 <= B <= 8); Y fp32 [B, N]."""
    B = _check_x(X, W.K)
    if Y is None:
        Y = torch.empty((B, W.N), dtype=torch.float32, device=X.device)
    _check_y(Y, B, W.N)
    if workspace is None and workspace_bytes(W.N, W.K, B):
        workspace = Workspace(workspace_bytes(W.N, W.K, B), X.device)
    ws_p, ws_n = _ws_args(workspace)
    m = W.c_struct()
    st = lib.q4_gemm_skinny(ctypes.byref(m), _ptr(X), B, _ptr(Y), ws_p, ws_n, _stream_ptr(stream))
    check(st, "q4_gemm_skinny")
    return Y


def gemm_skinny_noalloc(W: QuantizedMatrix, X: torch.Tensor, Y: torch.Tensor, stream=None) -> torch.Tensor:
    """Y = W X with no workspace: the library's fixed scratch array instead (see q4.h for its
    limits and for the rule that calls overlapping on the GPU race)."""
    B = _check_x(X, W.K)
    _check_y(Y, B, W.N)
    m = W.c_struct()
    check(lib.q4_gemm_skinny_noalloc(ctypes.byref(m), _ptr(X), B, _ptr(Y), _stream_ptr(stream)),
          "q4_gemm_skinny_noalloc")
    return Y


def gemv(W: QuantizedMatrix, x: torch.Tensor, y: torch.Tensor | None = None,
         workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """y = W x for x bf16 [K]; y fp32 [N]."""
    if _check_x(x, W.K) != 1:
        raise ValueError("gemv takes one activation vector")
    if y is None:
        y = torch.empty((W.N,), dtype=torch.float32, device=x.device)
    _check_y(y, 1, W.N)
    if workspace is None and workspace_bytes(W.N, W.K, 1):
        workspace = Workspace(workspace_bytes(W.N, W.K, 1), x.device)
    ws_p, ws_n = _ws_args(workspace)
    m = W.c_struct()
    check(lib.q4_gemv(ctypes.byref(m), _ptr(x), _ptr(y), ws_p, ws_n, _stream_ptr(stream)), "q4_gemv")
    return y


def _check_i32(t: torch.Tensor, n: int, name: str) -> None:
    if t.dtype != torch.int32 or not t.is_contiguous() or t.numel() < n:
        raise ValueError(f"{name} must be a contiguous int32 tensor of at least {n} elements")


def _check_list(mats, Xs, Ys=None) -> int:
    """One batch size for every matrix of a list, activations and outputs sized for each."""
    if len(Xs) != len(mats) or (Ys is not None and len(Ys) != len(mats)):
        raise ValueError("one activation tensor (and one output tensor) per matrix")
    Bs = {_check_x(x, m.K) for x, m in zip(Xs, mats)}
    if len(Bs) != 1:
        raise ValueError(f"every activation tensor must have the same batch size, got {sorted(Bs)}")
    B = Bs.pop()
    for y, m in zip(Ys or [], mats):
        _check_y(y, B, m.N)
    return B


def decode_step(mats, Xs, Ys, workspace: Workspace | None = None, stream=None, independent: bool = True) -> None:
    """Enqueue one decode step: Ys[i] = mats[i] Xs[i] for every matrix, in list order.

    independent=True: one persistent launch for the whole list (no Xs[j] may overlap any Ys[i]);
    False: one launch per matrix, so Ys[i] may feed Xs[j] for j > i."""
    n = len(mats)
    B = _check_list(mats, Xs, Ys)
    if workspace is None:
        need = decode_step_workspace_bytes([(m.N, m.K) for m in mats], B, independent)
        if need:
            workspace = Workspace(need, Xs[0].device)
    arr = (q4_matrix * n)(*[m.c_struct() for m in mats])
    xp = (c_vp * n)(*[_ptr(x) for x in Xs])
    yp = (c_vp * n)(*[_ptr(y) for y in Ys])
    ws_p, ws_n = _ws_args(workspace)
    flags = Q4_STEP_INDEPENDENT if independent else 0
    check(lib.q4_decode_step(arr, n, xp, yp, B, ws_p, ws_n, flags, _stream_ptr(stream)), "q4_decode_step")


def step_workspace_bytes(Ks, B: int) -> int:
    n = len(Ks)
    arr = (c_i64 * n)(*[int(K) for K in Ks])
    return int(lib.q4_step_workspace_bytes(arr, n, B))


def step_prepare(mats, Xs, workspace: Workspace, stream=None) -> None:
    """Phase 1 of an independent decode step: stage every activation once into the workspace."""
    n = len(mats)
    B = _check_list(mats, Xs)
    arr = (q4_matrix * n)(*[m.c_struct() for m in mats])
    xp = (c_vp * n)(*[_ptr(x) for x in Xs])
    check(lib.q4_step_prepare(arr, n, xp, B, workspace.ptr(), workspace.nbytes, _stream_ptr(stream)),
          "q4_step_prepare")


def step_stream(mats, Ys, B: int, workspace: Workspace, stream=None) -> None:
    """Phase 2: Ys[i] = mats[i] x_i from the activations the last step_prepare staged."""
    n = len(mats)
    if len(Ys) != n:
        raise ValueError("one output tensor per matrix")
    for y, m in zip(Ys, mats):
        _check_y(y, B, m.N)
    arr = (q4_matrix * n)(*[m.c_struct() for m in mats])
    yp = (c_vp * n)(*[_ptr(y) for y in Ys])
    check(lib.q4_step_stream(arr, n, yp, B, workspace.ptr(), workspace.nbytes, _stream_ptr(stream)),
          "q4_step_stream")


def step_stream_readonly(mats, Ys, B: int, workspace: Workspace, stream=None) -> None:
    """Measurement aid: the read-only twin of step_stream (same loads and stores, no arithmetic;
    the values it writes to Ys are meaningless)."""
    n = len(mats)
    if len(Ys) != n:
        raise ValueError("one output tensor per matrix")
    for y, m in zip(Ys, mats):
        _check_y(y, B, m.N)
    arr = (q4_matrix * n)(*[m.c_struct() for m in mats])
    yp = (c_vp * n)(*[_ptr(y) for y in Ys])
    check(lib.q4_step_stream_readonly(arr, n, yp, B, workspace.ptr(), workspace.nbytes, _stream_ptr(stream)),
          "q4_step_stream_readonly")


def argmax(Y: torch.Tensor, idx: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per batch row of fp32 logits [B, N]: index of the max, lowest index on ties (int32 [B])."""
    if Y.dtype != torch.float32 or not Y.is_contiguous():
        raise TypeError("logits must be a contiguous float32 CUDA tensor")
    Y2 = Y if Y.dim() == 2 else Y.view(1, -1)
    B, N = Y2.shape
    if idx is None:
        idx = torch.empty((B,), dtype=torch.int32, device=Y.device)
    _check_i32(idx, B, "idx")
    check(lib.q4_argmax_f32(_ptr(Y2), B, N, _ptr(idx), _stream_ptr(stream)), "q4_argmax_f32")
    return idx


def argmax_keys(Y: torch.Tensor, index_base: int = 0, keys: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Per batch row of fp32 logits [B, N] whose rows are global rows index_base.., the best one as a
    64-bit key (q4_argmax_key_f32): the largest key over several row slices is the argmax of the
    whole row."""
    if Y.dtype != torch.float32 or not Y.is_contiguous():
        raise TypeError("logits must be a contiguous float32 CUDA tensor")
    Y2 = Y if Y.dim() == 2 else Y.view(1, -1)
    B, N = Y2.shape
    if keys is None:
        keys = torch.empty((B,), dtype=torch.int64, device=Y.device)
    if keys.dtype != torch.int64 or not keys.is_contiguous() or keys.numel() < B:
        raise ValueError("keys must be a contiguous int64 tensor of at least B elements")
    check(lib.q4_argmax_key_f32(_ptr(Y2), B, N, int(index_base), _ptr(keys), _stream_ptr(stream)),
          "q4_argmax_key_f32")
    return keys


def argmax_key_index(keys: torch.Tensor, idx: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The global row index held in each argmax key (q4_argmax_key_index), int32 [B]."""
    if keys.dtype != torch.int64 or not keys.is_contiguous():
        raise TypeError("keys must be a contiguous int64 CUDA tensor")
    B = keys.numel()
    if idx is None:
        idx = torch.empty((B,), dtype=torch.int32, device=keys.device)
    _check_i32(idx, B, "idx")
    check(lib.q4_argmax_key_index(_ptr(keys), B, _ptr(idx), _stream_ptr(stream)), "q4_argmax_key_index")
    return idx


class Int8Head:
    """An int8 output head resident on the GPU (per-row fp16 scales, tiled copy of the codes):
    logits and/or their argmax per batch row in one call (q8_head)."""

    def __init__(self, codes: torch.Tensor | None, scales: torch.Tensor, N: int, K: int, tiled: torch.Tensor):
        self.codes, self.scales, self.N, self.K, self.tiled = codes, scales, N, K, tiled

    @classmethod
    def from_device(cls, codes: torch.Tensor, scales: torch.Tensor, keep_codes: bool = False, stream=None):
        """From device codes (int8 [N, K]) and scales (float16 [N], the fp16 bit patterns): builds the
        tiled copy (q8_tile)."""
        N, K = codes.shape
        nb = int(lib.q8_tiled_bytes(N, K))
        tiled = torch.empty(nb, dtype=torch.uint8, device=codes.device)
        H = cls(codes, scales, N, K, tiled)
        check(lib.q8_tile(ctypes.byref(H.c_struct()), _ptr(tiled), nb, _stream_ptr(stream)), "q8_tile")
        if not keep_codes:
            torch.cuda.current_stream(codes.device).synchronize()
            H.codes = None
        return H

    @classmethod
    def from_packed(cls, codes: np.ndarray, scales: np.ndarray, device="cuda", keep_codes: bool = False,
                    stream=None):
        c = torch.from_numpy(np.ascontiguousarray(codes)).to(device)
        s = torch.from_numpy(np.ascontiguousarray(scales).view(np.float16)).to(device)
        return cls.from_device(c, s, keep_codes, stream)

    @classmethod
    def from_float(cls, w: np.ndarray, device="cuda", n_threads: int = 0, keep_codes: bool = False):
        return cls.from_packed(*pack_int8_host(w, n_threads), device=device, keep_codes=keep_codes)

    def c_struct(self) -> q8_matrix:
        p = lambda t: _ptr(t) if t is not None else None
        return q8_matrix(p(self.codes), p(self.scales), self.N, self.K, p(self.tiled))

    def workspace(self, B: int, device="cuda") -> Workspace:
        return Workspace(int(lib.q8_head_workspace_bytes(self.N, self.K, B)), device)

    def __call__(self, X: torch.Tensor, Y: torch.Tensor | None = None, idx: torch.Tensor | None = None,
                 logits: bool = True, argmax: bool = True, workspace: Workspace | None = None, stream=None):
        """Returns (Y or None, idx or None) for X bf16 [B, K]."""
        B = _check_x(X, self.K)
        if logits and Y is None:
            Y = torch.empty((B, self.N), dtype=torch.float32, device=X.device)
        if argmax and idx is None:
            idx = torch.empty((B,), dtype=torch.int32, device=X.device)
        if logits:
            _check_y(Y, B, self.N)
        if argmax:
            _check_i32(idx, B, "idx")
        if workspace is None:
            workspace = self.workspace(B, X.device)
        ws_p, ws_n = _ws_args(workspace)
        m = self.c_struct()
        check(lib.q8_head(ctypes.byref(m), _ptr(X), B, _ptr(Y) if logits else None, _ptr(idx) if argmax else None,
                          ws_p, ws_n, _stream_ptr(stream)), "q8_head")
        return (Y if logits else None), (idx if argmax else None)


def prefill_kernel(K: int, M: int) -> str:
    """The kernel q4_gemm_prefill runs for (K, M) on the current device: "tcgen05" or "mma.sync"."""
    k = int(lib.q4_prefill_kernel(K, M))
    if k < 0:
        raise ValueError(f"invalid prefill sizes K={K} M={M}")
    return "tcgen05" if k == 1 else "mma.sync"


def gemm_prefill(W: QuantizedMatrix, X: torch.Tensor, Y: torch.Tensor | None = None,
                 workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """Y [M, N] = X [M, K] W^T for a prompt of M tokens (q4_gemm_prefill, tensor-core GEMM; the
    tcgen05 kernel for K <= 8192, see prefill_kernel)."""
    M = _check_x(X, W.K)
    X2 = X if X.dim() == 2 else X.view(1, -1)
    if Y is None:
        Y = torch.empty((M, W.N), dtype=torch.float32, device=X.device)
    _check_y(Y, M, W.N)
    if workspace is None:
        workspace = Workspace(int(lib.q4_prefill_workspace_bytes(W.K, M)), X.device)
    ws_p, ws_n = _ws_args(workspace)
    m = W.c_struct()
    check(lib.q4_gemm_prefill(ctypes.byref(m), _ptr(X2), M, _ptr(Y), ws_p, ws_n, _stream_ptr(stream)),
          "q4_gemm_prefill")
    return Y


def sample_topk(Y: torch.Tensor, k: int, inv_temperature: float, noise: torch.Tensor,
                token: torch.Tensor | None = None, topk: torch.Tensor | None = None, return_topk: bool = False,
                stream=None):
    """Top-k Gumbel-max sampling per row of fp32 logits [B, N] with caller-supplied noise [B, k]
    (q4_sample_topk).  Returns token int32 [B] (and the ranked top-k indices [B, k])."""
    if Y.dtype != torch.float32 or not Y.is_contiguous() or noise.dtype != torch.float32 or not noise.is_contiguous():
        raise TypeError("logits and noise must be contiguous float32 CUDA tensors")
    Y2 = Y if Y.dim() == 2 else Y.view(1, -1)
    B, N = Y2.shape
    if token is None:
        token = torch.empty((B,), dtype=torch.int32, device=Y.device)
    if return_topk and topk is None:
        topk = torch.empty((B, k), dtype=torch.int32, device=Y.device)
    if noise.numel() < B * k:
        raise ValueError(f"noise must hold B * k = {B} * {k} values")
    _check_i32(token, B, "token")
    if topk is not None:
        _check_i32(topk, B * k, "topk")
    check(lib.q4_sample_topk(_ptr(Y2), B, N, int(k), float(inv_temperature), _ptr(noise), _ptr(token),
                             _ptr(topk) if topk is not None else None, _stream_ptr(stream)), "q4_sample_topk")
    return (token, topk) if return_topk else token


def flash_decode_workspace(B: int, n_q_heads: int, n_kv_heads: int, head_dim: int, n_chunks: int = 0,
                           device="cuda") -> Workspace:
    """Workspace for flash_decode with these sizes (q4_flash_decode_workspace_bytes)."""
    n = int(lib.q4_flash_decode_workspace_bytes(B, n_q_heads, n_kv_heads, head_dim, n_chunks))
    if n == 0:
        raise Q4Error(1, "q4_flash_decode_workspace_bytes")
    return Workspace(n, device)


def flash_decode(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, lengths: torch.Tensor,
                 O: torch.Tensor | None = None, scale: float | None = None, n_chunks: int = 0,
                 workspace: Workspace | None = None, stream=None) -> torch.Tensor:
    """One decode step of grouped-query attention over a KV cache (q4_flash_decode).

    Q bf16 [B, Hq, D]; K, V bf16 [B, Hkv, Lmax, D]; lengths int32 [B] on the device; returns
    O fp32 [B, Hq, D].  scale defaults to 1/sqrt(D)."""
    for name, t in (("Q", Q), ("K", K), ("V", V)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous torch.bfloat16 CUDA tensor")
    if lengths.dtype != torch.int32 or not lengths.is_contiguous():
        raise TypeError("lengths must be a contiguous int32 CUDA tensor")
    B, Hq, D = Q.shape
    _, Hkv, Lmax, _ = K.shape
    if tuple(K.shape) != (B, Hkv, Lmax, D) or tuple(V.shape) != tuple(K.shape):
        raise ValueError("K and V must be [B, Hkv, Lmax, D] matching Q [B, Hq, D]")
    if O is None:
        O = torch.empty((B, Hq, D), dtype=torch.float32, device=Q.device)
    if workspace is None:
        workspace = flash_decode_workspace(B, Hq, Hkv, D, n_chunks, Q.device)
    sc = float(scale) if scale is not None else 1.0 / float(D) ** 0.5
    check(lib.q4_flash_decode(_ptr(Q), _ptr(K), _ptr(V), _ptr(lengths), B, Hq, Hkv, D, Lmax, sc, int(n_chunks),
                              _ptr(O), *_ws_args(workspace), _stream_ptr(stream)), "q4_flash_decode")
    return O


class DecodeStepGraph:
    """One decode step (all matrices, in order) captured once into a CUDA graph and replayed.

    The activations and outputs are fixed device buffers: write new activations
    into ``self.X[i]`` and read ``self.Y[i]`` after ``replay()``.  Unless X is
    given, the activations are views of one contiguous buffer ``self.X_flat``
    (matrix after matrix, [B, K] each), so a step's inputs arrive in one copy.
    """

    def __init__(self, mats, B: int, X=None, Y=None, workspace: Workspace | None = None, device="cuda",
                 with_argmax_of: int | None = None, independent: bool = True, after=None):
        self.after = after  # optional: after(stream) enqueues more library calls into the same graph
        self.mats = list(mats)
        self.B = B
        self.independent = independent
        if X is None:
            sizes = [B * m.K for m in self.mats]     # multiples of 128 elements: views stay 16-byte aligned
            self.X_flat = torch.zeros((sum(sizes),), dtype=torch.bfloat16, device=device)
            self.X = [v.view(B, m.K) for v, m in zip(torch.split(self.X_flat, sizes), self.mats)]
        else:
            self.X_flat = None
            self.X = X
        self.Y = Y if Y is not None else [torch.empty((B, m.N), dtype=torch.float32, device=device)
                                           for m in self.mats]
        self.ws = workspace if workspace is not None else \
            Workspace.for_shapes([(m.N, m.K) for m in self.mats], B, device, independent)
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
        decode_step(self.mats, self.X, self.Y, self.ws, stream=stream, independent=self.independent)
        if self.argmax_of is not None:
            argmax(self.Y[self.argmax_of], self.idx, stream=stream)
        if self.after is not None:
            self.after(stream)

    def replay(self):
        self.graph.replay()

    def run_host(self, X_host, Y_host=None, idx_host=None):
        """One step end to end: copy the activations from (pinned) host memory -- one tensor laid
        out like ``X_flat``, or one tensor per matrix -- replay, copy the outputs and/or the argmax
        indices back, and wait for them."""
        if isinstance(X_host, torch.Tensor):
            self.X_flat.copy_(X_host, non_blocking=True)
        else:
            for d, h in zip(self.X, X_host):
                d.copy_(h, non_blocking=True)
        self.graph.replay()
        for d, h in zip(self.Y, Y_host or []):
            h.copy_(d, non_blocking=True)
        if idx_host is not None and self.idx is not None:
            idx_host.copy_(self.idx, non_blocking=True)
        torch.cuda.current_stream().synchronize()
