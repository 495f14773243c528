"""Exact online-softmax attention on one GB300 (sm_103a), forward and backward.

PyTorch is used for device memory and streams only; every step of the
computation runs in the CUDA library ``_lib/libattn_gb300.so`` through its C
ABI (``include/attn.h``).  This module marshals tensors into the ABI's
argument structs:

* ``fwd(q, k, v, causal=..., cu_seqlens_q=...)`` -> ``(o, lse)``
* ``bwd(q, k, v, o, lse, dout, causal=...)`` -> ``(dq, dk, dv)``
* ``merge(o_parts, lse_parts)`` -> ``(o, lse)``: attention over the union of
  disjoint key sets from each set's result (the split-K merge)
* ``csr_fwd(row_ptr, col, v, scores=... | q=..., k=...)`` -> ``(o, lse)``:
  attention over a general CSR relation (softmax over each row's edges)
* ``FwdCall`` / ``BwdCall`` hold prepared argument structs for repeated
  launches (the benchmark and CUDA-graph capture use them).

Tensors are (tokens, heads, D) with the D axis contiguous; any token / head
strides whose rows stay 16-byte aligned are accepted (for example an (H, N, D)
tensor viewed as (N, H, D)).  ``cu_seqlens`` follow flash-attn's varlen
convention ``[0, L1, L1+L2, ...]`` as int32.
"""
from __future__ import annotations

import ctypes

import torch

from . import _abi
from ._abi import (ATTN_BF16, ATTN_CAUSAL, ATTN_F16, ATTN_F32, ATTN_FULL, ATTN_KERNEL_AUTO,
                   ATTN_KERNEL_SIMT, ATTN_KERNEL_TC, AttnError, check)

__all__ = ["fwd", "bwd", "merge", "csr_fwd", "FwdCall", "BwdCall", "MergeCall", "CsrCall",
           "device_status", "launch_count", "AttnError", "library_path"]

_DT = {torch.float16: ATTN_F16, torch.bfloat16: ATTN_BF16, torch.float32: ATTN_F32}
_E4M3 = getattr(torch, "float8_e4m3fn", None)
_KERNELS = {"auto": ATTN_KERNEL_AUTO, "simt": ATTN_KERNEL_SIMT, "tc": ATTN_KERNEL_TC}
# backward dq: "separate" (own kernel, deterministic), "fused" (dK/dV kernel adds
# f32 partial sums; tensor-core kernels only), "auto" (= separate)
_DQ_MODES = {"auto": _abi.ATTN_DQ_AUTO, "separate": _abi.ATTN_DQ_SEPARATE, "fused": _abi.ATTN_DQ_FUSED}


def library_path() -> str:
    return _abi.LIB_PATH


def launch_count() -> int:
    """Kernels launched by the library so far in this process."""
    return int(_abi.load().attn_launch_count())


def device_status(stream: torch.cuda.Stream | None = None) -> int:
    """Synchronise the stream and return / clear the device status word."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return int(_abi.load().attn_device_status(ctypes.c_void_p(s.cuda_stream)))


def strerror(code: int) -> str:
    """The library's message for a status code."""
    return _abi.load().attn_strerror(int(code)).decode()


def _dtype_code(dt: torch.dtype) -> int:
    if dt not in _DT:
        raise TypeError(f"unsupported dtype {dt}; use float16, bfloat16 or float32")
    return _DT[dt]


def _view(t: torch.Tensor | None, name: str) -> _abi.AttnTensor:
    if t is None:
        return _abi.AttnTensor(None, 0, 0)
    if t.dim() != 3:
        raise ValueError(f"{name} must be (tokens, heads, D), got {tuple(t.shape)}")
    if t.stride(2) != 1 and t.shape[2] > 1:
        raise ValueError(f"{name}: the D axis must be contiguous")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    # a size-1 axis is never stepped along, so any aligned stride describes it
    st = t.stride(0) if t.shape[0] > 1 else t.shape[1] * t.shape[2]
    sh = t.stride(1) if t.shape[1] > 1 else t.shape[2]
    return _abi.AttnTensor(t.data_ptr() if t.numel() else None, st, sh)


def _cu(cu, device) -> torch.Tensor | None:
    if cu is None:
        return None
    cu = torch.as_tensor(cu)
    if cu.dtype != torch.int32:
        cu = cu.to(torch.int32)
    return cu.to(device).contiguous()


def _workspace(nbytes: int, device) -> torch.Tensor:
    # torch's caching allocator returns 512-byte aligned blocks
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _selected(code: int, where: str) -> str:
    if code < 0:
        check(code, where)
    return "tc" if code == ATTN_KERNEL_TC else "simt"


class FwdCall:
    """Prepared forward: holds the argument struct, outputs and workspace."""

    def __init__(self, q, k, v, *, causal: bool = False, scale: float | None = None,
                 cu_seqlens_q=None, cu_seqlens_k=None, out_dtype: torch.dtype | None = None,
                 kernel: str = "auto", num_ctas: int = 0, num_splits: int = 0,
                 prune_threshold: float = 0.0, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, workspace: torch.Tensor | None = None):
        # fp8 (e4m3) queries and keys with a 16-bit v: the tensor-core kernel
        # contracts the scores in fp8 (attn.h, qk_fp8)
        qk_fp8 = q.dtype == _E4M3 and _E4M3 is not None
        if qk_fp8:
            if k.dtype != _E4M3:
                raise TypeError("fp8 queries need fp8 (float8_e4m3fn) keys")
        elif q.dtype != k.dtype or q.dtype != v.dtype:
            raise TypeError("q, k, v must share one dtype")
        dev = q.device
        Tq, H, D = q.shape
        Tk = k.shape[0]
        out_dtype = out_dtype or v.dtype
        self.cu_q = _cu(cu_seqlens_q, dev)
        self.cu_k = _cu(cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q, dev)
        self.o = out if out is not None else torch.empty((Tq, H, D), dtype=out_dtype, device=dev)
        self.lse = lse if lse is not None else torch.empty((H, Tq), dtype=torch.float32, device=dev)
        self.inputs = (q, k, v)
        a = _abi.FwdArgs()
        a.q, a.k, a.v, a.o = _view(q, "q"), _view(k, "k"), _view(v, "v"), _view(self.o, "out")
        a.lse = self.lse.data_ptr() if self.lse.numel() else None
        a.n_q, a.n_k, a.H, a.D = Tq, Tk, H, D
        a.scale = float(scale) if scale is not None else D ** -0.5
        a.relation = ATTN_CAUSAL if causal else ATTN_FULL
        a.dtype, a.o_dtype = _dtype_code(v.dtype), _dtype_code(self.o.dtype)
        a.qk_fp8 = 1 if qk_fp8 else 0
        a.n_seq = (self.cu_q.numel() - 1) if self.cu_q is not None else 1
        a.cu_seqlens_q = self.cu_q.data_ptr() if self.cu_q is not None else None
        a.cu_seqlens_k = self.cu_k.data_ptr() if self.cu_k is not None else None
        a.kernel = _KERNELS[kernel]
        a.num_ctas = int(num_ctas)
        a.num_splits = int(num_splits)
        a.prune_threshold = float(prune_threshold)
        # pruned-tile counter (device, int64 storage of the library's uint64)
        self.pruned_tiles = torch.zeros(1, dtype=torch.int64, device=dev) if prune_threshold else None
        a.pruned_tiles = self.pruned_tiles.data_ptr() if self.pruned_tiles is not None else None
        lib = _abi.load()
        need = lib.attn_fwd_workspace_bytes(ctypes.byref(a))
        self.workspace = workspace if workspace is not None else _workspace(need, dev)
        a.workspace = self.workspace.data_ptr()
        a.workspace_bytes = self.workspace.numel() * self.workspace.element_size()
        self.args = a
        self._fn = lib.attn_fwd

    def run(self, stream: torch.cuda.Stream | None = None):
        s = stream if stream is not None else torch.cuda.current_stream()
        check(self._fn(ctypes.byref(self.args), ctypes.c_void_p(s.cuda_stream)), "attn_fwd")
        return self.o, self.lse

    def selected_kernel(self) -> str:
        """"tc" or "simt": the kernel family these arguments run."""
        return _selected(_abi.load().attn_fwd_selected_kernel(ctypes.byref(self.args)),
                         "attn_fwd_selected_kernel")

    def pruned_count(self) -> int:
        """Tiles pruned by all runs of this call so far (0 without pruning)."""
        return int(self.pruned_tiles.item()) if self.pruned_tiles is not None else 0

    def num_splits(self) -> int:
        """Key splits (split-K chunks) these arguments run, 1 = none."""
        n = int(_abi.load().attn_fwd_num_splits(ctypes.byref(self.args)))
        if n < 0:
            check(n, "attn_fwd_num_splits")
        return n


class MergeCall:
    """Prepared merge of partial results over disjoint key sets.

    ``o_parts`` is (C, T, H, D) float32 contiguous, ``lse_parts`` (C, H, T)
    float32 contiguous (-inf marks a partial that admits no key).
    """

    def __init__(self, o_parts: torch.Tensor, lse_parts: torch.Tensor, *,
                 out_dtype: torch.dtype = torch.float32, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None):
        if o_parts.dtype != torch.float32 or lse_parts.dtype != torch.float32:
            raise TypeError("o_parts and lse_parts must be float32")
        if o_parts.dim() != 4 or not o_parts.is_contiguous() or not lse_parts.is_contiguous():
            raise ValueError("o_parts must be contiguous (C, T, H, D), lse_parts contiguous (C, H, T)")
        C, T, H, D = o_parts.shape
        if tuple(lse_parts.shape) != (C, H, T):
            raise ValueError(f"lse_parts must be {(C, H, T)}, got {tuple(lse_parts.shape)}")
        dev = o_parts.device
        self.o = out if out is not None else torch.empty((T, H, D), dtype=out_dtype, device=dev)
        self.lse = lse if lse is not None else torch.empty((H, T), dtype=torch.float32, device=dev)
        self.inputs = (o_parts, lse_parts)
        a = _abi.MergeArgs()
        a.o_parts = o_parts.data_ptr() if o_parts.numel() else None
        a.lse_parts = lse_parts.data_ptr() if lse_parts.numel() else None
        a.o = _view(self.o, "out")
        a.lse = self.lse.data_ptr() if self.lse.numel() else None
        a.n_parts, a.n_q, a.H, a.D = C, T, H, D
        a.o_dtype = _dtype_code(self.o.dtype)
        self.args = a
        self._fn = _abi.load().attn_merge

    def run(self, stream: torch.cuda.Stream | None = None):
        s = stream if stream is not None else torch.cuda.current_stream()
        check(self._fn(ctypes.byref(self.args), ctypes.c_void_p(s.cuda_stream)), "attn_merge")
        return self.o, self.lse


class BwdCall:
    """Prepared backward: holds the argument struct, gradients and workspace."""

    def __init__(self, q, k, v, o, lse, dout, *, causal: bool = False, scale: float | None = None,
                 cu_seqlens_q=None, cu_seqlens_k=None, grad_dtype: torch.dtype | None = None,
                 kernel: str = "auto", num_ctas: int = 0, dq=None, dk=None, dv=None,
                 workspace: torch.Tensor | None = None, prune_threshold: float = 0.0,
                 dq_mode: str = "auto"):
        dev = q.device
        Tq, H, D = q.shape
        Tk = k.shape[0]
        gdt = grad_dtype or q.dtype
        self.cu_q = _cu(cu_seqlens_q, dev)
        self.cu_k = _cu(cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q, dev)
        self.dq = dq if dq is not None else torch.empty((Tq, H, D), dtype=gdt, device=dev)
        self.dk = dk if dk is not None else torch.empty((Tk, H, D), dtype=gdt, device=dev)
        self.dv = dv if dv is not None else torch.empty((Tk, H, D), dtype=gdt, device=dev)
        self.inputs = (q, k, v, o, lse, dout)
        a = _abi.BwdArgs()
        a.q, a.k, a.v = _view(q, "q"), _view(k, "k"), _view(v, "v")
        a.o, a.dout = _view(o, "o"), _view(dout, "dout")
        a.lse = lse.data_ptr() if lse.numel() else None
        a.dq, a.dk, a.dv = _view(self.dq, "dq"), _view(self.dk, "dk"), _view(self.dv, "dv")
        a.n_q, a.n_k, a.H, a.D = Tq, Tk, H, D
        a.scale = float(scale) if scale is not None else D ** -0.5
        a.relation = ATTN_CAUSAL if causal else ATTN_FULL
        a.dtype, a.o_dtype = _dtype_code(q.dtype), _dtype_code(o.dtype)
        a.grad_dtype = _dtype_code(gdt)
        a.n_seq = (self.cu_q.numel() - 1) if self.cu_q is not None else 1
        a.cu_seqlens_q = self.cu_q.data_ptr() if self.cu_q is not None else None
        a.cu_seqlens_k = self.cu_k.data_ptr() if self.cu_k is not None else None
        a.kernel = _KERNELS[kernel]
        a.num_ctas = int(num_ctas)
        a.prune_threshold = float(prune_threshold)  # non-zero: the library refuses (fails closed)
        a.dq_mode = _DQ_MODES[dq_mode]
        lib = _abi.load()
        need = lib.attn_bwd_workspace_bytes(ctypes.byref(a))
        self.workspace = workspace if workspace is not None else _workspace(need, dev)
        a.workspace = self.workspace.data_ptr()
        a.workspace_bytes = self.workspace.numel() * self.workspace.element_size()
        self.args = a
        self._lib = lib

    def _call(self, fn, name, stream):
        s = stream if stream is not None else torch.cuda.current_stream()
        check(fn(ctypes.byref(self.args), ctypes.c_void_p(s.cuda_stream)), name)

    def preprocess(self, stream=None):
        self._call(self._lib.attn_bwd_preprocess, "attn_bwd_preprocess", stream)

    def dkdv(self, stream=None):
        self._call(self._lib.attn_bwd_dkdv, "attn_bwd_dkdv", stream)

    def dq_stage(self, stream=None):
        self._call(self._lib.attn_bwd_dq, "attn_bwd_dq", stream)

    def run(self, stream=None):
        self._call(self._lib.attn_bwd, "attn_bwd", stream)
        return self.dq, self.dk, self.dv

    def selected_kernel(self) -> str:
        """"tc" or "simt": the kernel family these arguments run."""
        return _selected(self._lib.attn_bwd_selected_kernel(ctypes.byref(self.args)),
                         "attn_bwd_selected_kernel")

    def selected_dq_mode(self) -> str:
        """"fused" or "separate": how these arguments compute dq."""
        code = self._lib.attn_bwd_selected_dq_mode(ctypes.byref(self.args))
        if code < 0:
            check(code, "attn_bwd_selected_dq_mode")
        return "fused" if code == _abi.ATTN_DQ_FUSED else "separate"


class CsrCall:
    """Prepared attention over a CSR relation.

    ``row_ptr`` (n_dst + 1) int64 and ``col`` (E) int32 on the device define
    the relation (row i's edges are ``col[row_ptr[i]:row_ptr[i+1]]``); ``v``
    is (n_src, H, D).  Scores: ``scores`` (E, H) float32 field scores, or
    ``q`` (n_dst, H, D) and ``k`` (n_src, H, D) for scale * <q_i, k_j>.
    ``row_order`` (n_dst) int32 on the device: the order in which the kernel
    takes the rows (results are the same bit for bit; an order that keeps
    rows with shared sources together makes their gathers L2 hits).
    """

    def __init__(self, row_ptr, col, v, *, scores=None, q=None, k=None, n_dst: int | None = None,
                 scale: float | None = None, out_dtype: torch.dtype | None = None,
                 out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 row_order: torch.Tensor | None = None):
        dev = v.device
        if row_ptr.dtype != torch.int64 or col.dtype != torch.int32:
            raise TypeError("row_ptr must be int64 and col int32")
        if not (row_ptr.is_cuda and col.is_cuda):
            raise ValueError("row_ptr and col must be CUDA tensors")
        n_src, H, D = v.shape
        n_dst = len(row_ptr) - 1 if n_dst is None else n_dst
        if scores is None and (q is None or k is None):
            raise ValueError("give either scores or both q and k")
        out_dtype = out_dtype or v.dtype
        self.o = out if out is not None else torch.empty((n_dst, H, D), dtype=out_dtype, device=dev)
        self.lse = lse if lse is not None else torch.empty((H, n_dst), dtype=torch.float32, device=dev)
        self.inputs = (row_ptr, col, v, scores, q, k)
        a = _abi.CsrArgs()
        a.row_ptr = row_ptr.data_ptr()
        a.col_idx = col.data_ptr() if col.numel() else None
        a.n_edges = col.numel()
        a.n_dst, a.n_src, a.H, a.D = n_dst, n_src, H, D
        if scores is not None:
            if scores.dtype != torch.float32 or tuple(scores.shape) != (col.numel(), H) \
                    or not scores.is_contiguous():
                raise ValueError("scores must be contiguous float32 (E, H)")
            a.edge_scores = scores.data_ptr() if scores.numel() else None
            if not scores.numel():
                a.edge_scores = row_ptr.data_ptr()  # no edge reads it; marks field scores
        else:
            a.q, a.k = _view(q, "q"), _view(k, "k")
        a.v, a.o = _view(v, "v"), _view(self.o, "out")
        a.lse = self.lse.data_ptr() if self.lse.numel() else None
        a.scale = float(scale) if scale is not None else D ** -0.5
        a.dtype, a.o_dtype = _dtype_code(v.dtype), _dtype_code(self.o.dtype)
        if row_order is not None:
            if row_order.dtype != torch.int32 or not row_order.is_cuda or row_order.numel() != n_dst \
                    or not row_order.is_contiguous():
                raise ValueError("row_order must be a contiguous int32 CUDA tensor of n_dst entries")
            a.row_order = row_order.data_ptr() if n_dst else None
            self.inputs = self.inputs + (row_order,)
        self.args = a
        self._fn = _abi.load().attn_csr_fwd

    def run(self, stream: torch.cuda.Stream | None = None):
        s = stream if stream is not None else torch.cuda.current_stream()
        check(self._fn(ctypes.byref(self.args), ctypes.c_void_p(s.cuda_stream)), "attn_csr_fwd")
        return self.o, self.lse


def csr_fwd(row_ptr, col, v, *, scores=None, q=None, k=None, scale: float | None = None,
            out_dtype: torch.dtype | None = None, row_order=None):
    """Attention over a CSR relation.  Returns ``(o, lse)``."""
    return CsrCall(row_ptr, col, v, scores=scores, q=q, k=k, scale=scale,
                   out_dtype=out_dtype, row_order=row_order).run()


def fwd(q, k, v, *, causal: bool = False, scale: float | None = None, cu_seqlens_q=None,
        cu_seqlens_k=None, out_dtype: torch.dtype | None = None, kernel: str = "auto",
        num_ctas: int = 0, num_splits: int = 0, prune_threshold: float = 0.0):
    """Attention forward.  Returns ``(o, lse)``; lse is (H, T_q) f32, natural log.

    ``num_splits``: key splits per query tile (split-K); 0 lets the library
    choose, 1 disables splitting.  ``prune_threshold``: 0 = exact; rho in
    (0, 1] enables approximate tile pruning (full relation, one sequence)."""
    return FwdCall(q, k, v, causal=causal, scale=scale, cu_seqlens_q=cu_seqlens_q,
                   cu_seqlens_k=cu_seqlens_k, out_dtype=out_dtype, kernel=kernel,
                   num_ctas=num_ctas, num_splits=num_splits,
                   prune_threshold=prune_threshold).run()


def merge(o_parts, lse_parts, *, out_dtype: torch.dtype = torch.float32):
    """Attention over the union of C disjoint key sets from each set's result:
    lse = ln sum_c exp(lse_c), o = sum_c exp(lse_c - lse) o_c.  Returns ``(o, lse)``."""
    return MergeCall(o_parts, lse_parts, out_dtype=out_dtype).run()


def bwd(q, k, v, o, lse, dout, *, causal: bool = False, scale: float | None = None,
        cu_seqlens_q=None, cu_seqlens_k=None, grad_dtype: torch.dtype | None = None,
        kernel: str = "auto", num_ctas: int = 0, dq_mode: str = "auto"):
    """Attention backward from the forward's o and lse.  Returns ``(dq, dk, dv)``."""
    return BwdCall(q, k, v, o, lse, dout, causal=causal, scale=scale, cu_seqlens_q=cu_seqlens_q,
                   cu_seqlens_k=cu_seqlens_k, grad_dtype=grad_dtype, kernel=kernel,
                   num_ctas=num_ctas, dq_mode=dq_mode).run()
