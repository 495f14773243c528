"""f64 CPU oracle for exact scaled dot-product attention -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline /
reference legs of ``bench.py`` may import this package.  The CUDA library in
``online_softmax_attention_gb300`` never imports it and shares no code with it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, OpenMP over
rows); this module only marshals arrays.  It defines the same operation as the
TIGA-lang attention examples page ("注意力与稠密关系", section "全量注意力，无掩码"
and its causal / varlen sections) and the composed two-pass softmax of the
OCANNL "Module Ir.Online_softmax" page.  See ``oracle.c`` for the citations of
each step.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` next to it (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        cmd = ["gcc", "-O2", "-ffp-contract=off", "-fopenmp", "-fPIC", "-shared",
               "-std=c11", "-o", _LIB + ".tmp", _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_fwd.argtypes = [
            ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp,
            ctypes.c_double, ctypes.c_int, _dp, _dp, ctypes.c_int]
        lib.oracle_attn_fwd_rows.restype = ctypes.c_int
        lib.oracle_attn_fwd_rows.argtypes = [
            ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp,
            ctypes.c_double, ctypes.c_int, ctypes.c_int, _i64p, _i32p, _dp, _dp, ctypes.c_int]
        lib.oracle_attn_bwd.restype = ctypes.c_int
        lib.oracle_attn_bwd.argtypes = [
            ctypes.c_int, _i32p, _i32p, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, _dp,
            ctypes.c_double, ctypes.c_int,
            ctypes.c_int, _i64p, _i32p, _dp,
            ctypes.c_int, _i64p, _i32p, _dp, _dp, ctypes.c_int]
        lib.oracle_attn_merge.restype = ctypes.c_int
        lib.oracle_attn_merge.argtypes = [
            ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp, _dp,
            ctypes.c_int]
        lib.oracle_attn_fwd_pruned.restype = ctypes.c_int
        lib.oracle_attn_fwd_pruned.argtypes = [
            ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _dp, _dp, _dp,
            ctypes.c_double, ctypes.c_double, ctypes.c_int, ctypes.c_int, _dp, _dp, _i64p, _dp,
            ctypes.c_int]
        lib.oracle_csr_fwd.restype = ctypes.c_int
        lib.oracle_csr_fwd.argtypes = [
            ctypes.c_int64, ctypes.c_int64, _i64p, _i32p, ctypes.c_int, ctypes.c_int, _dp, _dp,
            _dp, _dp, ctypes.c_double, _dp, _dp, ctypes.c_int]
        lib.oracle_max_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def max_threads() -> int:
    """Threads the oracle's OpenMP runtime uses by default on this host."""
    return int(_load().oracle_max_threads())


def _f64(x) -> np.ndarray:
    """Exact widening to a contiguous float64 numpy array (torch or numpy in)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch  # noqa: PLC0415  (only when torch tensors are passed)
        x = x.to(torch.float64).contiguous().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _cu(cu, total: int) -> np.ndarray:
    if cu is None:
        return np.array([0, total], dtype=np.int32)
    if hasattr(cu, "detach"):
        cu = cu.detach().to("cpu").numpy()
    return np.ascontiguousarray(np.asarray(cu, dtype=np.int32))


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


def _shape3(x: np.ndarray, name: str):
    if x.ndim != 3:
        raise ValueError(f"{name} must be (tokens, heads, dim), got shape {x.shape}")
    return x.shape


def fwd(q, k, v, *, causal: bool, scale: float | None = None, cu_seqlens_q=None,
        cu_seqlens_k=None, threads: int = 0):
    """Attention forward over (T, H, D) tensors.

    Returns ``(o, lse)``: o is float64 (T_q, H, D); lse is float64 (H, T_q),
    the natural log of the sum of exp(scaled score) over the admitted keys.
    ``cu_seqlens_*`` are cumulative segment offsets starting at 0 (None = one
    segment).  ``scale`` defaults to D^-1/2.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, H, D = _shape3(q, "q")
    Tk = _shape3(k, "k")[0]
    if v.shape != k.shape:
        raise ValueError("v must have k's shape")
    cq = _cu(cu_seqlens_q, Tq)
    ck = _cu(cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q, Tk)
    if scale is None:
        scale = D ** -0.5
    o = np.zeros((Tq, H, D), dtype=np.float64)
    lse = np.zeros((H, Tq), dtype=np.float64)
    rc = _load().oracle_attn_fwd(len(cq) - 1, _ptr(cq, _i32p), _ptr(ck, _i32p), H, D,
                                 _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), float(scale),
                                 int(bool(causal)), _ptr(o, _dp), _ptr(lse, _dp), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd rejected its arguments (rc={rc})")
    return o, lse


def fwd_rows(q, k, v, tokens, heads, *, causal: bool, scale: float | None = None,
             cu_seqlens_q=None, cu_seqlens_k=None, threads: int = 0):
    """Forward for listed (token, head) query rows only: ``(o_rows (n, D), lse (n,))``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, H, D = _shape3(q, "q")
    Tk = _shape3(k, "k")[0]
    cq = _cu(cu_seqlens_q, Tq)
    ck = _cu(cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q, Tk)
    if scale is None:
        scale = D ** -0.5
    tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int64))
    hd = np.ascontiguousarray(np.asarray(heads, dtype=np.int32))
    n = len(tok)
    o = np.zeros((n, D), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = _load().oracle_attn_fwd_rows(len(cq) - 1, _ptr(cq, _i32p), _ptr(ck, _i32p), H, D,
                                      _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), float(scale),
                                      int(bool(causal)), n, _ptr(tok, _i64p), _ptr(hd, _i32p),
                                      _ptr(o, _dp), _ptr(lse, _dp), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_rows rejected its arguments (rc={rc})")
    return o, lse


def bwd(q, k, v, dO, *, causal: bool, scale: float | None = None, cu_seqlens_q=None,
        cu_seqlens_k=None, q_rows=None, k_rows=None, threads: int = 0):
    """Backward by the explicit softmax Jacobian.

    With ``q_rows`` / ``k_rows`` None, returns full float64 ``(dq, dk, dv)``
    shaped like q, k, v.  Otherwise ``q_rows`` / ``k_rows`` are
    ``(tokens, heads)`` pairs and the matching outputs are ``(n, D)``.
    """
    q, k, v, dO = _f64(q), _f64(k), _f64(v), _f64(dO)
    Tq, H, D = _shape3(q, "q")
    Tk = _shape3(k, "k")[0]
    if dO.shape != q.shape:
        raise ValueError("dO must have q's shape")
    cq = _cu(cu_seqlens_q, Tq)
    ck = _cu(cu_seqlens_k if cu_seqlens_k is not None else cu_seqlens_q, Tk)
    if scale is None:
        scale = D ** -0.5

    def sel(rows, total):
        if rows is None:
            return 0, None, None, np.zeros((total, H, D), dtype=np.float64)
        tok = np.ascontiguousarray(np.asarray(rows[0], dtype=np.int64))
        hd = np.ascontiguousarray(np.asarray(rows[1], dtype=np.int32))
        return len(tok), tok, hd, np.zeros((len(tok), D), dtype=np.float64)

    nq, qt, qh, dq = sel(q_rows, Tq)
    nk, kt, kh, dk = sel(k_rows, Tk)
    dv = np.zeros_like(dk)
    lib = _load()
    rc = lib.oracle_attn_bwd(
        len(cq) - 1, _ptr(cq, _i32p), _ptr(ck, _i32p), H, D,
        _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(dO, _dp), float(scale), int(bool(causal)),
        nq, None if qt is None else _ptr(qt, _i64p), None if qh is None else _ptr(qh, _i32p),
        _ptr(dq, _dp),
        nk, None if kt is None else _ptr(kt, _i64p), None if kh is None else _ptr(kh, _i32p),
        _ptr(dk, _dp), _ptr(dv, _dp), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn_bwd rejected its arguments (rc={rc})")
    return dq, dk, dv


def merge(o_parts, lse_parts, *, threads: int = 0):
    """Attention over the union of C disjoint key sets from each set's result.

    ``o_parts`` is (C, T, H, D), ``lse_parts`` is (C, H, T); returns float64
    ``(o (T, H, D), lse (H, T))`` with lse = ln sum_c exp(lse_c) and
    o = sum_c exp(lse_c - lse) o_c (rows whose partials are all -inf: o = 0,
    lse = -inf).
    """
    op, lp = _f64(o_parts), _f64(lse_parts)
    if op.ndim != 4:
        raise ValueError(f"o_parts must be (C, T, H, D), got shape {op.shape}")
    C, T, H, D = op.shape
    if lp.shape != (C, H, T):
        raise ValueError(f"lse_parts must be (C, H, T) = {(C, H, T)}, got {lp.shape}")
    o = np.zeros((T, H, D), dtype=np.float64)
    lse = np.zeros((H, T), dtype=np.float64)
    rc = _load().oracle_attn_merge(C, T, H, D, _ptr(op, _dp), _ptr(lp, _dp), _ptr(o, _dp),
                                   _ptr(lse, _dp), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn_merge rejected its arguments (rc={rc})")
    return o, lse


def fwd_pruned(q, k, v, *, rho: float, block_q: int, block_k: int, scale: float | None = None,
               threads: int = 0):
    """Tile-pruned approximate forward, one sequence, full relation.

    Returns ``(o, lse, n_pruned, min_margin)``: o (T_q, H, D) and lse (H, T_q)
    float64; n_pruned = pruned (query block, key tile) pairs over all heads;
    min_margin = smallest |m_tile - (m_run + ln rho)| of the decisions taken
    against a finite rolling max (inf when there were none).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    Tq, H, D = _shape3(q, "q")
    Tk = _shape3(k, "k")[0]
    if v.shape != k.shape:
        raise ValueError("v must have k's shape")
    if scale is None:
        scale = D ** -0.5
    o = np.zeros((Tq, H, D), dtype=np.float64)
    lse = np.zeros((H, Tq), dtype=np.float64)
    n_pruned = np.zeros(1, dtype=np.int64)
    margin = np.zeros(1, dtype=np.float64)
    rc = _load().oracle_attn_fwd_pruned(Tq, Tk, H, D, _ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp),
                                        float(scale), float(rho), int(block_q), int(block_k),
                                        _ptr(o, _dp), _ptr(lse, _dp), _ptr(n_pruned, _i64p),
                                        _ptr(margin, _dp), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_attn_fwd_pruned rejected its arguments (rc={rc})")
    return o, lse, int(n_pruned[0]), float(margin[0])


def csr_fwd(row_ptr, col, v, *, scores=None, q=None, k=None, scale: float | None = None,
            threads: int = 0):
    """Attention over a CSR relation: softmax over each destination row's edges.

    ``row_ptr`` (n_dst + 1) and ``col`` (E) define the relation; ``v`` is
    (n_src, H, D).  Scores are ``scores`` (E, H) when given, else
    scale * <q_i, k_j> with q (n_dst, H, D), k (n_src, H, D), scale default
    D^-1/2.  Returns float64 ``(o (n_dst, H, D), lse (H, n_dst))``.
    """
    rp = np.ascontiguousarray(np.asarray(row_ptr.cpu() if hasattr(row_ptr, "cpu") else row_ptr,
                                         dtype=np.int64))
    cl = np.ascontiguousarray(np.asarray(col.cpu() if hasattr(col, "cpu") else col, dtype=np.int32))
    v = _f64(v)
    n_src, H, D = _shape3(v, "v")
    n_dst = len(rp) - 1
    sc = _f64(scores) if scores is not None else None
    if sc is not None and sc.shape != (len(cl), H):
        raise ValueError(f"scores must be (E, H) = {(len(cl), H)}, got {sc.shape}")
    qq = _f64(q) if q is not None else None
    kk = _f64(k) if k is not None else None
    if scale is None:
        scale = D ** -0.5
    o = np.zeros((n_dst, H, D), dtype=np.float64)
    lse = np.zeros((H, n_dst), dtype=np.float64)
    rc = _load().oracle_csr_fwd(n_dst, n_src, _ptr(rp, _i64p), _ptr(cl, _i32p), H, D,
                                None if sc is None else _ptr(sc, _dp),
                                None if qq is None else _ptr(qq, _dp),
                                None if kk is None else _ptr(kk, _dp), _ptr(v, _dp), float(scale),
                                _ptr(o, _dp), _ptr(lse, _dp), int(threads))
    if rc != 0:
        raise ValueError(f"oracle_csr_fwd rejected its arguments (rc={rc})")
    return o, lse


if __name__ == "__main__":  # pragma: no cover - manual build hook
    print(build(force="--force" in sys.argv))
