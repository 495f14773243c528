"""ctypes mirror of include/attn.h and the loader of the in-tree library.

Argument marshalling only: every step of the attention computation runs in
the CUDA library.  Importing this module fails loudly when the library has
not been built; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_lib", "libattn_gb300.so")

ABI_VERSION = 6

ATTN_OK, ATTN_EINVAL, ATTN_EUNSUPPORTED, ATTN_ECUDA, ATTN_ETIMEOUT, ATTN_EWORKSPACE = 0, -1, -2, -3, -4, -5
ATTN_F16, ATTN_BF16, ATTN_F32 = 0, 1, 2
ATTN_FULL, ATTN_CAUSAL = 0, 1
ATTN_KERNEL_AUTO, ATTN_KERNEL_SIMT, ATTN_KERNEL_TC = 0, 1, 2
ATTN_DQ_AUTO, ATTN_DQ_SEPARATE, ATTN_DQ_FUSED = 0, 1, 2
ATTN_NOALLOC_MAX_SEQ = 16367
ATTN_MAX_SPLITS = 64

# every symbol include/attn.h declares
EXPORTS = (
    "attn_abi_version", "attn_fwd_args_size", "attn_bwd_args_size",
    "attn_fwd_workspace_bytes", "attn_bwd_workspace_bytes", "attn_fwd", "attn_bwd",
    "attn_bwd_preprocess", "attn_bwd_dkdv", "attn_bwd_dq", "attn_fwd_simple",
    "attn_device_status", "attn_launch_count", "attn_strerror", "attn_last_error_string",
    "attn_fwd_selected_kernel", "attn_bwd_selected_kernel", "attn_fwd_noalloc",
    "attn_selftest_exp2", "attn_set_watchdog_cycles", "attn_merge_args_size",
    "attn_fwd_num_splits", "attn_merge", "attn_csr_args_size", "attn_csr_fwd",
    "attn_bwd_selected_dq_mode", "attn_fwd_simple_workspace_bytes",
)


class AttnTensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("stride_tok", ctypes.c_int64),
                ("stride_head", ctypes.c_int64)]


class FwdArgs(ctypes.Structure):
    _fields_ = [
        ("q", AttnTensor), ("k", AttnTensor), ("v", AttnTensor), ("o", AttnTensor),
        ("lse", ctypes.c_void_p),
        ("n_q", ctypes.c_int32), ("n_k", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
        ("scale", ctypes.c_float), ("relation", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("o_dtype", ctypes.c_int32), ("n_seq", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("kernel", ctypes.c_int32), ("num_ctas", ctypes.c_int32), ("num_splits", ctypes.c_int32),
        ("prune_threshold", ctypes.c_float), ("pruned_tiles", ctypes.c_void_p),
        ("qk_fp8", ctypes.c_int32),
    ]


class MergeArgs(ctypes.Structure):
    _fields_ = [
        ("o_parts", ctypes.c_void_p), ("lse_parts", ctypes.c_void_p), ("o", AttnTensor),
        ("lse", ctypes.c_void_p), ("n_parts", ctypes.c_int32), ("n_q", ctypes.c_int32),
        ("H", ctypes.c_int32), ("D", ctypes.c_int32), ("o_dtype", ctypes.c_int32),
    ]


class CsrArgs(ctypes.Structure):
    _fields_ = [
        ("row_ptr", ctypes.c_void_p), ("col_idx", ctypes.c_void_p), ("n_edges", ctypes.c_int64),
        ("n_dst", ctypes.c_int32), ("n_src", ctypes.c_int32), ("H", ctypes.c_int32),
        ("D", ctypes.c_int32), ("edge_scores", ctypes.c_void_p),
        ("q", AttnTensor), ("k", AttnTensor), ("v", AttnTensor), ("o", AttnTensor),
        ("lse", ctypes.c_void_p), ("scale", ctypes.c_float), ("dtype", ctypes.c_int32),
        ("o_dtype", ctypes.c_int32), ("row_order", ctypes.c_void_p),
    ]


class BwdArgs(ctypes.Structure):
    _fields_ = [
        ("q", AttnTensor), ("k", AttnTensor), ("v", AttnTensor), ("o", AttnTensor),
        ("dout", AttnTensor), ("lse", ctypes.c_void_p),
        ("dq", AttnTensor), ("dk", AttnTensor), ("dv", AttnTensor),
        ("n_q", ctypes.c_int32), ("n_k", ctypes.c_int32), ("H", ctypes.c_int32), ("D", ctypes.c_int32),
        ("scale", ctypes.c_float), ("relation", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("o_dtype", ctypes.c_int32), ("grad_dtype", ctypes.c_int32), ("n_seq", ctypes.c_int32),
        ("cu_seqlens_q", ctypes.c_void_p), ("cu_seqlens_k", ctypes.c_void_p),
        ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
        ("kernel", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
        ("prune_threshold", ctypes.c_float), ("dq_mode", ctypes.c_int32),
    ]


_lib = None


def load() -> ctypes.CDLL:
    """Load the library (once).  Raises if it is missing or mismatched."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"CUDA attention library not built ({LIB_PATH} missing); run "
            "`python -c 'import __graft_entry__ as g; g.build()'` or "
            "`python online_softmax_attention_gb300/build.py`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    fa, ba, ma = ctypes.POINTER(FwdArgs), ctypes.POINTER(BwdArgs), ctypes.POINTER(MergeArgs)
    ca = ctypes.POINTER(CsrArgs)
    sigs = {
        "attn_abi_version": (ctypes.c_int, []),
        "attn_fwd_args_size": (sz, []),
        "attn_bwd_args_size": (sz, []),
        "attn_merge_args_size": (sz, []),
        "attn_fwd_num_splits": (ctypes.c_int, [fa]),
        "attn_merge": (ctypes.c_int, [ma, vp]),
        "attn_csr_args_size": (sz, []),
        "attn_csr_fwd": (ctypes.c_int, [ca, vp]),
        "attn_fwd_workspace_bytes": (sz, [fa]),
        "attn_bwd_workspace_bytes": (sz, [ba]),
        "attn_fwd": (ctypes.c_int, [fa, vp]),
        "attn_bwd": (ctypes.c_int, [ba, vp]),
        "attn_bwd_preprocess": (ctypes.c_int, [ba, vp]),
        "attn_bwd_dkdv": (ctypes.c_int, [ba, vp]),
        "attn_bwd_dq": (ctypes.c_int, [ba, vp]),
        "attn_fwd_simple": (ctypes.c_int, [vp, vp, vp, vp, vp, i32, i32, i32, ctypes.c_float, i32,
                                           vp, i32, i32, vp, sz, vp]),
        "attn_fwd_simple_workspace_bytes": (sz, [i32, i32, i32, i32, i32, i32]),
        "attn_device_status": (ctypes.c_int, [vp]),
        "attn_fwd_selected_kernel": (ctypes.c_int, [fa]),
        "attn_fwd_noalloc": (ctypes.c_int, [fa, vp]),
        "attn_selftest_exp2": (ctypes.c_int, [vp, vp, i32, vp]),
        "attn_set_watchdog_cycles": (ctypes.c_longlong, [ctypes.c_longlong]),
        "attn_bwd_selected_kernel": (ctypes.c_int, [ba]),
        "attn_bwd_selected_dq_mode": (ctypes.c_int, [ba]),
        "attn_launch_count": (ctypes.c_uint64, []),
        "attn_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "attn_last_error_string": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if lib.attn_abi_version() != ABI_VERSION:
        raise ImportError(f"libattn_gb300 ABI {lib.attn_abi_version()} != binding ABI {ABI_VERSION}")
    if lib.attn_fwd_args_size() != ctypes.sizeof(FwdArgs) or \
            lib.attn_bwd_args_size() != ctypes.sizeof(BwdArgs) or \
            lib.attn_merge_args_size() != ctypes.sizeof(MergeArgs) or \
            lib.attn_csr_args_size() != ctypes.sizeof(CsrArgs):
        raise ImportError("libattn_gb300 struct layout does not match the binding")
    _lib = lib
    return lib


class AttnError(RuntimeError):
    def __init__(self, code: int, where: str):
        lib = load()
        msg = lib.attn_strerror(code).decode()
        if code == ATTN_ECUDA:
            msg += ": " + lib.attn_last_error_string().decode()
        super().__init__(f"{where} failed ({code}): {msg}")
        self.code = code


def check(code: int, where: str) -> None:
    if code != ATTN_OK:
        raise AttnError(code, where)
