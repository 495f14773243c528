"""The C-ABI library loads, exports what include/attn.h declares, and rejects
bad arguments before touching the GPU (CPU only: no kernel is launched)."""
import ctypes
import os
import re

import pytest

import online_softmax_attention_gb300 as attn
from online_softmax_attention_gb300 import _abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(autouse=True)
def _no_launch():
    """The calls here pass fake device pointers: none may reach a launch (on
    a machine with a GPU it would read and write those addresses)."""
    lib = _abi.load()
    before = lib.attn_launch_count()
    yield
    assert lib.attn_launch_count() == before, "a validation test launched a kernel"


def _declared():
    with open(os.path.join(ROOT, "include", "attn.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)))


def test_library_loads_and_abi_matches():
    lib = _abi.load()
    assert lib.attn_abi_version() == _abi.ABI_VERSION
    assert lib.attn_fwd_args_size() == ctypes.sizeof(_abi.FwdArgs)
    assert lib.attn_bwd_args_size() == ctypes.sizeof(_abi.BwdArgs)
    assert lib.attn_merge_args_size() == ctypes.sizeof(_abi.MergeArgs)


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert len(names) >= 15
    lib = _abi.load()
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/attn.h but not exported"
    assert set(names) == set(_abi.EXPORTS)


def test_strerror_texts():
    lib = _abi.load()
    for code in (0, -1, -2, -3, -4, -5):
        assert lib.attn_strerror(code)
    assert lib.attn_strerror(-99) == b"unknown status"


FAKE = 1 << 20  # 256-byte aligned host integer; never dereferenced by these calls


def _fwd_args(**kw):
    a = _abi.FwdArgs()
    H, D, N = kw.get("H", 2), kw.get("D", 64), kw.get("N", 256)
    es = 4 if kw.get("dtype", _abi.ATTN_F16) == _abi.ATTN_F32 else 2
    for name in ("q", "k", "v", "o"):
        setattr(a, name, _abi.AttnTensor(FAKE, H * D, D))
    a.lse = FAKE
    a.n_q = kw.get("n_q", N)
    a.n_k = kw.get("n_k", N)
    a.H, a.D = H, D
    a.scale = kw.get("scale", D ** -0.5)
    a.relation = kw.get("relation", _abi.ATTN_CAUSAL)
    a.dtype = kw.get("dtype", _abi.ATTN_F16)
    a.o_dtype = kw.get("o_dtype", a.dtype)
    a.n_seq = 1
    a.kernel = kw.get("kernel", _abi.ATTN_KERNEL_AUTO)
    a.num_splits = kw.get("num_splits", 0)
    a.prune_threshold = kw.get("prune", 0.0)
    a.qk_fp8 = kw.get("qk_fp8", 0)
    lib = _abi.load()
    a.workspace = FAKE
    a.workspace_bytes = kw.get("ws", lib.attn_fwd_workspace_bytes(ctypes.byref(a)))
    del es
    return a


@pytest.mark.parametrize("kw,code", [
    ({"D": 96}, _abi.ATTN_EUNSUPPORTED),
    ({"D": 256}, _abi.ATTN_EUNSUPPORTED),
    ({"n_q": 256, "n_k": 128}, _abi.ATTN_EUNSUPPORTED),      # causal needs equal lengths
    ({"relation": 7}, _abi.ATTN_EINVAL),
    ({"dtype": 9}, _abi.ATTN_EINVAL),
    ({"o_dtype": _abi.ATTN_BF16}, _abi.ATTN_EINVAL),         # fp16 in, bf16 out
    ({"ws": 16}, _abi.ATTN_EWORKSPACE),
    ({"num_splits": -1}, _abi.ATTN_EINVAL),
    ({"prune": -0.1}, _abi.ATTN_EINVAL),
    ({"prune": 1.5}, _abi.ATTN_EINVAL),
    ({"prune": float("nan")}, _abi.ATTN_EINVAL),
    ({"prune": 0.5}, _abi.ATTN_EUNSUPPORTED),                  # causal: fails closed
    ({"prune": 0.5, "relation": _abi.ATTN_FULL, "num_splits": 2}, _abi.ATTN_EUNSUPPORTED),
    ({"num_splits": _abi.ATTN_MAX_SPLITS + 1}, _abi.ATTN_EINVAL),
    ({"kernel": 42}, _abi.ATTN_EINVAL),
    ({"dtype": _abi.ATTN_F32, "kernel": _abi.ATTN_KERNEL_TC, "D": 128}, _abi.ATTN_EUNSUPPORTED),
    ({"qk_fp8": 2}, _abi.ATTN_EINVAL),
    ({"qk_fp8": 1}, _abi.ATTN_EUNSUPPORTED),                   # fp8 Q / K: D = 128 only
    ({"qk_fp8": 1, "D": 128, "dtype": _abi.ATTN_F32}, _abi.ATTN_EUNSUPPORTED),  # v 16-bit
    ({"qk_fp8": 1, "D": 128, "kernel": _abi.ATTN_KERNEL_SIMT}, _abi.ATTN_EUNSUPPORTED),
    ({"scale": float("nan")}, _abi.ATTN_EINVAL),
    ({"scale": float("inf")}, _abi.ATTN_EINVAL),
    ({"scale": float("-inf")}, _abi.ATTN_EINVAL),
    ({"qk_fp8": 1, "D": 128, "scale": 0.0}, _abi.ATTN_EUNSUPPORTED),  # fp8 Q / K: positive scales
])
def test_forward_argument_validation(kw, code):
    # every case is rejected on the host, before any launch: these arguments
    # hold fake pointers, so a launch on a machine with a GPU would fault
    lib = _abi.load()
    a = _fwd_args(**kw)
    before = lib.attn_launch_count()
    assert lib.attn_fwd(ctypes.byref(a), None) == code
    assert lib.attn_launch_count() == before


def test_forward_rejects_misaligned_strides_and_null_pointers():
    lib = _abi.load()
    a = _fwd_args()
    a.q = _abi.AttnTensor(FAKE, 2 * 64 + 1, 64)
    assert lib.attn_fwd(ctypes.byref(a), None) == _abi.ATTN_EINVAL
    a = _fwd_args()
    a.k = _abi.AttnTensor(FAKE + 2, 128, 64)
    assert lib.attn_fwd(ctypes.byref(a), None) == _abi.ATTN_EINVAL
    a = _fwd_args()
    a.v = _abi.AttnTensor(None, 128, 64)
    assert lib.attn_fwd(ctypes.byref(a), None) == _abi.ATTN_EINVAL
    assert lib.attn_fwd(None, None) == _abi.ATTN_EINVAL


def test_cu_seqlens_must_come_in_pairs():
    lib = _abi.load()
    a = _fwd_args()
    a.cu_seqlens_q = FAKE
    assert lib.attn_fwd(ctypes.byref(a), None) == _abi.ATTN_EINVAL
    a = _fwd_args()
    a.n_seq = 3  # several sequences need offsets
    assert lib.attn_fwd(ctypes.byref(a), None) == _abi.ATTN_EINVAL


def test_workspace_sizes_grow_with_sequences_and_rows():
    lib = _abi.load()
    a = _fwd_args()
    small = lib.attn_fwd_workspace_bytes(ctypes.byref(a))
    a.n_seq = 10000
    assert lib.attn_fwd_workspace_bytes(ctypes.byref(a)) > small
    b = _abi.BwdArgs()
    b.n_seq, b.H, b.n_q = 1, 32, 32768
    need = lib.attn_bwd_workspace_bytes(ctypes.byref(b))
    assert need >= 32 * 32768 * 4  # Dr is (H, n_q) f32
    assert need % 256 == 0


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    q = torch.zeros(8, 1, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        attn.fwd(q, q, q)


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("splits", [1, 2, 7, 64])
def test_explicit_splits_are_reported_and_size_the_workspace(splits):
    """num_splits > 1 adds the f32 partial outputs and partial lse of every
    split to the forward workspace; attn_fwd_num_splits reports the choice."""
    lib = _abi.load()
    H, D, N = 3, 128, 1000
    base = lib.attn_fwd_workspace_bytes(ctypes.byref(_fwd_args(H=H, D=D, N=N, num_splits=1)))
    a = _fwd_args(H=H, D=D, N=N, num_splits=splits)
    assert lib.attn_fwd_num_splits(ctypes.byref(a)) == splits
    extra = 0 if splits == 1 else (_align256(splits * N * H * D * 4) + _align256(splits * H * N * 4))
    assert lib.attn_fwd_workspace_bytes(ctypes.byref(a)) == base + extra


def test_num_splits_query_rejects_what_the_forward_rejects():
    lib = _abi.load()
    assert lib.attn_fwd_num_splits(ctypes.byref(_fwd_args(D=96))) == _abi.ATTN_EUNSUPPORTED
    assert lib.attn_fwd_num_splits(ctypes.byref(_fwd_args(num_splits=-3))) == _abi.ATTN_EINVAL
    assert lib.attn_fwd_num_splits(None) == _abi.ATTN_EINVAL
    # the automatic choice is a valid split count
    assert 1 <= lib.attn_fwd_num_splits(ctypes.byref(_fwd_args())) <= _abi.ATTN_MAX_SPLITS


def _merge_args(**kw):
    a = _abi.MergeArgs()
    H, D, n = kw.get("H", 2), kw.get("D", 64), kw.get("n_q", 16)
    a.o_parts = kw.get("o_parts", FAKE)
    a.lse_parts = kw.get("lse_parts", FAKE)
    a.o = _abi.AttnTensor(kw.get("o", FAKE), H * D, D)
    a.lse = FAKE
    a.n_parts, a.n_q, a.H, a.D = kw.get("n_parts", 4), n, H, D
    a.o_dtype = kw.get("o_dtype", _abi.ATTN_F32)
    return a


@pytest.mark.parametrize("kw", [
    {"n_parts": 0}, {"n_parts": _abi.ATTN_MAX_SPLITS + 1}, {"D": 6}, {"D": 260}, {"H": 0},
    {"n_q": -1}, {"o_dtype": 5}, {"o_parts": None}, {"o_parts": FAKE + 4}, {"lse_parts": None},
    {"lse_parts": FAKE + 2}, {"o": None}, {"o": FAKE + 8},
])
def test_merge_argument_validation(kw):
    lib = _abi.load()
    assert lib.attn_merge(ctypes.byref(_merge_args(**kw)), None) == _abi.ATTN_EINVAL
    assert lib.attn_merge(None, None) == _abi.ATTN_EINVAL


def test_merge_of_no_rows_launches_nothing():
    lib = _abi.load()
    before = lib.attn_launch_count()
    assert lib.attn_merge(ctypes.byref(_merge_args(n_q=0)), None) == _abi.ATTN_OK
    assert lib.attn_launch_count() == before


def test_pruning_fails_closed_on_varlen_and_backward():
    lib = _abi.load()
    a = _fwd_args(relation=_abi.ATTN_FULL, prune=0.5)
    a.cu_seqlens_q = a.cu_seqlens_k = FAKE
    assert lib.attn_fwd(ctypes.byref(a), None) == _abi.ATTN_EUNSUPPORTED
    # a pruned forward never runs split: the query reports one split
    a = _fwd_args(relation=_abi.ATTN_FULL, prune=0.5)
    assert lib.attn_fwd_num_splits(ctypes.byref(a)) == 1
    b = _abi.BwdArgs()
    for name in ("q", "k", "v", "o", "dout", "dq", "dk", "dv"):
        setattr(b, name, _abi.AttnTensor(FAKE, 128, 64))
    b.lse = FAKE
    b.n_q = b.n_k = 256
    b.H, b.D, b.scale, b.n_seq = 2, 64, 0.125, 1
    b.workspace = FAKE
    b.workspace_bytes = lib.attn_bwd_workspace_bytes(ctypes.byref(b))
    b.prune_threshold = 0.5
    for fn in (lib.attn_bwd, lib.attn_bwd_preprocess, lib.attn_bwd_dkdv, lib.attn_bwd_dq):
        assert fn(ctypes.byref(b), None) == _abi.ATTN_EUNSUPPORTED


def _csr_args(**kw):
    a = _abi.CsrArgs()
    H, D = kw.get("H", 2), kw.get("D", 64)
    a.row_ptr = kw.get("row_ptr", FAKE)
    a.col_idx = kw.get("col", FAKE)
    a.n_edges = kw.get("n_edges", 100)
    a.n_dst, a.n_src, a.H, a.D = kw.get("n_dst", 10), kw.get("n_src", 20), H, D
    a.edge_scores = kw.get("scores", FAKE)
    for name in ("q", "k", "v", "o"):
        setattr(a, name, _abi.AttnTensor(kw.get(name, FAKE), H * D, D))
    a.lse = FAKE
    a.scale = kw.get("scale", 0.125)
    a.dtype = kw.get("dtype", _abi.ATTN_BF16)
    a.o_dtype = kw.get("o_dtype", a.dtype)
    a.row_order = kw.get("row_order", None)
    return a


@pytest.mark.parametrize("kw", [
    {"row_order": FAKE + 2},
    {"D": 6}, {"D": 260}, {"D": 0}, {"H": 0}, {"n_dst": -1}, {"n_src": -1}, {"n_edges": -5},
    {"dtype": 7}, {"o_dtype": _abi.ATTN_F16}, {"row_ptr": None}, {"row_ptr": FAKE + 4},
    {"col": None}, {"col": FAKE + 2}, {"scores": FAKE + 1}, {"v": None}, {"o": FAKE + 8},
    {"scores": None, "q": None}, {"scores": None, "k": None},
    {"scores": None, "scale": float("inf")},
])
def test_csr_argument_validation(kw):
    lib = _abi.load()
    assert lib.attn_csr_fwd(ctypes.byref(_csr_args(**kw)), None) == _abi.ATTN_EINVAL
    assert lib.attn_csr_fwd(None, None) == _abi.ATTN_EINVAL


def test_csr_without_rows_launches_nothing():
    lib = _abi.load()
    before = lib.attn_launch_count()
    assert lib.attn_csr_fwd(ctypes.byref(_csr_args(n_dst=0)), None) == _abi.ATTN_OK
    assert lib.attn_launch_count() == before


def test_workspace_size_does_not_depend_on_the_pointers():
    """A caller may size the workspace before its tensors exist: the size
    depends on sizes, dtypes, relation and splits only."""
    lib = _abi.load()
    for splits in (0, 1, 5):
        a = _fwd_args(H=3, D=128, N=1000, num_splits=splits, relation=_abi.ATTN_FULL)
        with_ptrs = lib.attn_fwd_workspace_bytes(ctypes.byref(a))
        for name in ("q", "k", "v", "o"):
            setattr(a, name, _abi.AttnTensor(None, 0, 0))
        a.lse = None
        assert lib.attn_fwd_workspace_bytes(ctypes.byref(a)) == with_ptrs


@pytest.mark.parametrize("N,H,D,rel,n_seq,dt", [
    (256, 2, 64, _abi.ATTN_CAUSAL, 1, _abi.ATTN_F16),
    (1024, 4, 64, _abi.ATTN_FULL, 1, _abi.ATTN_F16),
    (1178, 4, 128, _abi.ATTN_CAUSAL, 5, _abi.ATTN_BF16),
    (8192, 1, 64, _abi.ATTN_FULL, 1, _abi.ATTN_F32),
])
def test_simple_form_workspace_matches_the_struct_form(N, H, D, rel, n_seq, dt):
    """attn_fwd_simple_workspace_bytes sizes exactly what attn_fwd needs for
    the flat form's arguments (contiguous (N, H, D), AUTO kernel and splits)."""
    lib = _abi.load()
    a = _fwd_args(H=H, D=D, N=N, relation=rel, dtype=dt, num_splits=0)
    if n_seq > 1:
        a.n_seq = n_seq
        a.cu_seqlens_q = a.cu_seqlens_k = FAKE
    want = lib.attn_fwd_workspace_bytes(ctypes.byref(a))
    got = lib.attn_fwd_simple_workspace_bytes(N, H, D, rel, n_seq, dt)
    assert got == want and got > 0 and got % 256 == 0
    assert lib.attn_fwd_simple_workspace_bytes(N, H, D, rel, 0, dt) == 0


def test_simple_form_rejects_a_short_workspace_before_launch():
    lib = _abi.load()
    need = lib.attn_fwd_simple_workspace_bytes(256, 2, 64, _abi.ATTN_CAUSAL, 1, _abi.ATTN_F16)
    before = lib.attn_launch_count()
    rc = lib.attn_fwd_simple(FAKE, FAKE, FAKE, FAKE, FAKE, 256, 2, 64, 0.125, _abi.ATTN_CAUSAL,
                             None, 1, _abi.ATTN_F16, FAKE, need - 256, None)
    assert rc == _abi.ATTN_EWORKSPACE
    assert lib.attn_launch_count() == before


def test_library_source_allocates_no_device_memory():
    """Every entry point works in caller-owned memory (workspace, or the fixed
    array of the allocation-free forward): no allocation or free call appears
    in the library's sources."""
    csrc = os.path.join(ROOT, "online_softmax_attention_gb300", "csrc")
    banned = re.compile(r"\b(cudaMalloc\w*|cudaFree\w*|cuMemAlloc\w*|cuMemFree\w*|"
                        r"cudaHostAlloc|cudaMallocHost|cuMemCreate|cuMemMap)\s*\(")
    seen = []
    for name in sorted(os.listdir(csrc)):
        with open(os.path.join(csrc, name)) as f:
            for i, line in enumerate(f, 1):
                if banned.search(line.split("//")[0]):
                    seen.append(f"{name}:{i}: {line.strip()}")
    assert not seen, "allocation calls in the library: " + "; ".join(seen)
