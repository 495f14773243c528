"""The flat entry point attn_fwd_simple (contiguous (N, H, D) self-attention,
the signature attn_fwd(q, k, v, out, lse, N, H, D, scale, relation,
cu_seqlens)) called through the C ABI and compared with the f64 oracle
element by element, its workspace sized by attn_fwd_simple_workspace_bytes.

Cases: the causal N=256 workload (TIGA-lang attention examples page, section
"因果稠密关系"), the full N=1024 one (section "全量注意力，无掩码"; the
library splits its keys, so the workspace holds split partials), and a varlen
causal batch on the pages' lengths [384, 1, 96, 640, 57] (section
"用图组合表达 varlen 因果注意力").  The flat form stores O in the input
dtype; for bf16 that storage alone is checked exactly: the bf16 O equals the
f32-stored O of the same call rounded to nearest even, and the f32 O meets
the 2e-3 bar against the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from online_softmax_attention_gb300 import _abi
from parity_util import check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda"
_DT = {torch.float16: _abi.ATTN_F16, torch.bfloat16: _abi.ATTN_BF16, torch.float32: _abi.ATTN_F32}


def _simple(x, causal, scale=None):
    q, k, v = (x[n].contiguous().to(DEV) for n in ("q", "k", "v"))
    N, H, D = q.shape
    rel = _abi.ATTN_CAUSAL if causal else _abi.ATTN_FULL
    cu = x["cu_seqlens_q"]
    n_seq = 1 if cu is None else len(cu) - 1
    cu_d = None if cu is None else cu.to(DEV)
    lib = _abi.load()
    need = lib.attn_fwd_simple_workspace_bytes(N, H, D, rel, n_seq, _DT[q.dtype])
    assert need > 0
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((H, N), float("nan"), dtype=torch.float32, device=DEV)
    s = torch.cuda.current_stream()
    rc = lib.attn_fwd_simple(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             N, H, D, D ** -0.5 if scale is None else scale, rel,
                             None if cu_d is None else cu_d.data_ptr(), n_seq, _DT[q.dtype],
                             ws.data_ptr(), need, ctypes.c_void_p(s.cuda_stream))
    assert rc == _abi.ATTN_OK, attn.strerror(rc)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return o, lse


@pytest.mark.parametrize("name", ["causal_fp16_n256", "full_fp16_n1024"])
def test_simple_form_on_the_small_workloads(name):
    w = attn_inputs.WORKLOADS[name]
    x = attn_inputs.make_workload(w)
    o, lse = _simple(x, w.causal)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=w.causal)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("dtype,D", [("fp16", 64), ("bf16", 128)])
def test_simple_form_varlen_pages_lengths(dtype, D):
    x = attn_inputs.make(dtype=dtype, H=4, D=D, seed=41, lengths=[384, 1, 96, 640, 57])
    o, lse = _simple(x, True)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=True,
                                cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)
    if dtype == "bf16":
        # the bf16-stored O is exactly the f32-stored O rounded to nearest even
        q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
        o32, lse32 = attn.fwd(q, k, v, causal=True, cu_seqlens_q=x["cu_seqlens_q"],
                              cu_seqlens_k=x["cu_seqlens_k"], out_dtype=torch.float32)
        torch.cuda.synchronize()
        check_o(o32, o_ref, x["q"].dtype, o32.dtype)
        assert torch.equal(o, o32.to(torch.bfloat16))
        assert torch.equal(lse, lse32)


def test_simple_form_single_sequence_ragged_tail_f32():
    x = attn_inputs.make(dtype="f32", H=2, D=64, seed=42, n_q=300)
    o, lse = _simple(x, False)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=False)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("name", ["varlen_causal_bf16"])
def test_bf16_stored_output_is_the_rounded_f32_output(name):
    """At the varlen workload's full size: O stored in bf16 equals O stored in
    f32 rounded to nearest even, bit for bit (the f32 O is the one compared
    with the oracle at 2e-3 in the workload tests)."""
    w = attn_inputs.WORKLOADS[name]
    x = attn_inputs.make_workload(w)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    kw = dict(causal=w.causal, cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])
    o16, lse16 = attn.fwd(q, k, v, **kw)
    o32, lse32 = attn.fwd(q, k, v, out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert o16.dtype == torch.bfloat16
    assert torch.equal(o16, o32.to(torch.bfloat16))
    assert torch.equal(lse16, lse32)
    assert bool(np.isfinite(lse32.cpu().numpy()).all())
