"""Element offsets past 2^31 (byte offsets past 2^32): every tensor is a
(tokens, 2, D) view whose second head starts 2^31 elements after its first,
all views of one call packed into one device buffer.  Every kernel's address
arithmetic on strided tensors must then be 64-bit, and a stray write lands in
a neighbouring view, which the tests re-read.  Results are compared element
by element with the oracle on the logical tensors."""
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu

DEV = "cuda"
FAR = 2 ** 31  # elements between head 0 and head 1 of every view


def _far_views(dtype, D, counts):
    """One buffer of FAR + sum(counts) * D elements; view i is (counts[i], 2, D)
    with head 0 at the packed offset and head 1 FAR elements further on."""
    total = sum(counts) * D
    assert total <= FAR
    buf = torch.empty(FAR + total, dtype=dtype, device=DEV)
    views, off = [], 0
    for n in counts:
        views.append(buf.as_strided((n, 2, D), (D, FAR, 1), off))
        off += n * D
    return buf, views


@pytest.fixture(autouse=True)
def _return_buffers():
    """Each test holds 4-8 GiB; give it back to the device afterwards."""
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# kernel family, dtype, D, dq mode
CASES = [("tc", "bf16", 128, "auto"), ("tc", "fp16", 64, "auto"), ("tc", "bf16", 128, "fused"),
         ("simt", "f32", 64, "auto"), ("simt", "bf16", 128, "auto")]


@pytest.mark.parametrize("kernel,dtype,D,dq_mode", CASES)
def test_forward_and_backward(kernel, dtype, D, dq_mode):
    x = attn_inputs.make(dtype=dtype, H=2, D=D, seed=820 + D, lengths=[300, 1, 257], backward=True)
    tdt = attn_inputs.DTYPES[dtype]
    T = x["q"].shape[0]
    buf, (q, k, v, dO, o, dq, dk, dv) = _far_views(tdt, D, [T] * 8)
    names = ("q", "k", "v", "dO")
    for view, n in zip((q, k, v, dO), names):
        view.copy_(x[n].to(DEV))
    cu = x["cu_seqlens_q"]
    _, lse = attn.FwdCall(q, k, v, causal=True, cu_seqlens_q=cu, kernel=kernel, out=o).run()
    attn.BwdCall(q, k, v, o, lse, dO, causal=True, cu_seqlens_q=cu, kernel=kernel, dq=dq, dk=dk,
                 dv=dv, dq_mode=dq_mode).run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0

    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=True, cu_seqlens_q=cu)
    check_o(o, o_ref, tdt, o.dtype)
    check_lse(lse, lse_ref)
    ref = oracle.bwd(x["q"], x["k"], x["v"], x["dO"], causal=True, cu_seqlens_q=cu)
    for g, r, n in zip((dq, dk, dv), ref, ("dq", "dk", "dv")):
        check_grad(g, r, n)
    for view, n in zip((q, k, v, dO), names):
        assert torch.equal(view.cpu(), x[n]), f"{n} was written to"


@pytest.mark.parametrize("kernel,dtype,D", [("tc", "bf16", 128), ("simt", "f32", 64), ("tc", "f32", 64)])
def test_split_forward_and_merge(kernel, dtype, D):
    """Key splits write f32 partials to the workspace; the merge writes O
    through the far view."""
    x = attn_inputs.make(dtype=dtype, H=2, D=D, seed=830 + D, lengths=[200, 37], lengths_k=[1000, 300])
    tdt = attn_inputs.DTYPES[dtype]
    Tq, Tk = x["q"].shape[0], x["k"].shape[0]
    buf, (q, k, v, o) = _far_views(tdt, D, [Tq, Tk, Tk, Tq])
    for view, n in zip((q, k, v), ("q", "k", "v")):
        view.copy_(x[n].to(DEV))
    call = attn.FwdCall(q, k, v, causal=False, cu_seqlens_q=x["cu_seqlens_q"],
                        cu_seqlens_k=x["cu_seqlens_k"], kernel=kernel, num_splits=4, out=o)
    _, lse = call.run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert call.num_splits() == 4
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=False, cu_seqlens_q=x["cu_seqlens_q"],
                                cu_seqlens_k=x["cu_seqlens_k"])
    check_o(o, o_ref, tdt, o.dtype)
    check_lse(lse, lse_ref)


def test_fp8_queries_and_keys():
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=840, lengths=[300, 257], qk_fp8=True)
    T = x["q"].shape[0]
    buf8, (q, k) = _far_views(torch.float8_e4m3fn, 128, [T, T])
    buf16, (v, o) = _far_views(torch.bfloat16, 128, [T, T])
    q.copy_(x["q"].to(DEV))
    k.copy_(x["k"].to(DEV))
    v.copy_(x["v"].to(DEV))
    _, lse = attn.FwdCall(q, k, v, causal=True, cu_seqlens_q=x["cu_seqlens_q"], out=o).run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=True, cu_seqlens_q=x["cu_seqlens_q"])
    check_o(o, o_ref, torch.bfloat16, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("dot", [False, True])
def test_csr_relation(dot):
    """The general CSR kernel (strided views are not packed rows)."""
    _, rp, col = attn_inputs.radius_graph(1500, 0.12, seed=850)
    x = attn_inputs.make_csr(row_ptr=rp, col=col, n_src=1500, H=2, D=64, dtype="bf16", seed=851,
                             field_scores=not dot, score_std=2.0)
    buf, (q, k, v, o) = _far_views(torch.bfloat16, 64, [1500] * 4)
    v.copy_(x["v"].to(DEV))
    kw = {}
    if dot:
        q.copy_(x["q"].to(DEV))
        k.copy_(x["k"].to(DEV))
        kw = {"q": q, "k": k}
    else:
        kw = {"scores": x["scores"].to(DEV)}
    _, lse = attn.CsrCall(x["row_ptr"].to(DEV), x["col"].to(DEV), v, out=o, **kw).run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    if dot:
        o_ref, lse_ref = oracle.csr_fwd(x["row_ptr"], x["col"], x["v"], q=x["q"], k=x["k"])
    else:
        o_ref, lse_ref = oracle.csr_fwd(x["row_ptr"], x["col"], x["v"], scores=x["scores"])
    check_o(o, o_ref, torch.bfloat16, o.dtype)
    check_lse(lse, lse_ref)
