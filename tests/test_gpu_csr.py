"""Attention over a general CSR relation (TIGA-lang attention examples page:
varlen section's explicit CSR relation, GAT section's softmax over incoming
edges), CUDA path through the C ABI vs the f64 oracle."""
import numpy as np
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_lse, check_o, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _gpu(x, *, dot, out_dtype=None, scale=None):
    rp, col, v = x["row_ptr"].to(DEV), x["col"].to(DEV), x["v"].to(DEV)
    if dot:
        o, lse = attn.csr_fwd(rp, col, v, q=x["q"].to(DEV), k=x["k"].to(DEV), scale=scale,
                              out_dtype=out_dtype)
    else:
        o, lse = attn.csr_fwd(rp, col, v, scores=x["scores"].to(DEV), out_dtype=out_dtype)
    torch.cuda.synchronize()
    return o, lse


def _ref(x, *, dot, scale=None):
    if dot:
        return oracle.csr_fwd(x["row_ptr"], x["col"], x["v"], q=x["q"], k=x["k"], scale=scale)
    return oracle.csr_fwd(x["row_ptr"], x["col"], x["v"], scores=x["scores"])


def _check(o, lse, o_ref, lse_ref, dtype, o_dtype):
    if dtype == torch.float32:
        # field scores arrive in f32 and are used as given; f32 arithmetic throughout
        assert float(np.abs(f64(o) - o_ref).max()) <= 1e-5
    else:
        check_o(o, o_ref, dtype, o_dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("dtype", ["f32", "bf16", "fp16"])
@pytest.mark.parametrize("D", [8, 64, 128, 200])
@pytest.mark.parametrize("dot", [False, True])
def test_radius_graph(dtype, D, dot):
    """The GAT example's graph family: points in the unit cube, an edge for
    every pair closer than the cutoff (2000 points, average degree ~9)."""
    _, rp, col = attn_inputs.radius_graph(2000, 0.1, seed=600 + D)
    x = attn_inputs.make_csr(row_ptr=rp, col=col, n_src=2000, H=3, D=D, dtype=dtype, seed=601,
                             field_scores=not dot, score_std=2.0)
    out = torch.float32 if dtype == "bf16" else None
    o, lse = _gpu(x, dot=dot, out_dtype=out)
    assert attn.device_status() == 0
    o_ref, lse_ref = _ref(x, dot=dot)
    _check(o, lse, o_ref, lse_ref, attn_inputs.DTYPES[dtype], o.dtype)


@pytest.mark.parametrize("causal,lengths_q,lengths_k", [
    (True, [384, 1, 96, 640, 57], None),   # the varlen example's relation, as CSR
    (False, [100, 3, 257], [31, 300, 128]),
    (True, [0, 5, 0, 70], None),
])
def test_segment_relations_as_csr_match_dense_attention(causal, lengths_q, lengths_k):
    """Rows with hundreds of edges (many blocks of 32), empty rows, and the
    same result as the cu_seqlens forward's oracle."""
    lk = lengths_k or lengths_q
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=602, lengths=lengths_q, lengths_k=lk)
    rp, col = attn_inputs.csr_of_segments(lengths_q, lk, causal)
    o, lse = attn.csr_fwd(rp.to(DEV), col.to(DEV), x["v"].to(DEV), q=x["q"].to(DEV),
                          k=x["k"].to(DEV))
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=causal,
                                cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])
    check_o(o, o_ref, torch.float16, o.dtype)
    check_lse(lse, lse_ref)


def test_repeated_edges_empty_rows_and_large_scores():
    rng = np.random.default_rng(603)
    deg = rng.integers(0, 80, 300)
    deg[::7] = 0
    rp = torch.tensor(np.concatenate([[0], np.cumsum(deg)]), dtype=torch.int64)
    col = torch.tensor(rng.integers(0, 40, int(deg.sum())), dtype=torch.int32)  # many repeats
    x = attn_inputs.make_csr(row_ptr=rp, col=col, n_src=40, H=2, D=128, dtype="bf16", seed=604,
                             field_scores=True, score_std=30.0)
    o, lse = _gpu(x, dot=False, out_dtype=torch.float32)
    assert attn.device_status() == 0
    o_ref, lse_ref = _ref(x, dot=False)
    _check(o, lse, o_ref, lse_ref, torch.bfloat16, o.dtype)
    assert not f64(o)[::7].any() and np.isneginf(f64(lse)[:, ::7]).all()


def test_malformed_relation_is_reported_and_skipped():
    """An out-of-range source and a decreasing offset: the kernel skips them
    (no out-of-bounds read) and reports ATTN_EINVAL; other rows are exact."""
    rp = torch.tensor([0, 3, 5, 4, 8], dtype=torch.int64)   # row 2 decreases
    col = torch.tensor([0, 1, 2, 1, 99, 0, 1, 2], dtype=torch.int32)  # 99 out of range
    x = attn_inputs.make_csr(row_ptr=rp, col=col, n_src=3, H=1, D=64, dtype="f32", seed=605,
                             field_scores=True)
    o, lse = _gpu(x, dot=False)
    assert attn.device_status() == attn._abi.ATTN_EINVAL
    assert attn.device_status() == 0  # cleared by the read
    good = oracle.csr_fwd([0, 3], col[:3], x["v"], scores=x["scores"][:3])
    assert float(np.abs(f64(o)[0] - good[0][0]).max()) <= 1e-5
    assert not f64(o)[2].any() and np.isneginf(f64(lse)[0, 2])
    row1 = oracle.csr_fwd([0, 1], col[3:4], x["v"], scores=x["scores"][3:4])  # edge 99 skipped
    assert float(np.abs(f64(o)[1] - row1[0][0]).max()) <= 1e-5


@pytest.mark.parametrize("dot", [False, True])
def test_strided_views_match_packed_rows(dot):
    """Tensors whose heads are not back to back in a row ((H, N, D) storage
    viewed as (N, H, D)) take the general kernel; packed rows take the
    row-centric one.  Both equal the oracle on the same relation."""
    _, rp, col = attn_inputs.radius_graph(1500, 0.1, seed=606)
    x = attn_inputs.make_csr(row_ptr=rp, col=col, n_src=1500, H=4, D=64, dtype="bf16", seed=607,
                             field_scores=not dot, score_std=2.0)
    o_ref, lse_ref = _ref(x, dot=dot)
    packed = _gpu(x, dot=dot, out_dtype=torch.float32)
    strided = dict(x)
    for name in ("v", "q", "k"):
        if x.get(name) is not None:
            strided[name] = x[name].permute(1, 0, 2).contiguous().permute(1, 0, 2)
    assert strided["v"].stride(1) != x["v"].shape[2]
    o_s, lse_s = _gpu(strided, dot=dot, out_dtype=torch.float32)
    assert attn.device_status() == 0
    for o, lse in (packed, (o_s, lse_s)):
        _check(o, lse, o_ref, lse_ref, torch.bfloat16, o.dtype)


@pytest.mark.parametrize("dot", [False, True])
@pytest.mark.parametrize("layout", ["packed", "strided"])
def test_row_order_leaves_results_unchanged(dot, layout):
    """Rows taken along a Z-order curve through the points, or in a random
    order: the same outputs, bit for bit, as index order, and the oracle's."""
    pos, rp, col = attn_inputs.radius_graph(3000, 0.08, seed=608)
    x = attn_inputs.make_csr(row_ptr=rp, col=col, n_src=3000, H=4, D=64, dtype="bf16", seed=609,
                             field_scores=not dot, score_std=2.0)
    if layout == "strided":  # the general kernel
        for name in ("v", "q", "k"):
            if x.get(name) is not None:
                x[name] = x[name].permute(1, 0, 2).contiguous().permute(1, 0, 2)
    args = dict(q=x["q"].to(DEV), k=x["k"].to(DEV)) if dot else dict(scores=x["scores"].to(DEV))
    rpd, cold, vd = rp.to(DEV), col.to(DEV), x["v"].to(DEV)
    base = attn.csr_fwd(rpd, cold, vd, out_dtype=torch.float32, **args)
    orders = [attn_inputs.curve_order(pos, 0.08),
              torch.randperm(3000, generator=torch.Generator().manual_seed(610)).to(torch.int32)]
    for order in orders:
        o, lse = attn.csr_fwd(rpd, cold, vd, out_dtype=torch.float32, row_order=order.to(DEV), **args)
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        assert torch.equal(o, base[0]) and torch.equal(lse, base[1])
    o_ref, lse_ref = _ref(x, dot=dot)
    _check(o, lse, o_ref, lse_ref, torch.bfloat16, o.dtype)


def test_row_order_entry_outside_the_rows_is_reported_and_skipped():
    """Entries -1 and n_dst + 93 are skipped (no out-of-bounds access) with
    ATTN_EINVAL; the rows the order names are exact, the two it omits untouched."""
    _, rp, col = attn_inputs.radius_graph(6, 0.9, seed=611)
    x = attn_inputs.make_csr(row_ptr=rp, col=col, n_src=6, H=2, D=64, dtype="f32", seed=612,
                             field_scores=True)
    order = torch.tensor([5, 0, -1, 3, 99, 1], dtype=torch.int32, device=DEV)
    out = torch.full((6, 2, 64), 7.0, device=DEV)
    lse = torch.full((2, 6), 7.0, device=DEV)
    attn.CsrCall(rp.to(DEV), col.to(DEV), x["v"].to(DEV), scores=x["scores"].to(DEV), out=out,
                 lse=lse, row_order=order).run()
    assert attn.device_status() == attn._abi.ATTN_EINVAL
    o_ref, lse_ref = _ref(x, dot=False)
    done = [0, 1, 3, 5]
    assert float(np.abs(f64(out)[done] - o_ref[done]).max()) <= 1e-5
    assert float(np.abs(f64(lse)[:, done] - lse_ref[:, done]).max()) <= 1e-5
    assert (f64(out)[[2, 4]] == 7.0).all() and (f64(lse)[:, [2, 4]] == 7.0).all()
