"""Split-K forward and the partial-result merge, through the C ABI, against the
f64 oracle (split-K of the Vx issue "Chunked-dot Reduce lowering: shorten the
reduction dependency chain", measurement section, C = 8)."""
import numpy as np
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_lse, check_o, f64

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(x, *, causal, kernel, splits, out_dtype=None, num_ctas=0):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    call = attn.FwdCall(q, k, v, causal=causal, cu_seqlens_q=x["cu_seqlens_q"],
                        cu_seqlens_k=x["cu_seqlens_k"], out_dtype=out_dtype, kernel=kernel,
                        num_ctas=num_ctas, num_splits=splits)
    assert call.num_splits() == splits
    o, lse = call.run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return o, lse


def _ref(x, *, causal):
    return oracle.fwd(x["q"], x["k"], x["v"], causal=causal, cu_seqlens_q=x["cu_seqlens_q"],
                      cu_seqlens_k=x["cu_seqlens_k"])


def _out(dtype):
    return torch.float32 if dtype == "bf16" else None


@pytest.mark.parametrize("kernel,dtype", [("simt", "f32"), ("simt", "fp16"), ("tc", "fp16"),
                                          ("tc", "bf16"), ("tc", "f32")])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("splits", [2, 3, 8])
def test_split_forward_single_sequence(kernel, dtype, D, causal, splits):
    """N = 700: 11 SIMT / 6 tensor-core key tiles, split unevenly, ragged tail;
    at 8 splits some chunks of the short causal rows are empty."""
    if kernel == "tc" and dtype == "f32" and D != 64:
        pytest.skip("the tensor-core kernels take f32 inputs at D = 64 only")
    x = attn_inputs.make(dtype=dtype, H=2, D=D, seed=300 + splits, n_q=700)
    o, lse = _run(x, causal=causal, kernel=kernel, splits=splits, out_dtype=_out(dtype))
    o_ref, lse_ref = _ref(x, causal=causal)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel,dtype", [("simt", "f32"), ("tc", "bf16"), ("tc", "f32")])
def test_split_forward_varlen_cross_with_empty_sequences(kernel, dtype):
    x = attn_inputs.make(dtype=dtype, H=3, D=64 if dtype == "f32" else 128, seed=310,
                         lengths=[130, 0, 1, 257, 64], lengths_k=[900, 40, 0, 1, 300])
    o, lse = _run(x, causal=False, kernel=kernel, splits=5, out_dtype=_out(dtype))
    o_ref, lse_ref = _ref(x, causal=False)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel,dtype", [("simt", "fp16"), ("tc", "bf16")])
def test_split_forward_varlen_causal_pages_lengths(kernel, dtype):
    x = attn_inputs.make(dtype=dtype, H=2, D=128, seed=311, lengths=[384, 1, 96, 640, 57])
    o, lse = _run(x, causal=True, kernel=kernel, splits=4, out_dtype=_out(dtype))
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


def test_split_more_chunks_than_key_tiles():
    """64 chunks over 2 key tiles: 62 chunks admit nothing and merge away."""
    x = attn_inputs.make(dtype="fp16", H=1, D=64, seed=312, lengths=[200], lengths_k=[150])
    for kernel in ("simt", "tc"):
        o, lse = _run(x, causal=False, kernel=kernel, splits=64)
        o_ref, lse_ref = _ref(x, causal=False)
        check_o(o, o_ref, x["q"].dtype, o.dtype)
        check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", ["simt", "tc"])
def test_split_forward_is_deterministic_and_grid_independent(kernel):
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=313, lengths=[500, 70])
    runs = [_run(x, causal=True, kernel=kernel, splits=3, out_dtype=torch.float32, num_ctas=n)
            for n in (0, 5, 0)]
    for o, lse in runs[1:]:
        assert torch.equal(o, runs[0][0]) and torch.equal(lse, runs[0][1])


def test_split_bf16_output_storage():
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=314, n_q=600)
    o, lse = _run(x, causal=True, kernel="tc", splits=4, out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


def test_cross_f32_workload_auto_splits():
    """The f32 cross-attention workload (SQ=8192, SK=2048, H=1, D=64): 128 query
    tiles leave most SMs idle, so the library splits the keys."""
    w = attn_inputs.WORKLOADS["cross_f32_8192x2048"]
    x = attn_inputs.make_workload(w)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    call = attn.FwdCall(q, k, v, causal=w.causal)
    assert call.num_splits() > 1
    o, lse = call.run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=w.causal)
    check_o(o, o_ref, torch.float32, o.dtype)
    check_lse(lse, lse_ref)


# --- the public merge entry point ------------------------------------------------

def _partials(C, T, H, D, seed, empty_frac=0.2):
    """Seeded partial results: O_c ~ N(0, 1), lse_c ~ 4 N(0, 1), some -inf."""
    g = torch.Generator().manual_seed(seed)
    op = torch.randn((C, T, H, D), generator=g, dtype=torch.float32)
    lp = 4 * torch.randn((C, H, T), generator=g, dtype=torch.float32)
    drop = torch.rand((C, H, T), generator=g) < empty_frac
    lp[drop] = -float("inf")
    return op, lp


@pytest.mark.parametrize("C", [1, 2, 8, 33, 64])
@pytest.mark.parametrize("D", [64, 128, 4, 200])
def test_merge_matches_oracle(C, D):
    op, lp = _partials(C, 77, 3, D, seed=400 + C + D)
    lp[:, 1, 5] = -float("inf")  # a row with no admitted key at all
    o, lse = attn.merge(op.to(DEV), lp.to(DEV))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge(op, lp)
    assert float(np.abs(f64(o) - o_ref).max()) <= 1e-5
    assert not f64(o)[5, 1].any()
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("out_dtype", [torch.float16, torch.bfloat16])
def test_merge_16_bit_output(out_dtype):
    op, lp = _partials(6, 300, 2, 128, seed=420)
    o, lse = attn.merge(op.to(DEV), lp.to(DEV), out_dtype=out_dtype)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.merge(op, lp)
    check_o(o, o_ref, torch.float16, out_dtype)
    check_lse(lse, lse_ref)


def test_merge_of_oracle_key_chunks_equals_attention_over_all_keys():
    """Merging per-chunk attention (computed by the oracle over disjoint key
    chunks) on the GPU gives attention over all keys."""
    x = attn_inputs.make(dtype="f32", H=2, D=64, seed=421, lengths=[90], lengths_k=[500])
    bounds = [0, 130, 131, 400, 500]
    parts = [oracle.fwd(x["q"], x["k"][a:b], x["v"][a:b], causal=False)
             for a, b in zip(bounds[:-1], bounds[1:])]
    op = torch.from_numpy(np.stack([p[0] for p in parts])).float()
    lp = torch.from_numpy(np.stack([p[1] for p in parts])).float()
    o, lse = attn.merge(op.to(DEV), lp.to(DEV))
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=False)
    assert float(np.abs(f64(o) - o_ref).max()) <= 1e-5
    check_lse(lse, lse_ref)
