"""f32 inputs on the tensor cores (D = 64): every input value split into bf16
parts (two for q and k, three for v), three bf16 products for the scores and
six for the values, f32 accumulation.  Compared with the f64 oracle at the f32
bound (max |err| <= 1e-5 on O, 1e-3 on lse) on the cases where the split
matters most: attention concentrated on one key (O is then one row of v, so
the representation error of v is not averaged away), large input magnitudes,
negative and zero scales, long key ranges; and against the CUDA-core f32
kernel."""
import numpy as np
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(q, k, v, **kw):
    o, lse = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), kernel="tc", **kw)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return o, lse


def test_one_dominant_key_per_query():
    """q_i = 6 k_{pi(i)}: each query's score on its own key exceeds the others
    by tens (natural log units), so O_i is close to the one row v_{pi(i)}."""
    g = torch.Generator().manual_seed(901)
    N, H, D = 300, 2, 64
    k = torch.randn((N, H, D), generator=g)
    v = torch.randn((N, H, D), generator=g) * 3.0
    perm = torch.randperm(N, generator=g)
    q = 6.0 * k[perm]
    o, lse = _run(q, k, v, causal=False)
    o_ref, lse_ref = oracle.fwd(q, k, v, causal=False)
    check_o(o, o_ref, torch.float32, o.dtype)
    check_lse(lse, lse_ref)
    # the case is what it claims: nearly all weight on one key
    assert np.abs(o_ref - v[perm].double().numpy()).max() < 1e-3


@pytest.mark.parametrize("gain", [0.01, 3.0])
def test_input_magnitudes(gain):
    """Inputs scaled by `gain` (scores by gain^2).  Much larger scores are
    outside what f32 arithmetic can hold to 1e-5 at all: the rounding of a
    score of magnitude ~100 alone moves O by about that much."""
    x = attn_inputs.make(dtype="f32", H=3, D=64, seed=902, n_q=400)
    q, k, v = (x[n] * gain for n in ("q", "k", "v"))
    o, lse = _run(q, k, v, causal=True)
    o_ref, lse_ref = oracle.fwd(q, k, v, causal=True)
    # O scales with v: compare relative to the gain
    check_o(o / gain, o_ref / gain, torch.float32, o.dtype)
    check_lse(lse, lse_ref)
    # no less accurate than the CUDA-core f32 kernel on the same inputs
    o_simt, _ = attn.fwd(q.to(DEV), k.to(DEV), v.to(DEV), causal=True, kernel="simt")
    e_tc = float(np.abs(o.double().cpu().numpy() - o_ref).max())
    e_simt = float(np.abs(o_simt.double().cpu().numpy() - o_ref).max())
    assert e_tc <= 2.0 * e_simt + 1e-6 * gain, (e_tc, e_simt)


@pytest.mark.parametrize("scale", [-0.2, 0.0, 0.5])
def test_scales(scale):
    x = attn_inputs.make(dtype="f32", H=2, D=64, seed=903, lengths=[300, 1, 129])
    o, lse = _run(x["q"], x["k"], x["v"], causal=True, scale=scale, cu_seqlens_q=x["cu_seqlens_q"])
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=True, scale=scale,
                                cu_seqlens_q=x["cu_seqlens_q"])
    check_o(o, o_ref, torch.float32, o.dtype)
    check_lse(lse, lse_ref)


def test_long_key_range_unsplit():
    """8192 keys in one scan (no key splits): 64 value partials added in f32."""
    x = attn_inputs.make(dtype="f32", H=1, D=64, seed=904, n_q=256, n_k=8192)
    o, lse = _run(x["q"], x["k"], x["v"], causal=False, num_splits=1)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=False)
    check_o(o, o_ref, torch.float32, o.dtype)
    check_lse(lse, lse_ref)


def test_agrees_with_the_cuda_core_kernel_and_repeats_bitwise():
    x = attn_inputs.make(dtype="f32", H=4, D=64, seed=905, lengths=[1000, 3, 517])
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    kw = dict(causal=True, cu_seqlens_q=x["cu_seqlens_q"])
    o1, l1 = attn.fwd(q, k, v, kernel="tc", **kw)
    o2, l2 = attn.fwd(q, k, v, kernel="simt", **kw)
    o3, l3 = attn.fwd(q, k, v, kernel="tc", **kw)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert (o1 - o2).abs().max().item() < 2e-5
    assert (l1 - l2).abs().max().item() < 1e-4
    assert torch.equal(o1, o3) and torch.equal(l1, l3)
