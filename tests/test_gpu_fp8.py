"""fp8 (e4m3) queries and keys on the tensor-core forward (attn.h, qk_fp8),
through the C ABI, against the f64 oracle on the same e4m3 values (which f64
holds exactly), at the same tolerances as the 16-bit path."""
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_lse, check_o

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(x, *, causal, out_dtype=torch.float32, num_splits=0, scale=None, kernel="auto"):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = attn.fwd(q, k, v, causal=causal, scale=scale, cu_seqlens_q=x["cu_seqlens_q"],
                      cu_seqlens_k=x["cu_seqlens_k"], out_dtype=out_dtype, num_splits=num_splits,
                      kernel=kernel)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return o, lse


def _ref(x, *, causal, scale=None):
    return oracle.fwd(x["q"], x["k"], x["v"], causal=causal, scale=scale,
                      cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])


@pytest.mark.parametrize("vdt", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300, 1000])
def test_single_sequence(vdt, causal, N):
    x = attn_inputs.make(dtype=vdt, H=2, D=128, seed=700 + N, n_q=N, qk_fp8=True)
    o, lse = _run(x, causal=causal)
    o_ref, lse_ref = _ref(x, causal=causal)
    check_o(o, o_ref, attn_inputs.DTYPES[vdt], o.dtype)
    check_lse(lse, lse_ref)


def test_varlen_pages_lengths():
    x = attn_inputs.make(dtype="bf16", H=4, D=128, seed=710, lengths=[384, 1, 96, 640, 57], qk_fp8=True)
    o, lse = _run(x, causal=True)
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, torch.bfloat16, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("splits", [1, 4])
def test_cross_attention_and_key_splits(splits):
    x = attn_inputs.make(dtype="fp16", H=2, D=128, seed=711, lengths=[100, 3, 257],
                         lengths_k=[31, 300, 1000], qk_fp8=True)
    o, lse = _run(x, causal=False, num_splits=splits, scale=0.07)
    o_ref, lse_ref = _ref(x, causal=False, scale=0.07)
    check_o(o, o_ref, torch.float16, o.dtype)
    check_lse(lse, lse_ref)


def test_output_in_the_value_dtype():
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=712, n_q=700, qk_fp8=True)
    o, lse = _run(x, causal=True, out_dtype=torch.bfloat16)
    assert o.dtype == torch.bfloat16
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, torch.bfloat16, torch.bfloat16)
    check_lse(lse, lse_ref)


def test_same_scores_as_the_16_bit_path():
    """e4m3 values are exact in bf16, and both MMAs accumulate exact products
    in f32: the fp8 and bf16 score paths agree to f32 summation order."""
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=713, n_q=600, qk_fp8=True)
    o8, l8 = _run(x, causal=True)
    y = dict(x)
    y["q"], y["k"] = x["q"].to(torch.bfloat16), x["k"].to(torch.bfloat16)
    o16, l16 = _run(y, causal=True)
    assert float((o8 - o16).abs().max()) <= 1e-5
    assert float((l8 - l16).abs().max()) <= 1e-5


def test_unsupported_combinations_fail_closed():
    x = attn_inputs.make(dtype="bf16", H=2, D=64, seed=714, n_q=64, qk_fp8=True)
    with pytest.raises(attn.AttnError):  # D = 64
        _run(x, causal=False)
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=715, n_q=64, qk_fp8=True)
    with pytest.raises(attn.AttnError):  # no CUDA-core fp8 path
        _run(x, causal=False, kernel="simt")
    with pytest.raises(attn.AttnError):  # negative scale
        _run(x, causal=False, scale=-0.1)


@pytest.mark.parametrize("seed,rho", [(501, 0.5), (502, 0.1)])
def test_tile_pruning(seed, rho):
    """The approximate tile-pruned forward on fp8 queries and keys: decisions
    (checked decisive on the oracle, margin > 0.01 in log units) and results
    equal the oracle's pruned forward with the kernel's 128 x 128 tiles."""
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=seed, lengths=[1000], lengths_k=[1500],
                         key_gain=(128, 0.2, 3.0), qk_fp8=True)
    o_ref, lse_ref, n_ref, margin = oracle.fwd_pruned(x["q"], x["k"], x["v"], rho=rho,
                                                      block_q=128, block_k=128)
    assert margin > 0.01 and n_ref > 0
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    call = attn.FwdCall(q, k, v, causal=False, prune_threshold=rho, out_dtype=torch.float32)
    o, lse = call.run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert call.pruned_count() == n_ref
    check_o(o, o_ref, torch.bfloat16, o.dtype)
    check_lse(lse, lse_ref)
