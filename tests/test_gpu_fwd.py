"""Forward parity: CUDA path (through the C ABI) vs the f64 oracle, element by
element, on seeded inputs spanning several tiles, ragged tails and edge cases."""
import numpy as np
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_lse, check_o, f64

pytestmark = pytest.mark.gpu

KERNELS = ["auto", "simt", "tc"]
DEV = "cuda"


def _skip_unsupported(kernel, dtype, D=64):
    if kernel == "tc" and dtype in ("f32", torch.float32) and D != 64:
        pytest.skip("the tensor-core kernels take f32 inputs at D = 64 only")


def _run(x, *, causal, kernel, out_dtype=None, scale=None, num_ctas=0):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    cq = x["cu_seqlens_q"]
    ck = x["cu_seqlens_k"]
    o, lse = attn.fwd(q, k, v, causal=causal, scale=scale, cu_seqlens_q=cq, cu_seqlens_k=ck,
                      out_dtype=out_dtype, kernel=kernel, num_ctas=num_ctas)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return o, lse


def _ref(x, *, causal, scale=None):
    return oracle.fwd(x["q"], x["k"], x["v"], causal=causal, scale=scale,
                      cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])


def _out_dtype(dtype):
    # bf16 inputs store O in f32 for the 2e-3 rel-RMS bar; others keep their dtype
    return torch.float32 if dtype == "bf16" else None


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16", "f32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 127, 129, 300])
def test_single_sequence(kernel, dtype, D, causal, N):
    _skip_unsupported(kernel, dtype, D)
    x = attn_inputs.make(dtype=dtype, H=3, D=D, seed=100 + N, n_q=N)
    o, lse = _run(x, causal=causal, kernel=kernel, out_dtype=_out_dtype(dtype))
    o_ref, lse_ref = _ref(x, causal=causal)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype,D", [("fp16", 64), ("bf16", 128), ("f32", 64)])
def test_varlen_pages_lengths(kernel, dtype, D):
    """The varlen example's lengths [384, 1, 96, 640, 57], block-diagonal causal."""
    _skip_unsupported(kernel, dtype)
    x = attn_inputs.make(dtype=dtype, H=4, D=D, seed=11, lengths=[384, 1, 96, 640, 57])
    o, lse = _run(x, causal=True, kernel=kernel, out_dtype=_out_dtype(dtype))
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_varlen_with_empty_and_tiny_sequences(kernel):
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=12, lengths=[0, 5, 0, 200, 1, 129, 0])
    o, lse = _run(x, causal=True, kernel=kernel, out_dtype=torch.float32)
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["fp16", "f32"])
def test_cross_attention_varlen_full(kernel, dtype):
    """Full relation with different query / key lengths per sequence."""
    _skip_unsupported(kernel, dtype)
    x = attn_inputs.make(dtype=dtype, H=2, D=64, seed=13, lengths=[100, 3, 257],
                         lengths_k=[31, 300, 128])
    o, lse = _run(x, causal=False, kernel=kernel)
    o_ref, lse_ref = _ref(x, causal=False)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_empty_key_sequence_gives_zero_and_minus_inf(kernel):
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=14, lengths=[70, 9], lengths_k=[0, 40])
    o, lse = _run(x, causal=False, kernel=kernel)
    o_ref, lse_ref = _ref(x, causal=False)
    assert (f64(o)[:70] == 0).all()
    assert np.isneginf(f64(lse)[:, :70]).all()
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_bf16_output_storage(kernel):
    x = attn_inputs.make(dtype="bf16", H=4, D=128, seed=15, n_q=777)
    o, lse = _run(x, causal=True, kernel=kernel)
    assert o.dtype == torch.bfloat16
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_hnd_storage_view_and_custom_scale(kernel):
    """(H, N, D) storage viewed as (N, H, D), as in the pages' examples."""
    x = attn_inputs.make(dtype="fp16", H=3, D=64, seed=16, n_q=333, layout="hnd")
    assert not x["q"].is_contiguous()
    o, lse = _run(x, causal=False, kernel=kernel, scale=0.3)
    o_ref, lse_ref = _ref(x, causal=False, scale=0.3)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_grid_size_independent_and_deterministic(kernel):
    x = attn_inputs.make(dtype="bf16", H=4, D=128, seed=17, lengths=[500, 37, 260])
    outs = [_run(x, causal=True, kernel=kernel, out_dtype=torch.float32, num_ctas=n)
            for n in (0, 1, 7, 0)]
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])


@pytest.mark.parametrize("kernel", KERNELS)
def test_invalid_cu_seqlens_reported_by_device_status(kernel):
    """Offsets past the tensor end are caught on the device: no work is done
    and the status word reads ATTN_EINVAL."""
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=18, n_q=64)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    bad = torch.tensor([0, 32, 96], dtype=torch.int32, device=DEV)  # 96 > 64 tokens
    attn.fwd(q, k, v, causal=True, cu_seqlens_q=bad, cu_seqlens_k=bad, kernel=kernel)
    assert attn.device_status() == attn._abi.ATTN_EINVAL
    assert attn.device_status() == 0  # cleared by the read
    bad2 = torch.tensor([0, 40, 20], dtype=torch.int32, device=DEV)  # decreasing
    attn.fwd(q, k, v, causal=False, cu_seqlens_q=bad2, cu_seqlens_k=bad2, kernel=kernel)
    assert attn.device_status() == attn._abi.ATTN_EINVAL


def test_zero_queries_is_a_no_op():
    q = torch.empty(0, 2, 64, dtype=torch.float16, device=DEV)
    k = torch.randn(10, 2, 64, dtype=torch.float16, device=DEV)
    o, lse = attn.fwd(q, k, k)
    assert o.shape == (0, 2, 64) and lse.shape == (2, 0)


@pytest.mark.parametrize("kernel", KERNELS)
def test_negative_scale(kernel):
    x = attn_inputs.make(dtype="fp16", H=2, D=128, seed=19, n_q=300)
    o, lse = _run(x, causal=True, kernel=kernel, scale=-0.09)
    o_ref, lse_ref = _ref(x, causal=True, scale=-0.09)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


def test_auto_selects_tensor_cores_for_16_bit():
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=20, n_q=256)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    assert attn.FwdCall(q, k, v, causal=True).selected_kernel() == "tc"
    q32 = q.float()  # f32 at D = 128: the CUDA-core kernel
    assert attn.FwdCall(q32, q32, q32, causal=True).selected_kernel() == "simt"
    q64 = q32[..., :64].contiguous()  # f32 at D = 64: the tensor cores (split operands)
    assert attn.FwdCall(q64, q64, q64, causal=True).selected_kernel() == "tc"


@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp16", 64)])
def test_tc_matches_simt_closely(dtype, D):
    """The two kernel families agree to well within the oracle tolerance."""
    x = attn_inputs.make(dtype=dtype, H=4, D=D, seed=21, lengths=[1000, 3, 517])
    o1, l1 = _run(x, causal=True, kernel="tc", out_dtype=torch.float32)
    o2, l2 = _run(x, causal=True, kernel="simt", out_dtype=torch.float32)
    assert (o1 - o2).abs().max().item() < 1e-2
    assert (l1 - l2).abs().max().item() < 1e-4


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype,D", [("fp16", 64), ("bf16", 128), ("f32", 64)])
@pytest.mark.parametrize("splits", [1, 3])
def test_zero_scale_is_uniform_attention(kernel, dtype, D, splits):
    """scale = 0: every admitted score is 0, so O is the mean of the admitted
    values and lse = ln(count); masked keys (causal diagonal, ragged tails)
    must still weigh nothing."""
    _skip_unsupported(kernel, dtype)
    x = attn_inputs.make(dtype=dtype, H=2, D=D, seed=23, lengths=[300, 1, 129])
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = attn.fwd(q, k, v, causal=True, scale=0.0, cu_seqlens_q=x["cu_seqlens_q"],
                      out_dtype=_out_dtype(dtype), kernel=kernel, num_splits=splits)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    o_ref, lse_ref = _ref(x, causal=True, scale=0.0)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
def test_many_short_sequences(kernel):
    """20000 sequences of 0 to 4 tokens: the schedule's prefix over many
    sequences, empty ones among them, and one partial tile per sequence."""
    lengths = np.random.default_rng(24).integers(0, 5, 20000).tolist()
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=24, lengths=lengths)
    o, lse = _run(x, causal=True, kernel=kernel)
    o_ref, lse_ref = _ref(x, causal=True)
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype,D,N,causal,splits", [
    ("fp16", 64, 256, True, 0), ("fp16", 64, 1024, False, 0), ("fp16", 64, 1024, False, 1),
    ("bf16", 128, 300, True, 1), ("f32", 64, 2048, False, 0)])
def test_single_launch_schedule_matches_the_dynamic_one(kernel, dtype, D, N, causal, splits):
    """One sequence whose items fit in one wave runs without the preparation
    kernel (CTA i runs item i): one attention launch, plus the merge when split
    (and the operand-splitting prepass for f32 on the tensor cores).  Its
    results equal those of the dynamic schedule (explicit grid) bit for bit
    and match the oracle."""
    _skip_unsupported(kernel, dtype)
    x = attn_inputs.make(dtype=dtype, H=3, D=D, seed=60 + N, n_q=N)
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    odt = _out_dtype(dtype)
    one = attn.FwdCall(q, k, v, causal=causal, kernel=kernel, num_splits=splits, out_dtype=odt)
    dyn = attn.FwdCall(q, k, v, causal=causal, kernel=kernel, num_splits=splits, out_dtype=odt,
                       num_ctas=sms)
    n0 = attn.launch_count()
    one.run()
    launched = attn.launch_count() - n0
    dyn.run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    # f32 on the tensor cores adds the operand-splitting prepass
    prepass = 1 if (dtype == "f32" and one.selected_kernel() == "tc") else 0
    assert launched == (1 if one.num_splits() == 1 else 2) + prepass
    assert torch.equal(one.o, dyn.o) and torch.equal(one.lse, dyn.lse)
    o_ref, lse_ref = _ref(x, causal=causal)
    check_o(one.o, o_ref, x["q"].dtype, one.o.dtype)
    check_lse(one.lse, lse_ref)
