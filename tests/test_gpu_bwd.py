"""Backward parity: CUDA dq, dk, dv (through the C ABI) vs the oracle's
explicit-Jacobian backward, on seeded inputs spanning tiles and ragged tails."""
import numpy as np
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_grad, check_lse, check_o

pytestmark = pytest.mark.gpu

# kernel family / dq mode: "auto" resolves to the separate (deterministic)
# dq kernel; "tc/fused" accumulates dq inside the dK/dV kernel
KERNELS = ["auto", "simt", "tc", "tc/fused"]
DEV = "cuda"


def _skip_unsupported(kernel, dtype):
    if kernel.startswith("tc") and dtype == "f32":
        pytest.skip("the tensor-core kernels take f16 / bf16 only")


def _split(kernel):
    fam, _, mode = kernel.partition("/")
    return fam, mode or "auto"


def _fwd_bwd(x, *, causal, kernel, out_dtype=None, grad_dtype=None, num_ctas=0, scale=None):
    fam, mode = _split(kernel)
    q, k, v, dO = (x[n].to(DEV) for n in ("q", "k", "v", "dO"))
    cq, ck = x["cu_seqlens_q"], x["cu_seqlens_k"]
    o, lse = attn.fwd(q, k, v, causal=causal, scale=scale, cu_seqlens_q=cq, cu_seqlens_k=ck,
                      out_dtype=out_dtype, kernel=fam)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, dO, causal=causal, scale=scale, cu_seqlens_q=cq,
                          cu_seqlens_k=ck, grad_dtype=grad_dtype, kernel=fam, num_ctas=num_ctas,
                          dq_mode=mode)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return dq, dk, dv


def _ref(x, *, causal, scale=None):
    return oracle.bwd(x["q"], x["k"], x["v"], x["dO"], causal=causal, scale=scale,
                      cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])


def _check(got, ref):
    for g, r, n in zip(got, ref, ("dq", "dk", "dv")):
        check_grad(g, r, n)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("dtype", ["fp16", "bf16", "f32"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 129, 300])
def test_single_sequence(kernel, dtype, D, causal, N):
    _skip_unsupported(kernel, dtype)
    x = attn_inputs.make(dtype=dtype, H=2, D=D, seed=200 + N, n_q=N, backward=True)
    _check(_fwd_bwd(x, causal=causal, kernel=kernel), _ref(x, causal=causal))


@pytest.mark.parametrize("kernel", KERNELS)
def test_varlen_pages_lengths(kernel):
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=21, lengths=[384, 1, 96, 640, 57],
                         backward=True)
    _check(_fwd_bwd(x, causal=True, kernel=kernel, out_dtype=torch.float32), _ref(x, causal=True))


@pytest.mark.parametrize("kernel", KERNELS)
def test_cross_attention_full(kernel):
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=22, lengths=[100, 3, 257],
                         lengths_k=[31, 300, 128], backward=True)
    _check(_fwd_bwd(x, causal=False, kernel=kernel), _ref(x, causal=False))


@pytest.mark.parametrize("kernel", KERNELS)
def test_f32_gradients_and_custom_scale(kernel):
    x = attn_inputs.make(dtype="bf16", H=2, D=64, seed=23, n_q=200, backward=True)
    got = _fwd_bwd(x, causal=True, kernel=kernel, grad_dtype=torch.float32, scale=0.2)
    assert got[0].dtype == torch.float32
    _check(got, _ref(x, causal=True, scale=0.2))


@pytest.mark.parametrize("kernel", ["auto", "simt", "tc"])
def test_deterministic_and_grid_independent(kernel):
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=24, lengths=[300, 70], backward=True)
    runs = [_fwd_bwd(x, causal=True, kernel=kernel, num_ctas=n) for n in (0, 3, 0)]
    for r in runs[1:]:
        for a, b in zip(r, runs[0]):
            assert torch.equal(a, b)


@pytest.mark.parametrize("D", [64, 128])
def test_fused_dq_grid_independent(D):
    """Fused dq: dk and dv are written once (bitwise equal across grids); dq is a
    sum of f32 reductions in varying order (equal up to rounding)."""
    x = attn_inputs.make(dtype="bf16", H=2, D=D, seed=24, lengths=[300, 70], backward=True)
    runs = [_fwd_bwd(x, causal=True, kernel="tc/fused", num_ctas=n, grad_dtype=torch.float32)
            for n in (0, 3, 0)]
    for r in runs[1:]:
        assert torch.equal(r[1], runs[0][1]) and torch.equal(r[2], runs[0][2])
        rel = float((r[0] - runs[0][0]).norm() / runs[0][0].norm())
        assert rel < 1e-5, rel


def test_dq_mode_selection():
    x = attn_inputs.make(dtype="bf16", H=2, D=64, seed=27, n_q=130, backward=True)
    q, k, v, dO = (x[n].to(DEV) for n in ("q", "k", "v", "dO"))
    o, lse = attn.fwd(q, k, v, causal=True)
    assert attn.BwdCall(q, k, v, o, lse, dO, causal=True).selected_dq_mode() == "separate"
    assert attn.BwdCall(q, k, v, o, lse, dO, causal=True, dq_mode="fused").selected_dq_mode() == "fused"
    assert attn.BwdCall(q, k, v, o, lse, dO, causal=True, kernel="simt").selected_dq_mode() == "separate"
    with pytest.raises(attn.AttnError):
        attn.BwdCall(q, k, v, o, lse, dO, causal=True, kernel="simt", dq_mode="fused").run()
    # the fused mode's workspace holds the dq partial sums, n_q * H * D f32
    fused = attn.BwdCall(q, k, v, o, lse, dO, causal=True, dq_mode="fused")
    sep = attn.BwdCall(q, k, v, o, lse, dO, causal=True)
    assert fused.workspace.numel() - sep.workspace.numel() >= 130 * 2 * 64 * 4


def test_fused_dq_matches_separate_closely():
    x = attn_inputs.make(dtype="bf16", H=4, D=128, seed=28, lengths=[1000, 129, 384], backward=True)
    a = _fwd_bwd(x, causal=True, kernel="tc/fused", out_dtype=torch.float32, grad_dtype=torch.float32)
    b = _fwd_bwd(x, causal=True, kernel="tc", out_dtype=torch.float32, grad_dtype=torch.float32)
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2]), "dk / dv differ between dq modes"
    rel = float((a[0] - b[0]).norm() / b[0].norm())
    assert rel < 1e-3, rel


@pytest.mark.parametrize("kernel", KERNELS)
def test_empty_sequences_and_empty_keys(kernel):
    """Zero-length query / key sequences: their gradients are zero, others unaffected."""
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=25, lengths=[0, 70, 9, 130],
                         lengths_k=[40, 0, 33, 129], backward=True)
    got = _fwd_bwd(x, causal=False, kernel=kernel)
    ref = _ref(x, causal=False)
    _check(got, ref)
    assert float(got[1][:40].abs().max()) == 0.0 and float(got[2][:40].abs().max()) == 0.0


def test_tc_backward_matches_simt_closely():
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=26, lengths=[700, 129], backward=True)
    a = _fwd_bwd(x, causal=True, kernel="tc", out_dtype=torch.float32, grad_dtype=torch.float32)
    b = _fwd_bwd(x, causal=True, kernel="simt", out_dtype=torch.float32, grad_dtype=torch.float32)
    for u, v in zip(a, b):
        rel = float((u - v).norm() / v.norm())
        assert rel < 5e-3, rel


@pytest.mark.parametrize("kernel", KERNELS)
def test_zero_scale(kernel):
    """scale = 0: P is uniform over the admitted keys, dq = dk = 0."""
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=48, lengths=[300, 1, 129], backward=True)
    got = _fwd_bwd(x, causal=True, kernel=kernel, scale=0.0)
    _check(got, _ref(x, causal=True, scale=0.0))
    assert float(got[0].abs().max()) == 0.0 and float(got[1].abs().max()) == 0.0


@pytest.mark.parametrize("kernel", KERNELS)
def test_many_short_sequences(kernel):
    lengths = np.random.default_rng(49).integers(0, 5, 20000).tolist()
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=49, lengths=lengths, backward=True)
    _check(_fwd_bwd(x, causal=True, kernel=kernel), _ref(x, causal=True))



def _rel_rms_tiled(g, ref, copies, factor=1.0):
    """Relative RMS of g (copies x block rows) against `ref` (one block, f64)
    times `factor`, repeated over the copies; summed on the device in chunks."""
    r = torch.as_tensor(np.asarray(ref) * factor, dtype=torch.float32, device=DEV)
    gv = g.reshape(copies, *r.shape)
    num = den = 0.0
    for c in gv.split(4096):
        assert bool(torch.isfinite(c).all())
        d = c.float() - r
        num += float(torch.sum(d * d, dtype=torch.float64))
        den += float(torch.sum(r * r, dtype=torch.float64)) * c.shape[0]
    return (num / den) ** 0.5


@pytest.mark.parametrize("long_side", ["keys", "queries"])
def test_more_than_65536_blocks_in_one_item(long_side):
    """One work item spanning more than 2^16 blocks of 128 rows: the forward's
    and the dq kernel's key loops (long keys) or the dK/dV kernel's query loop
    (long queries) run 65540 blocks.  One block carries the problem, the other
    65539 contribute exactly nothing, so the answer is the single-block
    problem's: filler keys score -100 against every query after scaling (q's
    first component is 4, the fillers' -200, scale 1/8), so their softmax
    weights, e^-100 below the smallest normal float, flush to 0; filler query
    rows repeat the query block
    with dO = 0 (their dS is 0, their O and lse repeat the block's).  Adding
    zeros keeps the tensor core's f32 accumulators exact, so the ordinary bars
    apply however many blocks an accumulator spans."""
    m = 65540
    x = attn_inputs.make(dtype="bf16", H=1, D=64, seed=91, n_q=256 if long_side == "keys" else 128,
                         n_k=128, backward=True)
    if long_side == "keys":
        x["q"][:, :, 0] = 4.0
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=False)
    rq, rk, rv = oracle.bwd(x["q"], x["k"], x["v"], x["dO"], causal=False)
    q, k, v, dO = (x[n].to(DEV) for n in ("q", "k", "v", "dO"))
    if long_side == "keys":
        filler = torch.zeros(((m - 1) * 128, 1, 64), dtype=k.dtype, device=DEV)
        kf = filler.clone()
        kf[:, :, 0] = -200.0
        k, v = torch.cat([k, kf]), torch.cat([v, filler])
    else:
        q = q.repeat(m, 1, 1)
        dO = torch.cat([dO, torch.zeros(((m - 1) * 128, 1, 64), dtype=dO.dtype, device=DEV)])
    o, lse = attn.fwd(q, k, v, causal=False, out_dtype=torch.float32)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, dO, causal=False, grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    if long_side == "keys":
        check_o(o, o_ref, torch.bfloat16, o.dtype)
        check_lse(lse, lse_ref)
        check_grad(dq, rq, "dq")
        check_grad(dk[:128], rk, "dk")
        check_grad(dv[:128], rv, "dv")
        assert float(dk[128:].abs().max()) == 0.0 and float(dv[128:].abs().max()) == 0.0
    else:
        assert _rel_rms_tiled(o, o_ref, m) <= 2e-3
        lse_d = lse.reshape(1, m, 128) - torch.as_tensor(lse_ref, dtype=torch.float32, device=DEV)[:, None, :]
        assert float(lse_d.abs().max()) <= 1e-3
        check_grad(dq[:128], rq, "dq")
        assert float(dq[128:].abs().max()) == 0.0
        check_grad(dk, rk, "dk")
        check_grad(dv, rv, "dv")
