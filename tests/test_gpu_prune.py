"""Tile-pruned approximate forward (TIGA-lang attention examples page, section
"基于 tile 剪枝的稀疏注意力"), CUDA path through the C ABI vs the oracle's
pruned forward with the kernel's own tile sizes.

The admission decisions are discrete and taken in floating point.  Every case
here is checked first on the oracle to be decisive: the smallest distance of a
decision's m_tile from its threshold m_run + ln(rho) (min_margin) is far above
the f32 rounding of the kernel's scores (~1e-5 at these magnitudes), so the
kernel must take exactly the oracle's decisions.  The pruned-tile counts are
then compared exactly, and O and lse element by element at the usual
tolerances.
"""
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_lse, check_o

pytestmark = pytest.mark.gpu

DEV = "cuda"
TILE = {"tc": 128, "simt": 64}  # query rows x keys of a tile, per kernel family
DECISIVE = 0.01


def _run(x, kernel, rho, out_dtype=None):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    call = attn.FwdCall(q, k, v, causal=False, kernel=kernel, prune_threshold=rho,
                        out_dtype=out_dtype)
    assert call.selected_kernel() == kernel
    o, lse = call.run()
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return o, lse, call.pruned_count()


def _ref(x, kernel, rho):
    b = TILE[kernel]
    o, lse, n, margin = oracle.fwd_pruned(x["q"], x["k"], x["v"], rho=rho, block_q=b, block_k=b)
    assert margin > DECISIVE, f"inputs not decisive for rho={rho}: min margin {margin}"
    return o, lse, n


# (kernel, dtype, D, seed, n_q, n_k, rho): seeds chosen so the oracle's min
# margin exceeds DECISIVE and some tiles are pruned
STRUCTURED = [
    ("tc", "bf16", 128, 501, 1000, 1500, 0.5),
    ("tc", "bf16", 128, 507, 1000, 1500, 0.05),
    ("tc", "fp16", 64, 503, 1000, 1000, 0.2),
    ("simt", "f32", 64, 500, 700, 900, 0.5),
    ("simt", "fp16", 128, 500, 700, 900, 0.1),
]


@pytest.mark.parametrize("kernel,dtype,D,seed,n_q,n_k,rho", STRUCTURED)
def test_pruned_forward_matches_oracle(kernel, dtype, D, seed, n_q, n_k, rho):
    b = TILE[kernel]
    x = attn_inputs.make(dtype=dtype, H=2, D=D, seed=seed, lengths=[n_q], lengths_k=[n_k],
                         key_gain=(b, 0.2, 3.0))
    o_ref, lse_ref, n_ref = _ref(x, kernel, rho)
    assert n_ref > 0
    out = torch.float32 if dtype == "bf16" else None
    o, lse, n = _run(x, kernel, rho, out_dtype=out)
    assert n == n_ref
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


def test_page_configuration_threshold_width_over_nodes():
    """The page's example: N = 1024, H = 4, D = 64, fp16 N(0, 1) in (H, N, D)
    storage, full relation, threshold width / nodes = 1 / 16.  On such inputs
    no tile falls below the threshold, so the result is the exact attention."""
    x = attn_inputs.make_workload("full_fp16_n1024")
    o_ref, lse_ref, n_ref = _ref(x, "tc", 64 / 1024)
    o, lse, n = _run(x, "tc", 64 / 1024)
    assert n == n_ref == 0
    check_o(o, o_ref, torch.float16, o.dtype)
    check_lse(lse, lse_ref)
    # nothing pruned: bit-identical to the exact forward run unsplit, like the pruned one
    o_exact, lse_exact = attn.fwd(*(x[m].to(DEV) for m in ("q", "k", "v")), kernel="tc",
                                  num_splits=1)
    assert torch.equal(o, o_exact) and torch.equal(lse, lse_exact)


def test_counter_accumulates_over_runs():
    x = attn_inputs.make(dtype="bf16", H=2, D=128, seed=501, lengths=[1000], lengths_k=[1500],
                         key_gain=(128, 0.2, 3.0))
    _, _, n_ref = _ref(x, "tc", 0.5)
    q, k, v = (x[m].to(DEV) for m in ("q", "k", "v"))
    call = attn.FwdCall(q, k, v, prune_threshold=0.5, out_dtype=torch.float32)
    call.run()
    call.run()
    torch.cuda.synchronize()
    assert call.pruned_count() == 2 * n_ref


@pytest.mark.parametrize("kernel", ["tc", "simt"])
def test_pruning_fails_closed_outside_the_dense_forward(kernel):
    x = attn_inputs.make(dtype="fp16", H=2, D=64, seed=520, n_q=300, backward=True)
    q, k, v, dO = (x[m].to(DEV) for m in ("q", "k", "v", "dO"))
    with pytest.raises(attn.AttnError):
        attn.fwd(q, k, v, causal=True, kernel=kernel, prune_threshold=0.5)
    cu = torch.tensor([0, 100, 300], dtype=torch.int32)
    with pytest.raises(attn.AttnError):
        attn.fwd(q, k, v, cu_seqlens_q=cu, kernel=kernel, prune_threshold=0.5)
    o, lse = attn.fwd(q, k, v, kernel=kernel, prune_threshold=0.5)
    with pytest.raises(attn.AttnError):
        attn.BwdCall(q, k, v, o, lse, dO, kernel=kernel, prune_threshold=0.5).run()
