"""Parity at the five benchmark workloads' full sizes, in the launch
configuration the benchmark uses (AUTO kernel choice, one CTA per SM).

Small workloads are compared element by element with the oracle; the large
ones on sampled (token, head) rows that the oracle computes one by one:
segment ends, tile edges and random rows for O / lse / dq, and sampled key
rows of six (sequence, head) pairs of the training workload -- the first and
the last head among them -- for dk / dv, each pair held to the gradient bar
on its own."""
import numpy as np
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from parity_util import check_grad, check_lse, check_o, sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _at(t, a, b):
    return t[torch.from_numpy(np.asarray(a)), torch.from_numpy(np.asarray(b))]


def _fwd(x, w, out_dtype=None):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    o, lse = attn.fwd(q, k, v, causal=w.causal, cu_seqlens_q=x["cu_seqlens_q"],
                      cu_seqlens_k=x["cu_seqlens_k"], out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    return o, lse


@pytest.mark.parametrize("name", ["causal_fp16_n256", "full_fp16_n1024", "cross_f32_8192x2048"])
def test_small_workloads_elementwise(name):
    w = attn_inputs.WORKLOADS[name]
    x = attn_inputs.make_workload(w)
    o, lse = _fwd(x, w)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=w.causal,
                                cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])
    check_o(o, o_ref, x["q"].dtype, o.dtype)
    check_lse(lse, lse_ref)


def test_varlen_causal_workload_sampled_rows():
    w = attn_inputs.WORKLOADS["varlen_causal_bf16"]
    x = attn_inputs.make_workload(w)
    assert any(L % 128 for L in x["lengths_q"]), "lengths must exercise the -inf tail"
    assert all(64 <= L <= 4096 for L in x["lengths_q"])
    o, lse = _fwd(x, w, out_dtype=torch.float32)
    toks, heads = sample_rows(x["lengths_q"], w.H, n_random=400, seed=1)
    o_ref, lse_ref = oracle.fwd_rows(x["q"], x["k"], x["v"], toks, heads, causal=True,
                                     cu_seqlens_q=x["cu_seqlens_q"])
    check_o(_at(o, toks, heads), o_ref, x["q"].dtype, o.dtype)
    check_lse(_at(lse, heads, toks), lse_ref)
    # the bf16-stored output too, at its bar
    o16, _ = _fwd(x, w)
    check_o(_at(o16, toks, heads), o_ref, x["q"].dtype, o16.dtype)


@pytest.mark.slow
def test_causal_training_workload_sampled():
    w = attn_inputs.WORKLOADS["causal_train_bf16_b4_n8192"]
    x = attn_inputs.make_workload(w)
    q, k, v, dO = (x[n].to(DEV) for n in ("q", "k", "v", "dO"))
    cu = x["cu_seqlens_q"]
    o, lse = attn.fwd(q, k, v, causal=True, cu_seqlens_q=cu, out_dtype=torch.float32)
    dq, dk, dv = attn.bwd(q, k, v, o, lse, dO, causal=True, cu_seqlens_q=cu)
    torch.cuda.synchronize()
    assert attn.device_status() == 0

    toks, heads = sample_rows(x["lengths_q"], w.H, n_random=300, seed=5)
    o_ref, lse_ref = oracle.fwd_rows(x["q"], x["k"], x["v"], toks, heads, causal=True,
                                     cu_seqlens_q=cu)
    check_o(_at(o, toks, heads), o_ref, x["q"].dtype, o.dtype)
    check_lse(_at(lse, heads, toks), lse_ref)

    # gradients on six (sequence, head) pairs, (b0, h0) and the last head (b3,
    # h31) among them: dk, dv on sampled keys (tile edges and random keys) of
    # every pair; dq on the sampled rows above plus tile-edge rows of every pair
    L = w.n_q
    pairs = [(0, 0), (0, 31), (1, 11), (2, 22), (3, 0), (3, 31)]
    rng = np.random.default_rng(55)
    kt, kh, qt, qh = [], [], [], []
    for b, h in pairs:
        keys = np.concatenate([rng.integers(0, L, 12), [0, 127, 128, L - 1]])
        kt += list(b * L + keys)
        kh += [h] * len(keys)
        rows = np.concatenate([rng.integers(0, L, 6), [0, 255, 256, L - 1]])
        qt += list(b * L + rows)
        qh += [h] * len(rows)
    kt, kh = np.array(kt, dtype=np.int64), np.array(kh, dtype=np.int32)
    qt = np.concatenate([np.array(qt, dtype=np.int64), toks[:120]])
    qh = np.concatenate([np.array(qh, dtype=np.int32), heads[:120]])
    rq, rk, rv = oracle.bwd(x["q"], x["k"], x["v"], x["dO"], causal=True, cu_seqlens_q=cu,
                            q_rows=(qt, qh), k_rows=(kt, kh))
    check_grad(_at(dq, qt, qh), rq, "dq")
    for i, (b, h) in enumerate(pairs):
        sl = slice(16 * i, 16 * (i + 1))
        check_grad(_at(dk, kt[sl], kh[sl]), rk[sl], f"dk (b{b}, h{h})")
        check_grad(_at(dv, kt[sl], kh[sl]), rv[sl], f"dv (b{b}, h{h})")
    for g in (dq, dk, dv):
        assert bool(torch.isfinite(g).all())
