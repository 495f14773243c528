"""attn_fwd_noalloc: the forward for callers that cannot allocate device memory.

Such callers hold only their input and output buffers -- for example a plugin
that a host framework calls with tensors it owns, with no allocator or
workspace to hand, or a serving loop that must not call cudaMalloc.  The entry
point takes its scheduler scratch from a fixed array inside the library.

These tests call it through the C ABI on two calls in a row with different
problems (and the first problem once more after the second, since the shared
array keeps the last call's contents), and check each result against the f64
oracle element by element at the forward tolerances, and bit for bit against
the regular attn_fwd run with the same schedule (num_splits = 1, the only one
the fixed scratch allows).  They also check that a sequence count beyond the
fixed scratch is rejected.  The file sorts last so that a run stopping at the
first failure has already run every other test; it also passes on its own in
a fresh process (the first call sets up the scratch address).
"""
import ctypes

import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
import oracle
from online_softmax_attention_gb300 import _abi
from parity_util import check_lse, check_o

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(case):
    if case == "varlen":
        x = attn_inputs.make(dtype="bf16", H=4, D=128, seed=31, lengths=[384, 1, 96, 640, 57])
        return x, True, torch.float32
    x = attn_inputs.make(dtype="fp16", H=3, D=64, seed=32, n_q=700, layout="hnd")
    return x, False, None


def _call(x, causal, out_dtype, num_splits=1):
    q, k, v = (x[n].to(DEV) for n in ("q", "k", "v"))
    return attn.FwdCall(q, k, v, causal=causal, cu_seqlens_q=x["cu_seqlens_q"],
                        cu_seqlens_k=x["cu_seqlens_k"], out_dtype=out_dtype, num_splits=num_splits)


def _noalloc(call):
    lib = _abi.load()
    s = torch.cuda.current_stream()
    return lib.attn_fwd_noalloc(ctypes.byref(call.args), ctypes.c_void_p(s.cuda_stream))


def _check(call, x, causal, o_ref, lse_ref):
    # against the oracle at the forward bounds, and bit for bit against attn_fwd
    # with the same (unsplit) schedule
    ro, rl = oracle.fwd(x["q"], x["k"], x["v"], causal=causal, cu_seqlens_q=x["cu_seqlens_q"],
                        cu_seqlens_k=x["cu_seqlens_k"])
    check_o(call.o, ro, x["q"].dtype, call.o.dtype)
    check_lse(call.lse, rl)
    assert torch.equal(call.o, o_ref)
    assert torch.equal(call.lse, lse_ref)


def test_noalloc_matches_the_oracle_and_attn_fwd_on_two_calls_in_a_row():
    results = []
    for case in ("varlen", "single"):
        x, causal, odt = _inputs(case)
        ref = _call(x, causal, odt, num_splits=1)
        o_ref, lse_ref = (t.clone() for t in ref.run())
        torch.cuda.synchronize()
        call = _call(x, causal, odt)
        call.o.fill_(float("nan"))
        call.lse.fill_(float("nan"))
        assert _noalloc(call) == _abi.ATTN_OK
        torch.cuda.synchronize()
        assert attn.device_status() == 0
        _check(call, x, causal, o_ref, lse_ref)
        results.append((call, x, causal, o_ref, lse_ref))
    # the first problem again: the scratch keeps the second call's contents
    call, x, causal, o_ref, lse_ref = results[0]
    call.o.zero_()
    call.lse.zero_()
    assert _noalloc(call) == _abi.ATTN_OK
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    _check(call, x, causal, o_ref, lse_ref)


def test_noalloc_rejects_more_sequences_than_its_scratch_holds():
    x, causal, odt = _inputs("single")
    call = _call(x, causal, odt)
    args = _abi.FwdArgs.from_buffer_copy(call.args)
    args.cu_seqlens_q = args.cu_seqlens_k = call.o.data_ptr()  # never read: rejected first
    args.n_seq = _abi.ATTN_NOALLOC_MAX_SEQ + 1
    lib = _abi.load()
    rc = lib.attn_fwd_noalloc(ctypes.byref(args), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == _abi.ATTN_EUNSUPPORTED
