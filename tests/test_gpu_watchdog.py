"""Failure detection on the GPU without faulting it: with a tiny bounded-wait
budget the tensor-core kernels' mbarrier waits run out, the kernels stop,
drain their loads, free tensor memory and exit, and the status word reads
ATTN_ETIMEOUT; the context stays usable and the next calls succeed."""
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn
from online_softmax_attention_gb300 import _abi

pytestmark = pytest.mark.gpu


def test_watchdog_timeout_is_reported_and_recoverable():
    lib = _abi.load()
    x = attn_inputs.make(dtype="bf16", H=4, D=128, seed=41, n_q=2048, backward=True)
    q, k, v, dO = (x[n].cuda() for n in ("q", "k", "v", "dO"))
    good_o, good_lse = attn.fwd(q, k, v, causal=True, kernel="tc")
    good_o, good_lse = good_o.clone(), good_lse.clone()
    assert attn.device_status() == 0
    prev = lib.attn_set_watchdog_cycles(64)  # far below one tile's latency
    try:
        attn.fwd(q, k, v, causal=True, kernel="tc")
        assert attn.device_status() == _abi.ATTN_ETIMEOUT
        o, lse = attn.fwd(q, k, v, causal=True, kernel="tc")
        dq, dk, dv = attn.bwd(q, k, v, o, lse, dO, causal=True, kernel="tc")
        assert attn.device_status() == _abi.ATTN_ETIMEOUT
    finally:
        lib.attn_set_watchdog_cycles(prev if prev != 4000000000 else 0)
    # the context is intact: normal calls give the normal answer again
    o, lse = attn.fwd(q, k, v, causal=True, kernel="tc")
    torch.cuda.synchronize()
    assert attn.device_status() == 0
    assert torch.equal(o, good_o) and torch.equal(lse, good_lse)
