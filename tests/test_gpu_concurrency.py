"""Concurrent calls: per-sequence forward + backward of the training workload
alternating between two compute streams while pinned host copies run on two
more (the pattern of the benchmark's end-to-end leg), for a few hundred steps.
Every mbarrier wait in the kernels is bounded, so a barrier protocol that can
lose a phase under unlucky timing shows up as a watchdog status instead of a
hang; the status word must stay clear, and the last step's results must equal
the batched call's bit for bit."""
import pytest
import torch

import attn_inputs
import online_softmax_attention_gb300 as attn

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_two_compute_streams_with_host_copies():
    w = attn_inputs.WORKLOADS["causal_train_bf16_b4_n8192"]
    x = attn_inputs.make_workload(w)
    q, k, v, dO = (x[n].to(DEV) for n in ("q", "k", "v", "dO"))
    L = w.n_q
    stream = torch.cuda.current_stream()
    pin = {n: x[n].contiguous().pin_memory() for n in ("q", "k", "v", "dO")}
    dev_in = {"q": q, "k": k, "v": v, "dO": dO}
    seqs = []
    for b in range(w.batch):
        sl = slice(b * L, (b + 1) * L)
        fb = attn.FwdCall(q[sl], k[sl], v[sl], causal=True, out_dtype=torch.float32)
        bb = attn.BwdCall(q[sl], k[sl], v[sl], fb.o, fb.lse, dO[sl], causal=True)
        seqs.append((sl, fb, bb))
    dq_h = torch.empty(q.shape, dtype=q.dtype).pin_memory()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    s_comp = [stream, torch.cuda.Stream()]
    ev_in = [torch.cuda.Event() for _ in seqs]
    ev_done = [torch.cuda.Event() for _ in seqs]
    ev_out = [torch.cuda.Event() for _ in seqs]
    ev_used = [torch.cuda.Event() for _ in seqs]
    for e in ev_out + ev_used:
        e.record(stream)

    def step():
        for i, (sl, _, _) in enumerate(seqs):
            s_in.wait_event(ev_used[i])
            with torch.cuda.stream(s_in):
                for n in ("q", "k", "v", "dO"):
                    dev_in[n][sl].copy_(pin[n][sl], non_blocking=True)
            ev_in[i].record(s_in)
        for i, (sl, fb, bb) in enumerate(seqs):
            cs = s_comp[i % 2]
            cs.wait_event(ev_in[i])
            cs.wait_event(ev_out[i])
            fb.run(cs)
            bb.run(cs)
            ev_done[i].record(cs)
            ev_used[i].record(cs)
        for i, (sl, _, bb) in enumerate(seqs):
            s_out.wait_event(ev_done[i])
            with torch.cuda.stream(s_out):
                dq_h[sl].copy_(bb.dq, non_blocking=True)
            ev_out[i].record(s_out)

    for it in range(300):
        step()
        if (it + 1) % 50 == 0:
            torch.cuda.synchronize()
            status = attn.device_status()
            assert status == 0, f"status {status} ({attn.strerror(status)}) after step {it + 1}"
    torch.cuda.synchronize()
    cu = x["cu_seqlens_q"].to(DEV)
    o, lse = attn.fwd(q, k, v, causal=True, cu_seqlens_q=cu, out_dtype=torch.float32)
    dq, _, _ = attn.bwd(q, k, v, o, lse, dO, causal=True, cu_seqlens_q=cu)
    torch.cuda.synchronize()
    assert torch.equal(dq_h, dq.cpu())
    assert attn.device_status() == 0
