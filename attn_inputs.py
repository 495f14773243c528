"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and lays them out; it holds none of the
attention arithmetic.  Both the CUDA path's tests / benchmark and the oracle
take their inputs from here, so the two sides see bit-identical operands.

Recipe (the pages draw their examples with ``torch.randn`` on the GPU, which a
CPU oracle cannot replay, so every draw here uses a CPU generator instead):

* ``torch.Generator().manual_seed(seed)`` on the CPU.
* Varlen lengths, when drawn, come first: ``torch.randint(lo, hi + 1, (n_seq,))``.
* Then q, k, v (then dO) in that order, each ``torch.randn(..., float32)`` and
  then cast to the workload dtype (round to nearest even).
* ``layout="hnd"`` draws an (H, N, D) tensor and returns its (N, H, D) view,
  as the TIGA-lang full / causal examples do ("the streaming kernel reads
  lane-major storage"); ``layout="thd"`` draws (T, H, D) directly.
* ``key_gain=(block, lo, hi)`` (structured keys for the tile-pruning tests):
  after all other draws, one gain per (block of ``block`` keys, head) is
  drawn uniformly in [lo, hi] (``torch.rand`` on the same generator) and the
  keys of that block and head are multiplied by it in f32, then cast back.
  Blocks of large gain hold the large scores, so whole key tiles differ in
  their best score as on the tile-pruning page's picture.

The named workloads are the five benchmark configurations, plus one with
structured keys for the tile-pruning option; they carry their shapes, dtype,
relation and seed.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

DTYPES = {"fp16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


@dataclass(frozen=True)
class Workload:
    name: str
    dtype: str
    H: int
    D: int
    causal: bool
    seed: int
    n_q: int = 0              # single-sequence query length (0 when varlen)
    n_k: int = 0              # single-sequence key length
    batch: int = 1            # equal-length sequences packed back to back
    varlen: tuple = ()        # (n_seq, lo, hi): lengths drawn uniformly in [lo, hi]
    layout: str = "thd"
    backward: bool = False
    key_gain: tuple = ()      # (block, lo, hi): structured keys, see the recipe
    note: str = field(default="", compare=False)


WORKLOADS = {
    "causal_fp16_n256": Workload(
        "causal_fp16_n256", "fp16", H=2, D=64, causal=True, seed=7, n_q=256, n_k=256,
        layout="hnd", note="causal fwd, N=256, H=2, D=64, fp16, (H,N,D) storage"),
    "full_fp16_n1024": Workload(
        "full_fp16_n1024", "fp16", H=4, D=64, causal=False, seed=0, n_q=1024, n_k=1024,
        layout="hnd", note="full fwd, N=1024, H=4, D=64, fp16, (H,N,D) storage"),
    "varlen_causal_bf16": Workload(
        "varlen_causal_bf16", "bf16", H=16, D=128, causal=True, seed=1, varlen=(32, 64, 4096),
        note="varlen causal fwd, 32 sequences with lengths uniform in [64,4096], H=16, D=128, bf16"),
    "cross_f32_8192x2048": Workload(
        "cross_f32_8192x2048", "f32", H=1, D=64, causal=False, seed=3, n_q=8192, n_k=2048,
        note="cross fwd in f32, SQ=8192, SK=2048, H=1, D=64"),
    "causal_train_bf16_b4_n8192": Workload(
        "causal_train_bf16_b4_n8192", "bf16", H=32, D=128, causal=True, seed=5, n_q=8192,
        n_k=8192, batch=4, backward=True,
        note="causal fwd+bwd, batch 4 x N=8192, H=32, D=128, bf16"),
    # tile pruning (approximate forward): keys with one gain in [0.2, 3] per
    # 128-key tile and head, so that whole tiles differ in their best score
    "pruned_full_bf16_n8192": Workload(
        "pruned_full_bf16_n8192", "bf16", H=16, D=128, causal=False, seed=9, n_q=8192,
        n_k=8192, key_gain=(128, 0.2, 3.0),
        note="full fwd, N=8192, H=16, D=128, bf16, key gain per 128-key tile in [0.2, 3]"),
}


def _randn(gen: torch.Generator, shape, dtype: torch.dtype) -> torch.Tensor:
    return torch.randn(shape, generator=gen, dtype=torch.float32).to(dtype)


def make(*, dtype: str, H: int, D: int, seed: int, n_q: int | None = None,
         n_k: int | None = None, batch: int = 1, lengths=None, lengths_k=None,
         varlen: tuple = (), layout: str = "thd", backward: bool = False,
         key_gain: tuple = ()) -> dict:
    """Draw one input set.  Returns CPU tensors and host cu_seqlens.

    Keys: q, k, v, (dO), cu_seqlens_q, cu_seqlens_k (int32, or None for a
    single sequence), lengths_q, lengths_k (python lists).
    """
    gen = torch.Generator().manual_seed(seed)
    tdt = DTYPES[dtype]
    if varlen:
        n_seq, lo, hi = varlen
        lq = torch.randint(lo, hi + 1, (n_seq,), generator=gen).tolist()
        lk = list(lq)
    elif lengths is not None:
        lq = [int(x) for x in lengths]
        lk = [int(x) for x in (lengths_k if lengths_k is not None else lengths)]
    else:
        lq = [int(n_q)] * batch
        lk = [int(n_k if n_k is not None else n_q)] * batch
    Tq, Tk = sum(lq), sum(lk)

    def draw(T):
        if layout == "hnd":
            return _randn(gen, (H, T, D), tdt).permute(1, 0, 2)
        return _randn(gen, (T, H, D), tdt)

    out = {"q": draw(Tq), "k": draw(Tk), "v": draw(Tk)}
    if backward:
        out["dO"] = draw(Tq)
    if key_gain:
        block, lo, hi = key_gain
        n_blocks = (Tk + block - 1) // block
        g = lo + (hi - lo) * torch.rand((n_blocks, H), generator=gen, dtype=torch.float32)
        gain = g.repeat_interleave(block, dim=0)[:Tk].unsqueeze(-1)  # (Tk, H, 1)
        out["k"] = (out["k"].to(torch.float32) * gain).to(tdt)
    multi = len(lq) > 1 or varlen or lengths is not None
    if multi:
        out["cu_seqlens_q"] = torch.tensor([0] + lq, dtype=torch.int64).cumsum(0).to(torch.int32)
        out["cu_seqlens_k"] = torch.tensor([0] + lk, dtype=torch.int64).cumsum(0).to(torch.int32)
    else:
        out["cu_seqlens_q"] = None
        out["cu_seqlens_k"] = None
    out["lengths_q"], out["lengths_k"] = lq, lk
    return out


def make_workload(w: Workload | str) -> dict:
    """Inputs of one named workload, by the recipe above."""
    if isinstance(w, str):
        w = WORKLOADS[w]
    return make(dtype=w.dtype, H=w.H, D=w.D, seed=w.seed, n_q=w.n_q or None,
                n_k=w.n_k or None, batch=w.batch, varlen=w.varlen, layout=w.layout,
                backward=w.backward, key_gain=w.key_gain)
