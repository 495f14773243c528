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
    qk_fp8: bool = False      # q and k rounded to float8_e4m3fn (v stays `dtype`)
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
    # fp8 queries and keys: the training workload's forward with q, k in e4m3
    "causal_fp8qk_b4_n8192": Workload(
        "causal_fp8qk_b4_n8192", "bf16", H=32, D=128, causal=True, seed=5, n_q=8192, n_k=8192,
        batch=4, qk_fp8=True,
        note="causal fwd, batch 4 x N=8192, H=32, D=128, q and k e4m3, v bf16"),
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
         key_gain: tuple = (), qk_fp8: bool = False) -> dict:
    """Draw one input set.  Returns CPU tensors and host cu_seqlens.

    Keys: q, k, v, (dO), cu_seqlens_q, cu_seqlens_k (int32, or None for a
    single sequence), lengths_q, lengths_k (python lists).  With qk_fp8, q and
    k are the same N(0, 1) draws rounded to float8_e4m3fn instead of `dtype`.
    """
    gen = torch.Generator().manual_seed(seed)
    tdt = DTYPES[dtype]
    qkdt = torch.float8_e4m3fn if qk_fp8 else tdt
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

    def draw(T, dt=tdt):
        if layout == "hnd":
            return _randn(gen, (H, T, D), dt).permute(1, 0, 2)
        return _randn(gen, (T, H, D), dt)

    out = {"q": draw(Tq, qkdt), "k": draw(Tk, qkdt), "v": draw(Tk)}
    if backward:
        out["dO"] = draw(Tq)
    if key_gain:
        block, lo, hi = key_gain
        n_blocks = (Tk + block - 1) // block
        g = lo + (hi - lo) * torch.rand((n_blocks, H), generator=gen, dtype=torch.float32)
        gain = g.repeat_interleave(block, dim=0)[:Tk].unsqueeze(-1)  # (Tk, H, 1)
        out["k"] = (out["k"].to(torch.float32) * gain).to(qkdt)
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
                backward=w.backward, key_gain=w.key_gain, qk_fp8=w.qk_fp8)


# ---- CSR relations (general sparse attention / segment softmax) ---------------------
#
# Structure only: which (destination, source) edges exist.  The GAT example of
# the TIGA-lang attention page builds a radius graph over random points in the
# unit cube (cutoff 0.15 over 512 points, average degree about 7); the block-
# diagonal (causal) relation of the varlen section can also be written as CSR.


def radius_graph(n: int, cutoff: float, seed: int):
    """Points uniform in [0, 1)^3 (CPU generator `seed`); an edge j -> i for
    every pair with |p_i - p_j| < cutoff, i != j.  Returns (positions (n, 3)
    f32, row_ptr (n + 1) int64 over destinations i, col (E) int32 sources j,
    sorted within each row).  Pairs are found through a grid of cells of side
    >= cutoff (the 27 neighbouring cells of each point's cell); distances are
    compared in f64."""
    gen = torch.Generator().manual_seed(seed)
    pos = torch.rand((n, 3), generator=gen, dtype=torch.float32)
    p = pos.double()
    cells = max(1, int(1.0 / cutoff))
    cid = torch.clamp((p * cells).long(), max=cells - 1)
    key = (cid[:, 0] * cells + cid[:, 1]) * cells + cid[:, 2]
    skey, order = torch.sort(key, stable=True)
    grid = torch.arange(cells ** 3)
    starts = torch.searchsorted(skey, grid, right=False)
    counts = torch.searchsorted(skey, grid, right=True) - starts
    dst_all, src_all = [], []
    for a in (-1, 0, 1):
        for b in (-1, 0, 1):
            for c in (-1, 0, 1):
                nc = cid + torch.tensor([a, b, c])
                ok = ((nc >= 0) & (nc < cells)).all(dim=1)
                i_idx = torch.nonzero(ok).squeeze(1)
                kk = (nc[i_idx, 0] * cells + nc[i_idx, 1]) * cells + nc[i_idx, 2]
                cnt = counts[kk]
                i_rep = torch.repeat_interleave(i_idx, cnt)
                base = starts[kk] - (torch.cumsum(cnt, 0) - cnt)
                j = order[torch.repeat_interleave(base, cnt) + torch.arange(len(i_rep))]
                d2 = ((p[i_rep] - p[j]) ** 2).sum(dim=1)
                keep = (d2 < cutoff * cutoff) & (i_rep != j)
                dst_all.append(i_rep[keep])
                src_all.append(j[keep])
    dst = torch.cat(dst_all)
    src = torch.cat(src_all)
    srt = torch.argsort(dst * n + src)
    dst, src = dst[srt], src[srt]
    row_ptr = torch.cat([torch.zeros(1, dtype=torch.int64),
                         torch.cumsum(torch.bincount(dst, minlength=n), 0)])
    return pos, row_ptr, src.to(torch.int32)


def curve_order(pos: torch.Tensor, cell: float) -> torch.Tensor:
    """A processing order for the rows of a graph over points: the points
    sorted along a Z-order (Morton) curve through cells of side `cell`, ties
    by index.  Rows taken in this order have spatially close neighbours in
    flight together.  Returns an int32 permutation of range(len(pos))."""
    cells = max(1, int(1.0 / cell))
    bits = max(1, (cells - 1).bit_length())
    c = torch.clamp((pos.double() * cells).long(), 0, cells - 1)
    code = torch.zeros(len(pos), dtype=torch.int64)
    for b in range(bits):
        for axis in range(3):
            code |= ((c[:, axis] >> b) & 1) << (3 * b + axis)
    key = code * len(pos) + torch.arange(len(pos), dtype=torch.int64)
    return torch.argsort(key).to(torch.int32)


def csr_of_segments(lengths_q, lengths_k, causal: bool):
    """CSR of the block-diagonal relation of cu_seqlens-packed sequences:
    query i of sequence b has edges to keys of sequence b (j <= i if causal)."""
    rows, cols = [], []
    q0 = k0 = 0
    for lq, lk in zip(lengths_q, lengths_k):
        for i in range(lq):
            n = min(i + 1, lk) if causal else lk
            rows.append(n)
            cols.append(torch.arange(k0, k0 + n, dtype=torch.int32))
        q0 += lq
        k0 += lk
    row_ptr = torch.tensor([0] + rows, dtype=torch.int64).cumsum(0)
    col = torch.cat(cols) if cols else torch.zeros(0, dtype=torch.int32)
    return row_ptr, col


def make_csr(*, row_ptr, col, n_src: int, H: int, D: int, dtype: str, seed: int,
             field_scores: bool, score_std: float = 1.0) -> dict:
    """Tensors for a CSR attention: v (n_src, H, D) always; with field_scores,
    scores (E, H) f32 ~ score_std * N(0, 1); else q (n_dst, H, D) and
    k (n_src, H, D).  Draw order: v, then scores or q, k."""
    gen = torch.Generator().manual_seed(seed)
    tdt = DTYPES[dtype]
    n_dst = len(row_ptr) - 1
    out = {"row_ptr": row_ptr, "col": col, "v": _randn(gen, (n_src, H, D), tdt)}
    if field_scores:
        out["scores"] = score_std * torch.randn((len(col), H), generator=gen, dtype=torch.float32)
        out["q"] = out["k"] = None
    else:
        out["scores"] = None
        out["q"] = _randn(gen, (n_dst, H, D), tdt)
        out["k"] = _randn(gen, (n_src, H, D), tdt)
    return out


@dataclass(frozen=True)
class CsrWorkload:
    name: str
    n: int            # nodes (destination rows = source rows)
    degree: float     # target average degree of the radius graph
    H: int
    D: int
    dtype: str
    field_scores: bool
    seed: int
    note: str = field(default="", compare=False)

    @property
    def cutoff(self) -> float:
        # expected degree of an interior point: n * (4/3) pi r^3
        return (self.degree / (self.n * 4.0 / 3.0 * 3.141592653589793)) ** (1.0 / 3.0)


CSR_WORKLOADS = {
    # the GAT example's scale: 512 points, cutoff 0.15 (average degree ~6-7), 8 features
    "csr_gat_n512": CsrWorkload("csr_gat_n512", 512, 0.0, 1, 8, "f32", True, 0,
                                note="radius graph n=512, cutoff 0.15, field scores, H=1, D=8, f32"),
    "csr_radius_field_bf16": CsrWorkload(
        "csr_radius_field_bf16", 1 << 20, 32.0, 4, 64, "bf16", True, 11,
        note="radius graph n=2^20, average degree ~32, field scores, H=4, D=64, bf16"),
    "csr_radius_dot_bf16": CsrWorkload(
        "csr_radius_dot_bf16", 1 << 20, 32.0, 4, 64, "bf16", False, 12,
        note="radius graph n=2^20, average degree ~32, dot-product scores, H=4, D=64, bf16"),
}


def make_csr_workload(w: CsrWorkload | str) -> dict:
    """Graph and tensors of one named CSR workload (graph seed = w.seed,
    tensors seed = w.seed + 1)."""
    if isinstance(w, str):
        w = CSR_WORKLOADS[w]
    cutoff = 0.15 if w.degree == 0.0 else w.cutoff
    pos, row_ptr, col = radius_graph(w.n, cutoff, w.seed)
    x = make_csr(row_ptr=row_ptr, col=col, n_src=w.n, H=w.H, D=w.D, dtype=w.dtype,
                 seed=w.seed + 1, field_scores=w.field_scores)
    x["row_order"] = curve_order(pos, cutoff)
    return x
