"""Tolerances and comparison helpers shared by the GPU parity tests.

Tolerances (per output element; rel-RMS = ||x - ref||_2 / ||ref||_2 over the
compared set):
  O, f16/bf16 inputs, stored f32 or f16:  max|err| <= 1e-2, rel-RMS <= 2e-3
  O, bf16 inputs, stored bf16:            max|err| <= 1e-2, rel-RMS <= 4e-3
      (storing O in bf16 alone costs about 1.6e-3 rel-RMS -- round to nearest
      with 8 significant bits -- on top of the 2e-3 arithmetic budget)
  O, f32:                                 max|err| <= 1e-5
  lse:                                    max|err| <= 1e-3
  dq, dk, dv:                             rel-RMS <= 5e-3
"""
from __future__ import annotations

import numpy as np
import torch


def rel_rms(x: np.ndarray, ref: np.ndarray) -> float:
    den = float(np.sqrt((ref ** 2).sum()))
    num = float(np.sqrt(((x - ref) ** 2).sum()))
    return num / den if den > 0 else num


def f64(t) -> np.ndarray:
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu", torch.float64).numpy()


def o_bounds(in_dtype: torch.dtype, out_dtype: torch.dtype):
    if in_dtype == torch.float32:
        return 1e-5, None
    if out_dtype == torch.bfloat16:
        return 1e-2, 4e-3
    return 1e-2, 2e-3


def check_o(o, o_ref, in_dtype, out_dtype, what="O"):
    o = f64(o)
    amax, rrms = o_bounds(in_dtype, out_dtype)
    err = np.abs(o - o_ref).max() if o.size else 0.0
    assert np.isfinite(o).all(), f"{what}: non-finite values"
    assert err <= amax, f"{what}: max|err| {err:.3e} > {amax:.1e}"
    if rrms is not None and o.size:
        r = rel_rms(o, o_ref)
        assert r <= rrms, f"{what}: rel-RMS {r:.3e} > {rrms:.1e}"


def check_lse(lse, lse_ref, what="lse"):
    lse = f64(lse)
    fin = np.isfinite(lse_ref)
    assert (np.isfinite(lse) == fin).all(), f"{what}: finiteness differs"
    assert (lse[~fin] == lse_ref[~fin]).all(), f"{what}: -inf rows differ"
    if fin.any():
        err = np.abs(lse[fin] - lse_ref[fin]).max()
        assert err <= 1e-3, f"{what}: max|err| {err:.3e} > 1e-3"


def check_grad(g, g_ref, what):
    g = f64(g)
    assert np.isfinite(g).all(), f"{what}: non-finite values"
    r = rel_rms(g, g_ref)
    assert r <= 5e-3, f"{what}: rel-RMS {r:.3e} > 5e-3"


def sample_rows(lengths, H, n_random, seed, extra_offsets=(0, 1, 63, 64, 127, 128, 129, 255, 256)):
    """(token, head) pairs: segment ends, tile edges and random rows."""
    rng = np.random.default_rng(seed)
    cu = np.concatenate([[0], np.cumsum(lengths)])
    toks, heads = [], []
    for b, L in enumerate(lengths):
        if L == 0:
            continue
        offs = {o for o in extra_offsets if o < L} | {L - 1, L - 2 if L > 1 else 0}
        for o in sorted(offs):
            toks.append(cu[b] + o)
            heads.append(int(rng.integers(0, H)))
    total = int(cu[-1])
    toks += list(rng.integers(0, total, n_random))
    heads += list(rng.integers(0, H, n_random))
    return np.array(toks, dtype=np.int64), np.array(heads, dtype=np.int32)
