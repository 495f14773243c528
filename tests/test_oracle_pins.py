"""Pins for the f64 oracle, independent of the oracle itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix: hand-derived closed forms (tests/golden/hand_cases.json), invariants of
softmax attention, special cases that reduce to a library routine (torch's
scaled_dot_product_attention and autograd, scipy's logsumexp), and central
finite differences.  Together they fail on a dropped scale, a wrong sign, a
transposed operand, an off-by-one in the causal relation, a wrong log base or a
segment leak.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _ev(x):
    if isinstance(x, str):
        return eval(x, {"__builtins__": {}}, {"log": math.log, "exp": math.exp})  # noqa: S307
    if isinstance(x, list):
        return [_ev(y) for y in x]
    return x


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, causal, scale):
    """torch's own attention in f64 on (T, H, D) numpy arrays, one sequence."""
    Q, K, V = (torch.from_numpy(np.ascontiguousarray(x)).permute(1, 0, 2)[None] for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=causal, scale=scale)
    return out[0].permute(1, 0, 2).numpy()


# --- hand-derived closed forms -------------------------------------------------

def _hand():
    with open(os.path.join(GOLDEN, "hand_cases.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _hand()["cases"], ids=lambda c: c["name"])
def test_hand_cases_forward(case):
    q, k, v = (np.array(_ev(case[n]), dtype=np.float64) for n in ("q", "k", "v"))
    o, lse = oracle.fwd(q, k, v, causal=case["causal"], scale=case["scale"],
                        cu_seqlens_q=case["cu_seqlens"])
    np.testing.assert_allclose(o, np.array(_ev(case["o"])), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(_ev(case["lse"])), rtol=0, atol=1e-13)


@pytest.mark.parametrize("case", _hand()["backward_cases"], ids=lambda c: c["name"])
def test_hand_cases_backward(case):
    q, k, v, dO = (np.array(_ev(case[n]), dtype=np.float64) for n in ("q", "k", "v", "dO"))
    dq, dk, dv = oracle.bwd(q, k, v, dO, causal=case["causal"], scale=case["scale"])
    np.testing.assert_allclose(dq, np.array(_ev(case["dq"])), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk, np.array(_ev(case["dk"])), rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv, np.array(_ev(case["dv"])), rtol=0, atol=1e-13)


# --- closed forms and invariants -----------------------------------------------

def test_zero_scale_is_the_uniform_average():
    """scale = 0 makes every admitted score 0: O_i is the plain mean of the
    admitted values, lse_i = ln |A_i|, dq = dk = 0 and dv_j is the sum of
    dO_i / |A_i| over the rows that admit key j (causal, two segments)."""
    lengths = [5, 3]
    cu = [0, 5, 8]
    H, D = 2, 3
    q, k, v, dO = (_rand((8, H, D), s) for s in (61, 62, 63, 64))
    o, lse = oracle.fwd(q, k, v, causal=True, scale=0.0, cu_seqlens_q=cu)
    dq, dk, dv = oracle.bwd(q, k, v, dO, causal=True, scale=0.0, cu_seqlens_q=cu)
    dv_ref = np.zeros_like(v)
    for b, L in enumerate(lengths):
        s0 = cu[b]
        for i in range(L):
            n = i + 1  # keys 0..i of the segment
            np.testing.assert_allclose(o[s0 + i], v[s0:s0 + n].mean(axis=0), rtol=0, atol=1e-14)
            np.testing.assert_allclose(lse[:, s0 + i], math.log(n), rtol=0, atol=1e-14)
            dv_ref[s0:s0 + n] += dO[s0 + i] / n
    assert not dq.any() and not dk.any()
    np.testing.assert_allclose(dv, dv_ref, rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal", [False, True])
def test_identical_keys_give_mean_of_admitted_values(causal):
    T, H, D = 37, 3, 8
    q = _rand((T, H, D), 1)
    k = np.broadcast_to(_rand((1, H, D), 2), (T, H, D)).copy()
    v = _rand((T, H, D), 3)
    scale = 0.3
    o, lse = oracle.fwd(q, k, v, causal=causal, scale=scale)
    for i in range(T):
        n = i + 1 if causal else T
        np.testing.assert_allclose(o[i], v[:n].mean(axis=0), rtol=0, atol=1e-13)
        s = scale * np.einsum("hd,hd->h", q[i], k[0])
        np.testing.assert_allclose(lse[:, i], s + math.log(n), rtol=0, atol=1e-12)


def test_one_hot_dominant_score_selects_one_value():
    T, H, D = 12, 2, 16
    rng = np.random.default_rng(4)
    k = np.zeros((T, H, D))
    for j in range(T):
        k[j, :, j] = 1.0  # orthonormal keys
    target = rng.integers(0, T, size=(T, H))
    c = 40.0
    q = np.zeros((T, H, D))
    for i in range(T):
        for h in range(H):
            q[i, h, target[i, h]] = c
    v = rng.standard_normal((T, H, D))
    o, lse = oracle.fwd(q, k, v, causal=False, scale=1.0)
    # all other weights are exp(-c) relative to the selected one
    bound = (T - 1) * math.exp(-c) * 2 * np.abs(v).max()
    for i in range(T):
        for h in range(H):
            np.testing.assert_allclose(o[i, h], v[target[i, h], h], rtol=0, atol=bound + 1e-15)
            np.testing.assert_allclose(lse[h, i], c + math.log1p((T - 1) * math.exp(-c)),
                                       rtol=0, atol=1e-12)


def test_per_row_constant_shift():
    """Adding c_i to every score of row i leaves O unchanged and shifts lse by c_i.

    The shift is made with one extra dimension: k[:, D] = 1, q[i, D] = c_i / scale.
    """
    T, H, D = 29, 2, 6
    q, k, v = _rand((T, H, D), 5), _rand((T, H, D), 6), _rand((T, H, D), 7)
    scale = D ** -0.5
    c = 50.0 * _rand((T, H), 8)
    q2 = np.concatenate([q, (c / scale)[..., None]], axis=2)
    k2 = np.concatenate([k, np.ones((T, H, 1))], axis=2)
    v2 = np.concatenate([v, np.zeros((T, H, 1))], axis=2)
    for causal in (False, True):
        o, lse = oracle.fwd(q, k, v, causal=causal, scale=scale)
        o2, lse2 = oracle.fwd(q2, k2, v2, causal=causal, scale=scale)
        np.testing.assert_allclose(o2[..., :D], o, rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse2, lse + c.T, rtol=0, atol=1e-11)


def test_joint_key_value_permutation_full_relation():
    T, H, D = 41, 3, 5
    q, k, v = _rand((T, H, D), 9), _rand((T, H, D), 10), _rand((T, H, D), 11)
    perm = np.random.default_rng(12).permutation(T)
    o, lse = oracle.fwd(q, k, v, causal=False)
    o2, lse2 = oracle.fwd(q, k[perm], v[perm], causal=False)
    np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


def test_causal_first_row_is_first_value_exactly():
    T, H, D = 17, 2, 4
    q, k, v = _rand((T, H, D), 13), _rand((T, H, D), 14), _rand((T, H, D), 15)
    o, lse = oracle.fwd(q, k, v, causal=True, scale=0.7)
    np.testing.assert_array_equal(o[0], v[0])
    for h in range(H):
        acc = 0.0
        for d in range(D):  # in index order, as a plain loop sums
            acc += float(q[0, h, d]) * float(k[0, h, d])
        assert lse[h, 0] == 0.7 * acc  # m + ln(1) with the single admitted score


def test_varlen_equals_concatenation_of_independent_sequences():
    lengths = [5, 1, 9, 1, 13]  # includes length-1 sequences
    T, H, D = sum(lengths), 2, 4
    q, k, v = _rand((T, H, D), 16), _rand((T, H, D), 17), _rand((T, H, D), 18)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o, lse = oracle.fwd(q, k, v, causal=True, cu_seqlens_q=cu)
    for b in range(len(lengths)):
        a, e = cu[b], cu[b + 1]
        ob, lb = oracle.fwd(q[a:e], k[a:e], v[a:e], causal=True)
        np.testing.assert_array_equal(o[a:e], ob)
        np.testing.assert_array_equal(lse[:, a:e], lb)
    # and length-1 sequences return their own value row
    np.testing.assert_array_equal(o[5], v[5])


def test_large_scores_are_stable_and_match_library_logsumexp():
    from scipy.special import logsumexp, softmax
    T, H, D = 23, 2, 8
    q, k, v = _rand((T, H, D), 19), _rand((T, H, D), 20), _rand((T, H, D), 21)
    scale = 100.0 * D ** -0.5
    o, lse = oracle.fwd(q, k, v, causal=False, scale=scale)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    for h in range(H):
        s = scale * q[:, h] @ k[:, h].T
        np.testing.assert_allclose(lse[h], logsumexp(s, axis=1), rtol=1e-14, atol=1e-11)
        np.testing.assert_allclose(o[:, h], softmax(s, axis=1) @ v[:, h], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("T,D", [(1, 4), (7, 3), (64, 16), (130, 32)])
def test_matches_torch_sdpa_f64(causal, T, D):
    H = 3
    q, k, v = _rand((T, H, D), 22), _rand((T, H, D), 23), _rand((T, H, D), 24)
    o, lse = oracle.fwd(q, k, v, causal=causal)
    np.testing.assert_allclose(o, _sdpa(q, k, v, causal, D ** -0.5), rtol=0, atol=1e-12)


def test_cross_attention_matches_torch_sdpa_f64():
    Tq, Tk, H, D = 19, 7, 2, 8
    q, k, v = _rand((Tq, H, D), 25), _rand((Tk, H, D), 26), _rand((Tk, H, D), 27)
    o, _ = oracle.fwd(q, k, v, causal=False)
    np.testing.assert_allclose(o, _sdpa(q, k, v, False, D ** -0.5), rtol=0, atol=1e-12)


def test_causal_rejects_unequal_lengths():
    q, k = _rand((5, 1, 2), 0), _rand((4, 1, 2), 1)
    with pytest.raises(ValueError):
        oracle.fwd(q, k, k, causal=True)


def test_sampled_rows_equal_full_forward():
    lengths = [37, 1, 140]
    T, H, D = sum(lengths), 3, 8
    q, k, v = _rand((T, H, D), 28), _rand((T, H, D), 29), _rand((T, H, D), 30)
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    o, lse = oracle.fwd(q, k, v, causal=True, cu_seqlens_q=cu)
    tokens = np.array([0, 36, 37, 38, 177, 100])
    heads = np.array([0, 2, 1, 0, 2, 1])
    orow, lrow = oracle.fwd_rows(q, k, v, tokens, heads, causal=True, cu_seqlens_q=cu)
    np.testing.assert_array_equal(orow, o[tokens, heads])
    np.testing.assert_array_equal(lrow, lse[heads, tokens])


# --- backward ------------------------------------------------------------------

def _loss(q, k, v, dO, causal, scale, cu=None):
    o, _ = oracle.fwd(q, k, v, causal=causal, scale=scale, cu_seqlens_q=cu)
    return float(np.sum(o * dO))


@pytest.mark.parametrize("causal", [False, True])
def test_backward_central_finite_differences(causal):
    T, H, D = 6, 1, 4
    q, k, v, dO = (_rand((T, H, D), s) for s in (31, 32, 33, 34))
    scale = 0.6
    dq, dk, dv = oracle.bwd(q, k, v, dO, causal=causal, scale=scale)
    h = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        for idx in np.ndindex(x.shape):
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            args[name] = xp
            lp = _loss(args["q"], args["k"], args["v"], dO, causal, scale)
            args[name] = xm
            lm = _loss(args["q"], args["k"], args["v"], dO, causal, scale)
            num[idx] = (lp - lm) / (2 * h)
        rel = np.linalg.norm(num - g) / np.linalg.norm(g)
        assert rel <= 1e-7, (name, rel)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_torch_autograd_f64(causal):
    T, H, D = 45, 2, 8
    q, k, v, dO = (_rand((T, H, D), s) for s in (35, 36, 37, 38))
    dq, dk, dv = oracle.bwd(q, k, v, dO, causal=causal)
    Q, K, V = (torch.from_numpy(x).permute(1, 0, 2)[None].clone().requires_grad_() for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=causal)
    out.backward(torch.from_numpy(dO).permute(1, 0, 2)[None])
    for g, t in ((dq, Q), (dk, K), (dv, V)):
        np.testing.assert_allclose(g, t.grad[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_backward_varlen_equals_per_sequence():
    lengths = [4, 1, 11]
    T, H, D = sum(lengths), 2, 4
    q, k, v, dO = (_rand((T, H, D), s) for s in (39, 40, 41, 42))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    dq, dk, dv = oracle.bwd(q, k, v, dO, causal=True, cu_seqlens_q=cu)
    for b in range(len(lengths)):
        a, e = cu[b], cu[b + 1]
        gq, gk, gv = oracle.bwd(q[a:e], k[a:e], v[a:e], dO[a:e], causal=True)
        np.testing.assert_allclose(dq[a:e], gq, rtol=0, atol=1e-14)
        np.testing.assert_allclose(dk[a:e], gk, rtol=0, atol=1e-14)
        np.testing.assert_allclose(dv[a:e], gv, rtol=0, atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_row_dot_identity(causal):
    """sum_j P_ij dP_ij equals <dO_i, O_i> (the per-row D of the OCANNL page's
    fused backward): dq rebuilt from that shortcut equals the oracle's dq."""
    from scipy.special import softmax
    T, H, D = 21, 2, 6
    q, k, v, dO = (_rand((T, H, D), s) for s in (43, 44, 45, 46))
    scale = D ** -0.5
    o, _ = oracle.fwd(q, k, v, causal=causal)
    dq, _, _ = oracle.bwd(q, k, v, dO, causal=causal)
    for h in range(H):
        s = scale * q[:, h] @ k[:, h].T
        if causal:
            s = np.where(np.tril(np.ones((T, T), dtype=bool)), s, -np.inf)
        p = softmax(s, axis=1)
        dp = dO[:, h] @ v[:, h].T
        Drow = np.einsum("id,id->i", dO[:, h], o[:, h])
        ds = p * (dp - Drow[:, None])
        np.testing.assert_allclose(dq[:, h], scale * ds @ k[:, h], rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_sum_invariants(causal):
    """Softmax is invariant to a common shift of all keys, so sum_j dk_j = 0;
    the probabilities of a row sum to 1, so sum_j dv_j = sum_i dO_i."""
    T, H, D = 33, 3, 5
    q, k, v, dO = (_rand((T, H, D), s) for s in (47, 48, 49, 50))
    dq, dk, dv = oracle.bwd(q, k, v, dO, causal=causal)
    np.testing.assert_allclose(dk.sum(axis=0), 0.0, atol=1e-12)
    np.testing.assert_allclose(dv.sum(axis=0), dO.sum(axis=0), atol=1e-12)


def test_backward_sampled_rows_equal_full():
    lengths = [19, 1, 30]
    T, H, D = sum(lengths), 2, 4
    q, k, v, dO = (_rand((T, H, D), s) for s in (51, 52, 53, 54))
    cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    dq, dk, dv = oracle.bwd(q, k, v, dO, causal=True, cu_seqlens_q=cu)
    rows = (np.array([0, 18, 19, 49, 25]), np.array([1, 0, 1, 1, 0]))
    keys = (np.array([0, 19, 20, 49, 3]), np.array([0, 1, 0, 1, 1]))
    sq, sk, sv = oracle.bwd(q, k, v, dO, causal=True, cu_seqlens_q=cu, q_rows=rows, k_rows=keys)
    np.testing.assert_array_equal(sq, dq[rows[0], rows[1]])
    np.testing.assert_array_equal(sk, dk[keys[0], keys[1]])
    np.testing.assert_array_equal(sv, dv[keys[0], keys[1]])


# --- merge of partial results over disjoint key sets (split-K) -------------------

def _ev_inf(x):
    if x == "-inf":
        return -math.inf
    if isinstance(x, list):
        return [_ev_inf(y) for y in x]
    return _ev(x)


def _merge_cases():
    with open(os.path.join(GOLDEN, "merge_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _merge_cases(), ids=lambda c: c["name"])
def test_merge_hand_cases(case):
    op, lp = (np.array(_ev_inf(case[n]), dtype=np.float64) for n in ("o_parts", "lse_parts"))
    o, lse = oracle.merge(op, lp)
    np.testing.assert_allclose(o, np.array(_ev_inf(case["o"])), rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(np.array(_ev_inf(case["lse"]))))
    fin = np.isfinite(lse)
    np.testing.assert_allclose(lse[fin], np.array(_ev_inf(case["lse"]))[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("bounds", [(0, 40, 41, 97), (0, 1, 97), (0, 13, 26, 50, 77, 90, 97), (0, 97)])
def test_merge_of_key_chunks_equals_attention_over_all_keys(bounds):
    """Attention over keys split into disjoint chunks, each chunk attended on
    its own and then merged, is attention over all keys (full relation)."""
    q, k, v = _rand((23, 3, 16), 71), _rand((97, 3, 16), 72), _rand((97, 3, 16), 73)
    parts = [oracle.fwd(q, k[a:b], v[a:b], causal=False, scale=0.3)
             for a, b in zip(bounds[:-1], bounds[1:])]
    o, lse = oracle.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    o_ref, lse_ref = oracle.fwd(q, k, v, causal=False, scale=0.3)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


def test_merge_with_an_empty_key_chunk():
    """A chunk with no key (lse = -inf, O = 0 from the forward) changes nothing."""
    q, k, v = _rand((9, 2, 8), 74), _rand((30, 2, 8), 75), _rand((30, 2, 8), 76)
    a = oracle.fwd(q, k[:0], v[:0], causal=False)
    b = oracle.fwd(q, k, v, causal=False)
    assert np.all(np.isneginf(a[1])) and not np.any(a[0])
    o, lse = oracle.merge(np.stack([a[0], b[0]]), np.stack([a[1], b[1]]))
    np.testing.assert_array_equal(o, b[0])
    np.testing.assert_array_equal(lse, b[1])


def test_merge_is_invariant_to_part_order():
    rng = np.random.default_rng(77)
    op, lp = rng.standard_normal((5, 11, 2, 8)), 3 * rng.standard_normal((5, 2, 11))
    perm = [3, 0, 4, 2, 1]
    o1, l1 = oracle.merge(op, lp)
    o2, l2 = oracle.merge(op[perm], lp[perm])
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(l1, l2, rtol=0, atol=1e-13)


def test_merge_large_lse_is_stable_and_matches_library_logsumexp():
    from scipy.special import logsumexp, softmax
    rng = np.random.default_rng(78)
    op = rng.standard_normal((4, 6, 1, 8))
    lp = 2000.0 * rng.standard_normal((4, 1, 6))
    o, lse = oracle.merge(op, lp)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
    np.testing.assert_allclose(lse, logsumexp(lp, axis=0), rtol=1e-15, atol=1e-12)
    w = softmax(lp[:, 0, :], axis=0)  # (C, T)
    np.testing.assert_allclose(o[:, 0, :], np.einsum("ct,ctd->td", w, op[:, :, 0, :]), rtol=0,
                               atol=1e-12)


# --- tile-pruned approximate forward ----------------------------------------------

def _prune_cases():
    with open(os.path.join(GOLDEN, "tile_prune_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _prune_cases(), ids=lambda c: c["name"])
def test_pruned_hand_cases(case):
    q, k, v = (np.array(_ev(case[n]), dtype=np.float64) for n in ("q", "k", "v"))
    o, lse, n_pruned, _ = oracle.fwd_pruned(q, k, v, rho=case["rho"], block_q=case["block_q"],
                                            block_k=case["block_k"], scale=1.0)
    assert n_pruned == case["n_pruned"]
    np.testing.assert_allclose(o, np.array(_ev(case["o"])), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.array(_ev(case["lse"])), rtol=0, atol=1e-13)


def test_pruned_page_worked_value():
    """The page prints exp(1 - 10) ~ 0.00012 for a block whose best score is 1
    after a seen maximum of 10, skipped under threshold 0.01."""
    with open(os.path.join(GOLDEN, "tile_prune_worked_example.json")) as f:
        g = json.load(f)
    ratio = math.exp(g["tile_max"] - g["seen_max"])
    assert float(f"{ratio:.{g['printed_digits']}g}") == g["printed_ratio"]
    # the rule in log form: skipped iff m_tile < m_run + ln(rho), i.e. ratio < rho
    assert (ratio < g["threshold"]) == g["skipped"]
    q = np.ones((1, 1, 1))
    k = np.array([g["seen_max"], g["tile_max"]]).reshape(2, 1, 1)
    _, _, n_pruned, margin = oracle.fwd_pruned(q, k, np.ones((2, 1, 1)), rho=g["threshold"],
                                               block_q=1, block_k=1, scale=1.0)
    assert n_pruned == int(g["skipped"])
    assert margin == pytest.approx(abs(g["tile_max"] - g["seen_max"] - math.log(g["threshold"])))


@pytest.mark.parametrize("bq,bk", [(16, 16), (64, 64), (128, 128), (7, 33)])
def test_pruned_with_negligible_rho_is_exact_attention(bq, bk):
    q, k, v = _rand((150, 2, 16), 81), _rand((230, 2, 16), 82), _rand((230, 2, 16), 83)
    o, lse, n_pruned, _ = oracle.fwd_pruned(q, k, v, rho=1e-300, block_q=bq, block_k=bk)
    o_ref, lse_ref = oracle.fwd(q, k, v, causal=False)
    assert n_pruned == 0
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-13)


def test_pruned_cold_tile_is_dropped_from_every_block():
    """Keys of one tile set to zero (all its scores 0) among tiles of large
    scores: every query block prunes exactly that tile, and the result is exact
    attention over the remaining keys."""
    bq, bk, Tq, Tk, H, D = 32, 16, 100, 80, 2, 8
    q = _rand((Tq, H, D), 84)
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = 10.0 * q[np.random.default_rng(85).integers(0, Tq, Tk)]  # scores up to 10
    k[32:48] = 0.0                                               # the cold tile (tile 2)
    v = _rand((Tk, H, D), 86)
    scale = 1.0
    o, lse, n_pruned, margin = oracle.fwd_pruned(q, k, v, rho=0.01, block_q=bq, block_k=bk,
                                                 scale=scale)
    keep = np.r_[0:32, 48:80]
    o_ref, lse_ref = oracle.fwd(q, k[keep], v[keep], causal=False, scale=scale)
    assert n_pruned == H * ((Tq + bq - 1) // bq)
    assert margin > 0.5
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, lse_ref, rtol=0, atol=1e-12)


def test_pruned_rejects_rho_outside_unit_interval():
    q = np.zeros((2, 1, 4))
    for rho in (0.0, -0.5, 1.5, float("nan")):
        with pytest.raises(ValueError):
            oracle.fwd_pruned(q, q, q, rho=rho, block_q=2, block_k=2)


# --- attention over a general CSR relation -------------------------------------------

def _csr_cases():
    with open(os.path.join(GOLDEN, "csr_cases.json")) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", _csr_cases(), ids=lambda c: c["name"])
def test_csr_hand_cases(case):
    v = np.array(_ev_inf(case["v"]), dtype=np.float64)
    sc = np.array(_ev_inf(case["scores"]), dtype=np.float64)
    o, lse = oracle.csr_fwd(case["row_ptr"], case["col"], v, scores=sc)
    np.testing.assert_allclose(o, np.array(_ev_inf(case["o"])), rtol=0, atol=1e-13)
    ref = np.array(_ev_inf(case["lse"]))
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(ref))
    np.testing.assert_allclose(lse[np.isfinite(ref)], ref[np.isfinite(ref)], rtol=0, atol=1e-13)


@pytest.mark.parametrize("causal,lengths_q,lengths_k", [
    (True, [384, 1, 96, 640, 57], None),   # the varlen example's lengths
    (False, [100, 3, 257], [31, 300, 128]),
    (True, [0, 5, 0, 70], None),
])
def test_csr_of_segment_relations_equals_dense_attention(causal, lengths_q, lengths_k):
    """The block-diagonal (causal) relation written as CSR gives the same
    attention as the cu_seqlens form."""
    import attn_inputs
    lk = lengths_k or lengths_q
    x = attn_inputs.make(dtype="f32", H=2, D=16, seed=90, lengths=lengths_q, lengths_k=lk)
    row_ptr, col = attn_inputs.csr_of_segments(lengths_q, lk, causal)
    o, lse = oracle.csr_fwd(row_ptr, col, x["v"], q=x["q"], k=x["k"], scale=0.3)
    o_ref, lse_ref = oracle.fwd(x["q"], x["k"], x["v"], causal=causal, scale=0.3,
                                cu_seqlens_q=x["cu_seqlens_q"], cu_seqlens_k=x["cu_seqlens_k"])
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-13)
    np.testing.assert_array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=0, atol=1e-13)


def test_csr_field_scores_equal_dot_scores_given_as_a_field():
    import attn_inputs
    _, row_ptr, col = attn_inputs.radius_graph(300, 0.2, seed=91)
    x = attn_inputs.make_csr(row_ptr=row_ptr, col=col, n_src=300, H=3, D=8, dtype="f32", seed=92,
                             field_scores=False)
    q, k = x["q"].double().numpy(), x["k"].double().numpy()
    dst = np.repeat(np.arange(300), np.diff(row_ptr.numpy()))
    sc = 0.5 * np.einsum("ehd,ehd->eh", q[dst], k[col.numpy()])
    a = oracle.csr_fwd(row_ptr, col, x["v"], scores=sc)
    b = oracle.csr_fwd(row_ptr, col, x["v"], q=x["q"], k=x["k"], scale=0.5)
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-12)


def test_csr_edge_order_within_a_row_does_not_matter():
    import attn_inputs
    _, row_ptr, col = attn_inputs.radius_graph(200, 0.25, seed=93)
    x = attn_inputs.make_csr(row_ptr=row_ptr, col=col, n_src=200, H=2, D=4, dtype="f32", seed=94,
                             field_scores=True)
    rng = np.random.default_rng(95)
    perm = np.concatenate([a + rng.permutation(b - a) for a, b in
                           zip(row_ptr[:-1].tolist(), row_ptr[1:].tolist())]).astype(np.int64)
    a = oracle.csr_fwd(row_ptr, col, x["v"], scores=x["scores"])
    b = oracle.csr_fwd(row_ptr, col.numpy()[perm], x["v"], scores=x["scores"].numpy()[perm])
    np.testing.assert_allclose(a[0], b[0], rtol=0, atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], rtol=0, atol=1e-13)


def test_csr_rejects_malformed_relations():
    v = np.zeros((2, 1, 4))
    sc = np.zeros((2, 1))
    with pytest.raises(ValueError):
        oracle.csr_fwd([0, 2], [0, 2], v, scores=sc)    # source out of range
    with pytest.raises(ValueError):
        oracle.csr_fwd([0, 2, 1], [0, 1], v, scores=sc)  # decreasing offsets
    with pytest.raises(ValueError):
        oracle.csr_fwd([1, 2], [0, 1], v, scores=sc)     # not starting at 0


def test_radius_graph_matches_brute_force():
    """The input generator's cell search finds exactly the pairs closer than the cutoff."""
    import attn_inputs
    pos, row_ptr, col = attn_inputs.radius_graph(512, 0.15, seed=0)
    p = pos.double().numpy()
    d2 = ((p[:, None, :] - p[None, :, :]) ** 2).sum(-1)
    adj = (d2 < 0.15 ** 2) & ~np.eye(512, dtype=bool)
    for i in range(512):
        np.testing.assert_array_equal(col[row_ptr[i]:row_ptr[i + 1]].numpy(), np.nonzero(adj[i])[0])
