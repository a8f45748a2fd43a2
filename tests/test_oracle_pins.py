"""Pins for the fp64 oracle: values the pages print, closed forms, invariants,
library routines it must reduce to, and planted mistakes the pins must catch.

Nothing here calls the GPU library; these run on any CPU.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from exact_io_aware_30_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(x, printed, digits, slack=0.0):
    """x agrees with a value printed to `digits` decimals.

    ``slack`` allows for a hand trace that rounded its intermediates before
    combining them (the page's 6.6164 is 0.4698 + 6.1465 from 4-5 digit
    factors; the exact value is 6.61634).
    """
    return abs(float(x) - float(printed)) <= 0.5 * 10.0 ** (-digits) + slack + 1e-12


HAND = 1e-4  # rounding slack of the hand-traced intermediates


def _rand(rng, *shape):
    return rng.standard_normal(shape)


# ---------------------------------------------------------------------------
# 1. The pages' worked examples
# ---------------------------------------------------------------------------

def check_worked_example(orc):
    g = _load("worked_example.json")
    q = np.array(g["q"])
    K = np.array(g["K"])
    V = np.array(g["V"])
    tr = orc.online_trace(q, K, V, g["scale"], g["block_size"])
    for t, ref in enumerate(g["after_tile"]):
        assert _close(tr["m"][t], ref["m"], 6)
        assert _close(tr["l"][t], ref["l"], ref["l_digits"])
        for c in range(2):
            assert _close(tr["o_unnorm"][t][c], ref["o_unnorm"][c], ref["o_digits"], HAND)
    # the correction factor applied at tile 2 and tile 2's weights
    corr = math.exp(tr["m"][0] - tr["m"][1])
    assert _close(corr, g["correction_tile2"], g["correction_digits"])
    for c in range(2):
        assert _close(tr["o"][c], g["output"][c], g["output_digits"])
    # direct softmax probabilities of the naive form
    P = orc.probs(q[None, :], K, g["scale"])
    for j in range(4):
        assert _close(P[0, j], g["probs"][j], g["probs_digits"])
    assert abs(P.sum() - 1.0) < 1e-14
    # tile-2 unnormalised weights exp(s - m) = P * l
    for jj, j in enumerate((2, 3)):
        assert _close(P[0, j] * tr["l"][-1], g["tile2_p"][jj], g["tile2_p_digits"])
    # naive form on the same data, via the [B,H,S,d] entry point
    o, lse = orc.attention(q[None, None, None, :], K[None, None], V[None, None], g["scale"])
    for c in range(2):
        assert _close(o[0, 0, 0, c], g["output"][c], g["output_digits"])
    # lse = m + ln l with the printed l (derived, not printed)
    assert abs(lse[0, 0, 0] - (3.0 + math.log(g["after_tile"][1]["l"]))) < 1e-5
    # one block of four keys (the block_size = 4 question)
    b4 = g["block4"]
    tr4 = orc.online_trace(q, K, V, g["scale"], 4)
    assert _close(tr4["l"][0], b4["l"], b4["l_digits"])
    for j in range(4):
        assert _close(P[0, j] * tr4["l"][0], b4["p_unnorm"][j], b4["p_digits"])
    for c in range(2):
        assert _close(tr4["o"][c], b4["output"][c], b4["output_digits"])


def test_worked_example_trace():
    check_worked_example(oracle.default())


def check_online_softmax_1d(orc):
    g = _load("online_softmax_1d.json")
    s = np.array(g["scores"])
    # scores s_j = q . k_j with q = [1,0,0,0] and k_j = [s_j,0,0,0] (zero
    # padding leaves the scores unchanged); values are one-hot rows
    q = np.array([1.0, 0.0, 0.0, 0.0])
    K = np.zeros((4, 4))
    K[:, 0] = s
    V = np.eye(4)
    tr = orc.online_trace(q, K, V, 1.0, g["block_size"])
    dg = g["digits"]
    assert _close(tr["m"][0], g["block1_max"], dg)
    assert _close(tr["l"][0], g["block1_sum"], dg)
    assert _close(math.exp(tr["m"][0] - tr["m"][1]), g["rescale"], dg)
    # printed as 0.135 x 1.135 ~ 0.153 from the rounded factors (exact 0.15365)
    assert _close(math.exp(tr["m"][0] - tr["m"][1]) * tr["l"][0], g["rescaled_block1_sum"], dg,
                  1e-3)
    assert _close(tr["m"][1], g["final_max"], dg)
    assert _close(tr["l"][1], g["direct_denominator"], dg)
    # the output with one-hot values is the probability vector itself
    assert abs(tr["o"].sum() - 1.0) < 1e-14
    assert np.argmax(tr["o"]) == 3


def test_online_softmax_1d_example():
    check_online_softmax_1d(oracle.default())


# ---------------------------------------------------------------------------
# 2. Reductions to library routines (scipy softmax / logsumexp, torch SDPA)
# ---------------------------------------------------------------------------

def _window_bool(Sq, Sk, W):
    i = np.arange(Sq)[:, None]
    j = np.arange(Sk)[None, :]
    return (j <= i) & (j > i - W)


def check_library_reduction(orc, rng):
    sp = pytest.importorskip("scipy.special")
    for (B, H, Sq, Sk, d) in [(1, 2, 7, 7, 5), (2, 1, 5, 9, 3), (1, 1, 13, 6, 8)]:
        q, k, v = _rand(rng, B, H, Sq, d), _rand(rng, B, H, Sk, d), _rand(rng, B, H, Sk, d)
        scale = 0.37
        S = scale * np.einsum("bhid,bhjd->bhij", q, k)
        ref_o = sp.softmax(S, axis=-1) @ v
        ref_lse = sp.logsumexp(S, axis=-1)
        o, lse = orc.attention(q, k, v, scale, "none")
        np.testing.assert_allclose(o, ref_o, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, ref_lse, rtol=1e-12, atol=1e-13)


def test_reduces_to_scipy_softmax_no_mask():
    check_library_reduction(oracle.default(), np.random.default_rng(1))


def check_torch_sdpa(orc, rng):
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for (Sq, Sk, d, W) in [(9, 9, 4, 3), (6, 11, 3, 1), (12, 5, 2, 4)]:
        q, k, v = _rand(rng, 1, 2, Sq, d), _rand(rng, 1, 2, Sk, d), _rand(rng, 1, 2, Sk, d)
        scale = 1.0 / math.sqrt(d)
        tq, tk, tv = (torch.from_numpy(x) for x in (q, k, v))
        # causal: torch's is_causal is the top-left aligned lower triangle
        ref = F.scaled_dot_product_attention(tq, tk, tv, is_causal=True, scale=scale).numpy()
        o, _ = orc.attention(q, k, v, scale, "causal")
        rows_ok = np.arange(Sq) < Sk  # torch leaves no row empty with Sq <= Sk
        np.testing.assert_allclose(o[:, :, rows_ok], ref[:, :, rows_ok], rtol=1e-12, atol=1e-12)
        # sliding window: the same boolean band handed to torch explicitly
        band = _window_bool(Sq, Sk, W)
        full = band.any(axis=1)
        ref_w = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=torch.from_numpy(band),
                                               scale=scale).numpy()
        o_w, lse_w = orc.attention(q, k, v, scale, "window", W)
        np.testing.assert_allclose(o_w[:, :, full], ref_w[:, :, full], rtol=1e-12, atol=1e-12)
        # rows that see no key: guarded to zero output and -inf lse
        assert np.all(o_w[:, :, ~full] == 0.0)
        assert np.all(np.isneginf(lse_w[:, :, ~full]))


def test_matches_torch_sdpa_causal_and_window():
    check_torch_sdpa(oracle.default(), np.random.default_rng(2))


# ---------------------------------------------------------------------------
# 3. Closed forms and special cases
# ---------------------------------------------------------------------------

def check_closed_forms(orc, rng):
    d = 6
    # one key: O = v0, lse = scale * q . k0
    q, k, v = _rand(rng, 1, 1, 4, d), _rand(rng, 1, 1, 1, d), _rand(rng, 1, 1, 1, d)
    o, lse = orc.attention(q, k, v, 0.5, "none")
    np.testing.assert_allclose(o[0, 0], np.repeat(v[0, 0], 4, axis=0), rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], 0.5 * q[0, 0] @ k[0, 0, 0], rtol=1e-14)
    # identical keys under a causal mask: row i averages v_0..v_i, lse = s + ln(i+1)
    Sq = 7
    q = _rand(rng, 1, 1, Sq, d)
    k = np.repeat(_rand(rng, 1, 1, 1, d), Sq, axis=2)
    v = _rand(rng, 1, 1, Sq, d)
    o, lse = orc.attention(q, k, v, 0.3, "causal")
    for i in range(Sq):
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :i + 1].mean(axis=0), rtol=1e-13, atol=1e-14)
        s = 0.3 * q[0, 0, i] @ k[0, 0, 0]
        assert abs(lse[0, 0, i] - (s + math.log(i + 1))) < 1e-12
    # scale = 0: every visible key has the same weight
    q, k, v = _rand(rng, 1, 1, 5, d), _rand(rng, 1, 1, 8, d), _rand(rng, 1, 1, 8, d)
    o, lse = orc.attention(q, k, v, 0.0, "none")
    np.testing.assert_allclose(o[0, 0], np.tile(v[0, 0].mean(axis=0), (5, 1)), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(8), rtol=1e-14)
    # causal row 0 sees only key 0
    q, k, v = _rand(rng, 1, 1, 6, d), _rand(rng, 1, 1, 6, d), _rand(rng, 1, 1, 6, d)
    o, _ = orc.attention(q, k, v, 0.4, "causal")
    assert np.array_equal(o[0, 0, 0], v[0, 0, 0])
    # window of one key: O_i = v_i exactly, lse_i = scale q_i . k_i
    o, lse = orc.attention(q, k, v, 0.4, "window", 1)
    assert np.array_equal(o[0, 0], v[0, 0])
    np.testing.assert_allclose(lse[0, 0], 0.4 * np.einsum("id,id->i", q[0, 0], k[0, 0]), rtol=1e-14)
    # a window at least as wide as the sequence is the causal mask
    o_c, lse_c = orc.attention(q, k, v, 0.4, "causal")
    o_w, lse_w = orc.attention(q, k, v, 0.4, "window", 6)
    assert np.array_equal(o_c, o_w) and np.array_equal(lse_c, lse_w)
    # one dominant key: the output is (almost exactly) that key's value row
    q = np.ones((1, 1, 3, d))
    k = np.zeros((1, 1, 5, d))
    k[0, 0, 2] = 40.0
    v = _rand(rng, 1, 1, 5, d)
    o, _ = orc.attention(q, k, v, 1.0, "none")
    np.testing.assert_allclose(o[0, 0], np.tile(v[0, 0, 2], (3, 1)), rtol=0, atol=1e-90)


def test_closed_forms():
    check_closed_forms(oracle.default(), np.random.default_rng(3))


# ---------------------------------------------------------------------------
# 4. Invariants
# ---------------------------------------------------------------------------

def check_invariants(orc, rng):
    d = 5
    for mask, W in (("none", 0), ("causal", 0), ("window", 3)):
        q, k, v = _rand(rng, 1, 1, 9, d), _rand(rng, 1, 1, 9, d), _rand(rng, 1, 1, 9, d)
        P = orc.probs(q[0, 0], k[0, 0], 0.45, mask, W)
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        # invisible pairs carry exactly zero weight
        i = np.arange(9)[:, None]
        j = np.arange(9)[None, :]
        vis = np.ones((9, 9), bool) if mask == "none" else (j <= i) & ((j > i - W) if W else True)
        assert np.all(P[~vis] == 0.0) and np.all(P[vis] > 0.0)
        # lse equals an independently ordered log-sum-exp of the visible scores
        _, lse = orc.attention(q, k, v, 0.45, mask, W)
        for r in range(9):
            s = np.sort(0.45 * (k[0, 0][vis[r]] @ q[0, 0, r]))[::-1]
            ref = s[0] + math.log(math.fsum(math.exp(x - s[0]) for x in s))
            assert abs(lse[0, 0, r] - ref) < 1e-13
    # keys a row cannot see do not affect it: overwrite them with large garbage
    q, k, v = _rand(rng, 1, 1, 8, d), _rand(rng, 1, 1, 8, d), _rand(rng, 1, 1, 8, d)
    o1, l1 = orc.attention(q, k, v, 0.5, "causal")
    k2, v2 = k.copy(), v.copy()
    k2[0, 0, 5:] = 1e6
    v2[0, 0, 5:] = -3e7
    o2, l2 = orc.attention(q, k2, v2, 0.5, "causal")
    assert np.array_equal(o1[0, 0, :5], o2[0, 0, :5]) and np.array_equal(l1[0, 0, :5], l2[0, 0, :5])
    # permuting query rows permutes the output (no mask)
    perm = rng.permutation(8)
    o3, l3 = orc.attention(q[:, :, perm], k, v, 0.5, "none")
    o4, l4 = orc.attention(q, k, v, 0.5, "none")
    assert np.array_equal(o3, o4[:, :, perm]) and np.array_equal(l3, l4[:, :, perm])
    # permuting key/value rows together changes only the summation order
    o5, l5 = orc.attention(q, k[:, :, perm], v[:, :, perm], 0.5, "none")
    np.testing.assert_allclose(o5, o4, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l5, l4, rtol=1e-13)


def test_invariants():
    check_invariants(oracle.default(), np.random.default_rng(4))


def check_blocked_equals_naive(orc, rng):
    for (B, H, Sq, Sk, d) in [(1, 2, 9, 9, 3), (2, 1, 5, 11, 4), (1, 1, 14, 6, 2)]:
        q, k, v = _rand(rng, B, H, Sq, d), _rand(rng, B, H, Sk, d), _rand(rng, B, H, Sk, d)
        for mask, W in (("none", 0), ("causal", 0), ("window", 1), ("window", 4)):
            o_ref, l_ref = orc.attention(q, k, v, 0.6, mask, W)
            for bs in list(range(1, Sk + 2)):
                o, l = orc.attention_blocked(q, k, v, 0.6, mask, W, block_size=bs)
                np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
                fin = np.isfinite(l_ref)
                assert np.array_equal(fin, np.isfinite(l))
                np.testing.assert_allclose(l[fin], l_ref[fin], rtol=1e-12, atol=1e-13)


def test_blocked_equals_naive_every_block_size():
    check_blocked_equals_naive(oracle.default(), np.random.default_rng(5))


def check_brute_force(orc, rng):
    """Exhaustive tiny shapes against a straight triple loop in Python floats."""
    for Sq in (1, 3, 5):
        for Sk in (1, 2, 4):
            for d in (1, 3):
                q, k, v = _rand(rng, 1, 1, Sq, d), _rand(rng, 1, 1, Sk, d), _rand(rng, 1, 1, Sk, d)
                for mask, W in (("none", 0), ("causal", 0), ("window", 2)):
                    o, lse = orc.attention(q, k, v, 0.8, mask, W)
                    for i in range(Sq):
                        vis = [j for j in range(Sk)
                               if mask == "none" or (j <= i and (mask != "window" or j > i - W))]
                        if not vis:
                            assert np.all(o[0, 0, i] == 0) and lse[0, 0, i] == -math.inf
                            continue
                        s = {j: 0.8 * sum(q[0, 0, i, c] * k[0, 0, j, c] for c in range(d)) for j in vis}
                        w = {j: math.exp(s[j]) for j in vis}
                        tot = math.fsum(w.values())
                        for c in range(d):
                            ref = math.fsum(w[j] * v[0, 0, j, c] for j in vis) / tot
                            assert abs(o[0, 0, i, c] - ref) <= 1e-12 * (1 + abs(ref))
                        assert abs(lse[0, 0, i] - math.log(tot)) < 1e-12


def test_brute_force_tiny():
    check_brute_force(oracle.default(), np.random.default_rng(6))


def check_gqa(orc, rng):
    """Grouped-query attention: query head h reads K/V head h // (H // Hkv).

    Pinned three ways that do not use the oracle's own head indexing: against
    the multi-head oracle on K/V with each head repeated H // Hkv times in a row
    (the grouping PyTorch's enable_gqa uses), against torch's SDPA on the same
    repeated K/V, and one query head at a time against a one-head call on the
    K/V head named explicitly.  The blocked form must agree too.
    """
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for (H, Hkv, Sq, Sk, d) in ((4, 2, 7, 9, 3), (6, 3, 5, 5, 4), (4, 1, 6, 8, 2), (3, 3, 4, 4, 2)):
        B = 2
        q = _rand(rng, B, H, Sq, d)
        k, v = _rand(rng, B, Hkv, Sk, d), _rand(rng, B, Hkv, Sk, d)
        g = H // Hkv
        k_rep, v_rep = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
        for mask, W in (("none", 0), ("causal", 0), ("window", 3)):
            o, lse = orc.attention(q, k, v, 0.7, mask, W)
            o_m, lse_m = orc.attention(q, k_rep, v_rep, 0.7, mask, W)
            np.testing.assert_allclose(o, o_m, rtol=1e-13, atol=1e-13)
            np.testing.assert_allclose(lse, lse_m, rtol=1e-13, atol=1e-13)
            ob, lb = orc.attention_blocked(q, k, v, 0.7, mask, W, block_size=2)
            np.testing.assert_allclose(ob, o, rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(lb, lse, rtol=1e-11, atol=1e-12)
            for b in range(B):
                for h in range(H):
                    o1, l1 = orc.attention(q[b:b + 1, h:h + 1], k[b:b + 1, h // g:h // g + 1],
                                           v[b:b + 1, h // g:h // g + 1], 0.7, mask, W)
                    np.testing.assert_allclose(o[b, h], o1[0, 0], rtol=1e-13, atol=1e-13)
                    np.testing.assert_allclose(lse[b, h], l1[0, 0], rtol=1e-13, atol=1e-13)
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(k).repeat_interleave(g, dim=1),
            torch.from_numpy(v).repeat_interleave(g, dim=1), scale=0.7).numpy()
        o, _ = orc.attention(q, k, v, 0.7, "none")
        np.testing.assert_allclose(o, ref, rtol=1e-12, atol=1e-12)


def test_grouped_query_heads():
    check_gqa(oracle.default(), np.random.default_rng(8))


# ---------------------------------------------------------------------------
# Backward: gradients of sum(O * dO)
# ---------------------------------------------------------------------------

def _loss(orc, q, k, v, g, scale, mask, W):
    o, _ = orc.attention(q, k, v, scale, mask, W)
    return math.fsum((o * g).ravel())


def check_bwd_finite_differences(orc, rng):
    """Every gradient element against a central difference of the forward."""
    h = 1e-6
    for (H, Hkv, Sq, Sk, d, mask, W) in ((2, 2, 4, 5, 3, "none", 0), (2, 1, 5, 4, 2, "causal", 0),
                                         (2, 2, 6, 3, 2, "window", 2)):
        q, k, v = _rand(rng, 1, H, Sq, d), _rand(rng, 1, Hkv, Sk, d), _rand(rng, 1, Hkv, Sk, d)
        g = _rand(rng, 1, H, Sq, d)
        grads = orc.attention_bwd(q, k, v, g, 0.6, mask, W)
        for x, gx in zip((q, k, v), grads):
            for idx in np.ndindex(x.shape):
                old = x[idx]
                x[idx] = old + h
                lp = _loss(orc, q, k, v, g, 0.6, mask, W)
                x[idx] = old - h
                lm = _loss(orc, q, k, v, g, 0.6, mask, W)
                x[idx] = old
                assert abs(gx[idx] - (lp - lm) / (2 * h)) < 1e-7, (mask, idx)


def test_bwd_matches_finite_differences():
    check_bwd_finite_differences(oracle.default(), np.random.default_rng(21))


def check_bwd_torch(orc, rng):
    """fp64 autograd through torch's SDPA (band masks passed explicitly)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for (H, Hkv, Sq, Sk, d, mask, W) in ((2, 2, 7, 9, 4, "none", 0), (4, 2, 9, 9, 3, "causal", 0),
                                         (3, 1, 8, 10, 5, "window", 3)):
        q, k, v = _rand(rng, 2, H, Sq, d), _rand(rng, 2, Hkv, Sk, d), _rand(rng, 2, Hkv, Sk, d)
        g = _rand(rng, 2, H, Sq, d)
        tq, tk, tv = (torch.from_numpy(x.copy()).requires_grad_(True) for x in (q, k, v))
        rep = H // Hkv
        if mask == "none":
            am = None
        elif mask == "causal":
            am = torch.from_numpy(np.tril(np.ones((Sq, Sk), bool)))
        else:
            am = torch.from_numpy(_window_bool(Sq, Sk, W))
        o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(rep, dim=1),
                                           tv.repeat_interleave(rep, dim=1), attn_mask=am,
                                           scale=0.45)
        o.backward(torch.from_numpy(g))
        dq, dk, dv = orc.attention_bwd(q, k, v, g, 0.45, mask, W)
        np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_bwd_matches_torch_autograd():
    check_bwd_torch(oracle.default(), np.random.default_rng(22))


def check_bwd_closed_forms(orc, rng):
    # one key: every P is 1, so dS = 0 (dQ = dK = 0) and dV = sum_i dO_i
    q, k, v, g = _rand(rng, 1, 2, 6, 3), _rand(rng, 1, 2, 1, 3), _rand(rng, 1, 2, 1, 3), \
        _rand(rng, 1, 2, 6, 3)
    dq, dk, dv = orc.attention_bwd(q, k, v, g, 0.9, "none")
    assert np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    np.testing.assert_allclose(dv[:, :, 0], g.sum(axis=2), rtol=1e-13, atol=1e-14)
    # scale 0: uniform weights 1/Sk, no gradient reaches q or k
    q, k, v, g = _rand(rng, 1, 1, 5, 4), _rand(rng, 1, 1, 7, 4), _rand(rng, 1, 1, 7, 4), \
        _rand(rng, 1, 1, 5, 4)
    dq, dk, dv = orc.attention_bwd(q, k, v, g, 0.0, "none")
    assert np.abs(dq).max() == 0 and np.abs(dk).max() == 0
    np.testing.assert_allclose(dv[0, 0], np.tile(g[0, 0].sum(axis=0) / 7, (7, 1)), rtol=1e-13)
    # causal, scale 0: key j is seen by rows i >= j, each with weight 1/(i+1)
    dq, dk, dv = orc.attention_bwd(q[:, :, :5], k[:, :, :5], v[:, :, :5], g, 0.0, "causal")
    for j in range(5):
        ref = sum(g[0, 0, i] / (i + 1) for i in range(j, 5))
        np.testing.assert_allclose(dv[0, 0, j], ref, rtol=1e-13)
    # rows of P sum to one, so sum_j dV_j = sum over rows that see a key of dO_i,
    # and the softmax Jacobian's rows sum to zero, so sum_j dK_j = 0
    for mask, W in (("none", 0), ("causal", 0), ("window", 2)):
        q, k, v, g = _rand(rng, 2, 3, 9, 4), _rand(rng, 2, 3, 6, 4), _rand(rng, 2, 3, 6, 4), \
            _rand(rng, 2, 3, 9, 4)
        dq, dk, dv = orc.attention_bwd(q, k, v, g, 0.8, mask, W)
        _, lse = orc.attention(q, k, v, 0.8, mask, W)
        seen = np.isfinite(lse)[..., None]
        np.testing.assert_allclose(dv.sum(axis=2), (g * seen).sum(axis=2), rtol=1e-12, atol=1e-12)
        assert np.abs(dk.sum(axis=2)).max() < 1e-12
        assert np.all(dq[~np.isfinite(lse)] == 0)


def test_bwd_closed_forms():
    check_bwd_closed_forms(oracle.default(), np.random.default_rng(23))


# ---------------------------------------------------------------------------
# Paged K/V cache (decoding)
# ---------------------------------------------------------------------------

def _paged_case(rng, B, H, Hkv, Sq, d, bs, lens, num_blocks):
    max_blocks = max(-(-L // bs) for L in lens) + 1
    perm = rng.permutation(num_blocks)
    table = np.full((B, max_blocks), -7, np.int32)  # entries past a request's blocks: junk
    used = 0
    for b, L in enumerate(lens):
        n = -(-L // bs)
        table[b, :n] = perm[used:used + n]
        used += n
    kc = rng.standard_normal((num_blocks, Hkv, bs, d))
    vc = rng.standard_normal((num_blocks, Hkv, bs, d))
    q = rng.standard_normal((B, H, Sq, d))
    return q, kc, vc, table, np.array(lens, np.int32)


def _gather(cache, table, b, L, bs):
    """[Hkv, L, d] of request b, gathered by numpy fancy indexing."""
    j = np.arange(L)
    return cache[table[b, j // bs], :, j % bs].transpose(1, 0, 2)


def check_paged(orc, rng):
    """Paged attention equals contiguous attention over the gathered cache."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    for (B, H, Hkv, Sq, d, bs, lens) in ((3, 4, 2, 1, 8, 4, (9, 1, 16)),
                                         (2, 2, 2, 3, 5, 8, (3, 30)),
                                         (2, 6, 1, 2, 4, 16, (17, 40))):
        q, kc, vc, table, sl = _paged_case(rng, B, H, Hkv, Sq, d, bs, lens, 40)
        for mask in ("none", "causal"):
            o, lse = orc.attention_paged(q, kc, vc, table, sl, 0.4, mask)
            for b, L in enumerate(lens):
                K, V = _gather(kc, table, b, L, bs), _gather(vc, table, b, L, bs)
                if mask == "none":
                    o_ref, l_ref = orc.attention(q[b:b + 1], K[None], V[None], 0.4, "none")
                    np.testing.assert_allclose(o[b], o_ref[0], rtol=1e-12, atol=1e-13)
                    np.testing.assert_allclose(lse[b], l_ref[0], rtol=1e-12, atol=1e-13)
                # query row i sits at position L - Sq + i: an explicit band for torch
                band = np.arange(L)[None, :] <= (L - Sq + np.arange(Sq))[:, None]
                am = torch.from_numpy(band) if mask == "causal" else None
                rep = H // Hkv
                ref = F.scaled_dot_product_attention(
                    torch.from_numpy(q[b:b + 1]),
                    torch.from_numpy(K[None]).repeat_interleave(rep, dim=1),
                    torch.from_numpy(V[None]).repeat_interleave(rep, dim=1),
                    attn_mask=am, scale=0.4).numpy()
                np.testing.assert_allclose(o[b], ref[0], rtol=1e-11, atol=1e-12)


def test_paged_matches_contiguous_attention():
    check_paged(oracle.default(), np.random.default_rng(24))


def test_paged_ignores_block_placement_and_unused_memory():
    rng = np.random.default_rng(25)
    q, kc, vc, table, sl = _paged_case(rng, 2, 2, 2, 2, 6, 4, (11, 7), 12)
    o, lse = oracle.attention_paged(q, kc, vc, table, sl, 0.5, "causal")
    # move every block elsewhere and rewrite the table
    perm = rng.permutation(12)
    kc2, vc2 = np.empty_like(kc), np.empty_like(vc)
    kc2[perm], vc2[perm] = kc, vc
    table2 = np.where(table >= 0, perm[np.clip(table, 0, None)], table).astype(np.int32)
    # blocks nobody references hold NaN
    used = set(int(x) for x in table2.ravel() if x >= 0)
    for blk in range(12):
        if blk not in used:
            kc2[blk] = np.nan
            vc2[blk] = np.nan
    o2, lse2 = oracle.attention_paged(q, kc2, vc2, table2, sl, 0.5, "causal")
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2)
    with pytest.raises(ValueError):  # a length past the table's blocks
        oracle.attention_paged(q, kc, vc, table, np.array([11, 99], np.int32), 0.5)


def test_row_subset_matches_full():
    rng = np.random.default_rng(7)
    q, k, v = _rand(rng, 2, 3, 10, 4), _rand(rng, 2, 3, 10, 4), _rand(rng, 2, 3, 10, 4)
    o, lse = oracle.attention(q, k, v, 0.5, "window", 3)
    rows = np.array([0, 17, 59, 33, 9])
    o_s, l_s = oracle.attention(q, k, v, 0.5, "window", 3, rows=rows)
    assert np.array_equal(o_s, o.reshape(-1, 4)[rows])
    assert np.array_equal(l_s, lse.reshape(-1)[rows])


def test_rejects_bad_arguments():
    z = np.zeros((1, 1, 2, 2))
    with pytest.raises(ValueError):
        oracle.attention(z, z, z, 1.0, "window", 0)
    with pytest.raises(ValueError):
        oracle.attention(z, z, z, 1.0, 7)
    with pytest.raises(ValueError):
        oracle.attention(z, z, z, 1.0, "none", rows=[4])
    q3, k2 = np.zeros((1, 3, 2, 2)), np.zeros((1, 2, 2, 2))
    with pytest.raises(ValueError):  # K/V head count must divide the query head count
        oracle.attention(q3, k2, k2, 1.0, "none")
    with pytest.raises(ValueError):
        oracle.attention_blocked(q3, k2, k2, 1.0, "none")


def test_visible_pair_counts_agree():
    from exact_io_aware_30_gb300 import metrics
    for Sq, Sk in ((1, 1), (7, 7), (9, 4), (4, 9), (300, 300), (257, 130)):
        for mask, W in (("none", 0), ("causal", 0), ("window", 1), ("window", 5), ("window", 400)):
            assert metrics.visible_pairs_closed_form(Sq, Sk, mask, W) == \
                oracle.visible_pairs(Sq, Sk, mask, W)
    # the causal count is S(S+1)/2
    assert metrics.visible_pairs_closed_form(8192, 8192, "causal") == 8192 * 8193 // 2


# ---------------------------------------------------------------------------
# 5. Planted mistakes: each mutation of the oracle's C source must fail a pin
# ---------------------------------------------------------------------------

MUTATIONS = [
    ("dropped scale", "Si[j] = scale * dot;", "Si[j] = dot;"),
    ("causal off by one", "if (j > i)\n        return 0;", "if (j >= i)\n        return 0;"),
    ("window off by one", "j <= i - (int64_t)window", "j < i - (int64_t)window"),
    ("transposed score (k.q over wrong row)", "const double *qi = q + flat * (int64_t)d;",
     "const double *qi = q + (flat / Sq * Sq) * (int64_t)d;"),
    ("wrong correction sign", "exp(m - m_new)", "exp(m_new - m)"),
    ("lse without max", "mrow[r - r0] + log(lrow[r - r0])", "log(lrow[r - r0])"),
    ("no normalisation", "Si[j] /= l;\n                lrow", "Si[j] /= 1.0;\n                lrow"),
    ("unguarded empty row", "if (m == -INFINITY) { /* no visible key: guarded row */",
     "if (0) {"),
    ("K/V head by modulo", "const int64_t kvh = h / (H / Hkv);", "const int64_t kvh = h % Hkv;"),
    ("K/V head ignores batch", "return (b * Hkv + kvh)", "return (kvh)"),
    ("bwd: Jacobian row term dropped (dQ pass)", "const double ds = P[j] * (dP[j] - rowdot);",
     "const double ds = P[j] * dP[j];"),
    ("bwd: Jacobian row term sign (dK/dV pass)", "const double ds = Pij * (orc_dot(doi, vj, d) - rt[r]);",
     "const double ds = Pij * (orc_dot(doi, vj, d) + rt[r]);"),
    ("bwd: dK without scale", "dkj[c] += scale * ds * qi[c];", "dkj[c] += ds * qi[c];"),
    ("bwd: dQ from q", "dqi[c] += scale * ds * kj[c];", "dqi[c] += scale * ds * qi[c];"),
    ("bwd: dV from dS", "dvj[c] += Pij * doi[c];", "dvj[c] += ds * doi[c];"),
    ("bwd: unnormalised P (dQ pass)", "P[j] /= l;\n            double rowdot", "P[j] /= 1.0;\n            double rowdot"),
    ("bwd: P without the row sum (dK/dV pass)", "- rm[r]) / rl[r];", "- rm[r]);"),
    ("bwd: dP against k", "dP[j] = orc_dot(doi, vh + j * (int64_t)d, d);",
     "dP[j] = orc_dot(doi, kh + j * (int64_t)d, d);"),
    ("paged: token offset in block", "+ j % block_size) * (int64_t)d;\n                double dot",
     "+ j / block_size) * (int64_t)d;\n                double dot"),
    ("paged: causal row position off by one", "? L - Sq + i : L - 1;", "? L - Sq + i - 1 : L - 1;"),
    ("paged: wrong K/V head", "const int64_t kvh = h / group;", "const int64_t kvh = h % Hkv;"),
    ("bwd: key pass skips the causal mask", "if (rl[r] == 0.0 || !orc_visible(mask_kind, window, i, j))",
     "if (rl[r] == 0.0)"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(tmp_path, name, old, new):
    src = open(oracle._SRC).read()
    assert old in src, f"mutation anchor for '{name}' not found"
    mutated = tmp_path / "mutant.c"
    mutated.write_text(src.replace(old, new, 1))
    lib = oracle.compile_source(str(mutated), str(tmp_path / "libmutant.so"))
    orc = oracle.OracleLib(lib)
    checks = [check_worked_example, check_online_softmax_1d, check_library_reduction,
              check_torch_sdpa, check_closed_forms, check_invariants,
              check_blocked_equals_naive, check_brute_force, check_gqa,
              check_bwd_finite_differences, check_bwd_torch, check_bwd_closed_forms, check_paged]
    caught = 0
    for chk in checks:
        try:
            with np.errstate(all="ignore"):
                if chk in (check_worked_example, check_online_softmax_1d):
                    chk(orc)
                else:
                    chk(orc, np.random.default_rng(11))
        except (AssertionError, ValueError, FloatingPointError):
            caught += 1
    assert caught >= 1, f"no pin caught the planted mistake '{name}'"


# ---------------------------------------------------------------------------
# 6. Input generator sanity (storage rounding only)
# ---------------------------------------------------------------------------

def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5, 3.0e-3, 65504.0], np.float32)
    bits = inputs.f32_to_bf16_bits(x)
    back = inputs.bf16_bits_to_f64(bits)
    # ties go to even mantissa; torch's conversion agrees
    torch = pytest.importorskip("torch")
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(back, ref)


def test_generator_is_seeded_and_spiky():
    w = inputs.Workload("t", 1, 2, 300, 300, 64, inputs.BF16, "none", spiky_keys=True, seed=5)
    a, b = inputs.generate(w), inputs.generate(w)
    assert np.array_equal(a.k_bits, b.k_bits) and np.array_equal(a.q_bits, b.q_bits)
    k = inputs.bits_to_f64(a.k_bits, inputs.BF16)
    norms = np.abs(k).max(axis=-1)
    for h in range(2):
        assert (norms[0, h] > 8.0).sum() >= 1
    assert len(inputs.WORKLOADS) == 5


def test_e4m3_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    rng = np.random.default_rng(12)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32) * 40,
                        rng.standard_normal(20000).astype(np.float32) * 1e-2,
                        np.array([448, 0.0, -0.0, 2 ** -9, 2 ** -10, 3 * 2 ** -10, 1.0625, 1.1875,
                                  -17.0, 240.0, 232.0], np.float32)])
    x = x[np.abs(x) <= 448]  # above 448 the code saturates here
    bits = inputs.f32_to_e4m3_bits(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(bits, ref)
    assert np.array_equal(inputs.e4m3_bits_to_f64(bits),
                          torch.from_numpy(ref).view(torch.float8_e4m3fn).to(torch.float64).numpy())
    assert inputs.f32_to_e4m3_bits(np.array([1000.0, -1e6], np.float32)).tolist() == [0x7E, 0xFE]


def test_fp8_generator_dequantises_exactly():
    w = inputs.Fp8Workload("t", 1, 2, 1, 40, 48, 128, "causal", seed=3)
    a = inputs.generate_fp8(w)
    q, k, v = a.f64()
    assert q.shape == (1, 2, 40, 128) and k.shape == v.shape == (1, 1, 48, 128)
    # descales are powers of two and every value is an e4m3 value times its factor
    for f in (a.q_descale, a.k_descale, a.v_descale):
        assert 2.0 ** np.round(np.log2(f)) == f
    assert np.array_equal(inputs.e4m3_bits_to_f64(a.vt_bits).transpose(0, 1, 3, 2) * a.v_descale, v)
