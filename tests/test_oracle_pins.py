"""Pins of the fp64 oracle against what the source pages and mathematics fix.

Nothing here compares the oracle with itself: the expectations come from
exact enumeration of the uniform space, closed forms, library routines
(scipy softmax, numpy argmax / cumsum / searchsorted), brute force and the
hand-worked fixtures in tests/golden.  Sources:

  explainer: "Speculative decoding: guess a few tokens first - why the answer
             stays the same", sections "What happens in one round", "Why fixing
             wrong guesses does not leave the target distribution" (min(p,q)
             identity, residual p'), the greedy paragraph, and "Speed depends
             on two numbers" (E[N]).
  AdaPLD:    section 3.3 "Tree construction and verification", Algorithm 1.
"""
import itertools
import json
import os

import numpy as np
import pytest
from scipy.special import log_softmax, softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


# ----------------------------------------------------------------- helpers
def rand_logits(rng, shape, scale=1.5):
    return (rng.standard_normal(shape) * scale).astype(np.float32)


def enumerate_law(zt, zd, T, min_cell=1e-12):
    """Exact law of the oracle's output for one chain (B=1) with drafts drawn
    independently per position from q_i.  The oracle's output is piecewise
    constant in the uniforms: dimension i < gamma only matters through
    u_i < r_i, the last dimension through the CDF breakpoints of whichever
    final distribution is used.  Breakpoints are computed here with scipy /
    numpy (independently of the oracle); the oracle is evaluated once per cell
    at the cell midpoint and weighted by cell volume times the draft
    probability.  Returns {emitted token tuple: probability}."""
    g1, V = zt.shape
    g = g1 - 1
    p = softmax(zt.astype(np.float64) / T, axis=1)
    q = softmax(zd.astype(np.float64) / T, axis=1) if g > 0 else np.zeros((0, V))
    # final-dimension breakpoints: union over every possible final distribution
    bps = [0.0, 1.0]
    for k in range(g):
        w = np.maximum(0.0, p[k] - q[k])
        if w.sum() > 0:
            bps.extend(np.cumsum(w) / w.sum())
    bps.extend(np.cumsum(p[g]) / p[g].sum())
    for k in range(g1):   # fallback distributions are p_k themselves
        bps.extend(np.cumsum(p[k]) / p[k].sum())
    bps = np.unique(np.clip(np.array(bps), 0.0, 1.0))
    fin_lo, fin_hi = bps[:-1], bps[1:]
    keep = (fin_hi - fin_lo) > min_cell
    fin_lo, fin_hi = fin_lo[keep], fin_hi[keep]
    fin_mid, fin_w = 0.5 * (fin_lo + fin_hi), fin_hi - fin_lo

    xs, us, ws = [], [], []
    for x in itertools.product(range(V), repeat=g):
        wx = float(np.prod([q[i, x[i]] for i in range(g)])) if g else 1.0
        if wx == 0.0:
            continue
        r = [p[i, x[i]] / q[i, x[i]] for i in range(g)]
        # per accept dimension: the accept cell [0, min(r,1)) and the reject cell
        cells = []
        for i in range(g):
            a = min(r[i], 1.0)
            c = []
            if a > min_cell:
                c.append((0.5 * a, a))
            if 1.0 - a > min_cell:
                c.append((0.5 * (a + 1.0), 1.0 - a))
            cells.append(c)
        for combo in itertools.product(*cells) if g else [()]:
            wc = wx * float(np.prod([c[1] for c in combo])) if g else wx
            for m, wf in zip(fin_mid, fin_w):
                xs.append(x)
                us.append([c[0] for c in combo] + [m])
                ws.append(wc * wf)
    n = len(ws)
    tgt = np.broadcast_to(zt, (n, g1, V))
    drf = np.broadcast_to(zd, (n, g, V)) if g else np.zeros((n, 0, V), np.float32)
    out = oracle.verify_sample(tgt, drf, np.array(xs, np.int32).reshape(n, g),
                               np.array(us, np.float64).astype(np.float32),
                               T)
    assert out["bad"] == 0
    law = {}
    for row, acc, w in zip(out["tokens"], out["accepted"], ws):
        key = tuple(int(t) for t in row[: acc + 1])
        law[key] = law.get(key, 0.0) + w
    return law, p


def check_law_is_target(law, p, tol):
    """P(n > k, Y_<k = a, Y_k = b) = P(n > k, Y_<k = a) * p_k(b) for every k."""
    g1, V = p.shape
    total = sum(law.values())
    assert abs(total - 1.0) < tol
    for k in range(g1):
        pref = {}
        joint = {}
        for seq, w in law.items():
            if len(seq) > k:
                a = seq[:k]
                pref[a] = pref.get(a, 0.0) + w
                joint[(a, seq[k])] = joint.get((a, seq[k]), 0.0) + w
        for a, pa in pref.items():
            for b in range(V):
                got = joint.get((a, b), 0.0)
                assert abs(got - pa * p[k, b]) < tol, (k, a, b, got, pa * p[k, b])
    return total


# ------------------------------------------------ emitted law equals target
@pytest.mark.parametrize("V,gamma,T,seed", [
    (2, 1, 1.0, 0), (3, 2, 1.0, 1), (5, 1, 0.7, 2), (4, 3, 1.0, 3), (8, 2, 1.3, 4), (6, 0, 1.0, 5),
])
def test_enumerated_law_equals_target(V, gamma, T, seed):
    """explainer, 'Why fixing wrong guesses ...': accept path gives min(p,q),
    residual gives the rest, so every emitted token follows the target
    distribution, position by position and conditionally on the prefix."""
    rng = np.random.default_rng(seed)
    zt = rand_logits(rng, (gamma + 1, V))
    zd = rand_logits(rng, (gamma, V))
    law, p = enumerate_law(zt, zd, T)
    check_law_is_target(law, p, 1e-9)


def test_law_check_catches_plain_resample():
    """The law check has teeth: resampling from p instead of the residual
    (which the explainer rules out) breaks it.  Emulated here by enumerating a
    modified process on the CPU in numpy."""
    rng = np.random.default_rng(7)
    V = 3
    p = softmax(rng.standard_normal(V))
    q = softmax(rng.standard_normal(V))
    law = np.zeros(V)
    for x in range(V):
        a = min(1.0, p[x] / q[x])
        law[x] += q[x] * a
        law += q[x] * (1 - a) * p        # wrong: plain resample from p
    assert np.max(np.abs(law - p)) > 1e-3


# ------------------------------------------------------------- E[N] closed form
@pytest.mark.parametrize("V,gamma,seed", [(3, 1, 0), (4, 2, 1), (5, 3, 2)])
def test_expected_tokens_closed_form(V, gamma, seed):
    """explainer, 'Speed depends on two numbers': with the same (p, q) at
    every position acceptance is i.i.d. with alpha = sum_x min(p(x), q(x))
    and E[N] = (1 - alpha^(gamma+1)) / (1 - alpha)."""
    rng = np.random.default_rng(seed)
    zt1 = rand_logits(rng, (V,))
    zd1 = rand_logits(rng, (V,))
    zt = np.tile(zt1, (gamma + 1, 1))
    zd = np.tile(zd1, (gamma, 1))
    law, p = enumerate_law(zt, zd, 1.0)
    q = softmax(zd1.astype(np.float64))
    alpha = np.minimum(p[0], q).sum()
    en = sum(len(s) * w for s, w in law.items())
    assert abs(en - (1 - alpha ** (gamma + 1)) / (1 - alpha)) < 1e-9


def test_expected_tokens_monte_carlo():
    """Same closed form by seeded Monte Carlo through the oracle's public
    entry point (drafts drawn from q with numpy), within 4 standard errors."""
    rng = np.random.default_rng(11)
    V, gamma, R = 6, 3, 200_000
    zt1 = rand_logits(rng, (V,))
    zd1 = rand_logits(rng, (V,))
    q = softmax(zd1.astype(np.float64))
    p = softmax(zt1.astype(np.float64))
    alpha = np.minimum(p, q).sum()
    x = rng.choice(V, size=(R, gamma), p=q).astype(np.int32)
    u = rng.random((R, gamma + 1), dtype=np.float32)
    out = oracle.verify_sample(np.broadcast_to(zt1, (R, gamma + 1, V)),
                               np.broadcast_to(zd1, (R, gamma, V)), x, u, 1.0)
    n = out["accepted"].astype(np.float64) + 1
    en = (1 - alpha ** (gamma + 1)) / (1 - alpha)
    assert abs(n.mean() - en) < 4 * n.std() / np.sqrt(R)
    # 1 <= emitted <= gamma+1 on every round ('What happens in one round')
    assert n.min() >= 1 and n.max() <= gamma + 1


# ----------------------------------------------------- losslessness identity
@pytest.mark.parametrize("V,seed", [(4, 0), (7, 1), (8, 2)])
def test_overlap_plus_residual_is_target(V, seed):
    """explainer, 'Why fixing wrong guesses ...': q(x) min(1, p(x)/q(x)) =
    min(p(x), q(x)), and min(p,q) + (1 - alpha) p' = p with p' the residual.
    The oracle's residual is read from its CDF output after a forced
    rejection (u_0 close to 1, a draft token with q > p)."""
    rng = np.random.default_rng(seed)
    zt = rand_logits(rng, (2, V))
    zd = rand_logits(rng, (1, V))
    p = softmax(zt[0].astype(np.float64))
    q = softmax(zd[0].astype(np.float64))
    cand = np.where(q > p * 1.01)[0]
    assert cand.size > 0
    x = int(cand[0])
    out = oracle.verify_sample(zt[None], zd[None], np.array([[x]], np.int32),
                               np.array([[0.9999999, 0.5]], np.float32), 1.0,
                               want_cdf=True, want_ratio=True)
    assert out["accepted"][0] == 0
    assert abs(out["ratio"][0, 0] - p[x] / q[x]) < 1e-12
    cdf = out["cdf"][0]
    resid = np.diff(np.concatenate([[0.0], cdf]))
    alpha = np.minimum(p, q).sum()
    assert np.max(np.abs(np.minimum(p, q) + (1 - alpha) * resid - p)) < 1e-12
    assert np.max(np.abs(q * np.minimum(1.0, p / q) - np.minimum(p, q))) < 1e-15


# ------------------------------------------------------------ special cases
def test_identical_models_accept_everything():
    """q = p: every ratio is exactly 1, so every draft is accepted (u < 1)
    and the bonus token is the inverse CDF of p_gamma, i.e. numpy's
    searchsorted on cumsum (side='right')."""
    rng = np.random.default_rng(3)
    B, gamma, V = 64, 3, 50
    zt = rand_logits(rng, (B, gamma + 1, V), 2.0)
    zd = zt[:, :gamma, :].copy()
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = rng.random((B, gamma + 1), dtype=np.float32)
    out = oracle.verify_sample(zt, zd, x, u, 1.0)
    assert (out["accepted"] == gamma).all()
    assert (out["tokens"][:, :gamma] == x).all()
    for b in range(B):
        pg = softmax(zt[b, gamma].astype(np.float64))
        c = np.cumsum(pg)
        t = np.searchsorted(c, float(u[b, gamma]) * c[-1], side="right")
        assert out["tokens"][b, gamma] == t


def test_one_hot_draft_on_impossible_token_rejects():
    """q one-hot on x with p(x) = 0: ratio 0, rejection at position 0, and
    the residual max(0, p - q) is p itself, so the token follows p_0."""
    rng = np.random.default_rng(4)
    B, V = 40, 30
    zt = rand_logits(rng, (B, 2, V))
    zd = np.full((B, 1, V), -np.inf, np.float32)
    x = rng.integers(0, V, (B, 1)).astype(np.int32)
    for b in range(B):
        zd[b, 0, x[b, 0]] = 0.0
        zt[b, 0, x[b, 0]] = -np.inf
    u = rng.random((B, 2), dtype=np.float32)
    out = oracle.verify_sample(zt, zd, x, u, 1.0, want_ratio=True)
    assert (out["accepted"] == 0).all()
    assert (out["ratio"][:, 0] == 0.0).all()
    for b in range(B):
        p0 = softmax(zt[b, 0].astype(np.float64))
        c = np.cumsum(p0)
        assert out["tokens"][b, 0] == np.searchsorted(c, float(u[b, 1]) * c[-1], side="right")


def test_zero_draft_probability_always_accepts():
    """q(x) = 0 < p(x): the ratio is infinite and the draft is accepted."""
    V = 5
    zt = np.zeros((1, 2, V), np.float32)
    zd = np.zeros((1, 1, V), np.float32)
    zd[0, 0, 2] = -np.inf
    out = oracle.verify_sample(zt, zd, np.array([[2]], np.int32),
                               np.array([[0.999, 0.1]], np.float32), 1.0, want_ratio=True)
    assert out["accepted"][0] == 1 and np.isinf(out["ratio"][0, 0])


@pytest.mark.parametrize("T", [0.5, 2.0, 4.0])
def test_temperature_is_logit_scaling(T):
    """The temperature only rescales logits: verify(z, T) = verify(z / T, 1)
    whenever z / T is exact (T a power of two)."""
    rng = np.random.default_rng(5)
    B, gamma, V = 32, 3, 40
    zt = rand_logits(rng, (B, gamma + 1, V), 2.0)
    zd = rand_logits(rng, (B, gamma, V), 2.0)
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = rng.random((B, gamma + 1), dtype=np.float32)
    a = oracle.verify_sample(zt, zd, x, u, T, want_logprob=True)
    b = oracle.verify_sample(zt / np.float32(T), zd / np.float32(T), x, u, 1.0, want_logprob=True)
    assert (a["tokens"] == b["tokens"]).all() and (a["accepted"] == b["accepted"]).all()
    assert np.allclose(a["logprob"], b["logprob"], rtol=0, atol=1e-12)


def test_logprobs_match_library_log_softmax():
    rng = np.random.default_rng(6)
    B, gamma, V, T = 8, 4, 300, 0.6
    zt = rand_logits(rng, (B, gamma + 1, V), 3.0)
    zd = rand_logits(rng, (B, gamma, V), 3.0)
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = rng.random((B, gamma + 1), dtype=np.float32)
    out = oracle.verify_sample(zt, zd, x, u, T, want_logprob=True)
    for b in range(B):
        for i in range(gamma):
            lp = log_softmax(zt[b, i].astype(np.float64) / T)[x[b, i]]
            lq = log_softmax(zd[b, i].astype(np.float64) / T)[x[b, i]]
            assert abs(out["logprob"][b, i, 0] - lp) < 1e-12
            assert abs(out["logprob"][b, i, 1] - lq) < 1e-12


def test_inverse_cdf_is_searchsorted():
    """Bonus sampling (gamma = 0) is numpy.searchsorted(cumsum(p), u*S,
    side='right') away from breakpoints; exactly one uniform is consumed."""
    rng = np.random.default_rng(8)
    B, V = 500, 97
    zt = rand_logits(rng, (B, 1, V), 2.5)
    u = rng.random((B, 1), dtype=np.float32)
    out = oracle.verify_sample(zt, None, None, u, 1.0)
    n_checked = 0
    for b in range(B):
        p = softmax(zt[b, 0].astype(np.float64))
        c = np.cumsum(p)
        x = float(u[b, 0]) * c[-1]
        if np.min(np.abs(c - x)) < 1e-12:
            continue
        assert out["tokens"][b, 0] == np.searchsorted(c, x, side="right")
        n_checked += 1
    assert n_checked > 490
    assert (out["accepted"] == 0).all()


def test_token_count_and_padding_invariants():
    """Each round emits between 1 and gamma+1 tokens ('What happens in one
    round'); accepted tokens are the drafts; slots after the final token are -1."""
    rng = np.random.default_rng(9)
    B, gamma, V = 200, 5, 64
    zt = rand_logits(rng, (B, gamma + 1, V), 2.0)
    zd = zt[:, :gamma] + rand_logits(rng, (B, gamma, V), 0.7)
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    u = rng.random((B, gamma + 1), dtype=np.float32)
    out = oracle.verify_sample(zt, zd, x, u, 1.0)
    k = out["accepted"]
    assert k.min() >= 0 and k.max() <= gamma
    for b in range(B):
        row = out["tokens"][b]
        assert (row[: k[b]] == x[b, : k[b]]).all()
        assert 0 <= row[k[b]] < V
        assert (row[k[b] + 1:] == -1).all()


def test_bad_inputs_flagged():
    rng = np.random.default_rng(10)
    B, gamma, V = 4, 2, 10
    zt = rand_logits(rng, (B, gamma + 1, V))
    zd = rand_logits(rng, (B, gamma, V))
    x = rng.integers(0, V, (B, gamma)).astype(np.int32)
    x[1, 1] = V          # out of range
    x[2, 0] = -1
    zt[3, 2, :] = -np.inf  # a row with no distribution
    u = rng.random((B, gamma + 1), dtype=np.float32)
    out = oracle.verify_sample(zt, zd, x, u, 1.0)
    assert out["bad"] == 3
    assert out["accepted"][0] >= 0
    for b in (1, 2, 3):
        assert out["accepted"][b] == -1 and (out["tokens"][b] == -1).all()
    g = oracle.verify_greedy(zt, x)
    assert g["bad"] == 2 and g["accepted"][1] == -1 and g["accepted"][2] == -1


# --------------------------------------------------------------------- greedy
def test_greedy_matches_argmax_first_mismatch():
    """explainer, greedy paragraph; numpy.argmax returns the first maximum,
    which is the lowest-index tie-break."""
    rng = np.random.default_rng(12)
    B, gamma, V = 300, 4, 23
    zt = rng.integers(-3, 4, (B, gamma + 1, V)).astype(np.float32)   # many ties
    x = np.argmax(zt[:, :gamma], axis=2).astype(np.int32)
    flip = rng.random((B, gamma)) < 0.3
    x[flip] = rng.integers(0, V, flip.sum())
    out = oracle.verify_greedy(zt, x)
    for b in range(B):
        g = np.argmax(zt[b], axis=1)
        k = gamma
        for i in range(gamma):
            if x[b, i] != g[i]:
                k = i
                break
        assert out["accepted"][b] == k
        assert list(out["tokens"][b, :k]) == list(x[b, :k])
        assert out["tokens"][b, k] == g[k]
        assert (out["tokens"][b, k + 1:] == -1).all()
        assert (out["argmax"][b] == g).all()


def test_greedy_signed_zero_tie():
    """-0.0 and +0.0 are equal logits: the lower index wins."""
    zt = np.array([[[-1.0, -0.0, 0.0, -2.0]]], np.float32)
    out = oracle.verify_greedy(zt, np.zeros((1, 0), np.int32))
    assert out["tokens"][0, 0] == 1


# ----------------------------------------------------------------------- tree
def brute_force_tree(g, tok, par):
    N = len(par)
    best = ()
    for n in range(N):
        path = []
        m = n
        while m > 0:
            path.append(m)
            m = par[m]
        path = tuple(reversed(path))
        ok = all(tok[v] == g[par[v]] for v in path)
        if not ok:
            continue
        if len(path) > len(best) or (len(path) == len(best) and path < best):
            best = path
    last = best[-1] if best else 0
    return list(best), [tok[v] for v in best] + [g[last]]


@pytest.mark.parametrize("seed", range(6))
def test_tree_matches_brute_force(seed):
    """AdaPLD 3.3 / Algorithm 1 VerifyAndAccept in its greedy form: the
    longest root path whose every node carries the target argmax of its
    parent, plus the bonus argmax.  Checked against enumeration of all root
    paths (ties: lexicographically smallest node ids)."""
    rng = np.random.default_rng(100 + seed)
    B, V = 40, 6
    N = int(rng.integers(1, 14))
    zt = rng.integers(-2, 3, (B, N, V)).astype(np.float32)
    par = np.empty((B, N), np.int32)
    tok = np.empty((B, N), np.int32)
    for b in range(B):
        par[b, 0] = -1
        tok[b, 0] = -1
        g = np.argmax(zt[b], axis=1)
        for n in range(1, N):
            par[b, n] = rng.integers(0, n)
            tok[b, n] = g[par[b, n]] if rng.random() < 0.7 else rng.integers(0, V)
    out = oracle.verify_tree_greedy(zt, tok, par)
    assert out["bad"] == 0
    for b in range(B):
        g = np.argmax(zt[b], axis=1)
        nodes, toks = brute_force_tree(g, tok[b], par[b])
        L = len(nodes)
        assert out["accepted"][b] == L
        assert list(out["nodes"][b, :L]) == nodes and (out["nodes"][b, L:] == -1).all()
        assert list(out["tokens"][b, :L + 1]) == toks and (out["tokens"][b, L + 1:] == -1).all()


def test_tree_chain_equals_greedy_chain():
    """A tree that is a single chain is ordinary greedy verification."""
    rng = np.random.default_rng(13)
    B, gamma, V = 50, 5, 17
    zt = rng.integers(-3, 4, (B, gamma + 1, V)).astype(np.float32)
    x = np.argmax(zt[:, :gamma], axis=2).astype(np.int32)
    flip = rng.random((B, gamma)) < 0.25
    x[flip] = rng.integers(0, V, flip.sum())
    gr = oracle.verify_greedy(zt, x)
    par = np.tile(np.arange(-1, gamma, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.full((B, 1), -1, np.int32), x], axis=1)
    tr = oracle.verify_tree_greedy(zt, tok, par)
    assert (tr["accepted"] == gr["accepted"]).all()
    assert (tr["tokens"] == gr["tokens"]).all()


def test_tree_bad_parents_flagged():
    zt = np.zeros((3, 3, 4), np.float32)
    tok = np.array([[-1, 0, 0]] * 3, np.int32)
    par = np.array([[-1, 0, 0], [-1, 0, 2], [0, 0, 1]], np.int32)
    out = oracle.verify_tree_greedy(zt, tok, par)
    assert out["bad"] == 2
    assert out["accepted"][0] >= 0 and out["accepted"][1] == -1 and out["accepted"][2] == -1


# --------------------------------------------------------------------- golden
def _load_golden():
    with open(GOLDEN) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _load_golden()["sample"], ids=lambda c: c["id"])
def test_golden_sample(case):
    scale = case.get("logit_scale", 1.0)
    zt = (scale * np.log(np.array(case["target_probs"], np.float64))).astype(np.float32)
    zd = (scale * np.log(np.array(case["draft_probs"], np.float64))).astype(np.float32)
    if case.get("batch_of_two"):
        B = 2
        x = np.array(case["draft_tokens"], np.int32)
        u = np.array(case["uniforms"], np.float32)
        zt = zt.reshape(B, -1, zt.shape[-1])
        zd = zd.reshape(B, -1, zd.shape[-1])
        exp_t = np.array(case["expect_tokens"])
        exp_a = np.array(case["expect_accepted"])
    else:
        x = np.array([case["draft_tokens"]], np.int32)
        u = np.array([case["uniforms"]], np.float32)
        zt, zd = zt[None], zd[None]
        exp_t = np.array([case["expect_tokens"]])
        exp_a = np.array([case["expect_accepted"]])
    out = oracle.verify_sample(zt, zd, x, u, case["T"], want_ratio=True, want_cdf=True)
    assert (out["tokens"] == exp_t).all(), out["tokens"]
    assert (out["accepted"] == exp_a).all()
    if "expect_ratio" in case:
        assert np.allclose(out["ratio"][0], case["expect_ratio"], rtol=1e-6)
    if "expect_residual" in case:
        resid = np.diff(np.concatenate([[0.0], out["cdf"][0]]))
        assert np.allclose(resid, case["expect_residual"], atol=1e-6)


@pytest.mark.parametrize("case", _load_golden()["greedy"], ids=lambda c: c["id"])
def test_golden_greedy(case):
    zt = np.array([case["logits"]], np.float32)
    out = oracle.verify_greedy(zt, np.array([case["draft_tokens"]], np.int32))
    assert list(out["tokens"][0]) == case["expect_tokens"]
    assert out["accepted"][0] == case["expect_accepted"]


@pytest.mark.parametrize("case", _load_golden()["tree"], ids=lambda c: c["id"])
def test_golden_tree(case):
    zt = np.array([case["logits"]], np.float32)
    out = oracle.verify_tree_greedy(zt, np.array([case["tokens"]], np.int32),
                                    np.array([case["parents"]], np.int32))
    assert list(out["nodes"][0]) == case["expect_nodes"]
    assert list(out["tokens"][0]) == case["expect_tokens"]
    assert out["accepted"][0] == case["expect_accepted"]


def residual_vanishing_case():
    """Two tokens, T = 1: p = softmax([0, -58]) puts ~6.5e-26 on token 1,
    q = softmax([0, -46]) ~1.1e-20.  Drafting token 1 gives r = p1/q1 ~ 6e-6,
    so u0 = 0.5 rejects it; in exact arithmetic the residual max(0, p - q) is
    (q1 - p1, 0): all of its mass sits on token 0, and the final token must be
    0 whatever u_gamma is.  In double precision p0 and q0 both round to 1.0, so
    the computed residual has no positive entry at all."""
    zt = np.array([[[0.0, -58.0], [0.0, -3.0]]], np.float32)     # [B=1, gamma+1=2, V=2]
    zd = np.array([[[0.0, -46.0]]], np.float32)                  # [B=1, gamma=1, V=2]
    x = np.array([[1]], np.int32)
    return zt, zd, x


@pytest.mark.parametrize("u_final", [0.0, 0.3, 0.999999])
def test_residual_without_double_mass_takes_token_zero(u_final):
    """The oracle's fallback for a residual whose positive mass vanishes in
    double precision (sample from p_k): here it must give token 0, the only
    token the exact residual can produce."""
    zt, zd, x = residual_vanishing_case()
    p = softmax(zt[0, 0].astype(np.float64))
    q = softmax(zd[0, 0].astype(np.float64))
    assert p[1] / q[1] < 1e-5 and p[0] - q[0] == 0.0 and p[1] - q[1] < 0.0   # the case holds
    u = np.array([[0.5, u_final]], np.float32)
    out = oracle.verify_sample(zt, zd, x, u, 1.0)
    assert out["accepted"].tolist() == [0]
    assert out["tokens"].tolist() == [[0, -1]]


def test_zero_mass_tokens_never_chosen_at_cdf_edges():
    """Inverse-CDF edge conventions: u = 0 picks the first token with positive
    mass (not a zero-mass token in front of it), and u = 1 (outside [0, 1),
    clamped) picks the last token with positive mass."""
    V = 6
    # residual max(0, p - q) is zero on tokens 0, 1 and 5
    p = np.array([0.05, 0.05, 0.3, 0.3, 0.25, 0.05])
    q = np.array([0.30, 0.30, 0.1, 0.1, 0.10, 0.10])
    zt = np.log(np.stack([p, np.full(V, 1.0 / V)])).astype(np.float32)[None]
    zd = np.log(q).astype(np.float32)[None, None]
    x = np.array([[0]], np.int32)                  # ratio 1/6: rejected for u0 = 0.9
    for u_last, expect in [(0.0, 2), (1.0, 4)]:
        out = oracle.verify_sample(zt, zd, x, np.array([[0.9, u_last]], np.float32), 1.0)
        assert out["accepted"][0] == 0 and out["tokens"][0, 0] == expect, (u_last, out)


# ------------------------------------------------------------- top-K branches
def _topk_brute(z, K, ex):
    """AdaPLD, Algorithm 1: TopKNextTokens(...) minus the excluded token, by
    sorting the whole row on (larger logit, lower index)."""
    order = sorted(range(len(z)), key=lambda j: (-float(z[j]), j))[:K]
    kept = [j for j in order if j != ex]
    return kept + [-1] * (K - len(kept))


@pytest.mark.parametrize("V,K", [(1, 1), (3, 4), (7, 2), (50, 4), (50, 8), (1000, 4), (300, 64)])
def test_topk_matches_sorted_definition(V, K):
    rng = np.random.default_rng(V * 131 + K)
    R = 40
    z = rng.integers(-4, 4, size=(R, V)).astype(np.float32)   # many equal logits
    ex = rng.integers(-1, V, size=R).astype(np.int32)
    ex[::3] = -1
    # half of the exclusions hit a token of the row's top K
    for r in range(0, R, 2):
        ex[r] = _topk_brute(z[r], K, -1)[min(K - 1, r % K)]
    got = oracle.topk_exclude(z, K, ex)
    for r in range(R):
        want = _topk_brute(z[r], K, int(ex[r]))
        assert got["idx"][r].tolist() == want, (r, want, got["idx"][r])
        for j, v in zip(want, got["val"][r]):
            assert (j < 0 and v == -np.inf) or v == z[r, j]


def test_topk_without_exclusion_k1_is_first_argmax():
    rng = np.random.default_rng(7)
    z = rng.integers(-2, 2, size=(30, 97)).astype(np.float32)
    got = oracle.topk_exclude(z, 1)["idx"][:, 0]
    assert (got == np.argmax(z, axis=1)).all()


def test_topk_signed_zero_and_masked_rows():
    z = np.array([[-0.0, 0.0, -np.inf, -np.inf],
                  [-np.inf, -np.inf, -np.inf, -np.inf],
                  [1.0, -np.inf, 1.0, 0.5]], np.float32)
    got = oracle.topk_exclude(z, 3, np.array([-1, 1, 0], np.int32))["idx"]
    assert got[0].tolist() == [0, 1, 2]        # -0.0 == +0.0: lower index first
    assert got[1].tolist() == [0, 2, -1]       # all masked: index order, 1 excluded
    assert got[2].tolist() == [2, 3, -1]       # 0 excluded from [0, 2, 3]


# ----------------------------------------------------- lexical (n-gram) retrieval
def test_ngram_hand_worked():
    # a b c a b c a b (a=1, b=2, c=3); query = last 2 tokens (a, b)
    t = np.array([[1, 2, 3, 1, 2, 3, 1, 2]], np.int32)
    r = oracle.ngram_retrieve(t, [8], w=2, L=3, max_matches=4)
    assert r["count"][0] == 2
    assert r["matches"][0].tolist() == [1, 4, -1, -1]     # windows (0,1) and (3,4); (6,7) is the query
    assert r["draft"][0].tolist() == [3, 1, 2]            # after p* = 4
    r = oracle.ngram_retrieve(t, [8], w=3, L=5, max_matches=1)
    assert r["count"][0] == 1 and r["matches"][0].tolist() == [4]   # (c, a, b) ends at 4 only
    assert r["draft"][0].tolist() == [3, 1, 2, -1, -1]   # clipped at the end of the context
    r = oracle.ngram_retrieve(t, [5], w=2, L=2, max_matches=2)      # context a b c a b
    assert r["count"][0] == 1 and r["draft"][0].tolist() == [3, 1]


def _ngram_brute(t, n, w, L, cap):
    q = list(t[n - w:n]) if n >= w else None
    ms = [p for p in range(w - 1, n - 1) if q is not None and list(t[p - w + 1:p + 1]) == q]
    draft = [-1] * L
    if ms:
        p = ms[-1]
        cont = list(t[p + 1:min(p + L, n - 1) + 1])
        draft = cont + [-1] * (L - len(cont))
    return len(ms), (ms[:cap] + [-1] * cap)[:cap], draft


@pytest.mark.parametrize("w", [1, 2, 3, 5, 8])
def test_ngram_matches_brute_force(w):
    rng = np.random.default_rng(w)
    B, n_max = 30, 300
    t = rng.integers(0, 4, size=(B, n_max)).astype(np.int32)   # 4-token alphabet: many matches
    lengths = rng.integers(1, n_max + 1, size=B).astype(np.int32)
    lengths[0], lengths[1] = 1, w                                # no room for a match
    r = oracle.ngram_retrieve(t, lengths, w=w, L=6, max_matches=7)
    for b in range(B):
        cnt, ms, dr = _ngram_brute(t[b], int(lengths[b]), w, 6, 7)
        assert r["count"][b] == cnt
        assert r["matches"][b].tolist() == ms
        assert r["draft"][b].tolist() == dr


# ------------------------------------------------ semantic fallback (cosine)
def test_cosine_special_vectors():
    q = np.array([[1.0, 2.0, -2.0, 0.5]], np.float32)
    H = np.stack([q[0], -q[0], 3 * q[0], np.array([2.0, -1.0, 0.0, 0.0], np.float32),
                  np.zeros(4, np.float32)])[None]
    r = oracle.cosine_topk(H, q, 5)
    s = r["scores"][0]
    assert s[0] == pytest.approx(1.0, abs=1e-15)      # identical
    assert s[1] == pytest.approx(-1.0, abs=1e-15)     # opposite
    assert s[2] == pytest.approx(1.0, abs=1e-15)      # scale does not matter
    assert s[3] == pytest.approx(0.0, abs=1e-15)      # orthogonal
    assert s[4] == 0.0                                # zero row scores 0
    assert r["idx"][0].tolist() == [0, 2, 3, 4, 1]    # ties: lower index first


def test_cosine_matches_scipy_distance():
    from scipy.spatial.distance import cdist
    rng = np.random.default_rng(3)
    B, W, d = 5, 37, 64
    H = rng.standard_normal((B, W, d)).astype(np.float32)
    q = rng.standard_normal((B, d)).astype(np.float32)
    pos = rng.integers(0, 10**6, size=(B, W)).astype(np.int32)
    r = oracle.cosine_topk(H, q, 6, positions=pos)
    for b in range(B):
        want = 1.0 - cdist(q[b:b + 1].astype(np.float64), H[b].astype(np.float64), "cosine")[0]
        assert np.allclose(r["scores"][b], want, rtol=0, atol=1e-12)
        top = sorted(range(W), key=lambda j: (-want[j], j))[:6]
        assert r["idx"][b].tolist() == top
        assert r["pos"][b].tolist() == [int(pos[b, j]) for j in top]
