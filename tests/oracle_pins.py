"""Pins for the fp64 oracle: checks against what the pages and the mathematics
fix, never against the oracle itself.  Each pin takes an oracle library handle
so that tests/test_oracle_mutants.py can run the same pins against builds of
the oracle with planted mistakes.

Sources (page title, section):
  Speculative Decoding overview page (猜想解码 (Speculative Decoding) 全景):
    考点2 acceptance probability, residual distribution, losslessness;
    考点4 expected tokens per step; 第二章 acceptance formula;
    第三章 NumPy operator and its self-test vectors.
"""
from __future__ import annotations

import json
import os

import numpy as np
from scipy.special import softmax

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F32, BF16 = 0, 1


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _ln(p):
    with np.errstate(divide="ignore"):
        return np.log(np.asarray(p, dtype=np.float64))


def _batch(B, target_rows, draft_rows, x, u_acc, u_res, temp):
    """Broadcast per-request row sets to a B-request fp32 batch."""
    tr = np.asarray(target_rows, dtype=np.float32)
    R, V = tr.shape
    g = R - 1
    dr = np.asarray(draft_rows, dtype=np.float32).reshape(g, V)
    Lt = np.ascontiguousarray(np.broadcast_to(tr, (B, R, V)))
    Ld = np.ascontiguousarray(np.broadcast_to(dr, (B, g, V)))
    x = np.ascontiguousarray(np.broadcast_to(np.asarray(x, np.int32), (B, g)))
    u_acc = np.ascontiguousarray(np.broadcast_to(np.asarray(u_acc, np.float32), (B, g)))
    u_res = np.ascontiguousarray(np.broadcast_to(np.asarray(u_res, np.float32), (B, R)))
    temp = np.ascontiguousarray(np.broadcast_to(np.asarray(temp, np.float32), (B,)))
    return Lt, Ld, x, u_acc, u_res, temp


def _midgrid(n):
    return ((np.arange(n) + 0.5) / n).astype(np.float32)


def _emitted(out):
    return (out["tokens"] >= 0).sum(axis=1)


# ---------------------------------------------------------------- page values

def pin_worked_example(lib):
    """考点2 / 第二章 worked example: P_draft = 0.5, P_target = 0.3 -> 0.6."""
    g = _golden("worked_example.json")
    pt, pd, pacc = g["p_target"], g["p_draft"], g["p_accept"]
    n = 20000
    u = _midgrid(n)
    Lt, Ld, x, ua, ur, T = _batch(n, [_ln([pt, 0.5, 0.2]), _ln([1 / 3] * 3)],
                                  [_ln([pd, 0.3, 0.2])], [0], 0.0, [0.5, 0.5], 1.0)
    ua = u.reshape(n, 1).copy()
    out = oracle.verify(Lt, Ld, x, ua, ur, T, F32, lib=lib)
    assert np.allclose(out["pt"][:, 0], pt, rtol=1e-6)
    assert np.allclose(out["pd"][:, 0], pd, rtol=1e-6)
    acc = out["n"] == 1
    assert abs(acc.mean() - pacc) <= 1.0 / n
    far = np.abs(u.astype(np.float64) - pacc) > 1e-6
    assert np.array_equal(acc[far], (u <= pacc)[far])
    assert np.all(out["tokens"][acc, 0] == 0)


def pin_numpy_operator_vectors(lib):
    """第三章 self-test vectors: token 1 (ratio 1.5) and token 0 (ratio 1) are
    always accepted; token 2 (ratio 1/3) is rejected for u > 1/3 and then the
    residual [0, .2, 0, 0, 0] makes the resampled token always 1."""
    g = _golden("numpy_operator_vectors.json")
    pt, pd = g["p_target"], g["p_draft"]
    d = g["derived_by_exact_arithmetic_from_the_vectors"]
    n = 4000
    u = _midgrid(n)
    for tok, ratio in ((1, d["ratio_token_1"]), (0, d["ratio_token_0"]),
                       (2, d["ratio_token_2"])):
        Lt, Ld, x, ua, ur, T = _batch(n, [_ln(pt), _ln([0.2] * 5)], [_ln(pd)], [tok], 0.0,
                                      [0.0, 0.5], 1.0)
        ua = u.reshape(n, 1).copy()
        ur = np.stack([u[::-1], np.full(n, 0.5, np.float32)], axis=1).copy()
        out = oracle.verify(Lt, Ld, x, ua, ur, T, F32, lib=lib)
        assert np.allclose(out["pt"][:, 0] / out["pd"][:, 0], ratio, rtol=1e-6)
        if ratio >= 1.0:
            assert np.all(out["n"] == 1) and np.all(out["tokens"][:, 0] == tok)
        else:
            far = np.abs(u.astype(np.float64) - ratio) > 1e-6
            rej = out["n"] == 0
            assert np.array_equal(rej[far], (u > ratio)[far])
            assert np.all(out["tokens"][rej, 0] == d["resample_token_after_any_rejection"])
            assert np.all(out["tokens"][rej, 1] == -1)
            assert np.allclose(out["Z"][rej], sum(d["residual_unnormalised"]), rtol=1e-6)


def pin_expected_tokens(lib):
    """考点4: with a per-position acceptance probability alpha, the mean number
    of emitted tokens is sum_{i=0..gamma} alpha^i; alpha -> 0 gives exactly 1.
    Construction: V=8, T=1, logits ln p with p_t = (a, 1-a-6e, e..e),
    p_d = (1-a-6e, a, e..e), a = (alpha-6e)/2, so sum_v min(p_t, p_d) = alpha,
    rows independent of one another."""
    g = _golden("expected_tokens.json")
    gamma = g["gamma"]
    rng = np.random.default_rng(7)
    eps = 1e-3
    for alpha_s, closed in g["closed_form_with_bonus"].items():
        alpha = float(alpha_s)
        a = (alpha - 6 * eps) / 2
        p_t = np.array([a, 1 - a - 6 * eps] + [eps] * 6)
        p_d = np.array([1 - a - 6 * eps, a] + [eps] * 6)
        N = 200000
        x = rng.choice(8, size=(N, gamma), p=p_d).astype(np.int32)
        Lt, Ld, _, _, _, T = _batch(N, [_ln(p_t)] * (gamma + 1), [_ln(p_d)] * gamma,
                                    [0] * gamma, 0.0, [0.0] * (gamma + 1), 1.0)
        ua = rng.random((N, gamma), dtype=np.float32)
        ur = rng.random((N, gamma + 1), dtype=np.float32)
        out = oracle.verify(Lt, Ld, x, ua, ur, T, F32, lib=lib)
        tokens = _emitted(out)
        assert np.all(tokens == out["n"] + 1)
        sd = tokens.std() / np.sqrt(N)
        assert abs(tokens.mean() - closed) < 4 * sd + 1e-9, (alpha, tokens.mean(), closed)
        nobonus = np.minimum(tokens, gamma)
        want_nb = (1 - alpha ** gamma) / (1 - alpha)
        assert abs(nobonus.mean() - want_nb) < 4 * nobonus.std() / np.sqrt(N) + 1e-9
        assert abs(want_nb - g["page_printed"][alpha_s]) < 0.01
    # alpha -> 0: disjoint supports, every step still emits exactly one token
    p_t = np.array([0.25] * 4 + [0.0] * 4)
    p_d = np.array([0.0] * 4 + [0.25] * 4)
    N = 5000
    x = rng.integers(4, 8, size=(N, gamma)).astype(np.int32)
    Lt, Ld, _, _, _, T = _batch(N, [_ln(p_t)] * (gamma + 1), [_ln(p_d)] * gamma,
                                [0] * gamma, 0.0, [0.0] * (gamma + 1), 1.0)
    ua = np.maximum(rng.random((N, gamma), dtype=np.float32), np.float32(1e-7))
    ur = rng.random((N, gamma + 1), dtype=np.float32)
    out = oracle.verify(Lt, Ld, x, ua, ur, T, F32, lib=lib)
    assert np.all(_emitted(out) == 1) and np.all(out["n"] == 0)
    assert np.all(out["tokens"][:, 0] < 4)


def pin_mixture_acceptance(lib):
    """考点2 / 考点4: a draft token x ~ P_d is accepted with probability
    sum_v min(P_t, P_d).  The softmax-mix draft rows of the large-batch
    workload, P_d = w P_t + (1 - w) q, make that at least w.  The oracle's
    acceptance frequency over draws from P_d must match the closed form within
    4 sigma for w = 0.3, 0.6, 0.9, with the rows stored as T ln p at T = 0.7
    (so the temperature must reach both rows)."""
    rng = np.random.default_rng(45)
    V, N, T = 40, 60000, np.float32(0.7)
    for w in (0.3, 0.6, 0.9):
        p_t = rng.dirichlet(np.full(V, 0.5))
        q = rng.dirichlet(np.full(V, 0.5))
        p_d = w * p_t + (1 - w) * q
        lt = (T * _ln(p_t)).astype(np.float32)
        ld = (T * _ln(p_d)).astype(np.float32)
        # the stored rows' own distributions (after fp32 rounding), in fp64
        pt = softmax(lt.astype(np.float64) / float(T))
        pd = softmax(ld.astype(np.float64) / float(T))
        alpha = float(np.minimum(pt, pd).sum())
        assert alpha >= w - 1e-6, (w, alpha)
        x = rng.choice(V, size=(N, 1), p=pd).astype(np.int32)
        Lt, Ld, _, _, _, temp = _batch(N, [lt, lt], [ld], [0], 0.0, [0.0, 0.0], T)
        ua = rng.random((N, 1), dtype=np.float32)
        ur = rng.random((N, 2), dtype=np.float32)
        out = oracle.verify(Lt, Ld, x, ua, ur, temp, F32, lib=lib)
        f = float(out["n"].mean())
        sd = np.sqrt(alpha * (1 - alpha) / N)
        assert abs(f - alpha) < 4 * sd, (w, f, alpha)


# ------------------------------------------------------------- mathematics

def pin_losslessness_chisq(lib, trials=1_000_000):
    """考点2 identity P_final == P_target: draft tokens drawn from P_draft, the
    token emitted at position 0 (always emitted) follows P_target[0]; the token
    at position 1, given that position 1 is reached, follows P_target[1].
    Chi-square with 7 degrees of freedom, rejected above 24.32 (p = 0.001)."""
    rng = np.random.default_rng(2026)
    V, gamma, T = 8, 2, float(np.float32(0.7))
    lt = rng.normal(0, 1.5, size=(gamma + 1, V)).astype(np.float32)
    ld = rng.normal(0, 1.5, size=(gamma, V)).astype(np.float32)
    Pt = softmax(lt.astype(np.float64) / T, axis=1)
    Pd = softmax(ld.astype(np.float64) / T, axis=1)
    x = np.stack([rng.choice(V, size=trials, p=Pd[i]) for i in range(gamma)], axis=1)
    Lt, Ld, _, _, _, Tb = _batch(trials, lt, ld, [0] * gamma, 0.0, [0.0] * (gamma + 1), T)
    ua = rng.random((trials, gamma), dtype=np.float32)
    ur = rng.random((trials, gamma + 1), dtype=np.float32)
    out = oracle.verify(Lt, Ld, x.astype(np.int32), ua, ur, Tb, F32, lib=lib)
    for pos in range(2):
        reached = out["n"] >= pos
        toks = out["tokens"][reached, pos]
        assert np.all(toks >= 0)
        obs = np.bincount(toks, minlength=V)
        exp_ = Pt[pos] * reached.sum()
        chi2 = float(((obs - exp_) ** 2 / exp_).sum())
        assert chi2 < 24.32, (pos, chi2)


def pin_brute_force_tiny(lib):
    """Brute force at V=4, gamma=3: every point of a u_acc grid gives the
    first-rejection index of the plain rule (u_i > r_i, r from the textbook
    softmax), the frequencies of k match prod r_i (1 - r_k) within grid
    resolution, and for each k the token over a u_res grid equals the
    index-order inverse CDF of max(0, P_t - P_d) (np.searchsorted on the
    cumulative sum, side='right'), with frequencies w/Z within 1/n."""
    rng = np.random.default_rng(11)
    V, gamma, T = 4, 3, float(np.float32(0.9))
    lt = rng.normal(0, 1.2, size=(gamma + 1, V)).astype(np.float32)
    ld = rng.normal(0, 1.2, size=(gamma, V)).astype(np.float32)
    Pt = softmax(lt.astype(np.float64) / T, axis=1)
    Pd = softmax(ld.astype(np.float64) / T, axis=1)
    xs = np.array([int(np.argmax(Pd[i])) for i in range(gamma)], np.int32)
    r = np.minimum(1.0, Pt[np.arange(gamma), xs] / Pd[np.arange(gamma), xs])
    n = 24
    grid = _midgrid(n)
    mesh = np.stack(np.meshgrid(*([grid] * gamma), indexing="ij"), -1).reshape(-1, gamma)
    N = mesh.shape[0]
    Lt, Ld, x, _, ur, Tb = _batch(N, lt, ld, xs, 0.0, [0.5] * (gamma + 1), T)
    out = oracle.verify(Lt, Ld, x, mesh.copy(), ur, Tb, F32, lib=lib)
    rej = mesh.astype(np.float64) > r[None, :]
    k_rule = np.where(rej.any(1), rej.argmax(1), gamma)
    far = np.all(np.abs(mesh.astype(np.float64) - r[None, :]) > 1e-6, axis=1)
    assert np.array_equal(out["n"][far], k_rule[far])
    for k in range(gamma + 1):
        want = np.prod(r[:k]) * ((1 - r[k]) if k < gamma else 1.0)
        assert abs((out["n"] == k).mean() - want) <= gamma * 0.5 / n + 1e-12
    m = 10000
    ug = _midgrid(m)
    for k in range(gamma + 1):
        ua = np.zeros((m, gamma), np.float32)
        if k < gamma:
            if r[k] >= 1.0:
                continue
            ua[:, k] = np.float32(0.9999999)
            w = np.maximum(0.0, Pt[k] - Pd[k])
        else:
            w = Pt[gamma].copy()
        ur = np.zeros((m, gamma + 1), np.float32)
        ur[:, k] = ug
        Lt, Ld, x, _, _, Tb = _batch(m, lt, ld, xs, 0.0, [0.0] * (gamma + 1), T)
        out = oracle.verify(Lt, Ld, x, ua, ur, Tb, F32, lib=lib)
        assert np.all(out["n"] == k)
        cum = np.cumsum(w)
        want = np.searchsorted(cum, ug.astype(np.float64) * cum[-1], side="right")
        nearb = np.min(np.abs(cum[None, :] / cum[-1] - ug.astype(np.float64)[:, None]), 1) < 1e-6
        got = out["tokens"][:, k]
        assert np.array_equal(got[~nearb], want[~nearb])
        freq = np.bincount(got, minlength=V) / m
        assert np.all(np.abs(freq - w / w.sum()) <= 1.0 / m + 1e-12)


def pin_accept_boundary(lib):
    """Reading R1 (accept iff u <= r) and R2 (P_draft(x) = 0 -> accept),
    on rows whose probabilities are exact in binary: p_t = 1/4 each,
    p_d = (1/2, 1/2, 0, 0), so r = 1/2 for token 0 exactly."""
    z = 0.0
    ninf = -np.inf
    lt = [[z, z, z, z], [z, z, z, z]]
    ld = [[z, z, ninf, ninf]]
    half = np.float32(0.5)
    above = np.nextafter(half, np.float32(1))
    ua = np.array([[half], [above], [0.0], [0.999]], np.float32)
    Lt, Ld, x, _, ur, T = _batch(4, lt, ld, [0], 0.0, [0.3, 0.3], 1.0)
    x = np.array([[0], [0], [2], [2]], np.int32)  # token 2: P_draft = 0 -> r = 1
    out = oracle.verify(Lt, Ld, x, ua, ur, T, F32, lib=lib)
    assert list(out["n"]) == [1, 0, 1, 1]
    # P_target(x) = 0 gives r = 0: only u = 0 is accepted
    lt2 = [[ninf, z, z, z], [z, z, z, z]]
    Lt, Ld, x, _, ur, T = _batch(2, lt2, [[z, z, z, z]], [0], 0.0, [0.3, 0.3], 1.0)
    out = oracle.verify(Lt, Ld, x, np.array([[0.0], [1e-7]], np.float32), ur, T, F32, lib=lib)
    assert list(out["n"]) == [1, 0]


def pin_inverse_cdf_strict(lib):
    """Reading R5: the token is the smallest v whose running residual mass
    exceeds u * Z (strict), so a zero-mass token is never emitted, even at
    u = 0.  p_t = (.2, .5, .3), p_d = (.4, .1, .5): residual (0, .4, 0)."""
    lt = [_ln([0.2, 0.5, 0.3]), _ln([1 / 3] * 3)]
    ld = [_ln([0.4, 0.1, 0.5])]
    us = np.array([0.0, 0.25, 0.5, 0.9999999], np.float32)
    Lt, Ld, x, _, _, T = _batch(len(us), lt, ld, [0], 0.0, [0.0, 0.0], 1.0)
    ur = np.stack([us, us], 1).copy()
    out = oracle.verify(Lt, Ld, x, np.full((len(us), 1), 0.9999, np.float32), ur, T, F32,
                        lib=lib)
    assert np.all(out["n"] == 0) and np.all(out["tokens"][:, 0] == 1)
    # residual (0.1, 0, 0.3): u = 0 -> token 0; u = 0.2 -> 0; u = 0.3 -> 2
    lt = [_ln([0.3, 0.2, 0.5]), _ln([1 / 3] * 3)]
    ld = [_ln([0.2, 0.6, 0.2])]
    us = np.array([0.0, 0.2, 0.3, 0.9], np.float32)
    Lt, Ld, x, _, _, T = _batch(len(us), lt, ld, [1], 0.0, [0.0, 0.0], 1.0)
    ur = np.stack([us, us], 1).copy()
    out = oracle.verify(Lt, Ld, x, np.full((len(us), 1), 0.9999, np.float32), ur, T, F32,
                        lib=lib)
    assert list(out["tokens"][:, 0]) == [0, 0, 2, 2]


def pin_softmax_textbook(lib):
    """Softmax against the textbook definition: ln p logits at T = 1 give p
    back; tempered rows match softmax(l / T); logits near 1000 (which overflow
    exp without the max shift) and -inf entries stay exact."""
    rng = np.random.default_rng(5)
    V = 7
    p = rng.dirichlet(np.ones(V))
    lt = np.stack([_ln(p), _ln(p)])
    ld = rng.normal(0, 2, size=(1, V))
    xs = np.arange(V, dtype=np.int32).reshape(V, 1)
    Lt, Ld, _, _, ur, T = _batch(V, lt, ld, [0], 0.0, [0.5, 0.5], 1.0)
    out = oracle.verify(Lt, Ld, xs, np.zeros((V, 1), np.float32), ur, T, F32, lib=lib)
    assert np.allclose(out["pt"][:, 0], p, rtol=2e-6)
    for T, shift in ((0.37, 0.0), (2.5, 0.0), (1.0, 1000.0), (0.8, -1000.0)):
        lt = (rng.normal(0, 3, size=(2, V)) + shift).astype(np.float32)
        lt[0, 3] = -np.inf
        ld = (rng.normal(0, 3, size=(1, V)) + shift).astype(np.float32)
        Lt, Ld, _, _, ur, Tb = _batch(V, lt, ld, [0], 0.0, [0.5, 0.5], T)
        out = oracle.verify(Lt, Ld, xs, np.zeros((V, 1), np.float32), ur, Tb, F32, lib=lib)
        assert np.all(out["flags"] & oracle.INVALID_ANY == 0)
        T32 = float(np.float32(T))  # the oracle sees the stored fp32 temperature
        wt = softmax(lt[0].astype(np.float64) / T32)
        wd = softmax(ld[0].astype(np.float64) / T32)
        assert np.allclose(out["pt"][:, 0], wt, rtol=1e-12, atol=0)
        assert np.allclose(out["pd"][:, 0], wd, rtol=1e-12, atol=0)


def pin_degenerate_shapes(lib):
    """gamma = 0 (plain sampling from target row 0: over a u grid the token
    frequencies are P_t[0] within 1/n) and V = 1 (every draft accepted)."""
    rng = np.random.default_rng(3)
    V, n = 6, 6000
    lt = rng.normal(0, 1, size=(1, V)).astype(np.float32)
    Lt = np.ascontiguousarray(np.broadcast_to(lt, (n, 1, V)))
    Ld = np.zeros((n, 0, V), np.float32)
    ur = _midgrid(n).reshape(n, 1)
    out = oracle.verify(Lt, Ld, np.zeros((n, 0), np.int32), np.zeros((n, 0), np.float32), ur,
                        np.ones(n, np.float32), F32, lib=lib)
    assert np.all(out["n"] == 0)
    freq = np.bincount(out["tokens"][:, 0], minlength=V) / n
    assert np.all(np.abs(freq - softmax(lt[0].astype(np.float64))) <= 1.0 / n + 1e-12)
    g = 3
    Lt = rng.normal(0, 1, size=(5, g + 1, 1)).astype(np.float32)
    Ld = rng.normal(0, 1, size=(5, g, 1)).astype(np.float32)
    out = oracle.verify(Lt, Ld, np.zeros((5, g), np.int32), rng.random((5, g), np.float32),
                        rng.random((5, g + 1), np.float32), np.ones(5, np.float32), F32, lib=lib)
    assert np.all(out["n"] == g) and np.all(out["tokens"] == 0)


def pin_invalid_inputs(lib):
    """Reading R7/R8: bad temperature, NaN / +inf / all -inf rows and
    out-of-range draft tokens invalidate only their own request."""
    rng = np.random.default_rng(9)
    B, g, V = 12, 2, 16
    Lt = rng.normal(0, 1, size=(B, g + 1, V)).astype(np.float32)
    Ld = rng.normal(0, 1, size=(B, g, V)).astype(np.float32)
    x = rng.integers(0, V, size=(B, g)).astype(np.int32)
    T = np.ones(B, np.float32)
    Lt[1, 0, 5] = np.nan
    Ld[2, 1, 0] = np.inf
    Lt[3, 2, :] = -np.inf
    x[4, 1] = V
    x[5, 0] = -1
    T[6], T[7], T[8], T[9] = 0.0, -1.0, np.nan, np.float32(1e-39)
    T[10] = np.inf
    Lt[11, 1, :] = -np.inf
    Lt[11, 1, 3] = 0.0  # -inf entries are legal while one entry is finite
    out = oracle.verify(Lt, Ld, x, rng.random((B, g), np.float32),
                        rng.random((B, g + 1), np.float32), T, F32, lib=lib)
    fl = out["flags"]
    assert fl[0] & oracle.INVALID_ANY == 0 and fl[11] & oracle.INVALID_ANY == 0
    for b in (1, 2, 3):
        assert fl[b] & oracle.INVALID_NONFINITE
    for b in (4, 5):
        assert fl[b] & oracle.INVALID_TOKEN
    for b in (6, 7, 8, 9, 10):
        assert fl[b] & oracle.INVALID_TEMP
    for b in range(1, 11):
        assert out["n"][b] == 0 and np.all(out["tokens"][b] == -1)


def pin_greedy(lib):
    """Reading R9 against the textbook argmax (np.argmax returns the first
    maximal index), with planted ties, on bf16 logits."""
    rng = np.random.default_rng(13)
    B, g, V = 40, 5, 300
    lt = rng.normal(0, 3, size=(B, g + 1, V)).astype(np.float32)
    bits = (lt.view(np.uint32) >> 16).astype(np.uint16)  # truncate to bf16
    wide = (bits.astype(np.uint32) << 16).view(np.float32)
    for b in range(0, B, 3):  # plant a tie: copy the max to a later and an earlier index
        for i in range(g + 1):
            a = int(np.argmax(wide[b, i]))
            bits[b, i, (a + 7) % V] = bits[b, i, a]
            if b % 2 == 0 and a > 0:
                bits[b, i, a - 1] = bits[b, i, a]
    wide = (bits.astype(np.uint32) << 16).view(np.float32)
    amax = np.argmax(wide, axis=2)
    x = amax[:, :g].copy().astype(np.int32)
    kk = rng.integers(0, g + 1, size=B)
    for b in range(B):
        if kk[b] < g:
            x[b, kk[b]] = (amax[b, kk[b]] + 1) % V
    out = oracle.greedy(bits, x, BF16, lib=lib)
    assert np.array_equal(out["argmax"], amax)
    assert np.array_equal(out["n"], kk)
    for b in range(B):
        k = kk[b]
        assert np.array_equal(out["tokens"][b, :k], amax[b, :k])
        assert out["tokens"][b, k] == amax[b, k]
        assert np.all(out["tokens"][b, k + 1:] == -1)
    bits[0, 2, 9] = 0x7FC0  # NaN
    bits[1, 0, :] = 0xFF80  # all -inf
    x[2, 0] = V
    out = oracle.greedy(bits, x, BF16, lib=lib)
    for b in range(3):
        assert out["flags"][b] & oracle.INVALID_ANY and out["n"][b] == 0
        assert np.all(out["tokens"][b] == -1)


ALL_PINS = [pin_worked_example, pin_numpy_operator_vectors, pin_expected_tokens,
            pin_mixture_acceptance,
            pin_losslessness_chisq, pin_brute_force_tiny, pin_accept_boundary,
            pin_inverse_cdf_strict, pin_softmax_textbook, pin_degenerate_shapes,
            pin_invalid_inputs, pin_greedy]


# ------------------------------------------------------- draft-row sampling

def _bf16_bits(a):
    """fp32 values -> bf16 bit patterns (truncation; the test's rows are
    built from these exact values)."""
    return (np.ascontiguousarray(a, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_wide(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pin_draft_sample_grid(lib):
    """考点2: the draft token is a sample of P_draft.  Brute force at V=5 over
    a u grid, fp32 and bf16 rows, T = 0.6: away from CDF edges the token is
    np.searchsorted(cumsum(P), u * sum(P), 'right') with P the textbook
    softmax(l / T); token frequencies are P within 1/n; m is the largest
    stored logit and S = sum exp((l - m) / T)."""
    rng = np.random.default_rng(21)
    V, n = 5, 10000
    T = float(np.float32(0.6))
    ug = _midgrid(n)
    for dt in (F32, BF16):
        l32 = rng.normal(0, 1.3, size=V).astype(np.float32)
        if dt == BF16:
            stored = _bf16_bits(l32)
            wide = _bf16_wide(stored)
        else:
            stored = l32
            wide = l32.astype(np.float64)
        L = np.ascontiguousarray(np.broadcast_to(stored, (n // 10, 10, V)))
        out = oracle.draft_sample(L, ug.reshape(n // 10, 10), np.full(n // 10, T, np.float32),
                                  dt, lib=lib)
        P = softmax(wide / T)
        cum = np.cumsum(P)
        u64 = ug.astype(np.float64)
        want = np.searchsorted(cum, u64 * cum[-1], side="right")
        nearb = np.min(np.abs(cum[None, :] / cum[-1] - u64[:, None]), 1) < 1e-6
        got = out["tokens"].reshape(-1)
        assert np.array_equal(got[~nearb], want[~nearb])
        freq = np.bincount(got, minlength=V) / n
        assert np.all(np.abs(freq - P) <= 1.0 / n + 1e-12)
        m = wide.max()
        assert np.all(out["m"] == m)
        assert np.allclose(out["S"], np.exp((wide - m) / T).sum(), rtol=1e-13, atol=0)
        assert np.all(out["flags"] & oracle.INVALID_ANY == 0)
    # ln p logits at T = 1: S = 1 / max p, m = ln max p + c
    p = rng.dirichlet(np.ones(7))
    c = 3.0
    L = (np.log(p) + c).astype(np.float32).reshape(1, 1, 7)
    out = oracle.draft_sample(L, np.array([[0.5]], np.float32), np.ones(1, np.float32), F32,
                              lib=lib)
    wide = L.astype(np.float64).reshape(-1)
    assert out["m"][0, 0] == wide.max()
    assert abs(out["S"][0, 0] - np.exp(wide - wide.max()).sum()) < 1e-13 * out["S"][0, 0]
    assert abs(out["S"][0, 0] * p.max() - 1.0) < 1e-6  # fp32 rounding of ln p + c


def pin_draft_then_verify_lossless(lib, trials=400_000):
    """考点2 identity with the draft tokens drawn by the draft-sampling oracle
    (T = 1.4): the token emitted at position 0 follows P_target[0], and the
    drafts follow P_draft.  Chi-square, 7 degrees of freedom, rejected above
    24.32 (p = 0.001)."""
    rng = np.random.default_rng(77)
    V, gamma = 8, 2
    T = float(np.float32(1.4))
    lt = rng.normal(0, 1.5, size=(gamma + 1, V)).astype(np.float32)
    ld = rng.normal(0, 1.5, size=(gamma, V)).astype(np.float32)
    Pt = softmax(lt.astype(np.float64) / T, axis=1)
    Pd = softmax(ld.astype(np.float64) / T, axis=1)
    Ld = np.ascontiguousarray(np.broadcast_to(ld, (trials, gamma, V)))
    temp = np.full(trials, T, np.float32)
    ds = oracle.draft_sample(Ld, rng.random((trials, gamma), dtype=np.float32), temp, F32,
                             lib=lib)
    x = ds["tokens"]
    for i in range(gamma):
        obs = np.bincount(x[:, i], minlength=V)
        chi2 = float(((obs - Pd[i] * trials) ** 2 / (Pd[i] * trials)).sum())
        assert chi2 < 24.32, ("draft", i, chi2)
    Lt = np.ascontiguousarray(np.broadcast_to(lt, (trials, gamma + 1, V)))
    out = oracle.verify(Lt, Ld, x, rng.random((trials, gamma), dtype=np.float32),
                        rng.random((trials, gamma + 1), dtype=np.float32), temp, F32, lib=lib)
    obs = np.bincount(out["tokens"][:, 0], minlength=V)
    chi2 = float(((obs - Pt[0] * trials) ** 2 / (Pt[0] * trials)).sum())
    assert chi2 < 24.32, ("emitted", chi2)


def pin_draft_sample_invalid(lib):
    """Readings R7/R8 on the draft side: a NaN or +inf logit, an all -inf row
    or a bad temperature gives token -1 and NaN statistics for that row only;
    a row with some -inf entries is legal and never emits them."""
    rng = np.random.default_rng(31)
    B, n, V = 4, 3, 9
    L = rng.normal(0, 1, size=(B, n, V)).astype(np.float32)
    L[0, 1, 4] = np.nan
    L[0, 2, 0] = np.inf
    L[1, 0, :] = -np.inf
    L[2, :, 1::2] = -np.inf
    T = np.array([1.0, 1.0, 0.9, 0.0], np.float32)
    u = rng.random((B, n), dtype=np.float32)
    out = oracle.draft_sample(L, u, T, F32, lib=lib)
    bad = np.zeros((B, n), bool)
    bad[0, 1] = bad[0, 2] = bad[1, 0] = True
    bad[3, :] = True
    assert np.all(out["tokens"][bad] == -1) and np.all(np.isnan(out["S"][bad]))
    assert np.all(out["flags"][0, 1:] & oracle.INVALID_NONFINITE)
    assert out["flags"][1, 0] & oracle.INVALID_NONFINITE
    assert np.all(out["flags"][3] & oracle.INVALID_TEMP)
    assert np.all(out["tokens"][~bad] >= 0)
    assert np.all(out["tokens"][2] % 2 == 0)


# ---------------------------------------------------- sink + ring KV cache

def pin_kv_slot_closed_form(lib):
    """Deferred-speculation page, "环形上下文与注意力沉淀机制": Slot(pos) is
    pos inside the S sink slots; past them, W consecutive positions fill the
    W ring slots S .. S+W-1 once each, and a position W later reuses the
    slot."""
    for S in (0, 1, 4):
        for W in (1, 3, 8):
            for p in range(S):
                assert oracle.kv_slot(p, S, W, lib=lib) == p
            assert oracle.kv_slot(S, S, W, lib=lib) == S
            for p0 in range(S, S + 3 * W):
                slots = sorted(oracle.kv_slot(p, S, W, lib=lib) for p in range(p0, p0 + W))
                assert slots == list(range(S, S + W))
                assert oracle.kv_slot(p0 + W, S, W, lib=lib) == oracle.kv_slot(p0, S, W, lib=lib)


def pin_kv_commit_content(lib):
    """The cache after a run of verification steps holds exactly what a plain
    model of a sink + sliding window holds: the first S positions, then the
    last W committed ones (a deque of length W), oldest first, read through
    the valid-slot list.  Each step commits k + 1 staged entries (the last
    emitted token and k accepted drafts, reading K1); entries of rejected
    drafts are never visible.  Every KV row carries a tag of its position."""
    from collections import deque
    rng = np.random.default_rng(41)
    B, LH, gamma, S, W = 3, 2, 3, 4, 6
    R = gamma + 1
    C = S + W
    kp = np.full((B, LH, C, 2), -99, np.int32)
    vp = kp.copy()
    pos = np.zeros(B, np.int32)
    models = [([], deque(maxlen=W)) for _ in range(B)]
    for step in range(12):
        k = rng.integers(-1, R, size=B).astype(np.int32)  # -1: a dropped request
        kn = np.empty((B, LH, R, 2), np.int32)
        for b in range(B):
            for j in range(R):
                tag = pos[b] + j if (k[b] >= 0 and j <= k[b]) else -1000 - j
                kn[b, :, j, 0] = tag
                kn[b, :, j, 1] = np.arange(LH) + 100 * b
        vn = kn.copy()
        vn[..., 0] = -vn[..., 0] - 1
        out = oracle.kv_commit(kp, vp, kn, vn, k, pos, S, W, lib=lib)
        kp, vp = out["k_pool"], out["v_pool"]
        for b in range(B):
            for j in range(int(k[b]) + 1):
                sinks, ring = models[b]
                p = int(pos[b]) + j
                (sinks if p < S else ring).append(p)
        pos = pos + np.maximum(k + 1, 0)
        assert np.array_equal(out["pos"], pos)
        assert np.all(out["flags"] == 0)
        vs = oracle.kv_valid_slots(pos, S, W, lib=lib)
        for b in range(B):
            sinks, ring = models[b]
            want = sinks + list(ring)
            n = int(vs["len"][b])
            assert n == len(want) == min(int(pos[b]), C)
            sl = vs["slots"][b, :n]
            assert len(set(sl.tolist())) == n and np.all(vs["slots"][b, n:] == -1)
            for lh in range(LH):
                assert np.array_equal(kp[b, lh, sl, 0], want)
                assert np.array_equal(vp[b, lh, sl, 0], [-t - 1 for t in want])
                assert np.all(kp[b, lh, sl, 1] == lh + 100 * b)
    # k past the staged entries is invalid and writes nothing
    out = oracle.kv_commit(kp, vp, kn, vn, np.array([R, 0, 0], np.int32), pos, S, W, lib=lib)
    assert out["flags"][0] == oracle.KV_INVALID and out["pos"][0] == pos[0]
    assert np.array_equal(out["k_pool"][0], kp[0])


# ------------------------------------------------ draft KV window block table

def pin_window_block_table(lib):
    """Draft KV sliding-window page: the unit-test example of "block table 的
    裁剪方式" ([10, 60, 200, 64] -> [10, 60, 72, 64] at W = 64, K = 3, block 16),
    the bounds of "窗口数学" (block-aligned start, windowed length <= W + b - 1,
    the window reaching back to seq + K - W; the clone's width is the page's
    W / b + 1, widened to ceil((W + b - 1) / b) where that is larger, reading
    K4), and what
    the clone is for: every position p in [start, seq) maps through the clone
    to the block the full table gives it, and columns past `needed` are 0."""
    g = _golden("draft_window_example.json")
    blk = g["block_size"]
    table = np.arange(4 * 16, dtype=np.int32).reshape(4, 16) + 1000
    out = oracle.window_block_table(g["seq_lens"], table, g["W"], blk, g["K"], lib=lib)
    assert list(out["seq"]) == g["windowed_seq_lens"]
    rng = np.random.default_rng(51)
    for W, blk, K in ((64, 16, 3), (100, 16, 0), (7, 4, 2), (32, 32, 5), (5, 1, 1)):
        B, full = 40, rng.integers(1, 30)
        seq = rng.integers(0, min(full * blk + 1, 1 << 20), size=B).astype(np.int32)
        seq[:3] = [0, 1, full * blk]
        table = rng.integers(1, 1 << 30, size=(B, full)).astype(np.int32)
        out = oracle.window_block_table(seq, table, W, blk, K, lib=lib)
        mc = max(W // blk + 1, -(-(W + blk - 1) // blk))
        assert out["table"].shape == (B, mc)
        for b in range(B):
            s_ = int(seq[b])
            start = int(out["start_block"][b]) * blk
            lo = max(s_ + K - W, 0)
            assert start % blk == 0 and start <= lo < start + blk
            assert int(out["seq"][b]) == s_ - start
            assert s_ - start <= W + blk - 1 or start == 0
            need = int(out["needed"][b])
            assert need == -(-(s_ - start) // blk) <= mc
            for p in range(start, s_):
                assert out["table"][b, (p - start) // blk] == table[b, p // blk]
            assert np.all(out["table"][b, need:] == 0)
    bad = oracle.window_block_table([-1, 5], np.ones((2, 3), np.int32), 8, 4, 0, lib=lib)
    assert bad["flags"][0] == oracle.KV_INVALID and bad["seq"][0] == 0
    assert np.all(bad["table"][0] == 0) and bad["flags"][1] == 0


ALL_PINS += [pin_draft_sample_grid, pin_draft_then_verify_lossless, pin_draft_sample_invalid,
             pin_kv_slot_closed_form, pin_kv_commit_content, pin_window_block_table]


# ------------------------------------------------------------ token trees
# Readings T1-T3 of the oracle (multi-branch verification): the pages name
# token trees but give no rule for siblings; the pins below hold for any
# correct multi-draft rejection sampler and reduce to the pinned chain rule.

def _tree_batch(B, Lt_rows, Ld_rows, parent, tokens, temp):
    N, V = np.asarray(Lt_rows).shape
    Lt = np.ascontiguousarray(np.broadcast_to(np.asarray(Lt_rows, np.float32), (B, N, V)))
    Ld = np.ascontiguousarray(np.broadcast_to(np.asarray(Ld_rows, np.float32), (B, N, V)))
    par = np.ascontiguousarray(np.broadcast_to(np.asarray(parent, np.int32), (B, N)))
    tok = np.ascontiguousarray(np.broadcast_to(np.asarray(tokens, np.int32), (B, N)))
    return Lt, Ld, par, tok, np.full(B, temp, np.float32)


def pin_tree_chain_is_verify(lib):
    """A chain (parent[n] = n - 1) is the plain verification of 考点2 / 第三章:
    node n's target row is position n, its draft row position n, its token
    the draft token n - 1; the leaf's draft row is never read (NaN there
    changes nothing).  Every output equals the pinned chain oracle's."""
    rng = np.random.default_rng(41)
    B, gamma, V = 300, 4, 11
    T = np.float32(0.8)
    Lt = rng.normal(0, 1.5, size=(B, gamma + 1, V)).astype(np.float32)
    Ld = (Lt[:, :gamma] + rng.normal(0, 0.8, size=(B, gamma, V))).astype(np.float32)
    x = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    ua = rng.random((B, gamma), dtype=np.float32)
    ur = rng.random((B, gamma + 1), dtype=np.float32)
    temp = np.full(B, T, np.float32)
    ref = oracle.verify(Lt, Ld, x, ua, ur, temp, F32, lib=lib)
    Ldt = np.concatenate([Ld, np.full((B, 1, V), np.nan, np.float32)], axis=1)
    par = np.broadcast_to(np.arange(-1, gamma, dtype=np.int32), (B, gamma + 1))
    tok = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    uat = np.concatenate([np.zeros((B, 1), np.float32), ua], axis=1)
    out = oracle.tree_verify(Lt, Ldt, par, tok, uat, ur, temp, F32, lib=lib)
    assert np.array_equal(out["n"], ref["n"])
    assert np.array_equal(out["tokens"], ref["tokens"])
    assert np.array_equal(out["flags"], ref["flags"])
    for b in range(B):  # a chain's accepted nodes are 1 .. n
        assert list(out["nodes"][b, :out["n"][b]]) == list(range(1, out["n"][b] + 1))


def pin_tree_single_node(lib):
    """N = 1: the walk ends at the root and draws from softmax(Lt[0] / T) by
    the index-order inverse CDF (np.searchsorted on the cumulative sum,
    side='right')."""
    rng = np.random.default_rng(42)
    V, m = 13, 4000
    T = float(np.float32(1.3))
    lt = rng.normal(0, 2, size=(1, V)).astype(np.float32)
    u = _midgrid(m)
    Lt, Ld, par, tok, temp = _tree_batch(m, lt, np.zeros((1, V)), [-1], [0], T)
    out = oracle.tree_verify(Lt, Ld, par, tok, np.zeros((m, 1), np.float32), u[:, None], temp,
                             F32, lib=lib)
    p = softmax(lt[0].astype(np.float64) / T)
    cum = np.cumsum(p)
    want = np.searchsorted(cum, u.astype(np.float64) * cum[-1], side="right")
    far = np.min(np.abs(cum[None, :] / cum[-1] - u.astype(np.float64)[:, None]), 1) >= 1e-6
    assert np.all(out["n"] == 0) and np.all(out["tokens"][:, 0] >= 0)
    assert np.array_equal(out["tokens"][far, 0], want[far])


def pin_tree_rejected_token_stays_rejected(lib):
    """After sibling c is rejected with token x (u > P_t(x) / P_d(x), so
    P_t(x) < P_d(x)), every later residual has r(x) = 0: a later sibling with
    the same token is rejected whenever its u is positive.  Tree: root with
    four siblings all carrying the token whose target / draft ratio is
    smallest."""
    rng = np.random.default_rng(43)
    B, V = 2000, 6
    lt = rng.normal(0, 1, size=(5, V)).astype(np.float32)
    ld = rng.normal(0, 1, size=(5, V)).astype(np.float32)
    p0 = softmax(lt[0].astype(np.float64))
    q0 = softmax(ld[0].astype(np.float64))
    x = int(np.argmin(p0 / q0))
    a = p0[x] / q0[x]
    assert a < 0.9
    Lt, Ld, par, tok, temp = _tree_batch(B, lt, ld, [-1, 0, 0, 0, 0], [0, x, x, x, x], 1.0)
    ua = rng.random((B, 5), dtype=np.float32) * np.float32(0.999) + np.float32(1e-4)
    out = oracle.tree_verify(Lt, Ld, par, tok, ua, rng.random((B, 5), dtype=np.float32), temp,
                             F32, lib=lib)
    first = ua[:, 1].astype(np.float64) <= a
    assert np.all(out["nodes"][first, 0] == 1)  # the first sibling is tested by P_t / P_d
    assert np.all(out["n"][~first] == 0)        # later copies of x are never accepted
    assert np.all(out["tokens"][~first, 0] != x)


def pin_tree_losslessness(lib, trials=400_000):
    """Multi-draft form of the 考点2 identity: the root has three siblings and
    each of them two children, every sibling drawn independently from its
    parent's draft distribution; the first emitted token follows P_t[root]
    and, given that a depth-1 node was accepted, the second follows that
    node's target row (all depth-1 nodes share their rows).  Chi-square, 7
    degrees of freedom, rejected above 24.32 (p = 0.001)."""
    rng = np.random.default_rng(44)
    V = 8
    T = float(np.float32(0.9))
    lt0, lt1 = (rng.normal(0, 1.5, size=V).astype(np.float32) for _ in range(2))
    ld0, ld1 = (rng.normal(0, 1.5, size=V).astype(np.float32) for _ in range(2))
    parent = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3]
    N = len(parent)
    rows_t = np.stack([lt0] + [lt1] * 3 + [lt0] * 6)
    rows_d = np.stack([ld0] + [ld1] * 3 + [ld0] * 6)
    Pt0, Pt1 = (softmax(r.astype(np.float64) / T) for r in (lt0, lt1))
    Q0, Q1 = (softmax(r.astype(np.float64) / T) for r in (ld0, ld1))
    tok = np.zeros((trials, N), np.int32)
    for n in range(1, 4):
        tok[:, n] = rng.choice(V, size=trials, p=Q0)
    for n in range(4, N):
        tok[:, n] = rng.choice(V, size=trials, p=Q1)
    Lt, Ld, par, _, temp = _tree_batch(trials, rows_t, rows_d, parent, np.zeros(N), T)
    out = oracle.tree_verify(Lt, Ld, par, tok, rng.random((trials, N), dtype=np.float32),
                             rng.random((trials, N), dtype=np.float32), temp, F32, lib=lib)
    assert np.all(out["tokens"][:, 0] >= 0)
    for pos, P, sel in ((0, Pt0, np.ones(trials, bool)), (1, Pt1, out["n"] >= 1)):
        obs = np.bincount(out["tokens"][sel, pos], minlength=V)
        exp_ = P * sel.sum()
        chi2 = float(((obs - exp_) ** 2 / exp_).sum())
        assert chi2 < 24.32, (pos, chi2)


def pin_tree_invalid(lib):
    """Readings T2/T3: a malformed parent array or an out-of-range token makes
    the request invalid; NaN in a row the walk reads invalidates it, NaN in a
    row off the walk does not."""
    V = 5
    lt = np.zeros((4, V), np.float32)
    lt[:, 2] = 3.0  # every target row puts nearly all mass on token 2
    ld = np.zeros((4, V), np.float32)
    ld[:, 2] = 3.0
    parent = [-1, 0, 0, 1]
    Lt, Ld, par, tok, temp = _tree_batch(6, lt, ld, parent, [0, 2, 1, 2], 1.0)
    Lt, Ld, par, tok = Lt.copy(), Ld.copy(), par.copy(), tok.copy()
    ua = np.full((6, 4), 0.01, np.float32)  # node 1 (token 2, ratio 1) is always accepted
    ur = np.full((6, 4), 0.5, np.float32)
    par[1, 2] = 2     # parent not before the node
    tok[2, 3] = V     # token out of range
    Lt[3, 2, 0] = np.nan  # node 2 is never visited: its row is not read
    Ld[3, 3, 1] = np.nan  # node 3 is a leaf: its draft row is not read
    Lt[4, 3, 4] = np.inf  # node 3's target row is read (the walk ends there)
    temp[5] = 0.0
    out = oracle.tree_verify(Lt, Ld, par, tok, ua, ur, temp, F32, lib=lib)
    assert out["flags"][1] & oracle.INVALID_TOKEN and out["flags"][2] & oracle.INVALID_TOKEN
    assert out["flags"][4] & oracle.INVALID_NONFINITE and out["flags"][5] & oracle.INVALID_TEMP
    for b in (1, 2, 4, 5):
        assert out["n"][b] == 0 and np.all(out["tokens"][b] == -1) and np.all(out["nodes"][b] == -1)
    for b in (0, 3):
        assert out["flags"][b] & oracle.INVALID_ANY == 0
        assert list(out["nodes"][b, :2]) == [1, 3] and list(out["tokens"][b, :3]) == [2, 2, 2]


ALL_PINS += [pin_tree_chain_is_verify, pin_tree_single_node,
             pin_tree_rejected_token_stays_rejected, pin_tree_losslessness, pin_tree_invalid]
