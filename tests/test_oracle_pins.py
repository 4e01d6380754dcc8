"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test checks the oracle against something the pages or the mathematics
fix: closed forms, library routines on special cases, brute force on tiny
inputs, the exactness theorem of speculative sampling ("SSD: drafting and
verification on separate GPUs", "What changes in SSD": the method is exact;
Leviathan et al. 2023 / Chen et al. 2023), and hand-worked examples stored
under tests/golden/.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import scipy.stats

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def softmax_ref(z, T):
    return scipy.special.softmax(np.asarray(z, dtype=np.float64) / T, axis=-1)


# ---------------------------------------------------------------------------
# temperature softmax
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 5, 1000])
@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_softmax_equal_logits_is_uniform(V, T):
    z = np.full((1, V), 3.75, dtype=np.float32)
    r = oracle.softmax_temp(z, [T])
    assert np.all(np.abs(r["probs"] - 1.0 / V) <= 1e-15)
    assert r["row_sum"][0] == V
    assert r["row_max"][0] == 3.75
    assert r["row_argmax"][0] == 0


def test_softmax_rational_closed_form():
    # z = ln(1..4): p = (1,2,3,4)/10 at T=1 and (1,4,9,16)/30 at T=1/2
    z = np.log(np.array([[1, 2, 3, 4]], dtype=np.float64)).astype(np.float32)
    r1 = oracle.softmax_temp(z, [1.0])["probs"][0]
    zz = z.astype(np.float64)[0]
    expect1 = np.exp(zz) / np.exp(zz).sum()
    assert np.allclose(r1, [0.1, 0.2, 0.3, 0.4], atol=2e-7)  # z rounded to binary32
    assert np.allclose(r1, expect1, atol=1e-15)
    r2 = oracle.softmax_temp(z, [0.5])["probs"][0]
    assert np.allclose(r2, np.array([1, 4, 9, 16]) / 30.0, atol=5e-7)


def test_softmax_matches_scipy():
    rng = np.random.default_rng(5)
    z = (rng.standard_normal((6, 777)) * 3).astype(np.float32)
    T = np.array([0.3, 0.5, 0.7, 1.0, 1.2, 4.0], dtype=np.float32)
    r = oracle.softmax_temp(z, T)
    ref = softmax_ref(z, T.astype(np.float64)[:, None])
    assert np.max(np.abs(r["probs"] - ref)) < 1e-14
    assert np.array_equal(r["row_argmax"], np.argmax(z, axis=1))
    assert np.array_equal(r["row_max"], z.max(axis=1).astype(np.float64))


def test_softmax_greedy_and_ties():
    z = np.array([[1.0, 5.0, 5.0, -2.0], [7.0, 7.0, 7.0, 7.0]], dtype=np.float32)
    r = oracle.softmax_temp(z, [0.0, 0.0])
    assert list(r["row_argmax"]) == [1, 0]  # lowest index wins ties
    assert np.array_equal(r["probs"], np.array([[0, 1, 0, 0], [1, 0, 0, 0]], dtype=np.float64))
    assert list(r["row_sum"]) == [1.0, 1.0]


def test_softmax_infinities_and_invalid_rows():
    ninf, nan = -np.inf, np.nan
    z = np.array([[0.0, ninf, 1.0, ninf],     # -inf -> probability 0
                  [ninf, ninf, ninf, ninf],   # all -inf at T>0: invalid
                  [0.0, nan, 1.0, 2.0],       # NaN: invalid
                  [0.0, 1.0, 2.0, 3.0],       # T < 0: invalid
                  [ninf, ninf, ninf, ninf]],  # all -inf at T=0: argmax 0
                 dtype=np.float32)
    r = oracle.softmax_temp(z, [1.0, 1.0, 1.0, -1.0, 0.0])
    p0 = r["probs"][0]
    assert p0[1] == 0 and p0[3] == 0
    assert abs(p0[2] / p0[0] - math.e) < 1e-12
    for i in (1, 2, 3):
        assert r["row_argmax"][i] == -1 and np.isnan(r["row_max"][i])
        assert np.all(np.isnan(r["probs"][i]))
    assert r["row_argmax"][4] == 0


def test_bf16_widening():
    # bf16 bit patterns: 1.0, -2.0, 0.5, 3.0 (0x4040)
    bits = np.array([[0x3F80, 0xC000, 0x3F00, 0x4040]], dtype=np.uint16)
    r = oracle.softmax_temp(bits, [1.0])
    assert r["row_max"][0] == 3.0 and r["row_argmax"][0] == 3
    ref = softmax_ref([1.0, -2.0, 0.5, 3.0], 1.0)
    assert np.max(np.abs(r["probs"][0] - ref)) < 1e-15


# ---------------------------------------------------------------------------
# exactness by exact enumeration (V = 4, k = 2)
# ---------------------------------------------------------------------------
def _call(Z, D, x, T, ua, us):
    r = oracle.verify_recover(Z[None], D[None], np.asarray(x, dtype=np.int32)[None],
                              [T], np.asarray(ua, dtype=np.float64)[None],
                              [us], f64_uniforms=True)
    return int(r["accept_len"][0]), [int(t) for t in r["out_tok"][0]]


def _boundary(pred, lo=0.0, hi=1.0, iters=64):
    """sup{u in [lo,hi) : pred(u) == pred(lo)} for a predicate that changes
    value at most once on [lo, hi)."""
    a = pred(lo)
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        if pred(mid) == a:
            lo = mid
        else:
            hi = mid
    return lo


def _measure(pred):
    """Lebesgue measure of {u in [0,1): pred(u)} for a one-switch predicate."""
    b = _boundary(pred)
    return b if pred(0.0) else 1.0 - b


def _token_distribution(tok_of_u, V):
    """Distribution of a non-decreasing token-valued function of u ~ U[0,1)."""
    probs = np.zeros(V)
    prev = 0.0
    for t in range(V):
        b = _boundary(lambda u: tok_of_u(u) <= t) if tok_of_u(0.0) <= t else 0.0
        if t == V - 1:
            b = 1.0
        probs[t] = max(0.0, b - prev)
        prev = max(prev, b)
    return probs


def _split(pred):
    """For a predicate on u in [0,1) that switches value at most once, return
    (measure of the True set, a point inside it, a point inside the False set);
    points are None for empty sets."""
    b = _boundary(pred)
    if pred(0.0):  # True on [0, b)
        t_pt, f_pt, m = b / 2, (b + 1.0) / 2, b
    else:          # True on [b, 1)
        t_pt, f_pt, m = (b + 1.0) / 2, b / 2, 1.0 - b
    return m, (t_pt if m > 0 else None), (f_pt if m < 1 else None)


def enumerate_output_distribution(Z, D, T, call=None, filt=None):
    """Exact law of the 3-token sequence produced by the oracle (one verify
    round, then completion from the target rows), draft tokens drawn from q.
    Acceptance probabilities are the measures of the accepting uniforms and
    token laws come from the break points of the oracle's draw as a function
    of u_smp, all located by bisection on the oracle itself.  `call` replaces
    the oracle entry point and `filt(z_row, p_row)` the distributions (for
    the filtered step)."""
    global _call
    V = Z.shape[1]
    p = softmax_ref(Z.astype(np.float64), T)
    q = softmax_ref(D.astype(np.float64), T)
    if filt is not None:
        p = np.stack([filt(Z[i], p[i]) for i in range(p.shape[0])])
        q = np.stack([filt(D[i], q[i]) for i in range(q.shape[0])])
    saved = _call
    if call is not None:
        _call = call
    try:
        return _enumerate(Z, D, T, V, p, q)
    finally:
        _call = saved


def _enumerate(Z, D, T, V, p, q):
    law = np.zeros((V,) * 3)
    for x0, x1 in itertools.product(range(V), repeat=2):
        wx = q[0, x0] * q[1, x1]
        if wx == 0:
            continue
        x = [x0, x1]
        a0, acc0, rej0 = _split(lambda u: _call(Z, D, x, T, [u, 0.5], 0.5)[0] >= 1)
        if rej0 is not None:  # one token from the residual of position 0
            dist = _token_distribution(lambda u: _call(Z, D, x, T, [rej0, 0.5], u)[1][0], V)
            law += wx * (1 - a0) * np.einsum("i,j,k->ijk", dist, p[1], p[2])
        if acc0 is not None:
            a1, acc1, rej1 = _split(lambda u: _call(Z, D, x, T, [acc0, u], 0.5)[0] >= 2)
            if rej1 is not None:
                dist = _token_distribution(lambda u: _call(Z, D, x, T, [acc0, rej1], u)[1][1], V)
                law[x0] += wx * a0 * (1 - a1) * np.outer(dist, p[2])
            if acc1 is not None:
                dist = _token_distribution(lambda u: _call(Z, D, x, T, [acc0, acc1], u)[1][2], V)
                law[x0, x1] += wx * a0 * a1 * dist
    return law, p, q


@pytest.mark.parametrize("seed", [0, 1, 2])
@pytest.mark.parametrize("T", [1.0, 0.6])
def test_exactness_by_enumeration(seed, T):
    T = float(np.float32(T))  # the oracle takes binary32 temperatures
    rng = np.random.default_rng(100 + seed)
    Z = (rng.standard_normal((3, 4)) * 1.5).astype(np.float32)
    D = (Z[:2] + rng.standard_normal((2, 4)) * 1.0).astype(np.float32)
    law, p, q = enumerate_output_distribution(Z, D, T)
    target = np.einsum("i,j,k->ijk", p[0], p[1], p[2])
    assert abs(law.sum() - 1.0) < 1e-12
    assert np.max(np.abs(law - target)) < 1e-12


def _filter_ref(z, p, K, top_p):
    """R9 written out independently: order by (logit desc, index asc), keep the
    first K, then the shortest prefix holding >= top_p of their mass."""
    order = sorted(range(len(z)), key=lambda v: (-float(z[v]), v))[:K]
    mass = sum(p[v] for v in order)
    keep, c = [], 0.0
    for v in order:
        keep.append(v)
        c += p[v]
        if c >= top_p * mass:
            break
    out = np.zeros_like(p)
    kept = sum(p[v] for v in keep)
    for v in keep:
        out[v] = p[v] / kept
    return out


@pytest.mark.parametrize("K,top_p", [(3, 1.0), (4, 0.7), (2, 0.5)])
def test_filtered_exactness_by_enumeration(K, top_p):
    """Over top-k / top-p filtered distributions the step reproduces the
    filtered target law exactly (V = 5, k = 2)."""
    rng = np.random.default_rng(7 + K)
    T = float(np.float32(0.9))
    Z = (rng.standard_normal((3, 5)) * 1.5).astype(np.float32)
    D = (Z[:2] + rng.standard_normal((2, 5))).astype(np.float32)

    def call(Z_, D_, x, T_, ua, us):
        r = oracle.verify_recover_filtered(Z_[None], D_[None], np.asarray(x, np.int32)[None], [T_],
                                           K, [top_p], np.asarray(ua, np.float64)[None], [us],
                                           f64_uniforms=True)
        return int(r["accept_len"][0]), [int(t) for t in r["out_tok"][0]]

    filt = lambda z, p: _filter_ref(z, p, K, top_p)
    law, p, q = enumerate_output_distribution(Z, D, T, call=call, filt=filt)
    target = np.einsum("i,j,k->ijk", p[0], p[1], p[2])
    assert abs(law.sum() - 1.0) < 1e-12
    assert np.max(np.abs(law - target)) < 1e-12
    assert (p > 0).sum(axis=1).max() <= K


def test_filtered_reduces_to_unfiltered_and_probabilities():
    rng = np.random.default_rng(5)
    B, k, V = 6, 3, 12
    Z = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    D = (Z[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    x = rng.integers(0, V, size=(B, k)).astype(np.int32)
    T = np.array([1.0, 0.7, 0.0, 1.3, 0.9, 0.5], np.float32)
    ua = rng.random((B, k)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    plain = oracle.verify_recover(Z, D, x, T, ua, us)
    full = oracle.verify_recover_filtered(Z, D, x, T, V, None, ua, us)
    for key in ("accept_len", "out_tok"):
        assert np.array_equal(plain[key], full[key])
    assert np.allclose(plain["p_at_x"], full["p_at_x"], atol=1e-15, equal_nan=True)
    K, tp = 4, np.full(B, 0.8, np.float32)
    r = oracle.verify_recover_filtered(Z, D, x, T, K, tp, ua, us)
    for b in range(B):
        if T[b] == 0:
            continue
        for i in range(k):
            if i > 0 and r["accept_len"][b] < i:
                break
            p = _filter_ref(Z[b, i], softmax_ref(Z[b, i].astype(np.float64)[None], T[b])[0], K, 0.8)
            assert abs(r["p_at_x"][b, i] - p[x[b, i]]) < 1e-12


def test_exactness_detects_a_wrong_residual():
    """The enumeration is sensitive: drawing the recovery token from p_n
    (dropping the -q_n term) breaks the law.  Computed here in numpy from the
    same enumeration formula, not from the oracle."""
    rng = np.random.default_rng(7)
    Z = (rng.standard_normal((3, 4)) * 1.5).astype(np.float32)
    D = (Z[:2] + rng.standard_normal((2, 4))).astype(np.float32)
    p = softmax_ref(Z.astype(np.float64), 1.0)
    q = softmax_ref(D.astype(np.float64), 1.0)
    acc = np.minimum(1.0, p[0] / q[0])
    first = (q[0] * acc) + (1 - (q[0] * acc).sum()) * p[0]  # wrong residual
    assert np.max(np.abs(first - p[0])) > 1e-3


# ---------------------------------------------------------------------------
# statistics on the uniform-driven path (V = 8, k = 2, 10^6 rows)
# ---------------------------------------------------------------------------
def _draw_from(probs, u):
    c = np.cumsum(probs, axis=-1)
    return np.minimum((u[..., None] >= c[None, :]).sum(-1), len(probs) - 1)


@pytest.fixture(scope="module")
def stat_run():
    rng = np.random.default_rng(2024)
    V, k, N = 8, 2, 1_000_000
    Z = (rng.standard_normal((k + 1, V)) * 1.2).astype(np.float32)
    D = (Z[:k] + rng.standard_normal((k, V)) * 0.8).astype(np.float32)
    T = 0.9
    p = softmax_ref(Z.astype(np.float64), T)
    q = softmax_ref(D.astype(np.float64), T)
    x = np.stack([_draw_from(q[i], rng.random(N)) for i in range(k)], axis=1).astype(np.int32)
    ua = rng.random((N, k)).astype(np.float32)
    us = rng.random(N).astype(np.float32)
    Zb = np.broadcast_to(Z, (N, k + 1, V)).copy()
    Db = np.broadcast_to(D, (N, k, V)).copy()
    r = oracle.verify_recover(Zb, Db, x, np.full(N, T, np.float32), ua, us)
    # complete every row to 3 tokens with independent draws from the target
    seq = np.full((N, 3), -1, dtype=np.int64)
    n = r["accept_len"]
    out = r["out_tok"]
    for j in range(3):
        have = j <= n
        seq[have, j] = out[have, j]
        fill = ~have
        seq[fill, j] = _draw_from(p[j], rng.random(fill.sum()))
    return {"p": p, "q": q, "n": n, "seq": seq, "N": N, "V": V}


@pytest.mark.slow
def test_chi_square_sequences(stat_run):
    p, seq, N, V = stat_run["p"], stat_run["seq"], stat_run["N"], stat_run["V"]
    idx = seq[:, 0] * V * V + seq[:, 1] * V + seq[:, 2]
    obs = np.bincount(idx, minlength=V ** 3).astype(np.float64)
    exp = np.einsum("i,j,k->ijk", p[0], p[1], p[2]).reshape(-1) * N
    small = exp < 5
    o = np.append(obs[~small], obs[small].sum())
    e = np.append(exp[~small], exp[small].sum())
    if e[-1] == 0:
        o, e = o[:-1], e[:-1]
    pval = scipy.stats.chisquare(o, e).pvalue
    assert pval > 1e-3, pval
    first = np.bincount(seq[:, 0], minlength=V)
    assert scipy.stats.chisquare(first, p[0] * N).pvalue > 1e-3


@pytest.mark.slow
def test_acceptance_rate_closed_form(stat_run):
    p, q, n, N = stat_run["p"], stat_run["q"], stat_run["n"], stat_run["N"]
    rate = np.minimum(p[0], q[0]).sum()
    emp = (n >= 1).mean()
    sigma = math.sqrt(rate * (1 - rate) / N)
    assert abs(emp - rate) < 5 * sigma


def test_special_cases_p_equals_q_and_one_hot_q():
    rng = np.random.default_rng(3)
    V, k = 6, 3
    Z = (rng.standard_normal((1, k + 1, V))).astype(np.float32)
    # q == p: every draft token is accepted for every u < 1
    for u in (0.0, 0.5, 0.999999):
        r = oracle.verify_recover(Z, Z[:, :k].copy(), [[0, 3, 5]], [1.0], [[u] * k], [0.3])
        assert r["accept_len"][0] == k
    # one-hot q at a: accepted with probability p(a)
    a = 2
    D = np.full((1, k, V), -np.inf, dtype=np.float32)
    D[0, :, a] = 0.0
    pa = softmax_ref(Z[0, 0].astype(np.float64), 1.0)[a]
    grid = (np.arange(4000) + 0.5) / 4000
    acc = [oracle.verify_recover(Z, D, [[a] * k], [1.0], [[u, 0, 0]], [0.5])["accept_len"][0] >= 1
           for u in grid]
    assert abs(np.mean(acc) - pa) <= 1.0 / 4000
    # after rejecting the one-hot draft, the residual is p with a removed
    r = oracle.verify_recover(Z, D, [[a] * k], [1.0], [[0.999999, 0, 0]], [0.0])
    assert r["accept_len"][0] == 0
    w = softmax_ref(Z[0, 0].astype(np.float64), 1.0)
    w[a] = 0
    assert r["out_tok"][0, 0] == int(np.argmax(w > 0))


def test_inverse_cdf_brute_force_rational():
    """Logits ln(a), ln(b) with small integers make p, q rational; the drawn
    token must satisfy C_{j-1} <= u*W < C_j in exact arithmetic."""
    a = [3, 1, 4, 1, 5, 9, 2, 6]
    b = [2, 7, 1, 8, 2, 8, 1, 8]
    Z = np.log(np.array([a, a], dtype=np.float64)).astype(np.float32)[None]
    D = np.log(np.array([b], dtype=np.float64)).astype(np.float32)[None]
    # exact p, q of the binary32 logits: use the widened values
    zp = np.exp(Z[0, 0].astype(np.float64)); zp /= zp.sum()
    dq = np.exp(D[0, 0].astype(np.float64)); dq /= dq.sum()
    w = np.maximum(0, zp - dq)
    C = np.cumsum(w)
    x = 3  # q(3) = 8/37 > p(3) = 1/31: rejected for u close to 1
    for u in np.linspace(0.0, 0.999, 97):
        r = oracle.verify_recover(Z, D, [[x]], [1.0], [[0.99999]], [u], f64_uniforms=True)
        assert r["accept_len"][0] == 0
        j = int(r["out_tok"][0, 0])
        t = u * C[-1]
        lo = C[j - 1] if j > 0 else 0.0
        assert lo - 1e-15 <= t < C[j] + 1e-15 and w[j] > 0
    # u = 0 picks the first token with positive residual
    r = oracle.verify_recover(Z, D, [[x]], [1.0], [[0.99999]], [0.0])
    assert r["out_tok"][0, 0] == int(np.argmax(w > 0))
    # exact fractions for one interior point
    pa = [Fraction(v, sum(a)) for v in a]
    qb = [Fraction(v, sum(b)) for v in b]
    wf = [max(Fraction(0), pa[i] - qb[i]) for i in range(8)]
    Cf = list(itertools.accumulate(wf))
    u = 0.61
    r = oracle.verify_recover(Z, D, [[x]], [1.0], [[0.99999]], [u], f64_uniforms=True)
    j = int(r["out_tok"][0, 0])
    t = Fraction(u) * Cf[-1]
    assert (Cf[j - 1] if j else 0) <= t < Cf[j]


def test_residual_all_zero_falls_back_to_p():
    # x has p(x) = q(x) = 0 (logit -inf in both): rejected, w == 0 everywhere
    Z = np.array([[[0.0, 1.0, -np.inf, 2.0], [0.0, 0.0, 0.0, 0.0]]], dtype=np.float32)
    D = Z[:, :1].copy()
    p = softmax_ref(Z[0, 0].astype(np.float64), 1.0)
    for u in (0.0, 0.2, 0.5, 0.9):
        r = oracle.verify_recover(Z, D, [[2]], [1.0], [[0.1]], [u], f64_uniforms=True)
        assert r["accept_len"][0] == 0
        j = int(r["out_tok"][0, 0])
        C = np.cumsum(p)
        assert (C[j - 1] if j else 0) <= u * C[-1] < C[j]


# ---------------------------------------------------------------------------
# greedy
# ---------------------------------------------------------------------------
def test_greedy_matches_argmax_agreement():
    rng = np.random.default_rng(11)
    B, k, V = 64, 5, 50
    Z = rng.integers(-3, 4, size=(B, k + 1, V)).astype(np.float32)  # many ties
    D = rng.integers(-3, 4, size=(B, k, V)).astype(np.float32)
    am = np.argmax(Z, axis=2)  # numpy: first occurrence wins
    x = np.where(rng.random((B, k)) < 0.7, am[:, :k], rng.integers(0, V, (B, k))).astype(np.int32)
    r = oracle.verify_recover(Z, D, x, np.zeros(B, np.float32), rng.random((B, k)), rng.random(B))
    for b in range(B):
        n = 0
        while n < k and x[b, n] == am[b, n]:
            n += 1
        assert r["accept_len"][b] == n
        assert list(r["out_tok"][b, :n]) == list(x[b, :n])
        assert r["out_tok"][b, n] == am[b, n]
        assert all(t == -1 for t in r["out_tok"][b, n + 1:])
        for i in range(k):
            assert r["p_at_x"][b, i] == float(x[b, i] == am[b, i])
            assert r["q_at_x"][b, i] == float(x[b, i] == np.argmax(D[b, i]))


def test_sentinels():
    Z = np.zeros((4, 3, 5), dtype=np.float32)
    D = np.zeros((4, 2, 5), dtype=np.float32)
    x = np.array([[0, 1], [0, 7], [0, 1], [0, 1]], dtype=np.int32)
    T = np.array([-1.0, 1.0, 1.0, np.nan], dtype=np.float32)
    Z[2, 1, 3] = np.nan
    r = oracle.verify_recover(Z, D, x, T, np.zeros((4, 2)), np.zeros(4))
    assert list(r["accept_len"]) == [-1, -2, -1, -1]
    assert np.all(r["out_tok"] == -1)
    assert np.all(np.isnan(r["p_at_x"]))


# ---------------------------------------------------------------------------
# forked top-f
# ---------------------------------------------------------------------------
def test_topf_matches_full_sort():
    rng = np.random.default_rng(21)
    B, P, V, f, M = 3, 4, 300, 5, 2
    L = rng.integers(-20, 20, size=(B, P, V)).astype(np.float32) / 4  # ties
    mask = rng.integers(-1, V, size=(B, P, M)).astype(np.int32)
    r = oracle.forked_topf(L, f, mask)
    for b in range(B):
        for j in range(P):
            keep = np.ones(V, bool)
            for t in mask[b, j]:
                if t >= 0:
                    keep[t] = False
            idx = np.nonzero(keep)[0]
            order = idx[np.lexsort((idx, -L[b, j, idx]))][:f]
            assert list(r["fork_tok"][b, j]) == list(order)
            assert np.array_equal(r["fork_logit"][b, j], L[b, j, order].astype(np.float64))


def test_topf_variable_fanout_is_a_prefix_of_the_full_sort():
    rng = np.random.default_rng(12)
    B, P, V, F = 3, 5, 40, 4
    L = rng.integers(-6, 6, size=(B, P, V)).astype(np.float32)   # many ties
    fan = [4, 0, 2, 7, -1]
    r = oracle.forked_topf(L, F, fanout=fan)
    for b in range(B):
        for j in range(P):
            keep = min(max(fan[j], 0), F)
            order = sorted(range(V), key=lambda v: (-L[b, j, v], v))
            assert r["fork_tok"][b, j, :keep].tolist() == order[:keep]
            assert (r["fork_tok"][b, j, keep:] == -1).all()
            assert np.isneginf(r["fork_logit"][b, j, keep:]).all()


def test_topf_padding_and_nan():
    L = np.array([[[1.0, 2.0, 3.0], [1.0, np.nan, 0.0]]], dtype=np.float32)
    mask = np.array([[[0, 1], [-1, -1]]], dtype=np.int32)
    r = oracle.forked_topf(L, 2, mask)
    assert list(r["fork_tok"][0, 0]) == [2, -1]
    assert r["fork_logit"][0, 0, 1] == -np.inf
    assert list(r["fork_tok"][0, 1]) == [-1, -1]
    assert np.all(np.isnan(r["fork_logit"][0, 1]))


# ---------------------------------------------------------------------------
# golden hand-worked cases
# ---------------------------------------------------------------------------
def _golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def test_golden_verify_cases():
    g = _golden("verify_cases.json")
    for case in g["cases"]:
        Z = np.log(np.array(case["target_weights"], dtype=np.float64)).astype(np.float32)[None]
        D = np.log(np.array(case["draft_weights"], dtype=np.float64)).astype(np.float32)[None]
        r = oracle.verify_recover(Z, D, [case["x"]], [case["T"]], [case["u_acc"]],
                                  [case["u_smp"]], f64_uniforms=True)
        assert r["accept_len"][0] == case["accept_len"], case["name"]
        assert list(r["out_tok"][0]) == case["out_tok"], case["name"]
        for i, pv in enumerate(case["p_at_x"]):
            assert abs(r["p_at_x"][0, i] - pv) < 1e-6, case["name"]


def test_golden_cache_cases():
    g = _golden("cache_cases.json")
    c = oracle.SpecCacheOracle(g["depth"])
    for step in g["steps"]:
        if step["op"] == "insert":
            c.insert(step["b"], step["pos"], step["tok"], np.array(step["payload"]))
        elif step["op"] == "clear":
            c.clear()
        else:
            hit, out = c.lookup(step["b"], step["pos"], step["tok"])
            assert list(hit) == step["hit"]
            assert out.tolist() == step["tok_out"]


# ---------------------------------------------------------------------------
# draft-side sampling (Gumbel-max with Philox4x32-10 uniforms)
# ---------------------------------------------------------------------------
def test_philox_known_answers():
    """Known-answer vectors of Philox4x32-10 published with the generator's
    reference code (Salmon et al. 2011, "Parallel random numbers: as easy as
    1, 2, 3"; the Random123 known-answer tests)."""
    kat = [
        ([0, 0, 0, 0], [0, 0], [0x6627e8d5, 0xe169c58d, 0xbc57ac4c, 0x9b00dbd8]),
        ([0xffffffff] * 4, [0xffffffff] * 2, [0x408f276d, 0x41c83b0e, 0xa20bc7c6, 0x6d5451fd]),
        ([0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344], [0xa4093822, 0x299f31d0],
         [0xd16cfe09, 0x94fdcceb, 0x5001e420, 0x24126ea1]),
    ]
    for ctr, key, want in kat:
        assert oracle.philox4x32_10(ctr, key).tolist() == want


def test_gumbel_max_draws_follow_the_softmax():
    """argmax(z/T + Gumbel) is a draw from softmax(z/T): frequencies over
    200000 independent rows (distinct b) against the closed form."""
    V, N, T = 6, 200_000, 0.8
    z = np.array([0.3, -1.0, 2.0, 0.0, 1.1, -3.0], dtype=np.float32)
    D = np.broadcast_to(z, (N, 1, V)).copy()
    x = oracle.draft_sample(D, np.full(N, T, np.float32), seed=0x1234_5678_9abc, offset=3)
    p = softmax_ref(z.astype(np.float64)[None], T)[0]
    obs = np.bincount(x[:, 0], minlength=V)
    assert scipy.stats.chisquare(obs, p * N).pvalue > 1e-3
    # a different offset gives different draws (fresh uniforms), same law
    x2 = oracle.draft_sample(D, np.full(N, T, np.float32), seed=0x1234_5678_9abc, offset=4)
    assert (x2 != x).mean() > 0.3
    assert scipy.stats.chisquare(np.bincount(x2[:, 0], minlength=V), p * N).pvalue > 1e-3


def test_draft_sample_special_cases():
    V = 9
    z = np.array([[[1.0, 5.0, 5.0, -2.0, 0.0, 3.0, -np.inf, 4.0, 5.0]]], dtype=np.float32)
    D = np.repeat(z, 4, axis=0)
    T = np.array([0.0, -1.0, np.nan, 1.0], dtype=np.float32)
    x = oracle.draft_sample(D, T, seed=7, offset=0)
    assert x[:, 0].tolist()[:3] == [1, -1, -1]      # greedy: lowest index of the maximum
    assert 0 <= x[3, 0] < V and x[3, 0] != 6        # -inf is never drawn
    one = np.full((3, 1, V), -np.inf, dtype=np.float32)
    one[:, 0, 4] = 0.0                               # a one-hot row
    assert (oracle.draft_sample(one, np.ones(3, np.float32), seed=1, offset=1) == 4).all()
    bad = z.copy()
    bad[0, 0, 2] = np.nan
    assert oracle.draft_sample(bad, np.ones(1, np.float32), seed=1, offset=1)[0, 0] == -1


# ---------------------------------------------------------------------------
# token-tree verification (multi-step speculative sampling over a tree)
# ---------------------------------------------------------------------------
def _tree_call(Z, D, par, tok, T, ua, us):
    r = oracle.verify_tree(Z[None], D[None], np.asarray(par, np.int32)[None],
                           np.asarray(tok, np.int32)[None], [T],
                           np.asarray(ua, np.float64)[None], [us], f64_uniforms=True)
    return int(r["accept_len"][0]), [int(t) for t in r["out_tok"][0]], \
        [int(n) for n in r["out_node"][0]]


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_tree_exactness_by_enumeration(seed):
    """Exactness of the tree rule (SpecInfer's multi-step speculative
    sampling; "SSD: drafting and verification on separate GPUs": the method
    does not change the output law).  Tree: root with children 1 and 2
    (tokens drawn independently from the root's q), node 1 with child 3
    (token drawn from node 1's q).  The law of the first two output tokens
    (completed from the target when only one is produced) must be
    p_root(t1) * p_t1(t2), where p_v is the target law after token v.  All
    measures come from bisection on the oracle; V = 3."""
    rng = np.random.default_rng(300 + seed)
    V, T = 3, float(np.float32(0.8))
    Zr = (rng.standard_normal(V) * 1.5).astype(np.float32)
    Dr = (Zr + rng.standard_normal(V) * 1.5).astype(np.float32)
    Zc = (rng.standard_normal((V, V)) * 1.5).astype(np.float32)      # target after token v
    Dc = (Zc + rng.standard_normal((V, V)) * 1.5).astype(np.float32)
    Zg = rng.standard_normal(V).astype(np.float32)
    pr, qr = softmax_ref(Zr, T), softmax_ref(Dr, T)
    pc, qc = softmax_ref(Zc, T), softmax_ref(Dc, T)
    par = [-1, 0, 0, 1]
    law = np.zeros((V, V))
    for x1, x2, y in itertools.product(range(V), repeat=3):
        w = qr[x1] * qr[x2] * qc[x1, y]
        Z = np.stack([Zr, Zc[x1], Zc[x2], Zg])
        D = np.stack([Dr, Dc[x1], Dc[x2], Dr])
        tok = [0, x1, x2, y]
        call = lambda u1, u2, u3, us: _tree_call(Z, D, par, tok, T, [0.5, u1, u2, u3], us)
        a1, acc1, rej1 = _split(lambda u: call(u, 0.5, 0.5, 0.5)[2][0] == 1)
        if acc1 is not None:
            a3, acc3, rej3 = _split(lambda u: call(acc1, 0.5, u, 0.5)[2][1] == 3)
            if acc3 is not None:
                law[x1, y] += w * a1 * a3
            if rej3 is not None:
                dist = _token_distribution(lambda u: call(acc1, 0.5, rej3, u)[1][1], V)
                law[x1] += w * a1 * (1 - a3) * dist
        if rej1 is not None:
            a2, acc2, rej2 = _split(lambda u: call(rej1, u, 0.5, 0.5)[2][0] == 2)
            if acc2 is not None:
                dist = _token_distribution(lambda u: call(rej1, acc2, 0.5, u)[1][1], V)
                law[x2] += w * (1 - a1) * a2 * dist
            if rej2 is not None:
                dist = _token_distribution(lambda u: call(rej1, rej2, 0.5, u)[1][0], V)
                law += w * (1 - a1) * (1 - a2) * dist[:, None] * pc
    target = pr[:, None] * pc
    assert abs(law.sum() - 1.0) < 1e-12
    assert np.max(np.abs(law - target)) < 1e-12


def test_tree_exactness_detects_a_missing_residual_update():
    """The enumeration is sensitive: trying the second child against the
    unchanged p (no residual update after the first rejection) changes the
    law of the first token.  Computed here in numpy for two leaf children."""
    rng = np.random.default_rng(9)
    p = softmax_ref(rng.standard_normal(4) * 1.5, 1.0)
    q = softmax_ref(rng.standard_normal(4) * 1.5, 1.0)
    a = np.minimum(1.0, p / q)
    rej1 = 1 - (q * a).sum()
    wrong = q * a + rej1 * (q * a) + rej1 * (1 - (q * a).sum()) * p
    assert np.max(np.abs(wrong - p)) > 1e-3


def test_tree_chain_is_the_chain_rule():
    """A tree that is a chain (parent[j] = j - 1, tok[j] = x[j-1]) gives the
    chain verify-and-recover step's tokens."""
    rng = np.random.default_rng(41)
    B, k, V = 96, 4, 20
    Z = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    D = (Z + rng.standard_normal((B, k + 1, V))).astype(np.float32)
    x = rng.integers(0, V, (B, k)).astype(np.int32)
    x[::3] = np.argmax(Z[::3, :k], axis=2)          # some greedy agreement
    T = rng.choice(np.array([0.0, 0.6, 1.0, 1.4], np.float32), B)
    ua = rng.random((B, k)).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    chain = oracle.verify_recover(Z, D[:, :k], x, T, ua, us)
    par = np.tile(np.arange(-1, k, dtype=np.int32), (B, 1))
    tok = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    uat = np.concatenate([np.zeros((B, 1), np.float32), ua], axis=1)
    tree = oracle.verify_tree(Z, D, par, tok, T, uat, us)
    assert np.array_equal(tree["accept_len"], chain["accept_len"])
    assert np.array_equal(tree["out_tok"], chain["out_tok"])
    n = tree["accept_len"]
    for b in range(B):
        assert list(tree["out_node"][b, :n[b]]) == list(range(1, n[b] + 1))
    assert 0 < (n > 0).sum() < B


def test_tree_single_node_is_an_inverse_cdf_draw():
    """A tree of one node draws the token from softmax(z / T) by inverse CDF
    (scipy softmax, numpy cumulative sum and searchsorted)."""
    rng = np.random.default_rng(3)
    B, V = 400, 50
    Z = (rng.standard_normal((B, 1, V)) * 2).astype(np.float32)
    T = rng.uniform(0.5, 1.5, B).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    r = oracle.verify_tree(Z, Z, np.full((B, 1), -1, np.int32), np.zeros((B, 1), np.int32), T,
                           np.zeros((B, 1), np.float32), us)
    assert (r["accept_len"] == 0).all()
    for b in range(B):
        c = np.cumsum(softmax_ref(Z[b, 0], float(T[b])))
        assert r["out_tok"][b, 0] == np.searchsorted(c, float(us[b]) * c[-1], side="right")


def _random_trees(rng, B, N):
    par = np.full((B, N), -1, np.int32)
    for j in range(1, N):
        par[:, j] = rng.integers(0, j, B)
    return par


def test_tree_greedy_invariants():
    """T = 0: every accepted node's token is the argmax of its parent's
    target row and no earlier sibling carries it; the last node has no child
    with its argmax, and the final token is that argmax."""
    rng = np.random.default_rng(17)
    B, N, V = 300, 12, 6
    Z = rng.integers(-2, 3, (B, N, V)).astype(np.float32)             # ties
    D = rng.standard_normal((B, N, V)).astype(np.float32)
    par = _random_trees(rng, B, N)
    am = np.argmax(Z, axis=2)                                          # lowest index on ties
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    hit = rng.random((B, N)) < 0.6
    for b in range(B):
        for j in range(1, N):
            if hit[b, j]:
                tok[b, j] = am[b, par[b, j]]
    r = oracle.verify_tree(Z, D, par, tok, np.zeros(B, np.float32), rng.random((B, N)),
                           rng.random(B))
    n = r["accept_len"]
    assert (n >= 0).all() and (n >= 2).any()
    for b in range(B):
        cur = 0
        for i in range(n[b]):
            c = r["out_node"][b, i]
            assert par[b, c] == cur and tok[b, c] == am[b, cur] == r["out_tok"][b, i]
            assert not any(par[b, s] == cur and tok[b, s] == tok[b, c] for s in range(1, c))
            cur = c
        assert r["out_tok"][b, n[b]] == am[b, cur]
        assert not any(par[b, s] == cur and tok[b, s] == am[b, cur] for s in range(1, N))
        assert (r["out_tok"][b, n[b] + 1:] == -1).all() and (r["out_node"][b, n[b]:] == -1).all()


def test_tree_sentinels():
    rng = np.random.default_rng(5)
    B, N, V = 6, 4, 9
    Z = rng.standard_normal((B, N, V)).astype(np.float32)
    D = rng.standard_normal((B, N, V)).astype(np.float32)
    par = np.tile(np.array([-1, 0, 0, 1], np.int32), (B, 1))
    tok = rng.integers(0, V, (B, N)).astype(np.int32)
    T = np.ones(B, np.float32)
    T[0] = -1.0                      # invalid temperature
    par[1, 2] = 2                    # parent not before the node
    tok[2, 3] = V                    # token out of range
    par[3, 0] = 0                    # root with a parent
    D[4, 1, 2] = np.nan              # NaN in the draft row of node 1 (it has a child)
    D[5, 3, 2] = np.nan              # NaN in a leaf's draft row: never used, not read
    r = oracle.verify_tree(Z, D, par, tok, T, rng.random((B, N)), rng.random(B))
    assert list(r["accept_len"]) [:5] == [-1, -2, -2, -2, -1]
    assert r["accept_len"][5] >= 0
    assert (r["out_tok"][:5] == -1).all() and (r["out_node"][:5] == -1).all()


def test_tree_law_by_sampling():
    """Bushier tree (root with three children drawn from q, each with two
    children drawn from that child's q), 2 * 10^5 rows: the first two tokens
    follow p_root(t1) * p_t1(t2) (chi-square)."""
    rng = np.random.default_rng(23)
    B, V, T = 200_000, 5, 1.0
    Zr = rng.standard_normal(V).astype(np.float32) * 1.5
    Dr = (Zr + rng.standard_normal(V) * 1.5).astype(np.float32)
    Zc = (rng.standard_normal((V, V)) * 1.5).astype(np.float32)
    Dc = (Zc + rng.standard_normal((V, V)) * 1.5).astype(np.float32)
    pr, qr = softmax_ref(Zr, T), softmax_ref(Dr, T)
    pc, qc = softmax_ref(Zc, T), softmax_ref(Dc, T)
    par = np.tile(np.array([-1, 0, 0, 0, 1, 1, 2, 2, 3, 3], np.int32), (B, 1))
    N = par.shape[1]
    tok = np.zeros((B, N), np.int32)
    tok[:, 1:4] = _draw_from(qr, rng.random((B, 3)))
    for j in range(4, N):
        parent_tok = tok[:, par[0, j]]
        tok[:, j] = (np.cumsum(qc[parent_tok], axis=1) <= rng.random(B)[:, None]).sum(1).clip(0, V - 1)
    Z = np.empty((B, N, V), np.float32)
    D = np.empty((B, N, V), np.float32)
    Z[:, 0], D[:, 0] = Zr, Dr
    Z[:, 1:], D[:, 1:] = Zc[tok[:, 1:]], Dc[tok[:, 1:]]
    r = oracle.verify_tree(Z, D, par, tok, np.full(B, T, np.float32),
                           rng.random((B, N)).astype(np.float32),
                           rng.random(B).astype(np.float32))
    n, out = r["accept_len"], r["out_tok"]
    t1 = out[:, 0].astype(np.int64)
    t2 = np.where(n >= 1, out[:, 1],
                  (np.cumsum(pc[t1], axis=1) <= rng.random(B)[:, None]).sum(1).clip(0, V - 1))
    obs = np.bincount(t1 * V + t2, minlength=V * V)
    exp = (pr[:, None] * pc).reshape(-1) * B
    assert scipy.stats.chisquare(obs, exp).pvalue > 1e-4
    assert (n >= 1).mean() > 0.3 and (n == 0).any() and (n == 2).any()


def tree_golden_inputs(case):
    """Arrays of one hand-derived tree case (tests/golden/tree_cases.json)."""
    Z = np.log(np.array(case["target_weights"], dtype=np.float64)).astype(np.float32)[None]
    D = np.log(np.array(case["draft_weights"], dtype=np.float64)).astype(np.float32)[None]
    return (Z, D, np.array([case["parent"]], np.int32), np.array([case["tok"]], np.int32),
            np.array([case["T"]], np.float32), np.array([case["u_acc"]]),
            np.array([case["u_smp"]]))


def test_golden_tree_cases():
    g = _golden("tree_cases.json")
    for case in g["cases"]:
        Z, D, par, tok, T, ua, us = tree_golden_inputs(case)
        r = oracle.verify_tree(Z, D, par, tok, T, ua, us, f64_uniforms=True)
        assert r["accept_len"][0] == case["accept_len"], case["name"]
        assert list(r["out_tok"][0]) == case["out_tok"], case["name"]
        assert list(r["out_node"][0]) == case["out_node"], case["name"]
