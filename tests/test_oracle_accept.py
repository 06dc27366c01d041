"""Pins of the oracle accept step, Philox and the own exp.

* Philox4x32-10 against the Random123 known-answer vectors (golden file);
* the own exp against math.exp within 2 ulp, with exp(0) == 1 exactly;
* argmax ties and NaN, greedy special cases by hand;
* the integer-mass transform against a float softmax and a brute-force top-p;
* rejection sampling: T = 0 equals greedy, p == q accepts everything, the
  committed-token marginals pass a chi-square test against p (the defining
  property of Leviathan/Chen sampling) and the mean accepted length matches
  the closed form sum_j prod_{i<j} alpha_i, alpha_i = sum_x min(p_i, q_i).
"""
import math

import numpy as np
import pytest
from scipy import stats

import oracle
import synth
from conftest import golden_lines


def test_philox_known_answers():
    rows = list(golden_lines("philox4x32_10_kat.txt"))
    assert len(rows) == 3
    for r in rows:
        v = [int(x, 16) for x in r]
        out = oracle.philox4x32_10(v[0:4], v[4:6])
        assert list(out) == v[6:10]


def _ulp_err(got, ref):
    ulp = math.ulp(np.float32(ref)) if ref != 0 else 2.0 ** -149
    return abs(got - ref) / float(np.spacing(np.float32(ref)))


def test_own_exp_accuracy_and_special_points():
    assert oracle.own_exp(0.0) == 1.0
    assert oracle.own_exp(-0.0) == 1.0
    assert oracle.own_exp(-32.5) == 0.0
    assert oracle.own_exp(float("nan")) == 0.0
    g = np.random.default_rng(5)
    xs = np.concatenate([-g.random(20000) * 32.0, -g.random(5000) * 1e-3,
                         -np.arange(0, 32.0, 0.125)]).astype(np.float32)
    worst = 0.0
    for x in xs:
        got = oracle.own_exp(float(x))
        ref = math.exp(float(x))
        worst = max(worst, _ulp_err(got, ref))
    assert worst <= 2.0, worst
    # monotone on a sorted sample
    xs = np.sort(xs)
    vals = [oracle.own_exp(float(x)) for x in xs]
    assert all(a <= b for a, b in zip(vals, vals[1:]))


def test_argmax_ties_and_nan():
    assert oracle.argmax_f32(np.array([1, 3, 3, 2], np.float32)) == 1
    assert oracle.argmax_f32(np.array([np.nan, 0.5, 0.5], np.float32)) == 1
    assert oracle.argmax_f32(np.array([np.nan, np.nan], np.float32)) == 0
    assert oracle.argmax_f32(np.array([-np.inf, np.nan, -np.inf], np.float32)) == 0
    assert oracle.argmax_f32(np.array([-1, np.inf, np.inf], np.float32)) == 1


def _one_hot_rows(ids, V):
    rows = np.zeros((len(ids), V), np.float32)
    for i, t in enumerate(ids):
        rows[i, t] = 5.0
    return rows


def test_greedy_cases():
    V = 11
    tgt = _one_hot_rows([4, 7, 2, 9], V)[None]           # argmaxes 4, 7, 2, 9
    # all three drafts match: len = 4, bonus = 9
    tok, ln, bad = oracle.accept_greedy(tgt, np.array([[4, 7, 2]]))
    assert ln[0] == 4 and list(tok[0]) == [4, 7, 2, 9] and bad == 0
    # first mismatch at i = 1: commit draft 0 then the target's 7
    tok, ln, _ = oracle.accept_greedy(tgt, np.array([[4, 1, 2]]))
    assert ln[0] == 2 and list(tok[0]) == [4, 7, -1, -1]
    # mismatch at 0
    tok, ln, _ = oracle.accept_greedy(tgt, np.array([[0, 7, 2]]))
    assert ln[0] == 1 and list(tok[0]) == [4, -1, -1, -1]
    # out of range id is a rejection
    tok, ln, bad = oracle.accept_greedy(tgt, np.array([[4, 99, 2]]))
    assert ln[0] == 2 and list(tok[0]) == [4, 7, -1, -1] and bad == 1
    # Kd = 0 returns the argmax
    tok, ln, _ = oracle.accept_greedy(tgt[:, :1], np.zeros((1, 0), np.int32))
    assert ln[0] == 1 and list(tok[0]) == [4]


def test_row_mass_against_float_softmax_and_brute_force_top_p():
    g = np.random.default_rng(7)
    for trial in range(30):
        V = int(g.integers(2, 40))
        lg = (g.standard_normal(V) * 3).astype(np.float32)
        T, top_p = 0.6, float(g.choice([0.5, 0.8, 0.95, 1.0]))
        W, S = oracle.row_mass(lg, T, top_p)
        full, Sf = oracle.row_mass(lg, T, 1.0)
        assert int(full.max()) == 2 ** 40
        p = np.exp((lg.astype(np.float64) - lg.max()) / T)
        assert np.allclose(full.astype(np.float64) / 2.0 ** 40, p, rtol=2e-6, atol=2.0 ** -40)
        # brute-force top-p on the integer masses: shortest prefix in
        # (W desc, index asc) order with cum * 2^32 >= P * S_full
        P = oracle.top_p_fixed(top_p)
        order = sorted(range(V), key=lambda v: (-int(full[v]), v))
        if P >= 2 ** 32:
            keep = set(range(V))
        else:
            cum, keep = 0, set()
            for v in order:
                cum += int(full[v])
                keep.add(v)
                if cum * 2 ** 32 >= P * Sf:
                    break
        for v in range(V):
            assert int(W[v]) == (int(full[v]) if v in keep else 0)
        assert S == sum(int(full[v]) for v in keep)


def test_rejection_t0_is_greedy():
    g = np.random.default_rng(8)
    B, Kd, V = 20, 4, 50
    tgt = g.standard_normal((B, Kd + 1, V)).astype(np.float32)
    drf = g.standard_normal((B, Kd, V)).astype(np.float32)
    am = tgt.argmax(axis=2)
    drafts = np.where(g.random((B, Kd)) < 0.7, am[:, :Kd], g.integers(0, V, (B, Kd))).astype(np.int32)
    t1, l1, _ = oracle.accept_rejection(tgt, drf, drafts, 0.0, 0.95, 1, 0)
    t2, l2, _ = oracle.accept_greedy(tgt, drafts)
    assert np.array_equal(t1, t2) and np.array_equal(l1, l2)


def test_rejection_p_equals_q_accepts_everything():
    g = np.random.default_rng(9)
    B, Kd, V = 64, 5, 30
    tgt = (g.standard_normal((B, Kd + 1, V)) * 3).astype(np.float32)
    drf = tgt[:, :Kd].copy()
    drafts = oracle.sample_drafts(drf, 0.6, 0.95, 11, 1 << 32)
    tok, ln, bad = oracle.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 11, 0)
    assert bad == 0 and np.all(ln == Kd + 1)
    assert np.array_equal(tok[:, :Kd], drafts)


def _dist(lg, T, top_p):
    W, S = oracle.row_mass(lg, T, top_p)
    return W.astype(np.float64) / S


CHI_N = 1_000_000


@pytest.fixture(scope="module")
def sixteen_token_case():
    g = np.random.default_rng(12)
    V, Kd = 16, 3
    tgt = (g.standard_normal((Kd + 1, V)) * 3).astype(np.float32)
    drf = (tgt[:Kd] + g.standard_normal((Kd, V))).astype(np.float32)
    drafts = oracle.sample_drafts(drf, 0.6, 0.95, 13, 1 << 32, broadcast_rows=True, B=CHI_N)
    tok, ln, bad = oracle.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 13, 0,
                                           broadcast_rows=True, B=CHI_N)
    assert bad == 0
    return tgt, drf, drafts, tok, ln


def _chi2_against(counts, probs):
    nz = probs > 0
    assert counts[~nz].sum() == 0, "a token excluded by top-p was committed"
    exp = probs[nz] * counts.sum()
    return stats.chisquare(counts[nz], exp).pvalue


def test_first_token_marginal_matches_target(sixteen_token_case):
    tgt, drf, drafts, tok, ln = sixteen_token_case
    p0 = _dist(tgt[0], 0.6, 0.95)
    counts = np.bincount(tok[:, 0], minlength=16)
    assert _chi2_against(counts, p0) > 1e-4


def test_second_token_given_first_accepted_matches_target(sixteen_token_case):
    tgt, drf, drafts, tok, ln = sixteen_token_case
    sel = ln >= 2                     # position 0 was accepted (token 0 == draft 0)
    assert np.array_equal(tok[sel, 0], drafts[sel, 0])
    p1 = _dist(tgt[1], 0.6, 0.95)
    counts = np.bincount(tok[sel, 1], minlength=16)
    assert _chi2_against(counts, p1) > 1e-4


def test_mean_accepted_length_matches_closed_form(sixteen_token_case):
    tgt, drf, drafts, tok, ln = sixteen_token_case
    Kd = drf.shape[0]
    alpha = [np.minimum(_dist(tgt[i], 0.6, 0.95), _dist(drf[i], 0.6, 0.95)).sum()
             for i in range(Kd)]
    # P(n >= j) = prod_{i<j} alpha_i
    probs = [np.prod(alpha[:j]) for j in range(1, Kd + 1)]
    mean = sum(probs)
    # variance of n = sum_j P(n>=j) (2j - 1) - mean^2
    var = sum(pr * (2 * j - 1) for j, pr in enumerate(probs, start=1)) - mean ** 2
    got = float(np.mean(ln - 1))
    assert abs(got - mean) <= 4 * math.sqrt(var / len(ln)), (got, mean)


def test_row_mass_top_k_and_min_p_against_float_definitions():
    """top-k keeps the k largest logits (ties to the lower index) with their
    unchanged masses; min-p keeps the entries whose probability is at least
    min_p times the largest (checked against float64 away from the edge);
    with top-p as well the kept set is the shorter of the two prefixes."""
    g = np.random.default_rng(21)
    for trial in range(40):
        V = int(g.integers(3, 60))
        lg = (g.standard_normal(V) * 3).astype(np.float32)
        if trial % 5 == 0:
            lg[g.integers(0, V, 3)] = lg[0]          # some exact ties
        T = 0.6
        full, Sf = oracle.row_mass(lg, T, 1.0)
        k = int(g.integers(1, V))
        W, S = oracle.row_mass(lg, T, 1.0, top_k=k)
        order = np.lexsort((np.arange(V), -lg.astype(np.float64)))   # logit desc, index asc
        top = set(int(v) for v in order[:k])
        assert set(np.nonzero(W)[0].tolist()) <= top
        for v in range(V):
            assert int(W[v]) == (int(full[v]) if v in top else 0)
        assert S == sum(int(full[v]) for v in top)
        # min-p alone
        mp = float(g.choice([0.01, 0.05, 0.2, 0.5]))
        Wm, Sm = oracle.row_mass(lg, T, 1.0, min_p=mp)
        ratio = np.exp((lg.astype(np.float64) - lg.max()) / T)      # p_v / p_max
        for v in range(V):
            if ratio[v] > mp * (1 + 1e-5):
                assert int(Wm[v]) == int(full[v])
            elif ratio[v] < mp * (1 - 1e-5):
                assert int(Wm[v]) == 0
        # top-p and min-p: the shorter prefix of the (W desc, index asc) order
        top_p = float(g.choice([0.5, 0.8, 0.95]))
        Wb, Sb = oracle.row_mass(lg, T, top_p, min_p=mp)
        Wp, _ = oracle.row_mass(lg, T, top_p)
        for v in range(V):
            assert int(Wb[v]) == (int(full[v]) if (Wp[v] > 0 and Wm[v] > 0) else 0)
        assert Sb == int(Wb.sum())


def test_top_k_one_commits_the_argmax():
    g = np.random.default_rng(22)
    B, Kd, V = 200, 2, 40
    tgt = (g.standard_normal((B, Kd + 1, V)) * 3).astype(np.float32)
    drf = (tgt[:, :Kd] + g.standard_normal((B, Kd, V))).astype(np.float32)
    drafts = oracle.sample_drafts(drf, 0.6, 0.95, 5, 1 << 32, top_k=1)
    assert np.array_equal(drafts, drf.argmax(axis=2))
    tok, ln, bad = oracle.accept_rejection(tgt, drf, drafts, 0.6, 0.95, 5, 0, top_k=1)
    am = tgt.argmax(axis=2)
    for b in range(B):
        n = ln[b] - 1
        assert np.array_equal(tok[b, :n], drafts[b, :n])
        assert np.all(tok[b, :n] == am[b, :n])         # accepted drafts are the argmax
        assert tok[b, n] == am[b, n]                     # the committed token too


def _float_pipeline(lg, T, top_k, top_p, min_p):
    """The sampler pipeline in float64: top-k on the logits, softmax at T,
    top-p (shortest prefix by probability reaching top_p), min-p, normalize."""
    lg = lg.astype(np.float64)
    V = lg.size
    keep = np.zeros(V, bool)
    keep[np.lexsort((np.arange(V), -lg))[:top_k if top_k else V]] = True
    p = np.where(keep, np.exp((lg - lg.max()) / T), 0.0)
    p /= p.sum()
    order = np.lexsort((np.arange(V), -p))
    cum = np.cumsum(p[order])
    n = int(np.searchsorted(cum, top_p - 1e-12) + 1) if top_p < 1 else V
    kp = np.zeros(V, bool)
    kp[order[:n]] = True
    kp &= p >= min_p * p.max()
    q = np.where(kp, p, 0.0)
    return q / q.sum()


def test_first_token_marginal_with_top_k_and_min_p():
    """Chi-square of the first committed token, with the whole pipeline on
    (top-k 6, top-p 0.9, min-p 0.05), against its float64 definition."""
    g = np.random.default_rng(23)
    V, Kd = 16, 2
    tgt = (g.standard_normal((Kd + 1, V)) * 2).astype(np.float32)
    drf = (tgt[:Kd] + g.standard_normal((Kd, V))).astype(np.float32)
    kw = dict(top_k=6, min_p=0.05)
    drafts = oracle.sample_drafts(drf, 0.6, 0.9, 31, 1 << 32, broadcast_rows=True, B=CHI_N, **kw)
    tok, ln, bad = oracle.accept_rejection(tgt, drf, drafts, 0.6, 0.9, 31, 0,
                                           broadcast_rows=True, B=CHI_N, **kw)
    assert bad == 0
    p0 = _float_pipeline(tgt[0], 0.6, 6, 0.9, 0.05)
    W0, S0 = oracle.row_mass(tgt[0], 0.6, 0.9, **kw)
    assert np.array_equal(W0 > 0, p0 > 0)           # the same kept set as the float pipeline
    counts = np.bincount(tok[:, 0], minlength=V)
    assert _chi2_against(counts, p0) > 1e-4


# ------------------------------------------------------------ top-k lists
def _top_lists(rows, Kt, g):
    """The top-Kt entries of each row in (logit desc, index asc) order, then
    shuffled: ids int32, logits fp32 [B, R, Kt]."""
    B, R, V = rows.shape
    ids = np.empty((B, R, Kt), np.int32)
    vals = np.empty((B, R, Kt), np.float32)
    for b in range(B):
        for r in range(R):
            o = np.lexsort((np.arange(V), -rows[b, r].astype(np.float64)))[:Kt]
            o = o[g.permutation(Kt)]
            ids[b, r], vals[b, r] = o, rows[b, r, o]
    return ids, vals


@pytest.mark.parametrize("B,Kd,V,Kt,top_p,top_k,min_p", [
    (12, 3, 200, 16, 0.95, 0, 0.0), (8, 2, 1000, 50, 0.9, 0, 0.05), (6, 4, 500, 64, 1.0, 20, 0.0),
    (10, 1, 300, 1, 0.95, 0, 0.0), (7, 0, 400, 30, 0.8, 0, 0.1)])
def test_top_k_lists_equal_the_dense_top_k_stage(B, Kd, V, Kt, top_p, top_k, min_p):
    """Rows given as their top-Kt lists (any order) accept exactly as the
    dense rows with the top-k stage at Kt (and any further top-k / min-p):
    the scatter into -inf rows against the sampler's own top-k stage."""
    g = np.random.default_rng(B * 31 + Kt)
    target = (g.standard_normal((B, Kd + 1, V)) * 3).astype(np.float32)
    draft = (target[:, :Kd] + g.standard_normal((B, Kd, V))).astype(np.float32)
    kk = min(top_k, Kt) if top_k else Kt
    drafts = oracle.sample_drafts(draft, 0.6, top_p, 5, 1 << 32, top_k=kk, min_p=min_p) if Kd \
        else np.zeros((B, 0), np.int32)
    t_ids, t_vals = _top_lists(target, Kt, g)
    d_ids, d_vals = _top_lists(draft, Kt, g) if Kd else (None, None)
    lt, ll, lb = oracle.accept_rejection_topk(t_ids, t_vals, d_ids, d_vals, drafts, V, 0.6, top_p,
                                              5, 3, top_k=top_k, min_p=min_p)
    dt, dl, db = oracle.accept_rejection(target, draft, drafts, 0.6, top_p, 5, 3, top_k=kk,
                                         min_p=min_p)
    assert np.array_equal(ll, dl) and np.array_equal(lt, dt) and lb == db


def test_lists_to_rows_places_every_listed_logit():
    ids = np.array([[[3, 0, 7], [9, 2, 5]]], np.int32)
    vals = np.array([[[1.0, -2.0, 0.5], [4.0, np.nan, -np.inf]]], np.float32)
    rows = oracle.lists_to_rows(ids, vals, 10)
    assert rows.shape == (1, 2, 10)
    assert rows[0, 0, 3] == 1.0 and rows[0, 0, 0] == -2.0 and rows[0, 0, 7] == 0.5
    assert np.isnan(rows[0, 1, 2]) and rows[0, 1, 9] == 4.0
    assert np.isneginf(rows[0, 1, 5])
    assert np.isneginf(np.delete(rows[0, 0], [0, 3, 7])).all()
    # ids outside [0, V) are dropped
    rows = oracle.lists_to_rows(np.array([[[11, 1]]], np.int32), np.array([[[5.0, 6.0]]],
                                                                          np.float32), 10)
    assert rows[0, 0, 1] == 6.0 and np.isneginf(np.delete(rows[0, 0], [1])).all()


def test_topk_lists_case_follows_its_recipe():
    """The seeded list generator: distinct in-range ids per row, target logits
    sorted descending, drafts taken from their own draft lists, and the
    draft lists sharing most of the target row's ids."""
    B, Kd, Kt, V = 6, 3, 40, 500
    t_ids, t_vals, d_ids, d_vals, drafts = synth.topk_lists_case(1, B, Kd, Kt, V)
    assert t_ids.shape == (B, Kd + 1, Kt) and d_ids.shape == (B, Kd, Kt)
    for ids in (t_ids, d_ids):
        assert ids.min() >= 0 and ids.max() < V
        for row in ids.reshape(-1, Kt):
            assert np.unique(row).size == Kt
    assert np.all(np.diff(t_vals, axis=-1) <= 0)
    shared = [np.intersect1d(t_ids[b, i], d_ids[b, i]).size for b in range(B) for i in range(Kd)]
    assert np.mean(shared) > 0.6 * Kt
    for b in range(B):
        for i in range(Kd):
            assert drafts[b, i] in d_ids[b, i]
    again = synth.topk_lists_case(1, B, Kd, Kt, V)
    assert all(np.array_equal(a, c) for a, c in zip(again, (t_ids, t_vals, d_ids, d_vals, drafts)))
