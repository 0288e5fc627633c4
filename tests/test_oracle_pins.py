"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: values the
pages print (tests/golden/*.json, each with its citation), exact rational
enumeration of the output law (the distribution-preservation theorem),
closed forms, library routines, and published known-answer vectors.  No GPU.
"""

import itertools
import math
from fractions import Fraction as F

import numpy as np
import pytest
import scipy.special

from conftest import load_golden
from oracle import philox, policy, verify
from oracle.policy import Dist


def frac_array(values):
    return np.array([F(v) for v in values], dtype=object)


# ---------------------------------------------------------------------------
# Philox4x32-10 known answers
# ---------------------------------------------------------------------------

def test_philox_known_answer_vectors():
    g = load_golden("philox4x32_10_kat.json")
    for vec in g["vectors"]:
        ctr = [int(w, 16) for w in vec["counter"]]
        key = [int(w, 16) for w in vec["key"]]
        out = philox.philox4x32(ctr, key)
        assert [f"{w:08x}" for w in out] == vec["out"]


def test_philox_uniform_grid_and_range():
    us = [philox.uniform(1234, s, p, d) for s in range(8) for p in range(8) for d in range(2)]
    for u in us:
        assert 0.0 <= u < 1.0
        assert (u * 2 ** 24) == int(u * 2 ** 24)
    assert len(set(us)) == len(us)
    # seed halves both enter the key
    assert philox.uniform(1, 0, 0, 0) != philox.uniform(1 + (1 << 32), 0, 0, 0)


# ---------------------------------------------------------------------------
# the page's reference-function assertions and worked examples
# ---------------------------------------------------------------------------

def test_verify_candidate_asserts_exact():
    g = load_golden("verify_candidate_asserts.json")
    for case in g["cases"]:
        p, q = frac_array(case["target"]), frac_array(case["draft"])
        acc, alpha, flags = verify.accept_test(p, q, case["token"], F(case["uniform"]))
        assert flags == 0
        assert acc == case["accepted"]
        if case["residual"] is not None:
            r, Z, f = verify.positive_residual(p, q)
            assert f == 0
            assert list(r) == [F(v) for v in case["residual"]]
    bad = g["invalid_token"]
    acc, _, flags = verify.accept_test(frac_array(bad["target"]), frac_array(bad["draft"]),
                                       bad["token"], F(bad["uniform"]))
    assert not acc and flags == verify.FLAG_BAD_TOKEN


def test_verify_candidate_asserts_float64():
    g = load_golden("verify_candidate_asserts.json")
    for case in g["cases"]:
        p = np.array([float(v) for v in case["target"]])
        q = np.array([float(v) for v in case["draft"]])
        acc, _, _ = verify.accept_test(p, q, case["token"], float(F(case["uniform"])))
        assert acc == case["accepted"]
        if case["residual"] is not None:
            r, _, _ = verify.positive_residual(p, q)
            np.testing.assert_allclose(r, [float(F(v)) for v in case["residual"]], atol=1e-15)


def test_p_equals_q_accepts_every_legal_draft():
    rng = np.random.default_rng(3)
    for V in (2, 3, 7, 64):
        w = rng.integers(0, 5, V)
        w[0] += 1
        p = np.array([F(int(x), int(w.sum())) for x in w], dtype=object)
        for x in range(V):
            if p[x] > 0:
                for u in (F(0), F(1, 2), 1 - F(1, 2 ** 24)):
                    acc, alpha, flags = verify.accept_test(p, p, x, u)
                    assert acc and alpha == 1 and flags == 0


def test_zero_draft_probability_is_flagged():
    p, q = frac_array(["0.5", "0.5"]), frac_array(["1", "0"])
    acc, _, flags = verify.accept_test(p, q, 1, F(0))
    assert not acc and flags == verify.FLAG_ZERO_Q


def test_worked_example_a():
    g = load_golden("worked_examples.json")["example_a"]
    p, q = frac_array(g["p"]), frac_array(g["q"])
    for x in range(4):
        _, alpha, _ = verify.accept_test(p, q, x, F(0))
        assert alpha == F(g["alpha"][x])
        assert q[x] * alpha == F(g["accepted_mass"][x])
    r, Z, f = verify.positive_residual(p, q)
    assert Z == F(g["rejection_rate"])
    assert 1 - Z == F(g["beta"])
    assert list(r) == [F(v) for v in g["residual"]]
    assert [Z * v for v in r] == [F(v) for v in g["missing_mass"]]
    # the page's two uniforms for draft token A (index 0)
    assert verify.accept_test(p, q, 0, F(g["draw_A_u_accept"]))[0]
    assert not verify.accept_test(p, q, 0, F(g["draw_A_u_reject"]))[0]
    # after the rejection the correction comes from B or C only
    for k in range(100):
        tok, _ = verify.inverse_cdf(r, F(k, 100))
        assert tok in (1, 2)


def test_worked_example_b():
    g = load_golden("worked_examples.json")["example_b"]
    p, q = frac_array(g["p"]), frac_array(g["q"])
    for x in range(3):
        _, alpha, _ = verify.accept_test(p, q, x, F(0))
        assert alpha == F(g["alpha"][x])
        assert q[x] * alpha == F(g["accepted_mass"][x])
    r, Z, _ = verify.positive_residual(p, q)
    assert [Z * v for v in r] == [F(v) for v in g["missing_mass"]]
    # acceptance mass + missing mass gives back p
    assert [q[x] * verify.accept_test(p, q, x, F(0))[1] + Z * r[x] for x in range(3)] == list(p)


def random_rational_dist(rng, V, zero_prob=0.25, max_w=6):
    w = rng.integers(1, max_w + 1, V) * (rng.random(V) >= zero_prob)
    if w.sum() == 0:
        w[rng.integers(V)] = 1
    s = int(w.sum())
    return np.array([F(int(x), s) for x in w], dtype=object)


def test_residual_denominator_identity_and_overlap():
    """Sum(q - min(q, p)) = Sum [p - q]_+ and beta = Sum min(p, q) = 1 - TV(p, q).

    tannlonggtaoo.github.io "Speculative Decoding", § 验证方式：reject sampling
    (the reverse derivation's denominator equals the forward one);
    wineandchord.com "推测解码：接受规则、状态与收益边界", § 特征级 Draft
    (Sum min(p, q) = 1 - TV(p, q)).
    """
    rng = np.random.default_rng(11)
    for _ in range(200):
        V = int(rng.integers(2, 9))
        p, q = random_rational_dist(rng, V), random_rational_dist(rng, V)
        _, Z, _ = verify.positive_residual(p, q)
        assert Z == sum(qx - min(qx, px) for px, qx in zip(p, q))
        accept_rate = sum(q[x] * verify.accept_test(p, q, x, F(0))[1]
                          for x in range(V) if q[x] > 0)
        tv = sum(abs(px - qx) for px, qx in zip(p, q)) / 2
        assert accept_rate == 1 - tv == 1 - Z


# ---------------------------------------------------------------------------
# inverse-CDF draw
# ---------------------------------------------------------------------------

def test_inverse_cdf_boundaries_exact():
    rng = np.random.default_rng(5)
    for _ in range(100):
        V = int(rng.integers(1, 9))
        w = random_rational_dist(rng, V)
        c = np.cumsum(w)
        for v in range(V):
            lo = c[v - 1] if v else F(0)
            if w[v] == 0:
                continue
            # the interval [lo, c_v) maps to v: check its left end and midpoint
            assert verify.inverse_cdf(w, lo)[0] == v
            assert verify.inverse_cdf(w, (lo + c[v]) / 2)[0] == v
        for k in range(64):
            tok, _ = verify.inverse_cdf(w, F(k, 64))
            assert w[tok] > 0


def test_inverse_cdf_law_matches_weights():
    """Measure of u in [0,1) mapping to v equals w_v / sum(w) (library cumsum)."""
    w = np.array([0.0, 0.25, 0.0, 0.5, 0.25])
    grid = (np.arange(4096) + 0.5) / 4096
    counts = np.bincount([verify.inverse_cdf(w, u)[0] for u in grid], minlength=5)
    np.testing.assert_array_equal(counts, [0, 1024, 0, 2048, 1024])


def test_inverse_cdf_fallback_largest_positive():
    w = np.array([0.3, 0.0, 0.7, 0.0])
    tok, margin = verify.inverse_cdf(w, 1.0)  # beyond the last boundary
    assert tok == 2 and margin == 0


# ---------------------------------------------------------------------------
# policy
# ---------------------------------------------------------------------------

def test_softmax_matches_library():
    rng = np.random.default_rng(7)
    for T in (0.25, 0.7, 1.0, 2.5):
        z = rng.standard_normal(1000) * 3
        d = policy.policy_distribution(z, T, 0)
        np.testing.assert_allclose(d.probs, scipy.special.softmax(z / T), rtol=1e-12, atol=1e-300)


def test_topk_kept_set_by_counting():
    """Kept iff fewer than k entries are strictly larger (ties at the threshold kept)."""
    rng = np.random.default_rng(8)
    for _ in range(50):
        V = int(rng.integers(2, 300))
        z = np.round(rng.standard_normal(V) * 2, 1)  # many ties
        k = int(rng.integers(1, V + 2))
        d = policy.policy_distribution(z, 0.8, k)
        greater = (z[None, :] > z[:, None]).sum(axis=1)
        kept = greater < k if 0 < k < V else np.ones(V, bool)
        np.testing.assert_array_equal(d.probs > 0, kept)
        np.testing.assert_allclose(d.probs[kept], scipy.special.softmax(z[kept] / 0.8), rtol=1e-12)


def test_greedy_lowest_index():
    z = np.array([1.0, 3.0, -np.inf, 3.0, 2.0])
    d = policy.policy_distribution(z, 0.0)
    assert d.onehot and d.index == int(np.argmax(z)) == 1 and d.flags == 0


def test_nonfinite_rows():
    for z, T, idx in [([0.0, np.nan, 1.0], 1.0, 2), ([0.0, np.inf, 1.0], 1.0, 2),
                      ([-np.inf, -np.inf], 1.0, 0), ([0.5, 2.0], -1.0, 1),
                      ([0.5, 2.0], np.nan, 1), ([0.5, 2.0], np.inf, 1)]:
        d = policy.policy_distribution(np.array(z), T)
        assert d.onehot and d.index == idx and d.flags == policy.FLAG_NONFINITE
    d = policy.policy_distribution(np.array([-np.inf, 0.0, -np.inf]), 1.0)
    assert not d.onehot and list(d.probs) == [0.0, 1.0, 0.0]


# ---------------------------------------------------------------------------
# exact enumeration: the output law of a chain equals the target's
# ---------------------------------------------------------------------------

def make_tables(rng, V, depth, zero_prob=0.25):
    """Random rational next-token tables keyed by prefix tuples up to ``depth``."""
    tables = {}
    for L in range(depth + 1):
        for prefix in itertools.product(range(V), repeat=L):
            tables[prefix] = random_rational_dist(rng, V, zero_prob)
    return tables


def ar_law(P, prefix, length):
    """Law of the next ``length`` tokens under autoregressive sampling from P."""
    law = {(): F(1)}
    for _ in range(length):
        nxt = {}
        for seq, w in law.items():
            row = P[prefix + seq]
            for v, pv in enumerate(row):
                if pv:
                    nxt[seq + (v,)] = nxt.get(seq + (v,), 0) + w * pv
        law = nxt
    return law


def representative_uniform(weights, v):
    c = np.cumsum(weights)
    lo = c[v - 1] if v else F(0)
    return (lo + c[v]) / (2 * c[-1])


def chain_law(P, Q, V, gamma):
    """Law of (round output + autoregressive continuation) over gamma+1 tokens.

    Enumerates every draft sequence (weight prod q_i(x_i)), every first
    rejection position j (weight prod_{i<j} alpha_i (1 - alpha_j), from the
    oracle's accept_test) and every drawn token (weight from the distribution
    the round draws from: the oracle's residual at j, or p_gamma for the
    bonus).  For each branch the oracle's chain walk is *run* with uniforms
    inside that branch's interval, and its output is recorded.
    """
    law = {}
    for xs in itertools.product(range(V), repeat=gamma):
        wq = F(1)
        for i in range(gamma):
            wq *= Q[xs[:i]][xs[i]]
        if wq == 0:
            continue
        prows = [P[xs[:i]] for i in range(gamma + 1)]
        qrows = [Q[xs[:i]] for i in range(gamma)]
        alphas = [verify.accept_test(prows[i], qrows[i], xs[i], F(0))[1] for i in range(gamma)]
        for j in range(gamma + 1):
            w = wq
            for i in range(j):
                w *= alphas[i]
            if j < gamma:
                w *= 1 - alphas[j]
                r, _, f = verify.positive_residual(prows[j], qrows[j])
                draw_dist = prows[j] if f else r
            else:
                draw_dist = prows[gamma]
            if w == 0:
                continue
            ua = [alphas[i] / 2 if i < j else (1 + alphas[i]) / 2 for i in range(gamma)]
            for v in range(V):
                if draw_dist[v] == 0:
                    continue
                ud = representative_uniform(draw_dist, v)
                res = verify.walk_chain(
                    gamma, V, lambda i: Dist(False, probs=prows[i]),
                    lambda i: Dist(False, probs=qrows[i]), xs,
                    lambda i: ua[i], lambda i: ud)
                assert res["flags"] == 0 and res["j"] == j
                out = tuple(t for t in res["tokens"] if t >= 0)
                bw = w * draw_dist[v] / sum(draw_dist)
                for cont, cw in ar_law(P, out, gamma + 1 - len(out)).items():
                    key = out + cont
                    law[key] = law.get(key, 0) + bw * cw
    return law


@pytest.mark.parametrize("V,gamma", [(2, 1), (2, 2), (2, 3), (3, 1), (3, 2), (3, 3),
                                     (4, 2), (5, 1), (5, 2), (6, 3), (8, 1), (8, 2), (8, 3)])
def test_chain_output_law_is_target_law(V, gamma):
    rng = np.random.default_rng(100 * V + gamma)
    P = make_tables(rng, V, gamma)
    Q = make_tables(rng, V, gamma - 1)
    got = chain_law(P, Q, V, gamma)
    want = ar_law(P, (), gamma + 1)
    assert {k: v for k, v in got.items() if v} == want


def test_chain_output_law_detects_planted_sign_error(monkeypatch):
    """A residual built from [q - p]_+ instead of [p - q]_+ breaks the law."""
    real = verify.positive_residual

    def wrong(p, q):
        return real(q, p)

    rng = np.random.default_rng(202)
    P = make_tables(rng, 3, 2, zero_prob=0.0)
    Q = make_tables(rng, 3, 1, zero_prob=0.0)
    monkeypatch.setattr(verify, "positive_residual", wrong)
    try:
        got = chain_law(P, Q, 3, 2)
    except AssertionError:
        return
    assert {k: v for k, v in got.items() if v} != ar_law(P, (), 3)


def test_greedy_rule_equals_general_rule():
    """Temperature 0: accept iff draft == argmax p, correction = argmax p.

    tannlonggtaoo.github.io "Speculative Decoding", § Greedy Sampling: the
    general proof still applies, so the greedy comparison is lossless.  Here
    the greedy short-cut of the walk (one-hot Dist) is compared with the
    general rule run on the same one-hot p as a probability vector.
    """
    rng = np.random.default_rng(13)
    for _ in range(300):
        V = int(rng.integers(2, 7))
        gamma = int(rng.integers(1, 4))
        a = [int(rng.integers(V)) for _ in range(gamma + 1)]
        qrows = [random_rational_dist(rng, V, 0.0) for _ in range(gamma)]
        xs = [int(rng.integers(V)) for _ in range(gamma)]
        us = [F(int(rng.integers(1000)), 1000) for _ in range(2 * gamma + 2)]

        def onehot(i):
            return Dist(True, index=a[i])

        def dense(i):
            v = np.array([F(0)] * V, dtype=object)
            v[a[i]] = F(1)
            return Dist(False, probs=v)

        args = (lambda i: Dist(False, probs=qrows[i]), xs,
                lambda i: us[2 * i], lambda i: us[2 * i + 1])
        g = verify.walk_chain(gamma, V, onehot, *args)
        h = verify.walk_chain(gamma, V, dense, *args)
        assert g["tokens"] == h["tokens"] and g["num_accepted"] == h["num_accepted"]


# ---------------------------------------------------------------------------
# expected output length
# ---------------------------------------------------------------------------

def expected_output_length(alphas):
    """E[accepted + 1] of the chain walk, exactly, for an acceptance profile.

    V = 2, q_i = (1, 0) so the draft always proposes token 0, and
    p_i = (alpha_i, 1 - alpha_i) so the oracle's acceptance probability at
    position i is alpha_i.  The walk is run once per branch.
    """
    gamma = len(alphas)
    prows = [np.array([a, 1 - a], dtype=object) for a in alphas]
    prows.append(np.array([F(1, 2), F(1, 2)], dtype=object))
    qrow = np.array([F(1), F(0)], dtype=object)
    total = F(0)
    for j in range(gamma + 1):
        w = F(1)
        for i in range(j):
            w *= alphas[i]
        if j < gamma:
            w *= 1 - alphas[j]
        if w == 0:
            continue
        ua = [alphas[i] / 2 if i < j else (1 + alphas[i]) / 2 for i in range(gamma)]
        res = verify.walk_chain(gamma, 2, lambda i: Dist(False, probs=prows[i]),
                                lambda i: Dist(False, probs=qrow), [0] * gamma,
                                lambda i: ua[i], lambda i: F(1, 3))
        total += w * (res["num_accepted"] + 1)
    return total


def test_expected_output_length_page_examples():
    g = load_golden("expected_output_length.json")
    for prof in g["profiles"]:
        alphas = [F(a) for a in prof["alpha"]]
        printed = F(prof["expected"])
        decimals = len(prof["expected"].split(".")[1])
        # the pages print E[N] rounded to the shown decimals (2.3056 -> 2.306)
        assert abs(expected_output_length(alphas) - printed) <= F(1, 2 * 10 ** decimals)


@pytest.mark.parametrize("a,gamma", [(F(1, 2), 3), (F(4, 5), 5), (F(9, 10), 7)])
def test_expected_output_length_closed_form(a, gamma):
    assert expected_output_length([a] * gamma) == (1 - a ** (gamma + 1)) / (1 - a)


def test_expected_output_length_monte_carlo_philox():
    """Constant acceptance a: the mean over Philox-driven rounds is within 4 sigma."""
    a, gamma, rounds = 0.8, 4, 20000
    p = np.array([a, 1 - a])
    q = np.array([1.0, 0.0])
    pb = np.array([0.5, 0.5])
    lengths = np.empty(rounds)
    for s in range(rounds):
        res = verify.walk_chain(
            gamma, 2, lambda i: Dist(False, probs=(p if i < gamma else pb)),
            lambda i: Dist(False, probs=q), [0] * gamma,
            lambda i, s=s: philox.uniform(99, s, i, 0), lambda i, s=s: philox.uniform(99, s, i, 1))
        lengths[s] = res["num_accepted"] + 1
    want = (1 - a ** (gamma + 1)) / (1 - a)
    sigma = lengths.std() / math.sqrt(rounds)
    assert abs(lengths.mean() - want) < 4 * sigma


# ---------------------------------------------------------------------------
# chain edge cases
# ---------------------------------------------------------------------------

def test_chain_bad_token_with_equal_rows_is_degenerate():
    p = np.array([0.25, 0.75])
    res = verify.walk_chain(1, 2, lambda i: Dist(False, probs=p), lambda i: Dist(False, probs=p),
                            [5], lambda i: 0.0, lambda i: 0.5)
    assert res["flags"] == verify.FLAG_BAD_TOKEN | verify.FLAG_DEGENERATE_RESIDUAL
    assert res["num_accepted"] == 0 and res["tokens"] == [1, -1]


def test_chain_gamma_zero_is_plain_sampling():
    p = np.array([0.25, 0.5, 0.25])
    for u, tok in [(0.0, 0), (0.3, 1), (0.8, 2)]:
        res = verify.walk_chain(0, 3, lambda i: Dist(False, probs=p), None, [],
                                None, lambda i, u=u: u)
        assert res["tokens"] == [tok] and res["num_accepted"] == 0


def test_chain_logit_level_uses_override_and_lazy_rows():
    rng = np.random.default_rng(21)
    B, gamma, V = 3, 4, 50
    target = rng.standard_normal((B, gamma + 1, V))
    draft = target[:, :gamma] + 0.3 * rng.standard_normal((B, gamma, V))
    tokens = rng.integers(0, V, (B, gamma)).astype(np.int32)
    ov = np.zeros((B, gamma + 1, 2))  # u = 0 accepts every draft with p(x) > 0
    res = verify.verify_chain(target, draft, tokens, np.ones(B), np.ones(B),
                              uniform_override=ov)
    for b in range(B):
        assert res[b]["num_accepted"] == gamma
        assert res[b]["tokens"][:gamma] == list(tokens[b])
        # u = 0 draws the smallest index with positive mass: token 0
        assert res[b]["tokens"][gamma] == 0


# ---------------------------------------------------------------------------
# tree: exact law, closed form of the repeated residual, masks
# ---------------------------------------------------------------------------

def tree_law(P, Q, V, shape_parent, max_depth):
    """Law of the first max_depth+1 tokens (tree round + AR continuation).

    Children of a node are drawn i.i.d. from that node's draft row (with
    replacement, so duplicate siblings occur).  Branch weights follow the
    multi-step rule step by step using the oracle's accept_test and
    positive_residual; the oracle's tree walk is run on each branch with
    uniforms inside the branch and its output recorded.
    """
    N = len(shape_parent)
    kids = [[c for c in range(N) if shape_parent[c] == n] for n in range(N)]
    law = {}
    L = max_depth + 1

    def assignments(n, prefix):
        """All token assignments of n's subtree (children drawn from Q[prefix])."""
        if not kids[n]:
            yield {}, F(1)
            return
        q = Q[prefix]
        for toks in itertools.product(range(V), repeat=len(kids[n])):
            w = F(1)
            for t in toks:
                w *= q[t]
            if w == 0:
                continue
            subs = [list(assignments(c, prefix + (t,))) for c, t in zip(kids[n], toks)]
            for combo in itertools.product(*subs):
                a = {c: t for c, t in zip(kids[n], toks)}
                ww = w
                for sub, sw in combo:
                    a.update(sub)
                    ww *= sw
                yield a, ww

    for assign, wa in assignments(0, ()):
        tokens = [0] + [assign[c] for c in range(1, N)]
        prefix_of = {0: ()}
        for c in range(1, N):
            prefix_of[c] = prefix_of[shape_parent[c]] + (tokens[c],)

        def branches(n, weight, ua):
            dist = P[prefix_of[n]]
            for c in kids[n]:
                _, alpha, f = verify.accept_test(dist, Q[prefix_of[n]], tokens[c], F(0))
                assert f == 0
                if alpha > 0:
                    yield from branches(c, weight * alpha, {**ua, c: alpha / 2})
                if alpha == 1:
                    return
                weight = weight * (1 - alpha)
                ua = {**ua, c: (1 + alpha) / 2}
                r, _, f = verify.positive_residual(dist, Q[prefix_of[n]])
                if not f:
                    dist = r
            for v in range(V):
                if dist[v]:
                    yield n, weight * dist[v] / sum(dist), ua, representative_uniform(dist, v)

        for node, w, ua, ud in branches(0, wa, {}):
            res = verify.walk_tree(
                N, V, shape_parent, tokens,
                lambda n: Dist(False, probs=P[prefix_of[n]]),
                lambda n: Dist(False, probs=Q[prefix_of[n]]),
                lambda c: ua.get(c, F(0)), lambda n: ud, max_depth)
            assert res["flags"] == 0 and res["path"][res["num_accepted"]] == node
            out = tuple(t for t in res["tokens"] if t >= 0)
            for cont, cw in ar_law(P, out, L - len(out)).items():
                key = out + cont
                law[key] = law.get(key, 0) + w * cw
    return law


@pytest.mark.parametrize("V,shape,depth", [
    (2, [-1, 0, 0], 1), (3, [-1, 0, 0], 1), (3, [-1, 0, 0, 0], 1), (5, [-1, 0, 0], 1),
    (2, [-1, 0, 0, 1, 1], 2), (3, [-1, 0, 0, 1], 2), (2, [-1, 0, 1, 1, 0], 2),
])
def test_tree_output_law_is_target_law(V, shape, depth):
    rng = np.random.default_rng(7 * V + len(shape))
    P = make_tables(rng, V, depth + 1)
    Q = make_tables(rng, V, depth)
    got = tree_law(P, Q, V, shape, depth)
    assert {k: v for k, v in got.items() if v} == ar_law(P, (), depth + 1)


def test_tree_law_detects_independent_sibling_retries(monkeypatch):
    """Testing every sibling against the original p (no residual update) is wrong.

    The planted mistake replaces the residual update by "keep p"; the branch
    weights and the walk then both follow the mistaken rule, and the law of
    the output is no longer the target's.
    """
    rng = np.random.default_rng(31)
    P = make_tables(rng, 3, 2, zero_prob=0.0)
    Q = make_tables(rng, 3, 1, zero_prob=0.0)
    monkeypatch.setattr(verify, "positive_residual", lambda p, q: (p, F(1), 0))
    got = tree_law(P, Q, 3, [-1, 0, 0], 1)
    assert {k: v for k, v in got.items() if v} != ar_law(P, (), 2)


def test_repeated_residual_closed_form():
    """s rejections at one node give [p - c_s q]_+ / W_s, c_1 = 1, c_{s+1} = c_s + W_s.

    The kernel uses this closed form; the oracle iterates p <- norm([p - q]_+)
    as the pages state.  Exact rationals.
    """
    rng = np.random.default_rng(17)
    for _ in range(200):
        V = int(rng.integers(2, 10))
        p, q = random_rational_dist(rng, V, 0.2), random_rational_dist(rng, V, 0.2)
        dist, c = p, F(1)
        for s in range(1, 6):
            r, Z, f = verify.positive_residual(dist, q)
            if f:
                break
            dist = r
            w = np.maximum(p - c * q, 0)
            W = w.sum()
            assert list(dist) == list(w / W)
            c = c + W


def test_tree_walk_leaf_root_is_bonus():
    p = np.array([0.1, 0.6, 0.3])
    res = verify.walk_tree(1, 3, [-1], [0], lambda n: Dist(False, probs=p), None,
                           None, lambda n: 0.5, 3)
    assert res["num_accepted"] == 0 and res["path"][:2] == [0, -1] and res["tokens"][:2] == [1, -1]


def test_tree_check_flags():
    assert verify.tree_check([-1, 0, 1], 2) == (0, [0, 1, 2])
    assert verify.tree_check([-1, 0, 1], 1)[0] == verify.FLAG_DEPTH
    assert verify.tree_check([0, 0, 1], 5)[0] == verify.FLAG_BAD_TREE
    assert verify.tree_check([-1, 2, 0], 5)[0] == verify.FLAG_BAD_TREE
    res = verify.walk_tree(3, 2, [-1, 0, 1], [0, 0, 0], None, None, None, None, 1)
    assert res["num_accepted"] == -1 and res["flags"] == verify.FLAG_DEPTH


def test_tree_mask_page_examples():
    g = load_golden("tree_examples.json")
    for tree in g["trees"]:
        mask, pos, flags = verify.tree_mask(tree["parent"], max_depth=8)
        assert flags == 0
        assert list(pos) == tree["depth"]
        for n, vis in enumerate(tree["visible"]):
            got = [m for m in range(len(tree["parent"])) if (int(mask[n, m // 64]) >> (m % 64)) & 1]
            assert got == vis


def test_tree_mask_matches_reachability_closure():
    """Ancestor-or-self sets from the boolean closure of the parent matrix."""
    from speculative_decoding_verification_temp_gb300 import workloads
    rng = np.random.default_rng(23)
    for N in (1, 2, 7, 60, 130):
        parent = workloads.tree_shape(rng, (4, 3, 2, 2, 1, 1, 1), N) if N <= 185 else None
        A = np.zeros((N, N), dtype=bool)
        for n in range(1, N):
            A[n, parent[n]] = True
        R = np.eye(N, dtype=bool)
        for _ in range(N):
            R = R | (R.astype(np.int64) @ A.astype(np.int64) > 0)
        mask, pos, flags = verify.tree_mask(parent, max_depth=64)
        assert flags == 0
        for n in range(N):
            got = np.array([(int(mask[n, m // 64]) >> (m % 64)) & 1 for m in range(N)], bool)
            np.testing.assert_array_equal(got, R[n])
            assert pos[n] == R[n].sum() - 1


def test_tree_mask_invalid_links():
    mask, pos, flags = verify.tree_mask([-1, 0, 5, 2], max_depth=4)
    assert flags == verify.FLAG_BAD_TREE
    assert list(pos) == [0, 1, -1, -1]
    mask, pos, flags = verify.tree_mask([-1, 0, 1, 2], max_depth=2)
    assert flags == verify.FLAG_DEPTH and list(pos) == [0, 1, 2, 3]


def test_overlap_page_examples():
    g = load_golden("worked_examples.json")
    a = g["example_a"]
    p, q = frac_array(a["p"]), frac_array(a["q"])
    assert verify.overlap(p, q) == F(a["beta"])
    # the second example: the accepted mass (0.4, 0.2, 0.1) sums to 0.7
    b = g["example_b"]
    p, q = frac_array(b["p"]), frac_array(b["q"])
    assert verify.overlap(p, q) == sum(F(v) for v in b["accepted_mass"])


def test_overlap_identities():
    rng = np.random.default_rng(21)
    for V in (2, 3, 5, 8):
        for _ in range(20):
            p, q = random_rational_dist(rng, V), random_rational_dist(rng, V)
            _, Z, _ = verify.positive_residual(p, q)
            assert verify.overlap(p, q) + Z == 1
            assert verify.overlap(p, p) == 1
            assert verify.overlap(p, q) == verify.overlap(q, p)
    # disjoint supports share no mass
    assert verify.overlap(frac_array(["1", "0"]), frac_array(["0", "1"])) == 0


def test_chain_overlap_matches_per_row_policy():
    rng = np.random.default_rng(22)
    B, gamma, V = 3, 2, 40
    zt = rng.normal(size=(B, gamma + 1, V))
    zd = zt[:, :gamma] + 0.5 * rng.normal(size=(B, gamma, V))
    t = np.array([1.0, 0.0, 0.7])
    beta = verify.chain_overlap(zt, zd, t, t)
    # sequence 1 is greedy on both sides: beta is 1 where the argmaxes agree
    for i in range(gamma):
        assert beta[1, i] == float(np.argmax(zt[1, i]) == np.argmax(zd[1, i]))
    # a softmax pair: beta is the expected acceptance probability under q
    p = np.exp(zt[0, 0] - zt[0, 0].max()); p /= p.sum()
    q = np.exp(zd[0, 0] - zd[0, 0].max()); q /= q.sum()
    assert abs(beta[0, 0] - np.sum(q * np.minimum(1.0, p / q))) < 1e-12


# ---------------------------------------------------------------------------
# typical acceptance: whoami-wesleyyou.top "Speculative Decoding" notes,
# § Medusa-1 与 typical acceptance
# ---------------------------------------------------------------------------

def test_entropy_closed_forms_and_library():
    import math
    from scipy.stats import entropy as scipy_entropy
    for V in (1, 2, 7, 128):
        assert abs(verify.entropy(np.full(V, 1.0 / V)) - math.log(V)) < 1e-12
    assert verify.entropy(np.array([0.0, 1.0, 0.0])) == 0.0
    rng = np.random.default_rng(31)
    for _ in range(20):
        p = rng.dirichlet(np.full(50, 0.3))
        p[rng.integers(0, 50, 5)] = 0.0  # zero entries contribute nothing
        p /= p.sum()
        assert abs(verify.entropy(p) - scipy_entropy(p)) < 1e-12


def test_typical_threshold_branches():
    u = np.full(4, 0.25)  # exp(-H) = 1/4
    assert abs(verify.typical_threshold(u, 1.0, 0.5) - 0.125) < 1e-15
    assert abs(verify.typical_threshold(u, 0.1, 0.5) - 0.1) < 1e-15
    # p(x) = 1/4 passes 1/8 and fails 3/8
    assert 0.25 > verify.typical_threshold(u, 1.0, 0.5)
    assert not 0.25 > verify.typical_threshold(u, 1.0, 1.5)
    # a one-hot row has H = 0: the threshold is min(epsilon, delta)
    assert verify.typical_threshold(np.array([0.0, 1.0]), 0.3, 0.9) == 0.3
    # a more spread target lowers the entropy-dependent threshold
    rng = np.random.default_rng(32)
    z = rng.normal(size=64)
    thr = []
    for T in (0.3, 0.6, 1.0, 2.0, 4.0):
        p = np.exp((z - z.max()) / T)
        thr.append(verify.typical_threshold(p / p.sum(), 1.0, 0.8))
    assert all(a > b for a, b in zip(thr, thr[1:]))


def _rows(*dists):
    return [Dist(False, probs=np.asarray(d, np.float64)) for d in dists]


def test_walk_typical_longest_prefix_then_greedy_token():
    V = 4
    # thresholds min(0.2, 0.5 exp(-H)): 0.195 for (.7, .1, .1, .1) (H = 0.9405),
    # 0.125 for the uniform row; every draft passes, the bonus is argmax 1
    rows = _rows([0.7, 0.1, 0.1, 0.1],
                 [0.25, 0.25, 0.25, 0.25],
                 [0.1, 0.1, 0.1, 0.7],
                 [0.1, 0.6, 0.2, 0.1])
    logits = [np.log(r.probs) for r in rows]
    get_p = lambda i: rows[i]
    get_z = lambda i: logits[i]
    res = verify.walk_typical(3, V, get_p, get_z, [0, 1, 3], 0.2, 0.5)
    assert res["num_accepted"] == 3 and res["tokens"] == [0, 1, 3, 1]
    # a failed test ends the prefix even when later drafts would pass: under
    # (.97, .01, .01, .01) the threshold is 0.2 and token 1 has 0.01
    rows2 = _rows([0.7, 0.1, 0.1, 0.1], [0.97, 0.01, 0.01, 0.01], [0.1, 0.1, 0.1, 0.7],
                  [0.1, 0.6, 0.2, 0.1])
    logits2 = [np.log(r.probs) for r in rows2]
    res = verify.walk_typical(3, V, lambda i: rows2[i], lambda i: logits2[i], [0, 1, 3], 0.2, 0.5)
    assert res["num_accepted"] == 1 and res["tokens"] == [0, 0, -1, -1]
    # a draft outside the vocabulary fails and is flagged
    res = verify.walk_typical(3, V, get_p, get_z, [0, 9, 3], 0.2, 0.5)
    assert res["num_accepted"] == 1 and res["tokens"] == [0, 0, -1, -1]
    assert res["flags"] == verify.FLAG_BAD_TOKEN


def test_typical_chain_greedy_and_threshold_one():
    rng = np.random.default_rng(33)
    B, gamma, V = 2, 3, 30
    z = rng.normal(size=(B, gamma + 1, V))
    arg = z.argmax(-1)
    toks = arg[:, :gamma].copy()
    toks[1, 1] = (arg[1, 1] + 1) % V
    t0 = np.zeros(B)
    # greedy rows: the test passes exactly for the argmax (threshold min(eps, delta) < 1)
    r = verify.typical_chain(z, toks, t0, 0.3, 0.5)
    assert r[0]["num_accepted"] == gamma and r[0]["tokens"] == list(arg[0])
    assert r[1]["num_accepted"] == 1 and r[1]["tokens"] == [arg[1, 0], arg[1, 1], -1, -1]
    # with epsilon = delta = 1 no probability exceeds the threshold
    r = verify.typical_chain(z, toks, t0, 1.0, 1.0)
    assert all(x["num_accepted"] == 0 for x in r)
    assert [x["tokens"][0] for x in r] == list(arg[:, 0])


# ---------------------------------------------------------------------------
# EAGLE-2 rerank: zzszmyf.github.io "LLM 推测解码精读笔记 · 04 EAGLE", § 10.3
# and § 题 5
# ---------------------------------------------------------------------------

def random_tree(rng, N):
    return np.array([-1] + [int(rng.integers(0, n)) for n in range(1, N)], np.int32)


def test_tree_values_are_path_products():
    from fractions import Fraction
    rng = np.random.default_rng(61)
    for _ in range(20):
        N = int(rng.integers(1, 40))
        par = random_tree(rng, N)
        c = rng.random(N).astype(np.float32)
        val = verify.tree_values(par, c)
        for n in range(N):
            path, a = Fraction(1), n
            while a != -1:
                path *= Fraction(float(c[a]))
                a = int(par[a])
            num, exp = val[n]
            assert Fraction(num) * Fraction(2) ** exp == path  # exact, no rounding
            assert verify.value_float(val[n]) == float(path)
            if n:  # value(child) <= value(parent)
                pn, pe = val[int(par[n])]
                assert Fraction(num) * Fraction(2) ** exp <= Fraction(pn) * Fraction(2) ** pe


def test_rerank_ranks_exact_products_not_rounded_ones():
    # Two nodes whose float32 path products are equal but whose exact products
    # differ: a deep node a * b just above a shallow node d = fl32(a * b).
    # Rounded products would tie and hand the place to the shallower node; the
    # page's value (the exact product) puts the deeper one first.
    a = np.float32(1 - 3 * 2.0 ** -24)
    exact = float(a) * float(a)
    d = np.float32(exact)
    assert float(d) < exact and np.float32(a * a) == d
    par = np.array([-1, 0, 1, 0], np.int32)       # 0 -> 1 -> 2 and 0 -> 3
    c = np.array([1.0, a, a, d], np.float32)      # values 1, a, a*a, d
    nodes, _, vals, _ = verify.tree_rerank(par, c, 3)
    assert nodes == [0, 1, 2] and vals[2] == exact
    # with the products exactly equal the shallower node wins the tie
    c = np.array([1.0, 0.5, 0.5, 0.25], np.float32)
    assert verify.tree_rerank(par, c, 3)[0] == [0, 1, 3]


def test_tree_values_do_not_underflow():
    # A chain of 400 nodes of confidence 0.5: the deepest value is 2^-399,
    # below every float32 and float64 normal, yet still ordered exactly.
    N = 400
    par = np.arange(-1, N - 1, dtype=np.int32)
    c = np.full(N, 0.5, np.float32)
    c[0] = 1.0
    val = verify.tree_values(par, c)
    assert val[N - 1] == (1, -(N - 1))
    order, _, _ = verify.rerank_order(par, c)
    assert order == list(range(N))


def test_rerank_is_connected_and_top_m():
    rng = np.random.default_rng(62)
    for _ in range(50):
        N = int(rng.integers(1, 30))
        par = random_tree(rng, N)
        c = rng.random(N).astype(np.float32)
        c[0] = 1.0
        c[rng.random(N) < 0.2] = 1.0  # ties along paths
        for m in (1, 3, N, N + 2):
            nodes, newp, vals, flags = verify.tree_rerank(par, c, m)
            assert flags == 0 and len(nodes) == min(m, N) and nodes[0] == 0
            chosen = set(nodes)
            for n in nodes:  # every chosen node's parent is chosen
                assert n == 0 or int(par[n]) in chosen
            for i, n in enumerate(nodes):  # the re-indexed parents match
                assert newp[i] == (-1 if n == 0 else nodes.index(int(par[n])))
            # no unchosen node beats a chosen one
            key = verify.value_keys(verify.tree_values(par, c))
            if len(nodes) < N:
                worst = min(key[n] for n in chosen)
                assert all(key[n] <= worst for n in range(N) if n not in chosen)


def test_rerank_page_properties_by_hand():
    # root 0 -> 1 (c .9) -> 2 (c .9) -> 3 (c .5); root -> 4 (c .6)
    par = np.array([-1, 0, 1, 2, 0], np.int32)
    c = np.array([1.0, 0.9, 0.9, 0.5, 0.6], np.float32)
    # values 1, .9, .81, .405, .6: with m = 4 the shallow unexpanded node 4
    # (.6) is kept and the deep node 3 (.405) is dropped
    nodes, newp, vals, _ = verify.tree_rerank(par, c, 4)
    assert nodes == [0, 1, 2, 4] and newp == [-1, 0, 1, 0]
    # a tie between a depth-1 and a depth-2 node goes to the shallower one
    par = np.array([-1, 0, 1, 0], np.int32)
    c = np.array([1.0, 1.0, 0.5, 0.5], np.float32)  # values 1, 1, .5, .5
    assert verify.tree_rerank(par, c, 3)[0] == [0, 1, 3]


def test_rerank_bad_inputs():
    assert verify.tree_rerank(np.array([0, 0], np.int32), np.ones(2), 2)[3] == verify.FLAG_BAD_TREE
    assert verify.tree_rerank(np.array([-1, 1], np.int32), np.ones(2), 2)[3] == verify.FLAG_BAD_TREE
    nodes, _, vals, flags = verify.tree_rerank(np.array([-1, 0, 0], np.int32),
                                               np.array([1.0, np.nan, 2.0]), 2)
    assert flags == verify.FLAG_NONFINITE and nodes == [0, 2] and vals == [1.0, 1.0]


# ---------------------------------------------------------------------------
# top-p and min-p (the published definitions; the pages only name them)
# ---------------------------------------------------------------------------

def test_topp_hand_cases():
    from oracle import policy as pol
    p = np.array([0.05, 0.5, 0.15, 0.3])
    # descending 0.5, 0.3, 0.15, 0.05: the mass reaches 0.8 at the second token
    assert np.allclose(pol.topp_filter(p, 0.8), [0, 0.5 / 0.8, 0, 0.3 / 0.8])
    assert np.allclose(pol.topp_filter(p, 0.81), [0, 0.5, 0.15, 0.3] / np.float64(0.95))
    assert np.array_equal(pol.topp_filter(p, 1.0), p)
    # the most probable token alone when top_p is below its mass
    assert np.allclose(pol.topp_filter(p, 0.3), [0, 1, 0, 0])
    # ties at the boundary are all kept
    q = np.array([0.4, 0.2, 0.2, 0.2])
    assert np.allclose(pol.topp_filter(q, 0.5), q)


def test_topp_minimal_prefix_property():
    from oracle import policy as pol
    rng = np.random.default_rng(71)
    for _ in range(200):
        V = int(rng.integers(2, 40))
        p = rng.dirichlet(np.full(V, 0.5))
        tp = float(rng.uniform(0.05, 0.99))
        f = pol.topp_filter(p, tp)
        kept = f > 0
        # a descending prefix, holding at least top_p of the mass ...
        assert p[kept].min() >= p[~kept].max(initial=0.0)
        assert p[kept].sum() >= tp - 1e-12
        # ... and minimal: without its smallest value it falls short
        assert p[kept].sum() - p[kept].min() * (p[kept] == p[kept].min()).sum() < tp
        assert abs(f.sum() - 1.0) < 1e-12


def test_minp_hand_cases_and_composition():
    from oracle import policy as pol
    p = np.array([0.5, 0.3, 0.15, 0.05])
    assert np.allclose(pol.minp_filter(p, 0.2), [0.5, 0.3, 0.15, 0] / np.float64(0.95))
    assert np.allclose(pol.minp_filter(p, 0.6), [0.5, 0.3, 0, 0] / np.float64(0.8))
    assert np.array_equal(pol.minp_filter(p, 0.0), p)
    # min-p at 1 keeps the maxima only; temperature first, then the filters
    z = np.log(np.array([0.5, 0.3, 0.15, 0.05]))
    d = pol.policy_distribution_ext(z, 1.0, 0, 1.0, 1.0)
    assert np.allclose(d.probs, [1, 0, 0, 0])
    d = pol.policy_distribution_ext(z, 2.0, 0, 0.8, 0.0)
    sm = np.exp(z / 2) / np.exp(z / 2).sum()
    assert np.allclose(d.probs, pol.topp_filter(sm, 0.8))
    # greedy rows stay one-hot
    assert pol.policy_distribution_ext(z, 0.0, 0, 0.5, 0.5).onehot


def test_topp_minp_out_of_range_readings():
    # the pages define neither filter: NaN switches a filter off, top_p <= 0
    # keeps the most probable value, min_p > 1 is taken as 1; the kept mass is
    # never empty, so every result is a distribution
    from oracle import policy as pol
    p = np.array([0.1, 0.4, 0.4, 0.1])
    assert np.array_equal(pol.topp_filter(p, np.nan), p)
    assert np.array_equal(pol.minp_filter(p, np.nan), p)
    assert np.allclose(pol.topp_filter(p, 0.0), [0, 0.5, 0.5, 0])    # ties with the top kept
    assert np.allclose(pol.topp_filter(p, -1.0), [0, 0.5, 0.5, 0])
    assert np.allclose(pol.minp_filter(p, 7.0), pol.minp_filter(p, 1.0))
    assert np.allclose(pol.minp_filter(p, 7.0), [0, 0.5, 0.5, 0])
    assert np.array_equal(pol.minp_filter(p, -0.5), p)
    z = np.log(p)
    for tp, mp in ((np.nan, 2.0), (-3.0, np.nan), (0.5, 1.5)):
        d = pol.policy_distribution_ext(z, 1.0, 0, tp, mp)
        assert np.isfinite(d.probs).all() and abs(d.probs.sum() - 1) < 1e-12


def test_filtered_policies_keep_the_verifier_exact():
    """With the same top-p / min-p on both sides the chain still returns the
    filtered target law exactly (enumeration over uniforms, exact arithmetic)."""
    from oracle import policy as pol
    rng = np.random.default_rng(72)
    for _ in range(10):
        V = 5
        p = pol.minp_filter(pol.topp_filter(rng.dirichlet(np.ones(V)), 0.85), 0.1)
        q = pol.minp_filter(pol.topp_filter(rng.dirichlet(np.ones(V)), 0.85), 0.1)
        pf = random_rational_from(p)
        qf = random_rational_from(q)
        law = [F(0)] * V
        for x in range(V):
            if qf[x] == 0:
                continue
            accepted, alpha, _ = verify.accept_test(pf, qf, x, F(0))
            law[x] += qf[x] * alpha
        r, Z, _ = verify.positive_residual(pf, qf)
        for y in range(V):
            law[y] += Z * r[y] if Z > 0 else 0
        assert law == list(pf)


def random_rational_from(p):
    # a nearby distribution in exact rationals with the same support
    w = [int(round(float(x) * 1000)) if x > 0 else 0 for x in p]
    w = [max(x, 1) if px > 0 else 0 for x, px in zip(w, p)]
    s = sum(w)
    return np.array([F(x, s) for x in w], dtype=object)


def test_verify_chain_with_topp_minp_defaults_and_filtering():
    """The new filters are off by default (identical results) and, when on,
    every emitted token lies in the filtered target support."""
    from oracle import policy as pol
    rng = np.random.default_rng(73)
    B, gamma, V = 6, 3, 50
    zt = rng.normal(size=(B, gamma + 1, V)) * 2
    zd = zt[:, :gamma] + 0.5 * rng.normal(size=(B, gamma, V))
    toks = zd.argmax(-1)
    t = np.ones(B)
    base = verify.verify_chain(zt, zd, toks, t, t, seed=5)
    same = verify.verify_chain(zt, zd, toks, t, t, seed=5, target_top_p=np.ones(B),
                               draft_top_p=np.ones(B), target_min_p=np.zeros(B),
                               draft_min_p=np.zeros(B))
    assert [r["tokens"] for r in base] == [r["tokens"] for r in same]
    tp, mp = np.full(B, 0.6), np.full(B, 0.05)
    res = verify.verify_chain(zt, zd, toks, t, t, seed=5, target_top_p=tp, draft_top_p=tp,
                              target_min_p=mp, draft_min_p=mp)
    for b, r in enumerate(res):
        for i, x in enumerate(r["tokens"]):
            if x < 0:
                break
            p = pol.policy_distribution_ext(zt[b, i], 1.0, 0, 0.6, 0.05).probs
            assert p[x] > 0, (b, i, x)
