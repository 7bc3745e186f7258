"""Pins of the CPU oracle against facts fixed by the pages and by mathematics.

No test here retypes an oracle formula and compares it with itself: each one
checks the oracle against a library routine, a closed form, an invariant or
an exact enumeration.

Sources (page title, section):
  [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈"
  [SD-7.3]   "7.3 Speculative Decoding：投机采样加速"
  [SD-blog]  "推测解码：用一个“小模型”骗出 3 倍推理速度"
"""

import itertools
import math

import numpy as np
import pytest
from scipy import optimize, special, stats

from ssd_inputs import WORKLOADS, make_batch


# --------------------------------------------------------------------------- Philox
def test_philox_round_structure_matches_numpy_philox4x64(orc):
    """The width-generic Philox of the oracle, instantiated at 64-bit words,
    reproduces numpy's Philox4x64-10 (numpy increments the counter before
    each block, so its first block is the oracle's counter + 1)."""
    rng = np.random.default_rng(5)
    for _ in range(20):
        key = [int(x) for x in rng.integers(0, 2 ** 63, size=2, dtype=np.uint64)]
        ctr = [int(x) for x in rng.integers(0, 2 ** 63, size=4, dtype=np.uint64)]
        bg = np.random.Philox(counter=ctr, key=key)
        raw = bg.random_raw(8)
        c1 = list(ctr)
        c1[0] += 1
        np.testing.assert_array_equal(orc.philox4x64(c1, key), raw[:4])
        c1[0] += 1
        np.testing.assert_array_equal(orc.philox4x64(c1, key), raw[4:])


def test_philox32_uniforms_are_uniform(orc):
    """u = (out0 >> 8) / 2^24: exact 24-bit grid, chi-square uniform over 256
    bins and over 32x32 serial pairs."""
    n = 1 << 20
    u = np.concatenate([orc.uniform_batch(12345, c1, 0, 7, n // 4) for c1 in range(4)])
    assert np.all(u >= 0) and np.all(u < 1)
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
    h, _ = np.histogram(u, bins=256, range=(0, 1))
    assert stats.chisquare(h).pvalue > 1e-4
    a = np.floor(u[0::2] * 32).astype(int)
    b = np.floor(u[1::2] * 32).astype(int)
    h2 = np.bincount(a * 32 + b, minlength=1024)
    assert stats.chisquare(h2).pvalue > 1e-4


def test_uniform_counter_words_are_distinct_streams(orc):
    base = orc.uniform(7, 3, 2, 0, 9)
    others = [orc.uniform(8, 3, 2, 0, 9), orc.uniform(7, 4, 2, 0, 9), orc.uniform(7, 3, 3, 0, 9),
              orc.uniform(7, 3, 2, 1, 9), orc.uniform(7, 3, 2, 0, 10)]
    assert all(o != base for o in others)


# --------------------------------------------------------------------------- softmax
def test_softmax_matches_scipy_and_temperature(orc):
    rng = np.random.default_rng(1)
    for V in (2, 7, 32, 1000):
        z = rng.normal(0, 3, V)
        for T in (0.3, 1.0, 2.5):
            p = orc.softmax(z, T)
            np.testing.assert_allclose(p, special.softmax(z / T), rtol=1e-13, atol=1e-300)
            assert abs(p.sum() - 1) < 1e-13
    assert np.allclose(orc.softmax(np.full(16, 3.25), 0.7), 1 / 16, rtol=0, atol=1e-16)
    # two-token case is the logistic function of the scaled difference
    p = orc.softmax(np.array([1.5, -0.5]), 0.8)
    assert abs(p[0] - special.expit(2.0 / 0.8)) < 1e-15


# --------------------------------------------------------------------------- top-F
def test_top_n_matches_stable_library_sort(orc):
    """Top-F by (logit desc, index asc) equals numpy's stable lexsort prefix,
    including heavy ties ([SSD-note] §"怎么猜奖励 token")."""
    rng = np.random.default_rng(2)
    for V in (5, 32, 257, 5000):
        for tie in (False, True):
            z = rng.integers(-3, 4, V).astype(float) if tie else rng.normal(size=V)
            order = np.lexsort((np.arange(V), -z))
            for n in (1, 2, 5, min(V, 9)):
                np.testing.assert_array_equal(orc.top_n(z, n), order[:n])


# --------------------------------------------------------------------------- Saguaro
@pytest.mark.parametrize("C", [1.0, 0.5, 0.3, 0.05])
def test_saguaro_closed_forms(orc, C):
    """q'(y) = q(y)*C/norm on the cached set S, q(y)/norm elsewhere, with
    norm = 1 - (1-C) Q_S ([SSD-note] §"Saguaro 优化二：Saguaro 采样").
    Closed form q'(S) = C Q_S / (1 - (1-C) Q_S); sum q' = 1; C = 1 leaves q
    bit-identical."""
    rng = np.random.default_rng(3)
    for V, F in ((8, 2), (32, 3), (500, 5)):
        z = rng.normal(0, 2, V)
        q = special.softmax(z)
        S = np.lexsort((np.arange(V), -z))[:F]
        qp = orc.saguaro_dist(z, 1.0, F, C)
        QS = q[S].sum()
        assert abs(qp.sum() - 1) < 1e-12
        assert abs(qp[S].sum() - C * QS / (1 - (1 - C) * QS)) < 1e-12
        notS = np.setdiff1d(np.arange(V), S)
        np.testing.assert_allclose(qp[notS], q[notS] / (1 - (1 - C) * QS), rtol=1e-12)
        if C == 1.0:
            assert np.array_equal(qp, orc.softmax(z, 1.0))


def test_saguaro_raises_residual_mass_on_cached_tokens(orc):
    """Lower C lowers q on S, so (p - q')^+ restricted to S cannot shrink
    ([SSD-note] §"解法：操纵草稿分布")."""
    rng = np.random.default_rng(4)
    for _ in range(20):
        zp = rng.normal(0, 2, 64)
        zq = zp + rng.normal(0, 1, 64)
        p = special.softmax(zp)
        S = np.lexsort((np.arange(64), -zq))[:4]
        prev = -1.0
        for C in (1.0, 0.8, 0.5, 0.3, 0.1):
            w, _ = orc.residual(p, orc.saguaro_dist(zq, 1.0, 4, C))
            assert w[S].sum() >= prev - 1e-15
            prev = w[S].sum()


# --------------------------------------------------------------------------- accept / residual
def test_accept_prob_rule(orc):
    """min(1, p/q): p >= q always accepts, else p/q ([SD-blog] §"三、接受概率为什么是对的")."""
    assert orc.accept_prob(0.3, 0.2) == 1.0
    assert orc.accept_prob(0.2, 0.2) == 1.0
    assert abs(orc.accept_prob(0.1, 0.4) - 0.25) < 1e-16


def test_residual_mass_is_total_variation(orc):
    """Z = sum (p-q)^+ = sum (q-p)^+ = 1 - sum min(p,q) (the rejection
    probability of the position)."""
    rng = np.random.default_rng(5)
    for V in (3, 32, 1000):
        p = special.softmax(rng.normal(0, 2, V))
        q = special.softmax(rng.normal(0, 2, V))
        w, Z = orc.residual(p, q)
        assert np.all(w >= 0)
        assert abs(Z - np.maximum(q - p, 0).sum()) < 1e-13
        assert abs(Z - (1 - np.minimum(p, q).sum())) < 1e-13
        assert abs(Z - 0.5 * np.abs(p - q).sum()) < 1e-13


def test_inverse_cdf_matches_library_search(orc):
    rng = np.random.default_rng(6)
    for _ in range(300):
        V = int(rng.integers(1, 60))
        w = rng.random(V) * (rng.random(V) < 0.6)
        if w.sum() == 0:
            w[rng.integers(V)] = 0.5
        Z = w.sum()
        u = float(np.floor(rng.random() * 2 ** 24)) / 2 ** 24
        y, m = orc.inverse_cdf(w, Z, u)
        expect = int(np.searchsorted(np.cumsum(w), u * Z, side="right"))
        if expect >= V:  # rounding left no index: last positive weight
            expect = int(np.nonzero(w > 0)[0][-1])
        assert y == expect
        assert w[y] > 0
    # exact CDF boundaries (dyadic weights) and u = 0 with leading zero weights:
    # the strict rule never returns a zero-weight token
    w = np.array([0.0, 0.25, 0.25, 0.0, 0.5])
    for u, expect in ((0.0, 1), (0.25, 2), (0.5, 4), (0.75, 4), (0.4999999, 2)):
        assert orc.inverse_cdf(w, 1.0, u)[0] == expect
        assert expect == int(np.searchsorted(np.cumsum(w), u, side="right"))


# --------------------------------------------------------------------------- losslessness
def _exact_emission_law(orc, zp, zq, F, C, T, accept=None):
    """Exact law of the emitted tokens by enumeration over every draft
    sequence x (weight prod_j q'_j(x_j)) and over the accept/reject branches,
    using the oracle's own step functions.  Returns reach[j] = P(position j
    reached) and law[j, y] = P(emitted token at position j = y, j reached)."""
    K = zq.shape[0] - 1
    V = zp.shape[1]
    accept = accept or orc.accept_prob
    p = [orc.softmax(zp[i], T) for i in range(K + 1)]
    qp = [orc.saguaro_dist(zq[j], T, int(F[j]), C) for j in range(K)]
    resid = []
    for i in range(K):
        w, Z = orc.residual(p[i], qp[i])
        resid.append(w / Z)
    law = np.zeros((K + 1, V))
    reach = np.zeros(K + 1)
    for xs in itertools.product(range(V), repeat=K):
        wgt = np.prod([qp[j][xs[j]] for j in range(K)])
        alive = wgt
        for i in range(K):
            reach[i] += alive
            a = accept(p[i][xs[i]], qp[i][xs[i]])
            law[i, xs[i]] += alive * a          # accepted draft is the emitted token
            law[i] += alive * (1 - a) * resid[i]  # rejected: bonus from the residual
            alive *= a
        reach[K] += alive
        law[K] += alive * p[K]                  # all accepted: bonus from p_K
    return p, reach, law


@pytest.mark.parametrize("V,K,C,T", [(4, 2, 1.0, 1.0), (5, 3, 0.5, 1.0), (8, 3, 1.0, 0.7),
                                     (6, 3, 0.3, 1.3), (8, 2, 0.5, 1.0)])
def test_losslessness_exact_enumeration(orc, V, K, C, T):
    """Every emitted token is distributed exactly as the target: P(emit_j = y
    | j reached) = p_j(y) ([SD-7.3] §7.3.3; [SD-blog] §"三、接受概率为什么是对的")."""
    rng = np.random.default_rng(V * 100 + K)
    zp = rng.normal(0, 2, (K + 1, V))
    zq = zp + rng.normal(0, 1, (K + 1, V))
    F = [min(2, V - 1)] * (K + 1)
    p, reach, law = _exact_emission_law(orc, zp, zq, F, C, T)
    for j in range(K + 1):
        np.testing.assert_allclose(law[j] / reach[j], p[j], rtol=0, atol=1e-12)
    # the acceptance probability of position i is alpha_i = sum min(p_i, q'_i)
    for i in range(K):
        alpha = np.minimum(p[i], orc.saguaro_dist(zq[i], T, F[i], C)).sum()
        assert abs(reach[i + 1] / reach[i] - alpha) < 1e-12


def test_losslessness_with_a_factor_per_position(orc):
    """Losslessness does not depend on C being shared by the positions: with a
    different Saguaro factor at every draft position ([SSD-note] §"关于逐位置 C
    的思考") the emitted token at every position still follows p_j exactly, and
    the acceptance of position i is sum min(p_i, q'_i(C_i))."""
    rng = np.random.default_rng(77)
    V, K, T = 6, 3, 1.0
    zp = rng.normal(0, 2, (K + 1, V))
    zq = zp + rng.normal(0, 1, (K + 1, V))
    F = [2, 2, 1, 1]
    Cs = (0.2, 0.7, 0.4)
    p = [orc.softmax(zp[i], T) for i in range(K + 1)]
    qp = [orc.saguaro_dist(zq[j], T, F[j], Cs[j]) for j in range(K)]
    law = np.zeros((K + 1, V))
    reach = np.zeros(K + 1)
    resid = []
    for i in range(K):
        w, Z = orc.residual(p[i], qp[i])
        resid.append(w / Z)
    for xs in itertools.product(range(V), repeat=K):
        alive = np.prod([qp[j][xs[j]] for j in range(K)])
        for i in range(K):
            reach[i] += alive
            a = orc.accept_prob(p[i][xs[i]], qp[i][xs[i]])
            law[i, xs[i]] += alive * a
            law[i] += alive * (1 - a) * resid[i]
            alive *= a
        reach[K] += alive
        law[K] += alive * p[K]
    for j in range(K + 1):
        np.testing.assert_allclose(law[j] / reach[j], p[j], rtol=0, atol=1e-12)
    for i in range(K):
        assert abs(reach[i + 1] / reach[i] - np.minimum(p[i], qp[i]).sum()) < 1e-12


def test_losslessness_enumeration_detects_wrong_accept_rule(orc):
    """The enumeration pin is sensitive: composing the same steps with an
    inverted ratio min(1, q/p) breaks losslessness."""
    rng = np.random.default_rng(9)
    zp = rng.normal(0, 2, (3, 5))
    zq = zp + rng.normal(0, 1, (3, 5))
    bad = lambda px, qx: min(1.0, qx / px)  # noqa: E731
    p, reach, law = _exact_emission_law(orc, zp, zq, [2, 2, 2], 1.0, 1.0, accept=bad)
    assert np.abs(law[0] / reach[0] - p[0]).max() > 1e-3


# --------------------------------------------------------------------------- Monte Carlo laws
def _replicated_batch(zp, zq, n):
    return (np.ascontiguousarray(np.broadcast_to(zp.astype(np.float32), (n,) + zp.shape)),
            np.ascontiguousarray(np.broadcast_to(zq.astype(np.float32), (n,) + zq.shape)))


def _accept_law(p, qp, K):
    """Exact law of k: P(k >= j) = prod_{i<j} alpha_i, alpha_i = sum min(p_i, q'_i)."""
    alpha = [np.minimum(p[i], qp[i]).sum() for i in range(K)]
    ge = np.cumprod([1.0] + alpha)  # P(k >= j), j = 0..K
    pk = np.append(ge[:-1] - ge[1:], ge[K])
    return pk


def test_accept_length_law_monte_carlo(orc):
    """Config-1 shapes (B=1 rows replicated, K=4, V=32, C=0.5, F=[3,3,2,2,2]):
    the histogram of k over 2*10^5 seeded rounds matches the closed-form
    law P(k >= j) = prod_{i<j} alpha_i (chi-square and a 4-sigma z-test on
    E[k]); positions are independent because the synthetic logits do not
    depend on the drafted prefix."""
    w = WORKLOADS["c1"]
    bt = make_batch(w)
    zp = bt["target"][0].astype(np.float64)
    zq = bt["draft"][0].astype(np.float64)
    K, F, C, T = w.K, bt["fanout"], w.C, w.T
    p = [orc.softmax(zp[i], T) for i in range(K + 1)]
    qp = [orc.saguaro_dist(zq[j], T, int(F[j]), C) for j in range(K)]
    pk = _accept_law(p, qp, K)
    n = 50_000
    tgt, dft = _replicated_batch(bt["target"][0], bt["draft"][0], n)
    seeds = np.arange(n, dtype=np.uint64) * 7919 + 11
    ks = []
    for rnd in range(4):
        tok = orc.draft_tokens(dft, F, C, T, seeds, round_=rnd, K=K)
        r = orc.verify(tgt, dft, tok, seeds, rnd, F, C, T, nthreads=8)
        ks.append(r["accept_len"])
    ks = np.concatenate(ks)
    hist = np.bincount(ks, minlength=K + 1)
    assert stats.chisquare(hist, pk * len(ks)).pvalue > 1e-4
    mean = (np.arange(K + 1) * pk).sum()
    var = ((np.arange(K + 1) - mean) ** 2 * pk).sum()
    z = (ks.mean() - mean) / math.sqrt(var / len(ks))
    assert abs(z) < 4


@pytest.mark.parametrize("Cv", [(0.3, 0.5, 0.8, 1.0), (1.0, 0.2, 1.0, 0.6)])
def test_accept_length_law_per_position_C(orc, Cv):
    """One Saguaro factor per draft position ([SSD-note] §"关于逐位置 C 的思考"
    proposes it): drafts drawn from q'_j built with C_j and verified against
    the same q'_j keep the accept-length law P(k >= j) = prod_{i<j} alpha_i,
    alpha_i = sum min(p_i, q'_i(C_i)), and every emitted token still follows
    p_j.  Config-1 shapes, 10^5 seeded rows."""
    w = WORKLOADS["c1"]
    bt = make_batch(w)
    zp = bt["target"][0].astype(np.float64)
    zq = bt["draft"][0].astype(np.float64)
    K, F, T = w.K, bt["fanout"], w.T
    p = [orc.softmax(zp[i], T) for i in range(K + 1)]
    qp = [orc.saguaro_dist(zq[j], T, int(F[j]), Cv[j]) for j in range(K)]
    pk = _accept_law(p, qp, K)
    n = 50_000
    tgt, dft = _replicated_batch(bt["target"][0], bt["draft"][0], n)
    seeds = np.arange(n, dtype=np.uint64) * 6007 + 5
    ks, ts, xs = [], [], []
    for rnd in range(2):
        tok = orc.draft_tokens(dft, F, Cv, T, seeds, round_=rnd, K=K)
        r = orc.verify(tgt, dft, tok, seeds, rnd, F, Cv, T, nthreads=8)
        ks.append(r["accept_len"]); ts.append(r["bonus"]); xs.append(tok)
    ks, ts, xs = np.concatenate(ks), np.concatenate(ts), np.concatenate(xs)
    hist = np.bincount(ks, minlength=K + 1)
    assert stats.chisquare(hist, pk * len(ks)).pvalue > 1e-4
    V = zp.shape[1]
    for j in range(K + 1):
        reached = ks >= j
        emit = np.where(ks[reached] > j, xs[reached][:, min(j, K - 1)], ts[reached])
        obs = np.bincount(emit, minlength=V)
        m = p[j] * reached.sum() > 5
        stat = stats.chisquare(obs[m], p[j][m] / p[j][m].sum() * obs[m].sum())
        assert stat.pvalue > 1e-4, (j, stat)


def _greedy_case(V=40, K=4, B=64, seed=31):
    """Logits whose two largest entries are at least 0.5 apart, with the
    draft's argmax equal to the target's at about half the positions."""
    rng = np.random.default_rng(seed)
    zp = rng.normal(0, 1, (B, K + 1, V))
    zq = zp + rng.normal(0, 0.5, (B, K + 1, V))
    for z in (zp, zq):
        top = z.argmax(-1)
        np.put_along_axis(z, top[..., None], z.max(-1, keepdims=True) + 0.5, -1)
    agree = rng.random((B, K + 1)) < 0.6
    ia = zp.argmax(-1)
    for b in range(B):
        for j in range(K + 1):
            if agree[b, j]:   # move the draft's peak onto the target's argmax
                zq[b, j, ia[b, j]] = zq[b, j].max() + 0.5
    return zp, zq


def test_greedy_is_the_low_temperature_limit(orc):
    """T = 0 is the limit T -> 0: with greedy drafts (x_j = argmax z_q[j])
    the stochastic verify at T = 0.005 (top-2 gaps >= 0.5, so p and q are
    one-hot to e^-100) gives the same accept lengths and bonus tokens as the
    greedy verify, for every seed and C."""
    zp, zq = _greedy_case()
    B, K1, V = zp.shape
    K = K1 - 1
    tok = zq[:, :K].argmax(-1).astype(np.int32)
    seeds = np.arange(B, dtype=np.uint64) * 977 + 1
    F = np.array([3, 2, 2, 1, 1], dtype=np.int32)
    for C in (1.0, 0.4):
        g = orc.verify(zp.astype(np.float32), zq.astype(np.float32), tok, seeds, 0, F, C, 0.0)
        for rnd in range(3):
            s_ = orc.verify(zp.astype(np.float32), zq.astype(np.float32), tok, seeds, rnd, F, C,
                            0.005)
            np.testing.assert_array_equal(g["accept_len"], s_["accept_len"])
            np.testing.assert_array_equal(g["bonus"], s_["bonus"])
            # the guesses' draft probabilities tend to 1 for the argmax, 0 otherwise
            np.testing.assert_array_equal(g["guesses"], s_["guesses"])
            np.testing.assert_allclose(g["guess_q"], s_["guess_q"], rtol=0, atol=1e-12)
    assert 0 < g["accept_len"].mean() < K
    np.testing.assert_array_equal(g["resid_mass"], 1.0)


def test_greedy_ties_go_to_the_lower_index(orc):
    """The greedy argmax breaks ties as numpy.argmax does (first occurrence),
    with heavily tied bf16-rounded logits."""
    rng = np.random.default_rng(5)
    B, K, V = 200, 3, 16
    zp = np.round(rng.normal(0, 1, (B, K + 1, V)) * 2) / 2    # many ties at the max
    zq = zp.copy()
    tok = rng.integers(0, V, (B, K)).astype(np.int32)
    tok[::2] = zp[::2, :K].argmax(-1)                         # half the rows accept early
    F = np.array([2, 2, 1, 1], dtype=np.int32)
    g = orc.verify(zp.astype(np.float32), zq.astype(np.float32), tok, np.zeros(B, np.uint64), 0,
                   F, 1.0, 0.0)
    am = zp.argmax(-1)
    for b in range(B):
        k = next((i for i in range(K) if tok[b, i] != am[b, i]), K)
        assert g["accept_len"][b] == k
        assert g["bonus"][b] == am[b, k]


def test_per_sequence_temperature_equals_separate_calls(orc):
    """A temperature per sequence (0 = greedy) gives each sequence the
    outputs of a call with that temperature alone (same Philox counters)."""
    w = WORKLOADS["c1"]
    bt = make_batch(w, B=6)
    F = bt["fanout"]
    Ts = np.array([1.0, 0.7, 0.0, 1.3, 0.0, 0.5])
    tok = orc.draft_tokens(bt["draft"], F, w.C, 1.0, bt["seeds"], K=w.K)
    both = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 4, F, w.C, Ts)
    for b in range(6):
        one = orc.verify(bt["target"][b:b + 1], bt["draft"][b:b + 1], tok[b:b + 1],
                         bt["seeds"][b:b + 1], 4, F, w.C, Ts[b], row_ids=[b])
        for key in ("accept_len", "bonus", "guesses", "guess_q"):
            np.testing.assert_array_equal(both[key][b:b + 1], one[key])
        np.testing.assert_allclose(both["resid_mass"][b], one["resid_mass"][0], rtol=0, atol=0)


def test_bonus_law_monte_carlo(orc):
    """Given rejection at i the bonus follows normalize((p_i - q'_i)^+); given
    all accepted it follows p_K ([SD-7.3] §7.3.3).  Chi-square over 10^6
    seeded trials at V = 32, plus the marginal of the emitted token at every
    position equals p_j."""
    w = WORKLOADS["c1"]
    rng = np.random.default_rng(21)
    K, V, C, T = 2, 32, 0.5, 1.0
    zp = rng.normal(0, 1.0, (K + 1, V))
    zq = zp + rng.normal(0, 0.7, (K + 1, V))
    F = np.array([3, 2, 2], dtype=np.int32)
    p = [orc.softmax(zp[i].astype(np.float32), T) for i in range(K + 1)]
    qp = [orc.saguaro_dist(zq[j].astype(np.float32), T, int(F[j]), C) for j in range(K)]
    n = 250_000
    tgt, dft = _replicated_batch(zp, zq, n)
    seeds = np.arange(n, dtype=np.uint64) * 104729 + 3
    ks, ts, xs = [], [], []
    for rnd in range(4):
        tok = orc.draft_tokens(dft, F, C, T, seeds, round_=rnd, K=K)
        r = orc.verify(tgt, dft, tok, seeds, rnd, F, C, T, nthreads=8)
        ks.append(r["accept_len"]); ts.append(r["bonus"]); xs.append(tok)
    ks, ts, xs = np.concatenate(ks), np.concatenate(ts), np.concatenate(xs)
    for i in range(K + 1):
        sel = ts[ks == i]
        if i < K:
            wres, Z = orc.residual(p[i], qp[i])
            expect = wres / Z
        else:
            expect = p[K]
        obs = np.bincount(sel, minlength=V)
        m = expect * len(sel) > 5
        assert np.all(obs[~m] <= max(5, 0.01 * len(sel)))
        stat = stats.chisquare(obs[m], expect[m] / expect[m].sum() * obs[m].sum())
        assert stat.pvalue > 1e-4, (i, stat)
    # the emitted token at position j (accepted draft or bonus) ~ p_j
    for j in range(K + 1):
        reached = ks >= j
        emit = np.where(ks[reached] > j, xs[reached][:, min(j, K - 1)], ts[reached])
        obs = np.bincount(emit, minlength=V)
        m = p[j] * reached.sum() > 5
        stat = stats.chisquare(obs[m], p[j][m] / p[j][m].sum() * obs[m].sum())
        assert stat.pvalue > 1e-4, (j, stat)
    _ = w


def test_verify_outputs_are_consistent(orc):
    """Structural facts: all K accepted -> K+1 tokens ([SD-7.3] §7.3.2);
    after a rejection at k the bonus differs from the rejected draft x_k
    (w(x_k) = 0 whenever x_k was rejected); guesses exclude x_j and are
    ordered by draft logit."""
    w = WORKLOADS["c1"]
    bt = make_batch(w, B=2000)
    F, C, T = bt["fanout"], w.C, w.T
    tok = orc.draft_tokens(bt["draft"], F, C, T, bt["seeds"], K=w.K)
    r = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 0, F, C, T, nthreads=8)
    k, t, g = r["accept_len"], r["bonus"], r["guesses"]
    assert k.min() >= 0 and k.max() <= w.K
    rej = k < w.K
    assert np.all(t[rej] != tok[rej, k[rej]])
    for b in range(200):
        for j in range(w.Kq):
            gj = g[b, j][g[b, j] >= 0]
            assert len(gj) == F[j]
            if j < w.K:
                assert tok[b, j] not in gj
            z = bt["draft"][b, j]
            assert np.all(np.diff(z[gj]) <= 0)


# --------------------------------------------------------------------------- cache
def test_cache_lookup_matches_dict(orc):
    rng = np.random.default_rng(8)
    B, K = 64, 4
    keys = {}
    while len(keys) < 500:
        keys[(int(rng.integers(B)), int(rng.integers(K + 1)), int(rng.integers(1000)))] = len(keys)
    row, k, t = (np.array(c) for c in zip(*keys.keys()))
    branch = np.array(list(keys.values()))
    acc = rng.integers(0, K + 1, B)
    bon = rng.integers(0, 1000, B)
    hit_rows = rng.choice(B, 40, replace=False)
    hit_keys = [kk for kk in keys if kk[0] in hit_rows]
    for kk in hit_keys:
        acc[kk[0]], bon[kk[0]] = kk[1], kk[2]
    out, all_hit = orc.cache_lookup(row, k, t, branch, acc, bon)
    expect = np.array([keys.get((b, int(acc[b]), int(bon[b])), -1) for b in range(B)])
    np.testing.assert_array_equal(out, expect)
    assert all_hit == int(np.all(expect >= 0))
    with pytest.raises(KeyError):
        orc.cache_lookup([0, 0], [1, 1], [2, 2], [0, 1], acc, bon)


# --------------------------------------------------------------------------- fan-out
def test_fanout_is_the_lagrange_optimum(orc):
    """F_k ~ a^(k/(1+r)) minimises sum_k a^k F_k^-r under sum F = budget
    ([SSD-note] §"最优扇出度分配"): the closed form equals a numerical
    minimisation of that objective."""
    for K, budget, a, r in ((4, 12, 0.7, 1.0), (8, 24, 0.6, 0.5), (8, 16, 0.9, 2.0)):
        x = orc.fanout_real(K, budget, a, r)
        P = a ** np.arange(K + 1)
        obj = lambda f: float((P * np.power(f, -r)).sum())  # noqa: E731
        res = optimize.minimize(obj, np.full(K + 1, budget / (K + 1)), method="SLSQP",
                                bounds=[(1e-6, budget)] * (K + 1),
                                constraints=[{"type": "eq", "fun": lambda f: f.sum() - budget}],
                                options={"ftol": 1e-14, "maxiter": 500})
        np.testing.assert_allclose(x, res.x, rtol=2e-4)
        assert abs(x.sum() - budget) < 1e-9


def test_fanout_integer_allocation(orc):
    """Integer fan-out sums to the budget, is non-increasing in k for a < 1,
    and stays within one of the real optimum (largest-remainder rounding)."""
    for K in (1, 4, 8, 16):
        for budget in (0, 1, 12, 16, 24, 100):
            for a in (0.3, 0.7, 0.95):
                F = orc.fanout(K, budget, a, 1.0)
                x = orc.fanout_real(K, budget, a, 1.0)
                assert F.sum() == budget
                assert np.all(np.abs(F - x) < 1)
                assert np.all(np.diff(F) <= 0)
    for wl in WORKLOADS.values():
        assert tuple(orc.fanout(wl.K, wl.budget, 0.7, 1.0)) == tuple(wl.fanout)
