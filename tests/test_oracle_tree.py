"""Pins of the oracle's tree-draft verification against facts fixed by the
mathematics and by the linear case.

[SD-7.3] "7.3 Speculative Decoding：投机采样加速" §7.3.9 item 3 names tree drafts
(several candidate continuations per position); §7.3.3 gives the per-token
rule that the tree walk applies to each candidate in turn, with the residual
(r - q)^+ renormalised after every rejection.  The pins:
  * a chain tree is the linear verification (C = 1), output for output;
  * exact enumeration over every assignment of the children's tokens, with
    the oracle's own step functions: the token emitted after reaching a node
    u follows p_u exactly (losslessness) for several topologies;
  * the enumeration is sensitive: without renormalising the residual, or
    testing later children against p instead of the residual, it breaks;
  * Monte Carlo of the whole oracle walk: the first emitted token follows
    p_root and the accepted-path law matches the enumeration (chi-square);
  * tree drafting: each node's token follows its parent's draft
    distribution (chi-square).
"""

import itertools

import numpy as np
import pytest
from scipy import stats

from ssd_inputs import WORKLOADS, make_batch

TOPOLOGIES = {
    "two-children": [-1, 0, 0],
    "three-children": [-1, 0, 0, 0],
    "two-by-two": [-1, 0, 0, 1, 1, 2],
    "uneven": [-1, 0, 0, 1, 3],
}


def children(parent, u):
    return [v for v in range(u + 1, len(parent)) if parent[v] == u]


def _node_law(orc, p, q, parent, u, accept=None, renorm=True, use_residual=True):
    """Exact law of the token emitted right after node u is reached, averaged
    over the i.i.d. draws of u's children from q_u, composed from the oracle's
    step functions (accept_prob, residual).  Returns (law, accept) where
    accept[i] = P(child i of u is accepted)."""
    accept = accept or orc.accept_prob
    ch = children(parent, u)
    V = len(p[u])
    law = np.zeros(V)
    acc = np.zeros(len(ch))
    if not ch:
        return p[u].copy(), acc
    for xs in itertools.product(range(V), repeat=len(ch)):
        w = np.prod([q[u][x] for x in xs])
        r = p[u].copy()
        alive = w
        for i, x in enumerate(xs):
            a = accept(r[x] if use_residual else p[u][x], q[u][x])
            law[x] += alive * a
            acc[i] += alive * a
            alive *= 1 - a
            res, Z = orc.residual(r, q[u])
            if Z > 0:
                r = res / Z if renorm else res
        law += alive * r
    return law, acc


def _tree_rows(V, N, seed):
    rng = np.random.default_rng(seed)
    zp = rng.normal(0, 1.5, (N, V))
    zq = zp + rng.normal(0, 1.0, (N, V))
    return zp, zq


@pytest.mark.parametrize("name", sorted(TOPOLOGIES))
@pytest.mark.parametrize("V", [3, 5])
def test_tree_emission_is_lossless_exact_enumeration(orc, name, V):
    """After reaching any node u the next emitted token -- an accepted child's
    token or the bonus -- follows p_u exactly, whatever the children drawn."""
    parent = TOPOLOGIES[name]
    N = len(parent)
    zp, zq = _tree_rows(V, N, 10 * V + N)
    for T in (1.0, 0.6):
        p = [orc.softmax(zp[u], T) for u in range(N)]
        q = [orc.softmax(zq[u], T) for u in range(N)]
        for u in range(N):
            law, _ = _node_law(orc, p, q, parent, u)
            np.testing.assert_allclose(law, p[u], rtol=0, atol=1e-12)


def test_tree_enumeration_detects_wrong_residuals(orc):
    """The enumeration pin is sensitive: without renormalising the residual,
    or with later children tested against p_u instead of the residual, the
    emission law is no longer p_u."""
    parent = TOPOLOGIES["three-children"]
    zp, zq = _tree_rows(4, 4, 3)
    p = [orc.softmax(zp[u], 1.0) for u in range(4)]
    q = [orc.softmax(zq[u], 1.0) for u in range(4)]
    bad1, _ = _node_law(orc, p, q, parent, 0, renorm=False)
    bad2, _ = _node_law(orc, p, q, parent, 0, use_residual=False)
    assert np.abs(bad1 - p[0]).max() > 1e-3
    assert np.abs(bad2 - p[0]).max() > 1e-3


def test_chain_tree_is_linear_verification(orc):
    """A chain (node v's parent is v - 1) verified as a tree gives the linear
    verification's outputs at C = 1: drafts, accept lengths, bonus tokens,
    residual masses and margins, row for row."""
    w = WORKLOADS["c2"]
    B, K, V = 200, 4, 600
    bt = make_batch(w, B=B, V=V, K=K, seed=5)
    parent = np.arange(-1, K)  # N = K + 1 nodes
    F = np.zeros(K + 1, dtype=np.int32)
    for rnd in (0, 3):
        tok_lin = orc.draft_tokens(bt["draft"], F, 1.0, w.T, bt["seeds"], round_=rnd, K=K)
        tok_tree = orc.tree_draft(bt["draft"], parent, bt["seeds"], rnd, w.T)
        np.testing.assert_array_equal(tok_tree[:, 1:], tok_lin)
        lin = orc.verify(bt["target"], bt["draft"], tok_lin, bt["seeds"], rnd, F, 1.0, w.T)
        tr = orc.tree_verify(bt["target"], bt["draft"], parent, tok_tree, bt["seeds"], rnd, w.T)
        np.testing.assert_array_equal(tr["accept_len"], lin["accept_len"])
        np.testing.assert_array_equal(tr["bonus"], lin["bonus"])
        np.testing.assert_allclose(tr["resid_mass"], lin["resid_mass"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(tr["margin_cdf"], lin["margin_cdf"], rtol=0, atol=1e-12)
        for b in range(B):
            k = tr["accept_len"][b]
            np.testing.assert_array_equal(tr["path"][b, :k], np.arange(1, k + 1))
            assert np.all(tr["path"][b, k:] == -1)


def _exact_path_law(orc, p, q, parent):
    """Exact law of the final node of the walk, by enumeration (oracle steps)."""
    N = len(parent)
    law = np.zeros(N)

    def walk(u, prob):
        _, acc = _node_law(orc, p, q, parent, u)
        ch = children(parent, u)
        law[u] += prob * (1 - acc.sum())
        for i, v in enumerate(ch):
            walk(v, prob * acc[i])

    walk(0, 1.0)
    return law


@pytest.mark.parametrize("name", ["two-by-two", "uneven"])
def test_tree_walk_laws_monte_carlo(orc, name):
    """The whole oracle walk over 60000 seeded trees: the first emitted token
    follows p_root, and the final node of the accepted path follows the
    exact enumeration law (chi-square)."""
    parent = np.array(TOPOLOGIES[name])
    N, V, n = len(parent), 6, 60000
    zp, zq = _tree_rows(V, N, 41)
    T = 1.0
    zp32, zq32 = zp.astype(np.float32), zq.astype(np.float32)
    p = [orc.softmax(zp32[u].astype(np.float64), T) for u in range(N)]
    q = [orc.softmax(zq32[u].astype(np.float64), T) for u in range(N)]
    tgt = np.ascontiguousarray(np.broadcast_to(zp32, (n, N, V)))
    dft = np.ascontiguousarray(np.broadcast_to(zq32, (n, N, V)))
    seeds = np.arange(n, dtype=np.uint64) * 13 + 7
    tok = orc.tree_draft(dft, parent, seeds, 2, T, nthreads=8)
    r = orc.tree_verify(tgt, dft, parent, tok, seeds, 2, T, nthreads=8)
    first = np.where(r["accept_len"] > 0, tok[np.arange(n), np.maximum(r["path"][:, 0], 0)],
                     r["bonus"])
    obs = np.bincount(first, minlength=V)
    assert stats.chisquare(obs, p[0] * n).pvalue > 1e-4
    final = np.array([r["path"][b, r["accept_len"][b] - 1] if r["accept_len"][b] > 0 else 0
                      for b in range(n)])
    expect = _exact_path_law(orc, p, q, list(parent))
    obs = np.bincount(final, minlength=N)
    m = expect * n > 5
    assert stats.chisquare(obs[m], expect[m] / expect[m].sum() * obs[m].sum()).pvalue > 1e-4
    # the token emitted after a node reached at depth >= 1 follows that node's p
    for u in range(1, N):
        sel = np.nonzero(final == u)[0]
        if len(sel) < 2000 or children(list(parent), u):
            continue
        obs = np.bincount(r["bonus"][sel], minlength=V)
        assert stats.chisquare(obs, p[u] * len(sel)).pvalue > 1e-4


def test_tree_draft_follows_parent_distribution(orc):
    """Tree drafting: node v's token is drawn from q_{parent(v)}."""
    parent = np.array(TOPOLOGIES["two-by-two"])
    N, V, n = len(parent), 7, 40000
    _, zq = _tree_rows(V, N, 77)
    zq32 = zq.astype(np.float32)
    dft = np.ascontiguousarray(np.broadcast_to(zq32, (n, N, V)))
    seeds = np.arange(n, dtype=np.uint64) + 3
    tok = orc.tree_draft(dft, parent, seeds, 1, 0.8, nthreads=8)
    assert np.all(tok[:, 0] == -1)
    for v in range(1, N):
        qv = orc.softmax(zq32[parent[v]].astype(np.float64), 0.8)
        assert stats.chisquare(np.bincount(tok[:, v], minlength=V), qv * n).pvalue > 1e-4


def test_tree_rejects_bad_topology_and_tokens(orc):
    zp, zq = _tree_rows(4, 3, 1)
    t, d = zp[None].astype(np.float32), zq[None].astype(np.float32)
    with pytest.raises(ValueError):
        orc.tree_verify(t, d, [-1, 1, 0], np.zeros((1, 3)), np.ones(1, np.uint64), 0, 1.0)
    with pytest.raises(ValueError):
        orc.tree_verify(t, d, [-1, 0, 0], np.array([[0, 1, 9]]), np.ones(1, np.uint64), 0, 1.0)
