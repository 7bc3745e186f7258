"""Checks against the few values the source pages print (tests/golden)."""

import json
import os

import numpy as np

GOLD = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "page_values.json")))


def test_all_hit_fraction_matches_page(orc):
    """[SSD-note] §Saguaro 优化三: with a per-row hit rate h the all-rows-hit
    probability is h^b; the page's 92%-with-a-miss figure is reproduced by the
    oracle's cache lookup over seeded rounds (each row hits with prob h)."""
    g = GOLD["all_hit_complement"]
    h, b = g["h"], g["b"]
    assert abs((1 - h ** b) - g["value"]) < g["tolerance"]
    rng = np.random.default_rng(11)
    rounds, misses = 20000, 0
    row = np.arange(b)
    kk = np.zeros(b, dtype=np.int32)
    tt = np.full(b, 7, dtype=np.int32)
    branch = np.arange(b, dtype=np.int32)
    for _ in range(rounds):
        hit = rng.random(b) < h
        bonus = np.where(hit, 7, 8).astype(np.int32)
        _, all_hit = orc.cache_lookup(row, kk, tt, branch, np.zeros(b, np.int32), bonus)
        misses += 1 - all_hit
    frac = misses / rounds
    assert abs(frac - g["value"]) < 4 * np.sqrt(g["value"] * (1 - g["value"]) / rounds) + 0.005


def test_low_acceptance_tokens_per_round(orc):
    """[SD-blog] §四 (坑 1): 20-30% acceptance at K=4 gives about one token per
    round; measured with the oracle's verify on logits tuned to that alpha."""
    g = GOLD["low_acceptance_k4"]
    K, V, n = g["K"], 16, 20000
    rng = np.random.default_rng(12)
    zp = rng.normal(0, 3, (K + 1, V)).astype(np.float32)
    zq = (zp + rng.normal(0, 6, (K + 1, V))).astype(np.float32)
    F = np.zeros(K + 1, dtype=np.int32)
    p = [orc.softmax(zp[i], 1.0) for i in range(K)]
    q = [orc.softmax(zq[i], 1.0) for i in range(K)]
    alpha = np.array([np.minimum(p[i], q[i]).sum() for i in range(K)])
    tgt = np.ascontiguousarray(np.broadcast_to(zp, (n, K + 1, V)))
    dft = np.ascontiguousarray(np.broadcast_to(zq, (n, K + 1, V)))
    seeds = np.arange(n, dtype=np.uint64) + 99
    tok = orc.draft_tokens(dft, F, 1.0, 1.0, seeds, K=K)
    r = orc.verify(tgt, dft, tok, seeds, 0, F, 1.0, 1.0, nthreads=8)
    tokens_per_round = r["accept_len"].mean() + 1
    expect = 1 + np.cumprod(alpha).sum()
    assert abs(tokens_per_round - expect) < 0.03
    if g["alpha_range"][0] <= alpha.mean() <= g["alpha_range"][1]:
        lo, hi = g["tokens_per_round_range"]
        assert lo <= tokens_per_round <= hi


def test_all_accepted_emits_k_plus_one(orc):
    """[SD-7.3] §7.3.2: identical target and draft distributions accept every
    draft, so each round emits K drafts plus one bonus from p_K."""
    K, V, n = 4, 32, 500
    rng = np.random.default_rng(13)
    z = rng.normal(0, 2, (K + 1, V)).astype(np.float32)
    tgt = np.ascontiguousarray(np.broadcast_to(z, (n, K + 1, V)))
    F = np.zeros(K + 1, dtype=np.int32)
    seeds = np.arange(n, dtype=np.uint64)
    tok = orc.draft_tokens(tgt, F, 1.0, 1.0, seeds, K=K)
    r = orc.verify(tgt, tgt, tok, seeds, 0, F, 1.0, 1.0)
    assert np.all(r["accept_len"] == K)
