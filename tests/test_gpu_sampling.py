"""GPU parity of ssd_topf_bonus, ssd_saguaro_sample and the outcome cache
against the CPU oracle, through the C ABI.

Sources (page title, section): [SSD-note] "论文阅读：Speculative Speculative Decoding —
消除推测解码的最后一个顺序瓶颈" §"怎么猜奖励 token", §"Saguaro 优化二：Saguaro 采样",
§"实现细节：缓存怎么建", §"SSD 的核心思想", §"Saguaro 优化三：自适应回退策略".
"""

import numpy as np
import pytest
from scipy import stats

import sampling_ssd_verify_gb300 as ssd
from ssd_inputs import WORKLOADS, bf16_bits, make_batch
from tests.parity import PROB_TOL, TIE, compare_draws, i32, seeds_t, to_np, torch_dev, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    ssd.build()
    ssd.lib()


# ----------------------------------------------------------------------------- top-F
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_topf_bonus_matches_full_sort(orc, dtype):
    """Guesses = top-(F_j+1) by raw logit minus x_j (ties to the lower
    index), q_j of each guess; c3-sized draft rows."""
    w = WORKLOADS["c3"]
    bt = make_batch(w, B=16, dtype=dtype)
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, 1.0, w.T, bt["seeds"], K=w.K, nthreads=16)
    g = to_np(ssd.topf_bonus(upload(bt["draft"], dtype), F, w.T, draft_tokens=i32(tok)))
    o = orc.topf_bonus(bt["draft"], F, w.T, tokens=tok, K=w.K, nthreads=16)
    np.testing.assert_array_equal(g["guesses"], o["guesses"])
    assert np.abs(g["guess_q"] - o["guess_q"]).max() < PROB_TOL


def test_topf_ties_break_to_lower_index(orc):
    """Integer-valued logits make thousands of exact ties; the guesses must
    follow (logit desc, index asc) even when a row is split across CTAs."""
    rng = np.random.default_rng(41)
    B, Kq, V = 3, 6, 50000
    z = rng.integers(-20, 4, (B, Kq, V)).astype(np.float32)
    F = np.array([15, 9, 5, 3, 1, 0], dtype=np.int32)
    for dtype in ("f32", "bf16"):
        arr = z if dtype == "f32" else bf16_bits(z)
        g = to_np(ssd.topf_bonus(upload(arr, dtype), F, 1.0, guess_q=False))
        o = orc.topf_bonus(arr, F, 1.0)
        np.testing.assert_array_equal(g["guesses"], o["guesses"])


def test_topf_without_exclusion_and_small_vocab(orc):
    rng = np.random.default_rng(42)
    for V, F in ((2, (1, 0, 1)), (5, (4, 2, 3)), (37, (7, 0, 15))):
        z = rng.normal(0, 2, (40, 3, V)).astype(np.float32)
        F = np.asarray(F, dtype=np.int32)
        g = to_np(ssd.topf_bonus(upload(z, "f32"), F, 0.8))
        o = orc.topf_bonus(z, F, 0.8)
        np.testing.assert_array_equal(g["guesses"], o["guesses"])
        assert np.abs(g["guess_q"] - o["guess_q"]).max() < PROB_TOL


# ----------------------------------------------------------------------------- Saguaro
def _branch_rows(w, R, V=None, dtype=None, seed=0):
    """R fresh G-generator rows (the continuation logits of R branches)."""
    bt = make_batch(w, B=R, V=V, K=0, seed=w.seed + 100 + seed, dtype=dtype)
    return np.ascontiguousarray(bt["target"][:, 0, :]), bt["seeds"]


def _check_saguaro(orc, rows, dtype, T, C, F, seeds, j, rnd):
    g = to_np(ssd.saguaro_sample(upload(rows, dtype), T, C, F, seeds_t(seeds), j, rnd))
    o = orc.saguaro_sample(rows, T, C, F, seeds, j, rnd, nthreads=16)
    ok = compare_draws(g["token"], o, V=rows.shape[-1])
    assert np.abs(g["qprime"][ok] - o["qprime"][ok]).max(initial=0) < PROB_TOL
    if np.max(F) > 0:
        np.testing.assert_array_equal(g["guesses"][ok], o["guesses"][ok])
    return g


def test_saguaro_sample_ssd_cache_build_rows(orc):
    """The SSD cache build: 32 outer rows x 12 branches = 384 branch rows,
    V = 151936 bf16, C = 0.3, F_j of the geometric fan-out, 4 continuation
    positions."""
    w = WORKLOADS["c4"]
    R = w.B * w.branches
    for j in range(w.cont_positions):
        rows, seeds = _branch_rows(w, R, seed=j)
        _check_saguaro(orc, rows, "bf16", w.T, w.C, int(w.fanout[j]), seeds, j, 11)


def test_saguaro_sample_per_row_fanout(orc):
    """Branch rows that continue different outcome positions take that
    position's fan-out ([SSD-note] §"最优扇出度分配"): 384 rows of the SSD
    cache build with F_row mixed over 0..3 in one call, against the oracle;
    a device F_row tensor gives the same results, and a value above Fmax is
    clamped and reported."""
    torch, dev = torch_dev()
    w = WORKLOADS["c4"]
    R = w.B * w.branches
    rows, seeds = _branch_rows(w, R, seed=5)
    F = np.asarray([w.fanout[r % (w.K + 1)] for r in range(R)], dtype=np.int32)
    F[::7] = 0
    for rnd in (0, 3):
        g = _check_saguaro(orc, rows, "bf16", w.T, w.C, F, seeds, 1, rnd)
    Fd = torch.from_numpy(F).to(dev)
    g2 = to_np(ssd.saguaro_sample(upload(rows, "bf16"), w.T, w.C, Fd, seeds_t(seeds), 1, 3,
                                  Fmax=int(F.max())))
    for k in ("token", "qprime", "guesses"):
        np.testing.assert_array_equal(g2[k], g[k])
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    bad = Fd.clone()
    bad[0] = 9
    ssd.saguaro_sample(upload(rows, "bf16"), w.T, w.C, bad, seeds_t(seeds), 1, 3,
                       Fmax=int(F.max()), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & ssd.DEV_BAD_FANOUT


@pytest.mark.parametrize("V,dtype,C,F,T", [(32, "f32", 0.5, 3, 1.0), (37, "bf16", 0.05, 7, 0.6),
                                           (2, "f32", 0.3, 1, 1.0), (4099, "bf16", 1.0, 5, 1.3),
                                           (50000, "f32", 0.2, 15, 1.0), (1000, "bf16", 0.7, 0, 1)])
def test_saguaro_sample_edges(orc, V, dtype, C, F, T):
    w = WORKLOADS["c2"]
    rows, seeds = _branch_rows(w, 300, V=V, dtype=dtype, seed=V)
    for rnd in (0, 1):
        _check_saguaro(orc, rows, dtype, T, C, F, seeds, 2, rnd)


def test_saguaro_draw_follows_q_prime(orc):
    """x ~ q' (cached tokens' probability times C, renormalised): chi-square
    over 4*10^5 draws of one V = 32 row."""
    rng = np.random.default_rng(43)
    z = rng.normal(0, 1.5, 32).astype(np.float32)
    C, F, T = 0.3, 4, 1.0
    n = 400_000
    rows = np.ascontiguousarray(np.broadcast_to(z, (n, 32)))
    seeds = np.arange(n, dtype=np.uint64) * 3 + 1
    g = to_np(ssd.saguaro_sample(upload(rows, "f32"), T, C, F, seeds_t(seeds), 0, 0,
                                 guesses=False))
    qp = orc.saguaro_dist(z, T, F, C)
    obs = np.bincount(g["token"], minlength=32)
    m = qp * n > 5
    assert stats.chisquare(obs[m], qp[m] / qp[m].sum() * obs[m].sum()).pvalue > 1e-4


# ----------------------------------------------------------------------------- cache
def test_cache_build_and_lookup_match_oracle(orc):
    torch, dev = torch_dev()
    rng = np.random.default_rng(44)
    B, K, V = 256, 8, 151936
    keys = {}
    while len(keys) < 6144:
        keys[(int(rng.integers(B)), int(rng.integers(K + 1)), int(rng.integers(V)))] = len(keys)
    row, k, t = (np.array(c, dtype=np.int32) for c in zip(*keys.keys()))
    branch = np.array(list(keys.values()), dtype=np.int32)
    acc = rng.integers(0, K + 1, B).astype(np.int32)
    bon = rng.integers(0, V, B).astype(np.int32)
    for kk in list(keys)[:3000]:
        acc[kk[0]], bon[kk[0]] = kk[1], kk[2]
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tab = ssd.cache_build(i32(row), i32(k), i32(t), i32(branch), dev_status=status)
    lk = ssd.cache_lookup(tab, i32(acc), i32(bon))
    eb, eall = orc.cache_lookup(row, k, t, branch, acc, bon)
    np.testing.assert_array_equal(lk["branch"].cpu().numpy(), eb)
    assert int(lk["all_hit"].item()) == eall
    assert int(status.item()) == 0
    # all rows hit
    for b in range(B):
        cand = [kk for kk in keys if kk[0] == b]
        if cand:
            acc[b], bon[b] = cand[0][1], cand[0][2]
    lk = ssd.cache_lookup(tab, i32(acc), i32(bon))
    eb, eall = orc.cache_lookup(row, k, t, branch, acc, bon)
    np.testing.assert_array_equal(lk["branch"].cpu().numpy(), eb)
    assert int(lk["all_hit"].item()) == eall


def test_cache_duplicate_keys_are_reported():
    torch, dev = torch_dev()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    row = i32(np.array([0, 1, 0], np.int32))
    k = i32(np.array([2, 2, 2], np.int32))
    t = i32(np.array([5, 5, 5], np.int32))
    br = i32(np.array([10, 11, 12], np.int32))
    tab = ssd.cache_build(row, k, t, br, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & ssd.DEV_DUPLICATE_KEY
    lk = ssd.cache_lookup(tab, i32(np.array([2, 2], np.int32)), i32(np.array([5, 5], np.int32)))
    b = lk["branch"].cpu().numpy()
    assert b[0] in (10, 12) and b[1] == 11


def test_cache_from_verify_guesses_round(orc):
    """A full SSD verification round (c4 outer rows): verify with fused
    guesses, cache built from those guesses, lookup of the outcomes -- all
    against the oracle's round."""
    torch, dev = torch_dev()
    w = WORKLOADS["c4"]
    bt = make_batch(w)
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], round_=2, K=w.K, nthreads=16)
    out = ssd.verify(upload(bt["target"], "bf16"), upload(bt["draft"], "bf16"), i32(tok),
                     seeds_t(bt["seeds"]), 2, F, w.C, w.T)
    tab = ssd.cache_build_guesses(out["guesses"])
    lk = ssd.cache_lookup(tab, out["accept_len"], out["bonus"])
    o = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 2, F, w.C, w.T, nthreads=16)
    tie = (o["margin_accept"] < TIE) | (o["margin_cdf"] < TIE)
    g = o["guesses"]
    Fm = g.shape[2]
    keys = [(b, k, int(g[b, k, f]), (b * w.Kq + k) * Fm + f) for b in range(w.B)
            for k in range(w.Kq) for f in range(Fm) if g[b, k, f] >= 0]
    r_, k_, t_, br_ = (np.array(c) for c in zip(*keys))
    eb, eall = orc.cache_lookup(r_, k_, t_, br_, o["accept_len"], o["bonus"])
    gb = lk["branch"].cpu().numpy()
    np.testing.assert_array_equal(gb[~tie], eb[~tie])
    if not tie.any():
        assert int(lk["all_hit"].item()) == eall
