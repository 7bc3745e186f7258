"""GPU parity of ssd_verify against the CPU oracle, through the C ABI.

Sources (page title, section): [SD-7.3] "7.3 Speculative Decoding：投机采样加速"
§7.3.2-7.3.3; [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个
顺序瓶颈" §"Saguaro 优化二：Saguaro 采样", §"怎么猜奖励 token".
"""

import dataclasses

import numpy as np
import pytest
from scipy import stats

import sampling_ssd_verify_gb300 as ssd
from ssd_inputs import WORKLOADS, make_batch
from tests.parity import compare_draws, compare_verify, i32, seeds_t, to_np, torch_dev, upload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    ssd.build()
    ssd.lib()


def _padded(arr, dtype, pad):
    """Upload [B, R, V] with `pad` extra elements per row (row stride V+pad)."""
    torch, dev = torch_dev()
    if pad == 0:
        return upload(arr, dtype)
    B, R, V = arr.shape
    big = np.zeros((B, R, V + pad), dtype=arr.dtype)
    big[:, :, :V] = arr
    return upload(big, dtype)[:, :, :V]


def run_verify(orc, w, B=None, V=None, K=None, dtype=None, rounds=(0,), seed=None, C=None,
               T=None, F=None, Kq=None, pad=0, offset=0, nthreads=16, batch=None):
    torch, dev = torch_dev()
    bt = batch if batch is not None else make_batch(w, B=B, V=V, K=K, seed=seed, dtype=dtype)
    K = bt["K"]
    dtype = bt["dtype"]
    C = w.C if C is None else C
    T = w.T if T is None else T
    Kq = K + 1 if Kq is None else Kq
    F = np.asarray(w.fanout if F is None else F, dtype=np.int32)[:Kq]
    target = bt["target"]
    draft = np.ascontiguousarray(bt["draft"][:, :Kq])
    seeds = bt["seeds"]
    if offset:
        # shift the whole batch by `offset` elements inside a larger buffer
        flat_t = np.concatenate([np.zeros(offset, target.dtype), target.ravel()])
        flat_d = np.concatenate([np.zeros(offset, draft.dtype), draft.ravel()])
        tg = upload(flat_t, dtype)[offset:].view(target.shape)
        dg = upload(flat_d, dtype)[offset:].view(draft.shape)
    else:
        tg = _padded(target, dtype, pad)
        dg = _padded(draft, dtype, pad)
    stats_all = []
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for r in rounds:
        tok = orc.draft_tokens(draft, F, C, T, seeds, round_=r, K=K, nthreads=nthreads)
        g = ssd.verify(tg, dg, i32(tok), seeds_t(seeds), r, F, C, T, dev_status=status)
        torch.cuda.synchronize()
        o = orc.verify(target, draft, tok, seeds, r, F, C, T, Fmax=max(1, int(F.max())),
                       nthreads=nthreads)
        stats_all.append(compare_verify(to_np(g), o, K, V=target.shape[-1]))
    assert int(status.item()) == 0
    return stats_all


@pytest.mark.parametrize("T", [1.0, 0.0], ids=["sampled", "greedy"])
def test_max_K_many_rows_with_rows_skipped(orc, T):
    """K = 32 (the largest) over 600 sequences of small rows: with this many
    rows every position streams after earlier positions are decided, so
    target rows past a rejection are dropped at every position up to 32."""
    w = dataclasses.replace(WORKLOADS["c1"], K=32)
    st = run_verify(orc, w, B=600, V=256, K=32, F=[2] * 33, C=0.5, T=T, rounds=(0, 1))
    assert sum(s["rows"] for s in st) == 1200


def test_c1_tiny_exactness_many_rows(orc):
    """B=1,K=4,V=32 fp32 (C=0.5, F=[3,3,2,2,2]) drawn for 20000 independent
    sequences x 5 rounds."""
    w = WORKLOADS["c1"]
    st = run_verify(orc, w, B=20000, rounds=range(5))
    assert sum(s["rows"] for s in st) == 100000


def test_c2_single_stream_llama_vocab(orc):
    """B=1, K=4, V=128256 bf16, T=0.7, C=0.5: 24 seeded rounds."""
    w = WORKLOADS["c2"]
    run_verify(orc, w, rounds=range(24))


def test_c3_batched_full_size(orc):
    """B=64, K=8, V=128256 bf16, C=1, budget 16: every row against the oracle."""
    w = WORKLOADS["c3"]
    st = run_verify(orc, w, rounds=(0, 1))
    for s in st:
        assert 0.5 < s["accept_mean"] < 8


def test_c4_outer_verify(orc):
    """The SSD round's verify of 32 outer rows: K=4, V=151936 bf16, C=0.3,
    over four rounds."""
    w = WORKLOADS["c4"]
    run_verify(orc, w, rounds=(0, 1, 2, 3))


def test_c5_full_round_all_rows(orc):
    """The benchmarked call at the benchmarked size: ssd_verify_round on the
    whole large-batch workload (B=256, K=8, V=151936 fp32, C=0.5, budget 24)
    against the oracle on every row -- accept lengths, bonus tokens,
    guesses, each sequence's outcome-cache branch and all-rows-hit."""
    torch, dev = torch_dev()
    w = WORKLOADS["c5"]
    bt = make_batch(w)
    K = w.K
    F = np.asarray(w.fanout, dtype=np.int32)
    tg, dg = upload(bt["target"], "f32"), upload(bt["draft"], "f32")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for rnd in (1000, 1001):
        tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], round_=rnd, K=K,
                               nthreads=16)
        r = ssd.verify_round(tg, dg, i32(tok), seeds_t(bt["seeds"]), rnd, F, w.C, w.T,
                             dev_status=status)
        g = {k: v.cpu().numpy() for k, v in r.items() if k != "table"}
        o = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], rnd, F, w.C, w.T,
                       nthreads=16)
        st = compare_verify({k: g[k] for k in ("accept_len", "bonus", "resid_mass", "guesses",
                                               "guess_q")}, o, K, V=w.V)
        assert st["rows"] == w.B
        gg = o["guesses"]
        b, k, f = np.nonzero(gg >= 0)
        branch = (b * gg.shape[1] + k) * gg.shape[2] + f
        eb, eall = orc.cache_lookup(b, k, gg[b, k, f], branch, o["accept_len"], o["bonus"])
        same = (g["accept_len"] == o["accept_len"]) & (g["bonus"] == o["bonus"])
        np.testing.assert_array_equal(g["branch"][same], eb[same])
        if same.all():
            assert int(g["all_hit"][0]) == eall
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_c5_large_batch_sampled_rows(orc):
    """B=256, K=8, V=151936 fp32, C=0.5, budget 24 at full size, in the launch
    configuration the benchmark times; the oracle checks a sample of rows."""
    torch, dev = torch_dev()
    w = WORKLOADS["c5"]
    bt = make_batch(w)
    K, Kq = w.K, w.Kq
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], round_=5, K=K, nthreads=16)
    tg = upload(bt["target"], "f32")
    dg = upload(bt["draft"], "f32")
    g = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 5, F, w.C, w.T))
    rows = np.array([0, 1, 17, 63, 64, 100, 127, 128, 200, 254, 255])
    o = orc.verify(bt["target"][rows], bt["draft"][rows], tok[rows], bt["seeds"][rows], 5, F,
                   w.C, w.T, nthreads=16, row_ids=rows)
    compare_verify({kk: v[rows] for kk, v in g.items()}, o, K, V=w.V)
    # properties every row must satisfy
    assert np.all((g["accept_len"] >= 0) & (g["accept_len"] <= K))
    assert np.all((g["bonus"] >= 0) & (g["bonus"] < w.V))
    rej = g["accept_len"] < K
    assert np.all(g["bonus"][rej] != tok[rej, g["accept_len"][rej]])
    assert np.all((g["resid_mass"] > 0) & (g["resid_mass"] <= 1 + 1e-5))


@dataclasses.dataclass
class Edge:
    name: str
    B: int
    K: int
    V: int
    dtype: str
    F: tuple
    C: float = 0.5
    T: float = 1.0
    Kq: int | None = None
    pad: int = 0
    offset: int = 0


EDGES = [
    Edge("V37 unaligned rows f32", 50, 3, 37, "f32", (2, 2, 1, 1)),
    Edge("V37 unaligned rows bf16", 50, 3, 37, "bf16", (2, 2, 1, 1)),
    Edge("V2 minimum vocab", 200, 1, 2, "f32", (1, 0), C=0.3),
    Edge("K1 no fan-out", 100, 1, 300, "bf16", (0, 0), C=0.4),
    Edge("K32 maximum drafts", 4, 32, 515, "f32", tuple([1] * 33)),
    Edge("Kq=K no draft row K", 40, 4, 1000, "bf16", (3, 2, 2, 1), Kq=4),
    Edge("padded row stride f32", 20, 4, 3001, "f32", (3, 3, 2, 2, 2), pad=5),
    Edge("padded row stride bf16", 20, 4, 3001, "bf16", (3, 3, 2, 2, 2), pad=3),
    Edge("odd element offset bf16", 8, 4, 4099, "bf16", (3, 3, 2, 2, 2), offset=1),
    Edge("rows split over many CTAs", 3, 7, 20000, "f32", (5, 4, 3, 3, 2, 2, 1, 1)),
    Edge("F up to 15", 6, 2, 700, "bf16", (15, 9, 4), C=0.2),
    Edge("high temperature", 30, 4, 2048, "f32", (3, 3, 2, 2, 2), T=2.5),
    Edge("low temperature", 30, 4, 2048, "bf16", (3, 3, 2, 2, 2), T=0.3),
    # more than 512 draw units per row: the bonus draw sums and searches its
    # unit sums in several rounds
    Edge("V300000 multi-round draw f32", 6, 3, 300000, "f32", (3, 2, 2, 1)),
    Edge("V300000 multi-round draw bf16", 6, 3, 300000, "bf16", (3, 2, 2, 1), C=1.0),
]


@pytest.mark.parametrize("e", EDGES, ids=[e.name for e in EDGES])
def test_edge_shapes(orc, e):
    w = dataclasses.replace(WORKLOADS["c2"], gen="G" if e.V > 64 else "gauss", T=e.T,
                            fanout=e.F, C=e.C, seed=77)
    run_verify(orc, w, B=e.B, V=e.V, K=e.K, dtype=e.dtype, rounds=(0, 1), F=e.F, Kq=e.Kq,
               pad=e.pad, offset=e.offset)


def test_plain_sd_is_bit_identical_with_c1_or_empty_sets(orc):
    """C = 1 (any F) and F = 0 (any C) are both plain speculative decoding:
    identical accept lengths, bonus tokens and residual masses."""
    torch, dev = torch_dev()
    w = WORKLOADS["c3"]
    bt = make_batch(w, B=16, V=20000)
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], np.zeros_like(F), 1.0, w.T, bt["seeds"], K=w.K)
    tg, dg = upload(bt["target"], "bf16"), upload(bt["draft"], "bf16")
    a = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 0, F, 1.0, w.T))
    b = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 0, np.zeros_like(F), 0.4, w.T,
                         guesses=False))
    for k in ("accept_len", "bonus", "resid_mass"):
        np.testing.assert_array_equal(a[k], b[k])


@pytest.mark.parametrize("name,B,V,dtype,Cv", [
    ("c1", 4000, 32, "f32", (0.3, 0.5, 0.8, 1.0)),
    ("c5", 24, 151936, "f32", (0.2, 0.3, 0.5, 0.5, 0.7, 0.9, 1.0, 1.0)),
    ("c3", 12, 128256, "bf16", (0.3, 1.0, 0.5, 1.0, 0.7, 0.2, 1.0, 0.4)),
], ids=["c1-shape", "c5-shape", "c3-shape"])
def test_per_position_C(orc, name, B, V, dtype, Cv):
    """ssd_verify_ck: one Saguaro factor per draft position ([SSD-note]
    §"关于逐位置 C 的思考"), drafts drawn with the same factors, against the
    oracle row by row."""
    run_verify(orc, WORKLOADS[name], B=B, V=V, dtype=dtype, C=np.array(Cv), rounds=(0, 1))


def test_per_position_C_equal_entries_match_scalar(orc):
    """Every per-position factor equal to C gives ssd_verify's outputs with C,
    bit for bit (guesses, their probabilities and residual masses included)."""
    torch, dev = torch_dev()
    w = WORKLOADS["c5"]
    bt = make_batch(w, B=16, V=30000)
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=w.K)
    tg, dg = upload(bt["target"], "f32"), upload(bt["draft"], "f32")
    a = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 2, F, w.C, w.T))
    b = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 2, F, np.full(w.K, w.C), w.T))
    for k in a:
        np.testing.assert_array_equal(a[k], b[k])


def _as_f32(a):
    """Logit array as float32 (bf16 arrays hold the raw 16-bit patterns)."""
    return (a.astype(np.uint32) << 16).view(np.float32) if a.dtype == np.uint16 else a


@pytest.mark.parametrize("name,B,V,dtype", [("c3", 16, 128256, "bf16"),
                                            ("c5", 12, 151936, "f32"),
                                            ("c1", 500, 32, "f32")])
def test_greedy_verify(orc, name, B, V, dtype):
    """T = 0, the greedy limit: a draft is accepted iff it is the target
    row's argmax (ties to the lower index) and the bonus is the argmax of the
    first rejected target row.  Greedy drafts (the draft rows' argmax) and
    sampled drafts, against the oracle, every output exact."""
    torch, dev = torch_dev()
    w = WORKLOADS[name]
    bt = make_batch(w, B=B, V=V, dtype=dtype)
    K = w.K
    F = np.asarray(w.fanout, dtype=np.int32)
    tg, dg = upload(bt["target"], dtype), upload(bt["draft"], dtype)
    greedy_tok = _as_f32(bt["draft"])[:, :K].argmax(-1).astype(np.int32)
    sampled_tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=K, nthreads=16)
    for tok in (greedy_tok, sampled_tok):
        g = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 0, F, w.C, 0.0))
        o = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 0, F, w.C, 0.0,
                       Fmax=max(1, int(F.max())), nthreads=16)
        for k in ("accept_len", "bonus", "guesses", "guess_q"):
            np.testing.assert_array_equal(g[k], o[k].astype(g[k].dtype), err_msg=k)
        np.testing.assert_array_equal(g["resid_mass"], 1.0)
    assert 0 < g["accept_len"].mean() <= K


def test_per_sequence_temperature(orc):
    """ssd_verify_ex: one temperature per sequence, greedy ones among them,
    against the oracle; a negative temperature is verified greedily and
    reported."""
    torch, dev = torch_dev()
    w = WORKLOADS["c5"]
    B, V = 16, 40000
    bt = make_batch(w, B=B, V=V)
    F = np.asarray(w.fanout, dtype=np.int32)
    Ts = np.array([1.0, 0.0, 0.7, 1.3, 0.0, 0.5, 1.0, 2.0] * 2, dtype=np.float32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, 1.0, bt["seeds"], K=w.K, nthreads=16)
    tg, dg = upload(bt["target"], "f32"), upload(bt["draft"], "f32")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for rnd in (0, 1):
        g = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), rnd, F, w.C,
                             torch.from_numpy(Ts).to(dev), dev_status=status))
        o = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], rnd, F, w.C,
                       Ts.astype(np.float64), Fmax=max(1, int(F.max())), nthreads=16)
        compare_verify(g, o, w.K, V=V)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    bad = Ts.copy()
    bad[3] = -1.0
    g = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 0, F, w.C,
                         torch.from_numpy(bad).to(dev), dev_status=status))
    torch.cuda.synchronize()
    assert int(status.item()) & ssd.DEV_BAD_TEMPERATURE
    bad[3] = 0.0
    o = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 0, F, w.C,
                   bad.astype(np.float64), Fmax=max(1, int(F.max())), nthreads=16)
    compare_verify(g, o, w.K, V=V)


def test_fanout_ablation_round_matches_oracle(orc):
    """One round of the fan-out ablation harness (library calls: Saguaro
    drafts, verify with guesses, cache build and lookup) against the oracle
    composed the same way, for the geometric and the uniform allocation."""
    from sampling_ssd_verify_gb300.ablation import round_hits, uniform_fanout

    w = dataclasses.replace(WORKLOADS["c5"], B=64, V=8192)
    for F in (ssd.fanout(w.K, 24), uniform_fanout(w.K, 24)):
        res = round_hits(w, F, 0.5, 1.0, seed=7, rnd=1)
        bt = res["batch"]
        # the library's drafts against the oracle's Saguaro draws, position by
        # position, with the near-tie rule
        for j in range(w.K):
            oj = orc.saguaro_sample(np.ascontiguousarray(bt["draft"][:, j, :]), 1.0, 0.5,
                                    int(F[j]), bt["seeds"], j, 1, nthreads=16)
            compare_draws(res["tokens"][:, j], oj, V=w.V)
        o = orc.verify(bt["target"], bt["draft"], res["tokens"], bt["seeds"], 1, F, 0.5, 1.0,
                       nthreads=16)
        compare_verify({"accept_len": res["accept_len"], "bonus": res["bonus"],
                        "guesses": res["guesses"]}, o, w.K, V=w.V)
        same = (o["accept_len"] == res["accept_len"]) & (o["bonus"] == res["bonus"])
        hit_o = np.array([o["bonus"][b] in o["guesses"][b, o["accept_len"][b]]
                          for b in range(w.B)])
        np.testing.assert_array_equal(res["hit"][same], hit_o[same])


@pytest.mark.parametrize("name,B,V,dtype,T", [("c5", 32, 151936, "f32", None),
                                              ("c3", 16, 128256, "bf16", None),
                                              ("c1", 64, 32, "f32", None),
                                              ("c1", 1, 32, "f32", None),
                                              ("c4", 32, 151936, "bf16", 0.0)],
                         ids=["c5-shape", "c3-shape", "c1-shape", "c1-one-row", "c4-greedy"])
def test_verify_round_equals_separate_calls(orc, name, B, V, dtype, T):
    """ssd_verify_round (verify, the round's outcome cache and its lookup in
    one launch) gives the outputs of ssd_verify, ssd_cache_build_guesses and
    ssd_cache_lookup called in sequence, bit for bit, over consecutive rounds
    on the same table (a round never sees the previous round's keys)."""
    torch, dev = torch_dev()
    w = WORKLOADS[name]
    T = w.T if T is None else T
    bt = make_batch(w, B=B, V=V, dtype=dtype)
    F = np.asarray(w.fanout, dtype=np.int32)
    tg, dg = upload(bt["target"], dtype), upload(bt["draft"], dtype)
    seeds = seeds_t(bt["seeds"])
    table = None
    hits = 0
    for rnd in range(3):
        tok = i32(orc.draft_tokens(bt["draft"], F, w.C, max(T, 0.5), bt["seeds"], round_=rnd,
                                   K=w.K))
        a = ssd.verify(tg, dg, tok, seeds, rnd, F, w.C, T)
        look = ssd.cache_lookup(ssd.cache_build_guesses(a["guesses"]), a["accept_len"],
                                a["bonus"])
        r = ssd.verify_round(tg, dg, tok, seeds, rnd, F, w.C, T, table=table)
        table = r["table"]
        torch.cuda.synchronize()
        for k in a:
            np.testing.assert_array_equal(r[k].cpu().numpy(), a[k].cpu().numpy(), err_msg=k)
        np.testing.assert_array_equal(r["branch"].cpu().numpy(), look["branch"].cpu().numpy())
        assert int(r["all_hit"].item()) == int(look["all_hit"].item())
        # the table holds the round's guesses in the cache format
        again = ssd.cache_lookup(table, r["accept_len"], r["bonus"])
        np.testing.assert_array_equal(again["branch"].cpu().numpy(), look["branch"].cpu().numpy())
        hits += int((r["branch"] >= 0).sum().item())
    assert hits > 0


def test_bad_token_sets_status(orc):
    torch, dev = torch_dev()
    w = WORKLOADS["c1"]
    bt = make_batch(w, B=4)
    tok = np.zeros((4, w.K), dtype=np.int32)
    tok[2, 1] = w.V + 5
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    ssd.verify(upload(bt["target"], "f32"), upload(bt["draft"], "f32"), i32(tok),
               seeds_t(bt["seeds"]), 0, w.fanout, w.C, w.T, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & ssd.DEV_BAD_TOKEN


def test_gpu_laws_chi_square(orc):
    """The library's own outputs follow the exact laws: accept length
    P(k >= j) = prod alpha_i and bonus ~ normalize((p_i - q'_i)^+) (or p_K),
    over 10^6 seeded trials at V = 32."""
    torch, dev = torch_dev()
    rng = np.random.default_rng(31)
    K, V, C, T = 2, 32, 0.5, 1.0
    zp = rng.normal(0, 1.0, (K + 1, V)).astype(np.float32)
    zq = (zp + rng.normal(0, 0.7, (K + 1, V))).astype(np.float32)
    F = np.array([3, 2, 2], dtype=np.int32)
    p = [orc.softmax(zp[i], T) for i in range(K + 1)]
    qp = [orc.saguaro_dist(zq[j], T, int(F[j]), C) for j in range(K)]
    n = 250_000
    tgt = np.ascontiguousarray(np.broadcast_to(zp, (n, K + 1, V)))
    dft = np.ascontiguousarray(np.broadcast_to(zq, (n, K + 1, V)))
    seeds = np.arange(n, dtype=np.uint64) * 7 + 5
    tg, dg = upload(tgt, "f32"), upload(dft, "f32")
    ks, ts = [], []
    for r in range(4):
        tok = orc.draft_tokens(dft, F, C, T, seeds, round_=r, K=K, nthreads=16)
        g = to_np(ssd.verify(tg, dg, i32(tok), seeds_t(seeds), r, F, C, T, guesses=False))
        ks.append(g["accept_len"])
        ts.append(g["bonus"])
    ks, ts = np.concatenate(ks), np.concatenate(ts)
    alpha = [np.minimum(p[i], qp[i]).sum() for i in range(K)]
    ge = np.cumprod([1.0] + alpha)
    pk = np.append(ge[:-1] - ge[1:], ge[K])
    assert stats.chisquare(np.bincount(ks, minlength=K + 1), pk * len(ks)).pvalue > 1e-4
    for i in range(K + 1):
        sel = ts[ks == i]
        if i < K:
            wr, Z = orc.residual(p[i], qp[i])
            expect = wr / Z
        else:
            expect = p[K]
        obs = np.bincount(sel, minlength=V)
        m = expect * len(sel) > 5
        st = stats.chisquare(obs[m], expect[m] / expect[m].sum() * obs[m].sum())
        assert st.pvalue > 1e-4, (i, st)


def test_target_rows_past_a_rejection_are_not_read(orc):
    """The bytes of target rows the round did not read: a multiple of the
    element size, at most the target rows past position 0 of every rejected
    sequence (rows past its first rejection), and some at the c5 shape, where
    most sequences stop early; the outputs equal the oracle (every test of
    this file runs with rows skipped)."""
    torch, dev = torch_dev()
    w = WORKLOADS["c5"]
    B = 64
    bt = make_batch(w, B=B, seed=21)
    tg, dg = upload(bt["target"], "f32"), upload(bt["draft"], "f32")
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=w.K, nthreads=16)
    ws = torch.zeros(ssd.lib().ssd_verify_workspace_size(B, w.K, w.Kq, w.V), dtype=torch.uint8,
                     device=dev)
    out = {}
    total = 0
    for rnd in range(4):
        g = ssd.verify_round(tg, dg, i32(tok), seeds_t(bt["seeds"]), rnd, F, w.C, w.T,
                             workspace=ws, out=out)
        sk = ssd.verify_skipped_bytes(ws, tg, w.K, w.Kq)
        al = g["accept_len"].cpu().numpy()
        bound = int(np.where(al < w.K, w.K - al, 0).sum()) * w.V * 4
        assert sk % 4 == 0 and 0 <= sk <= bound, (sk, bound)
        total += sk
        o = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], rnd, F, w.C, w.T, nthreads=16)
        compare_verify(to_np({k: g[k] for k in ("accept_len", "bonus", "resid_mass", "guesses")}),
                       o, w.K, V=w.V)
    assert total > 0
