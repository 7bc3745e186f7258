"""GPU parity of ssd_tree_verify (tree-draft verification) against the CPU
oracle, through the C ABI.

[SD-7.3] "7.3 Speculative Decoding：投机采样加速" §7.3.9 item 3 (tree drafts) and
§7.3.3 (the per-token rule applied to each candidate, residual renormalised
after every rejection).
"""

import dataclasses

import numpy as np
import pytest

import sampling_ssd_verify_gb300 as ssd
from ssd_inputs import WORKLOADS, make_batch
from tests.parity import TIE, i32, seeds_t, torch_dev, upload

pytestmark = pytest.mark.gpu

# SpecInfer-like shapes: a wide first level, narrower below
TREES = {
    "chain-4": [-1, 0, 1, 2, 3],
    "binary-depth-3": [-1, 0, 0, 1, 1, 2, 2],
    "wide-3x2": [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3],
    "uneven-11": [-1, 0, 0, 1, 1, 1, 2, 4, 4, 7, 8],
}


@pytest.fixture(scope="module", autouse=True)
def built():
    ssd.build()
    ssd.lib()


def _tree_batch(w, B, N, V, dtype, seed):
    """[B, N, V] target and draft rows from the workload's generator: row u
    of a tree is the generator's position u."""
    bt = make_batch(w, B=B, V=V, K=N - 1, seed=seed, dtype=dtype)
    return bt["target"], np.ascontiguousarray(bt["draft"][:, :N]), bt["seeds"]


def compare_tree(g, o, max_disagree_frac=2e-3):
    tie = (o["margin_accept"] < TIE) | (o["margin_cdf"] < TIE)
    same = (g["accept_len"] == o["accept_len"]) & (g["bonus"] == o["bonus"])
    same &= (g["path"] == o["path"]).all(axis=1)
    bad = ~same & ~tie
    assert not bad.any(), (np.nonzero(bad)[0][:8], g["accept_len"][bad][:5],
                           o["accept_len"][bad][:5], g["bonus"][bad][:5], o["bonus"][bad][:5])
    assert (~same).sum() <= max(2, max_disagree_frac * len(same))
    err = np.abs(g["resid_mass"][same] - o["resid_mass"][same])
    assert err.max(initial=0) < 1e-5, err.max()
    return int(tie.sum())


@pytest.mark.parametrize("tree", sorted(TREES))
@pytest.mark.parametrize("wl,B,V,dtype", [("c3", 24, 128256, "bf16"), ("c5", 16, 151936, "f32"),
                                          ("c1", 400, 32, "f32")],
                         ids=["c3-shape", "c5-shape", "c1-shape"])
def test_tree_verify_matches_oracle(orc, tree, wl, B, V, dtype):
    torch, dev = torch_dev()
    w = WORKLOADS[wl]
    parent = np.array(TREES[tree], dtype=np.int32)
    N = len(parent)
    tgt, dft, seeds = _tree_batch(w, B, N, V, dtype, seed=11)
    tg, dg = upload(tgt, dtype), upload(dft, dtype)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for rnd in (0, 1):
        tok = orc.tree_draft(dft, parent, seeds, rnd, w.T, nthreads=16)
        g = ssd.tree_verify(tg, dg, parent, i32(tok), seeds_t(seeds), rnd, w.T,
                            dev_status=status)
        g = {k: v.cpu().numpy() for k, v in g.items()}
        o = orc.tree_verify(tgt, dft, parent, tok, seeds, rnd, w.T, nthreads=16)
        compare_tree(g, o)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("B,V,dtype", [(70, 4099, "bf16"), (36, 1000, "f32")],
                         ids=["two-CTA-clusters-unaligned-rows", "four-CTA-clusters"])
def test_tree_cluster_sizes(orc, B, V, dtype):
    """Batches that give the walk clusters of 2 and 4 CTAs per tree; V = 4099
    bf16 rows alternate between 16-byte aligned (bulk-copy ring) and not
    (plain loads); V = 1000 (two units) leaves a partial last unit and two of
    the four CTAs of a cluster without a share of the rows."""
    torch, dev = torch_dev()
    w = WORKLOADS["c3"]
    parent = np.array(TREES["uneven-11"], dtype=np.int32)
    N = len(parent)
    tgt, dft, seeds = _tree_batch(w, B, N, V, dtype, seed=V)
    tg, dg = upload(tgt, dtype), upload(dft, dtype)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for rnd in (2, 3):
        tok = orc.tree_draft(dft, parent, seeds, rnd, w.T, nthreads=16)
        g = ssd.tree_verify(tg, dg, parent, i32(tok), seeds_t(seeds), rnd, w.T,
                            dev_status=status)
        g = {k: v.cpu().numpy() for k, v in g.items()}
        o = orc.tree_verify(tgt, dft, parent, tok, seeds, rnd, w.T, nthreads=16)
        compare_tree(g, o)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("shape", ["root-only", "one-edge", "star-255", "chain-255"])
def test_tree_extreme_shapes(orc, shape):
    """The degenerate and the largest trees: a root alone (the bonus from p_0,
    no test), one edge, a root with 255 children (up to 254 residual passes
    at one node) and a chain of 256 nodes (depth 255)."""
    torch, dev = torch_dev()
    N = {"root-only": 1, "one-edge": 2, "star-255": 256, "chain-255": 256}[shape]
    if shape == "star-255":
        parent = np.array([-1] + [0] * (N - 1), dtype=np.int32)
    else:
        parent = np.arange(-1, N - 1, dtype=np.int32)
    w = WORKLOADS["c1"]
    B, V = 3, 1000
    w = dataclasses.replace(w, V=V)
    tgt, dft, seeds = _tree_batch(w, B, N, V, "f32", seed=N)
    tg, dg = upload(tgt, "f32"), upload(dft, "f32")
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    tok = orc.tree_draft(dft, parent, seeds, 1, w.T, nthreads=4)
    g = ssd.tree_verify(tg, dg, parent, i32(tok), seeds_t(seeds), 1, w.T, dev_status=status)
    g = {k: v.cpu().numpy() for k, v in g.items()}
    o = orc.tree_verify(tgt, dft, parent, tok, seeds, 1, w.T, nthreads=4)
    compare_tree(g, o)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


@pytest.mark.parametrize("B,V", [(32, 50000), (600, 4096)], ids=["c3-rows", "many-rows"])
def test_chain_tree_equals_linear_verify(orc, B, V):
    """A chain verified as a tree gives ssd_verify's accept lengths and bonus
    tokens at C = 1, bit for bit.  With 600 sequences the linear verification
    drops the target rows past known rejections while the tree path reads
    every row: the two paths still agree."""
    torch, dev = torch_dev()
    w = WORKLOADS["c3"]
    K = 6
    bt = make_batch(w, B=B, V=V, K=K, seed=3)
    parent = np.arange(-1, K, dtype=np.int32)
    F = np.zeros(K + 1, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, 1.0, w.T, bt["seeds"], K=K)
    tg, dg = upload(bt["target"], "bf16"), upload(bt["draft"], "bf16")
    lin = ssd.verify(tg, dg, i32(tok), seeds_t(bt["seeds"]), 4, F, 1.0, w.T, guesses=False)
    tt = np.concatenate([np.full((B, 1), -1, np.int32), tok], axis=1)
    tr = ssd.tree_verify(tg, dg[:, :K + 1], parent, i32(tt), seeds_t(bt["seeds"]), 4, w.T)
    np.testing.assert_array_equal(tr["accept_len"].cpu().numpy(), lin["accept_len"].cpu().numpy())
    np.testing.assert_array_equal(tr["bonus"].cpu().numpy(), lin["bonus"].cpu().numpy())


def test_tree_bad_arguments():
    torch, dev = torch_dev()
    t = torch.zeros((2, 3, 64), device=dev)
    tok = torch.zeros((2, 3), dtype=torch.int32, device=dev)
    with pytest.raises(ssd.SSDError):
        ssd.tree_verify(t, t, [-1, 2, 0], tok, np.ones(2, np.uint64), 0)
    with pytest.raises(ssd.SSDError):
        ssd.tree_verify(t, t, [-1, 0, 0], tok, np.ones(2, np.uint64), 0, T=0.0)
