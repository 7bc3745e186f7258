"""The benchmark's host-side plumbing (CPU): the recorded DRAM traffic is only
reported for the kernel sources it was measured on, the oracle round does
what the GPU step does, and the per-rank inputs differ."""

import numpy as np

import bench
from ssd_inputs import WORKLOADS, make_batch


def _fake_tree(tmp_path, kernel_text):
    csrc = tmp_path / "sampling_ssd_verify_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (csrc / "k.cu").write_text(kernel_text)
    (tmp_path / "profiles").mkdir()
    return tmp_path


def test_traffic_is_reported_only_for_the_profiled_sources(tmp_path, monkeypatch):
    root = _fake_tree(tmp_path, "// kernel v1\n")
    monkeypatch.setattr(bench, "ROOT", str(root))
    sha = bench.csrc_hash()
    (root / "profiles" / "dram.md").write_text(
        f"# capture\n\ncsrc_sha: {sha}\ntraffic_bytes_per_launch[c5]: 3136955904\n")
    assert bench.traffic_from_profile("c5") == 3136955904.0
    assert bench.traffic_from_profile("c3") is None
    # any change to the kernel sources retires the recorded figure
    (root / "sampling_ssd_verify_gb300" / "csrc" / "k.cu").write_text("// kernel v2\n")
    assert bench.csrc_hash() != sha
    assert bench.traffic_from_profile("c5") is None


def test_oracle_round_is_verify_then_cache_lookup(orc):
    w = WORKLOADS["c1"]
    bt = make_batch(w, B=64)
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=w.K)
    rows = np.arange(64)
    branch, all_hit = bench.oracle_round(orc, bt, tok, 3, F, w, 2, rows)
    ref = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 3, F, w.C, w.T, row_ids=rows)
    g = ref["guesses"]
    for b in range(64):
        k, t = int(ref["accept_len"][b]), int(ref["bonus"][b])
        hits = np.nonzero(g[b, k] == t)[0]
        expect = (b * g.shape[1] + k) * g.shape[2] + int(hits[0]) if len(hits) else -1
        assert branch[b] == expect
    assert all_hit == int(np.all(branch >= 0))
    assert (branch >= 0).any()


def test_ranks_draw_different_batches():
    w = WORKLOADS["c5"]
    assert bench.rank_seed(w, 0) != bench.rank_seed(w, 1)
    a = make_batch(w, B=1, V=256, seed=bench.rank_seed(w, 0))
    b = make_batch(w, B=1, V=256, seed=bench.rank_seed(w, 1))
    assert not np.array_equal(a["target"], b["target"])


def test_roofline_counts_every_logit_and_reports_the_bytes_read_beside():
    # 2.8 GB of logits, 0.96 GB of them not read, one launch of 0.4 ms, a
    # 7000 GB/s peak: 7000 GB/s on every logit (frac 1.0), 4600 GB/s on the
    # 1.84 GB read (frac 4600 / 7000)
    r = bench.verify_roofline(2.8e9, 0.96e9, 0.4, 0.39, 7000.0, "measured", 2.3e9)
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] == 7000.0
    assert abs(r["achieved"] - 7000.0) < 1e-6 and abs(r["frac"] - 1.0) < 1e-12
    assert abs(r["bytes_read_per_launch"] - 1.84e9) < 1.0
    assert abs(r["gb_per_s_on_bytes_read"] - 4600.0) < 1e-6
    assert abs(r["frac_on_bytes_read"] - 4600.0 / 7000.0) < 1e-12
    assert r["algorithmic_bytes_per_launch"] == 2.8e9
    assert r["skipped_target_bytes_per_launch"] == 0.96e9
    assert r["traffic"] == 2.3e9 and r["launch_ms"] == 0.4 and r["launch_ms_median"] == 0.39
    # nothing skipped: both fractions agree
    r0 = bench.verify_roofline(1e9, 0.0, 1.0, 1.0, 1000.0, "fallback", None)
    assert r0["frac"] == r0["frac_on_bytes_read"] == 1.0 and r0["traffic"] is None
