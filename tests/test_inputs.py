"""The seeded synthetic inputs follow the stated recipe (CPU).

Generator G: per sequence a random vocabulary permutation, target logit of
the rank-r token = -zipf * ln r + 0.5 * Gumbel(0, 1), fresh Gumbel draws per
position; draft = target + N(0, sigma^2).  bf16 workloads store the
round-to-nearest-even bf16 of the fp32 values.  Every sequence is generated
from its own Philox stream, so any subset of rows can be regenerated alone.
"""

import numpy as np
import pytest

from ssd_inputs import WORKLOADS, make_batch
from ssd_inputs.generators import bf16_bits, bf16_to_f32, sequence_logits


def test_workload_shapes():
    expect = {"c1": (1, 4, 32, "f32"), "c2": (1, 4, 128256, "bf16"),
              "c3": (64, 8, 128256, "bf16"), "c4": (32, 4, 151936, "bf16"),
              "c5": (256, 8, 151936, "f32")}
    for name, (B, K, V, dt) in expect.items():
        w = WORKLOADS[name]
        assert (w.B, w.K, w.V, w.dtype) == (B, K, V, dt)
        assert w.Kq == K + 1 and len(w.fanout) == K + 1
        assert sum(w.fanout) == w.budget
        assert w.algorithmic_bytes() == B * (2 * K + 2) * V * w.elem_bytes


def test_batches_are_deterministic_and_row_independent():
    w = WORKLOADS["c3"]
    a = make_batch(w, B=6, V=4096)
    b = make_batch(w, B=6, V=4096)
    for k in ("target", "draft", "seeds"):
        np.testing.assert_array_equal(a[k], b[k])
    sub = make_batch(w, V=4096, rows=[4, 1])
    np.testing.assert_array_equal(sub["target"], a["target"][[4, 1]])
    np.testing.assert_array_equal(sub["draft"], a["draft"][[4, 1]])
    np.testing.assert_array_equal(sub["seeds"], a["seeds"][[4, 1]])
    assert len(set(a["seeds"].tolist())) == 6


def test_generator_g_structure():
    """Zipf head over a per-sequence permutation, Gumbel spread, draft noise."""
    w = WORKLOADS["c5"]
    V = 65536
    zp0, zq0, s0 = sequence_logits(w, 0, V=V)
    zp1, _, _ = sequence_logits(w, 1, V=V)
    # the permutation differs between sequences: their argmaxes differ
    assert zp0[0].argmax() != zp1[0].argmax()
    # rank r's token keeps its Zipf level at every position: the mean over
    # positions of the sorted logits falls like -zipf * ln r (plus the Gumbel mean)
    base = np.sort(zp0, axis=1)[:, ::-1].mean(axis=0)
    r = np.array([10, 100, 1000, 10000])
    slope = np.polyfit(np.log(r), base[r - 1], 1)[0]
    assert abs(slope + w.zipf) < 0.1
    # draft noise: std of (draft - target) equals sigma
    assert s0 == pytest.approx(w.sigma)
    assert np.std(zq0 - zp0) == pytest.approx(w.sigma, rel=0.02)
    # the Gumbel spread of one token across positions: std pi / sqrt(6) * scale
    spread = np.std(zp0[:, :2000], axis=0).mean()
    assert 0.3 * w.gumbel_scale < spread < 1.5 * w.gumbel_scale


def test_per_row_sigma_of_the_batched_workload():
    """c3: each sequence's draft noise std is drawn from U[0.3, 1.5]."""
    w = WORKLOADS["c3"]
    sig = [sequence_logits(w, b, V=2048)[2] for b in range(40)]
    assert min(sig) >= 0.3 and max(sig) <= 1.5
    assert max(sig) - min(sig) > 0.6


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0, 1.00390625, 1.01171875, -2.5e-3, 3.0e38, 0.0], dtype=np.float32)
    # 1 + 2^-8 is a tie between 1 and 1 + 2^-7: it rounds to the even mantissa (1.0);
    # 1 + 3 * 2^-8 is a tie that rounds up to 1 + 2^-6
    back = bf16_to_f32(bf16_bits(x))
    assert back[0] == 1.0 and back[1] == 1.0 and back[2] == np.float32(1.015625)
    assert np.all(np.abs(back - x) <= np.abs(x) * 2.0 ** -8)
    bt = make_batch(WORKLOADS["c2"], B=1, V=512)
    zp, zq, _ = sequence_logits(WORKLOADS["c2"], 0, V=512)
    np.testing.assert_array_equal(bt["target"][0], bf16_bits(zp))
    np.testing.assert_array_equal(bt["draft"][0], bf16_bits(zq))
