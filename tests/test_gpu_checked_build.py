"""The bounds-checked build (libssd_checks.so, -DSSD_CHECKS) on the paths the
benchmark and the SSD cache build use: every global, shared and workspace
access of the kernels is checked, a failed check is recorded in the last 256
bytes of the caller's workspace and the access is skipped.

Each call runs on both libraries with the same inputs and a workspace larger
than the call needs (so the record must sit at the caller's end, not at the
end of the launch's own layout): the record must stay zero and every output
must equal the product library's bit for bit.
"""

import ctypes

import numpy as np
import pytest

import sampling_ssd_verify_gb300 as ssd
from sampling_ssd_verify_gb300 import _build
from ssd_inputs import WORKLOADS, make_batch
from tests.parity import i32, seeds_t, torch_dev, upload

pytestmark = pytest.mark.gpu

EXTRA = 4096 + 40  # workspace bytes beyond the call's need (not a multiple of 256)


@pytest.fixture(scope="module")
def libs():
    ssd.build()
    main = ssd.lib()
    path = _build.build(checks=True)
    chk = ctypes.CDLL(path)
    for name, (args, res) in ssd._SIGS.items():
        fn = getattr(chk, name)
        fn.argtypes = args
        fn.restype = res
    yield main, chk
    ssd._lib = main


def _both(libs, call, nbytes):
    """Run call(workspace) on the product and the checked library; return
    both outputs (numpy) and the checked run's record."""
    torch, dev = torch_dev()
    main, chk = libs
    outs = []
    for L in (main, chk):
        ssd._lib = L
        ws = torch.zeros(nbytes + EXTRA, dtype=torch.uint8, device=dev)
        o = call(ws)
        torch.cuda.synchronize()
        outs.append({k: v.cpu().numpy() for k, v in o.items() if hasattr(v, "cpu")})
        rec = ws[-256:].cpu().numpy().view(np.uint64)
    ssd._lib = main
    return outs[0], outs[1], rec


def _assert_same(a, b, skip=("table",)):
    for k in a:
        if k in skip:
            continue
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)


def _draft_tokens(dg, w, F, seeds):
    tok = []
    for j in range(w.K):
        tok.append(ssd.saguaro_sample(dg[:, j, :], w.T, w.C, int(F[j]), seeds, j, 0,
                                      guesses=False, qprime=False)["token"])
    torch, _ = torch_dev()
    return torch.stack(tok, 1).contiguous()


@pytest.mark.parametrize("wl,B,V,dtype", [("c3", 8, 128256, "bf16"), ("c5", 4, 151936, "f32"),
                                          ("c1", 64, 37, "bf16")])
def test_checked_verify_round(libs, wl, B, V, dtype):
    """verify_round (streaming pass, draws, round cache), aligned rows with
    the block-sum draw and unaligned rows (V = 37 bf16) without it."""
    w = WORKLOADS[wl]
    bt = make_batch(w, B=B, V=V, dtype=dtype, seed=77)
    tg, dg = upload(bt["target"], dtype), upload(bt["draft"], dtype)
    seeds = seeds_t(bt["seeds"])
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = _draft_tokens(dg, w, F, seeds)
    nb = ssd.lib().ssd_verify_workspace_size(B, w.K, dg.shape[1], V)
    a, b, rec = _both(libs, lambda ws: ssd.verify_round(tg, dg, tok, seeds, 5, F, w.C, w.T,
                                                        workspace=ws), nb)
    assert not rec.any(), f"bounds check failed: code {rec[0]} a {rec[1]} b {rec[2]} n {rec[5]}"
    _assert_same(a, b)


@pytest.mark.parametrize("V,dtype", [(151936, "bf16"), (4099, "bf16"), (37, "f32")])
def test_checked_saguaro(libs, V, dtype):
    """ssd_saguaro_sample with per-row fan-out: aligned rows (block-sum draw)
    and unaligned ones (queued draws)."""
    w = WORKLOADS["c4"]
    R = 96
    bt = make_batch(w, B=R, K=0, V=V, dtype=dtype, seed=V)
    rows = upload(np.ascontiguousarray(bt["target"][:, 0, :]), dtype)
    seeds = seeds_t(bt["seeds"])
    F = np.asarray([w.fanout[r % len(w.fanout)] for r in range(R)], dtype=np.int32)
    nb = ssd.lib().ssd_saguaro_workspace_size(R, V)
    a, b, rec = _both(libs, lambda ws: ssd.saguaro_sample(rows, w.T, w.C, F, seeds, 1, 2,
                                                          workspace=ws), nb)
    assert not rec.any(), f"bounds check failed: code {rec[0]} a {rec[1]} b {rec[2]} n {rec[5]}"
    _assert_same(a, b)


def test_checked_tree(libs):
    w = WORKLOADS["c3"]
    parent = [-1, 0, 0, 1, 1, 2, 2]
    B, N, V = 6, len(parent), 128256
    bt = make_batch(w, B=B, V=V, K=N - 1, seed=3, dtype="bf16")
    tg = upload(bt["target"], "bf16")
    dg = upload(np.ascontiguousarray(bt["draft"][:, :N]), "bf16")
    torch, dev = torch_dev()
    rng = np.random.default_rng(3)
    tok = i32(rng.integers(0, V, (B, N)).astype(np.int32))
    nb = ssd.lib().ssd_tree_workspace_size(B, N, V)
    a, b, rec = _both(libs, lambda ws: ssd.tree_verify(tg, dg, parent, tok, seeds_t(bt["seeds"]),
                                                       4, w.T, workspace=ws), nb)
    assert not rec.any(), f"bounds check failed: code {rec[0]} a {rec[1]} b {rec[2]} n {rec[5]}"
    _assert_same(a, b)
