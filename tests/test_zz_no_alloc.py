"""ssd_verify_noalloc: verification for callers that cannot allocate.

Some callers cannot hand the library a device workspace -- an inference
runtime's plugin whose enqueue hook may not allocate, a process whose device
memory is entirely owned by a pool allocator, or a decode loop that cannot pay
for cudaMalloc and the synchronisation it brings.  ssd_verify_noalloc runs the
same verification on a scratch array built into the library.  This test calls
it through the C ABI twice in a row and checks each result against ssd_verify
with a caller workspace on the same inputs.  It lives in a file of its own,
collected last, and builds and loads everything it needs, so it runs the same
alone in a fresh process or after the rest of the suite.
"""

import ctypes

import numpy as np
import pytest

import sampling_ssd_verify_gb300 as ssd
from ssd_inputs import WORKLOADS, make_batch
from tests.parity import PROB_TOL, i32, seeds_t, torch_dev, upload

pytestmark = pytest.mark.gpu

SSD_ERR_WORKSPACE = 5


def _noalloc():
    ssd.build()
    f = ssd.lib().ssd_verify_noalloc
    vp, ci = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [ctypes.POINTER(ssd._Logits), ctypes.POINTER(ssd._Logits), ci, ci, ci, ci,
                  ctypes.c_float, vp, vp, ctypes.c_uint32, vp, ctypes.c_float, vp, vp, vp, vp,
                  vp, ci, vp, vp]
    f.restype = ci
    return f


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


@pytest.mark.parametrize("wname,B,V", [("c5", 32, 151936), ("c3", 16, 128256)])
def test_noalloc_matches_workspace_entry_point(wname, B, V):
    torch, dev = torch_dev()
    f = _noalloc()
    w = WORKLOADS[wname]
    K, Kq = w.K, w.Kq
    bt = make_batch(w, B=B, V=V)
    tg, dg = upload(bt["target"], w.dtype), upload(bt["draft"], w.dtype)
    seeds = seeds_t(bt["seeds"])
    F = np.asarray(w.fanout, dtype=np.int32)
    Fmax = int(F.max())
    gen = torch.Generator(device="cpu").manual_seed(5)
    tok = i32(torch.randint(0, V, (B, K), generator=gen, dtype=torch.int32).numpy())
    tl, dl = ssd._logits(tg), ssd._logits(dg)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    for rnd in (7, 8):  # two calls in a row share the scratch array
        torch.cuda.synchronize()
        alloc0, free0 = torch.cuda.memory_allocated(), torch.cuda.mem_get_info()[0]
        out = {"accept_len": torch.full((B,), -7, dtype=torch.int32, device=dev),
               "bonus": torch.full((B,), -7, dtype=torch.int32, device=dev),
               "resid_mass": torch.full((B,), -1.0, dtype=torch.float32, device=dev),
               "guesses": torch.full((B, Kq, Fmax), -7, dtype=torch.int32, device=dev),
               "guess_q": torch.full((B, Kq, Fmax), -1.0, dtype=torch.float32, device=dev)}
        st = f(ctypes.byref(tl), ctypes.byref(dl), B, K, Kq, V, float(w.T), _ptr(tok), _ptr(seeds),
               rnd, F.ctypes.data_as(ctypes.c_void_p), float(w.C), _ptr(out["accept_len"]),
               _ptr(out["bonus"]), _ptr(out["resid_mass"]), _ptr(out["guesses"]),
               _ptr(out["guess_q"]), Fmax, _ptr(status),
               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0, ssd.lib().ssd_status_string(st)
        torch.cuda.synchronize()
        if rnd == 8:
            # after the first call has loaded everything, a call takes no
            # device memory from torch's allocator or from the device
            assert torch.cuda.memory_allocated() == alloc0
            assert torch.cuda.mem_get_info()[0] == free0
        ref = ssd.verify(tg, dg, tok, seeds, rnd, F, w.C, w.T)
        torch.cuda.synchronize()
        for k in ("accept_len", "bonus", "guesses"):
            np.testing.assert_array_equal(out[k].cpu().numpy(), ref[k].cpu().numpy())
        for k in ("resid_mass", "guess_q"):
            assert np.abs(out[k].cpu().numpy() - ref[k].cpu().numpy()).max() < PROB_TOL
    assert int(status.item()) == 0


def test_noalloc_rejects_requests_beyond_its_scratch():
    f = _noalloc()
    assert ssd.lib().ssd_verify_workspace_size(4096, 8, 9, 151936) > (4 << 20)
    fake = ssd._Logits(ctypes.c_void_p(0x10000), 1, 0, 151936)
    F = np.zeros(9, dtype=np.int32)
    st = f(ctypes.byref(fake), ctypes.byref(fake), 4096, 8, 9, 151936, 1.0, 0x20000, 0x30000, 0,
           F.ctypes.data_as(ctypes.c_void_p), 1.0, 0x40000, 0x50000, None, None, None, 1, None,
           None)
    assert st == SSD_ERR_WORKSPACE
