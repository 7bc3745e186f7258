"""The C-ABI library: it builds, loads, exports every declared entry point,
and its host-side logic (argument validation, sizes, fan-out) is right.
No test here launches device work."""

import ctypes
import os
import re

import numpy as np
import pytest

import sampling_ssd_verify_gb300 as ssd

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ssd.h")


@pytest.fixture(scope="module")
def L():
    ssd.build()
    return ssd.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssd_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ("ssd_verify", "ssd_topf_bonus", "ssd_saguaro_sample", "ssd_cache_build",
              "ssd_cache_lookup", "ssd_fanout"):
        assert n in names


@pytest.mark.parametrize("lang,std", [("c", "c99"), ("c++", "c++17")])
def test_header_is_plain_c(tmp_path, lang, std):
    """ssd.h is a C ABI: it compiles as strict C99 and as C++ (no torch or
    C++-only types in the declarations)."""
    import shutil
    import subprocess

    cc = shutil.which("gcc") if lang == "c" else shutil.which("g++")
    if cc is None:
        pytest.skip("no host compiler")
    src = tmp_path / ("t.c" if lang == "c" else "t.cpp")
    src.write_text('#include "ssd.h"\nint main(void) { return ssd_version() < 0; }\n')
    r = subprocess.run([cc, "-x", lang, f"-std={std}", "-Wall", "-Wextra", "-pedantic", "-Werror",
                        "-I", os.path.dirname(HEADER), "-fsyntax-only", str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
        assert isinstance(getattr(L, name), ctypes._CFuncPtr)


def test_status_strings(L):
    assert L.ssd_status_string(0) == b"ok"
    assert b"invalid" in L.ssd_status_string(1)
    assert L.ssd_status_string(99) == b"unknown status"
    assert L.ssd_version() >= 100


def test_fanout_host_helper_matches_oracle(L, orc):
    """The library's own fan-out helper (host code) agrees with the oracle's
    restatement for many (K, budget, a, r)."""
    for K in (1, 2, 4, 8, 12, 32):
        for budget in (0, 1, 7, 12, 16, 24, 100):
            for a in (0.2, 0.5, 0.7, 0.9, 1.0):
                for r in (0.0, 0.5, 1.0, 2.0):
                    np.testing.assert_array_equal(ssd.fanout(K, budget, a, r),
                                                  orc.fanout(K, budget, a, r))
    F = np.zeros(5, dtype=np.int32)
    assert L.ssd_fanout(-1, 12, 0.7, 1.0, F.ctypes.data_as(ctypes.c_void_p)) == 1
    assert L.ssd_fanout(4, 12, 0.0, 1.0, F.ctypes.data_as(ctypes.c_void_p)) == 1
    assert L.ssd_fanout(4, 12, 0.7, -1.0, F.ctypes.data_as(ctypes.c_void_p)) == 1
    assert L.ssd_fanout(4, 12, 0.7, 1.0, None) == 1


def test_workspace_sizes(L):
    for B, K, Kq, V in ((1, 4, 5, 32), (64, 8, 9, 128256), (256, 8, 9, 151936), (3, 1, 1, 2)):
        n = L.ssd_verify_workspace_size(B, K, Kq, V)
        assert n > 0 and n % 256 == 0
    assert L.ssd_verify_workspace_size(0, 4, 5, 32) == 0
    assert L.ssd_verify_workspace_size(1, 33, 33, 32) == 0
    assert L.ssd_verify_workspace_size(1, 4, 6, 32) == 0
    assert L.ssd_verify_workspace_size(1, 4, 5, 1) == 0
    assert L.ssd_verify_workspace_size(1, 4, 5, 1 << 24) == 0
    assert L.ssd_topf_workspace_size(4, 5, 1000) > 0
    assert L.ssd_saguaro_workspace_size(384, 151936) > 0
    assert L.ssd_saguaro_workspace_size(0, 10) == 0


def test_cache_bytes(L):
    assert L.ssd_cache_bytes(0) == 256
    assert L.ssd_cache_bytes(384) == 16 * 1024
    assert L.ssd_cache_bytes(6144) == 16 * 16384
    assert L.ssd_cache_bytes(-1) == 0


def _fake(ptr=0x10000, dtype=0, stride=32):
    return ssd._Logits(ctypes.c_void_p(ptr), dtype, 0, stride)


def _verify(L, **kw):
    a = dict(target=_fake(), draft=_fake(), B=1, K=4, Kq=5, V=32, T=1.0, tok=0x20000,
             seeds=0x30000, fan=None, C=1.0, acc=0x40000, bonus=0x50000, Fmax=1, ws=None,
             wsb=0)
    a.update(kw)
    fan = None if a["fan"] is None else np.asarray(a["fan"], dtype=np.int32)
    return L.ssd_verify(ctypes.byref(a["target"]), ctypes.byref(a["draft"]), a["B"], a["K"],
                        a["Kq"], a["V"], a["T"], a["tok"], a["seeds"], 0,
                        None if fan is None else fan.ctypes.data_as(ctypes.c_void_p), a["C"],
                        a["acc"], a["bonus"], None, None, None, a["Fmax"], a["ws"], a["wsb"],
                        None, None)


def test_verify_rejects_bad_arguments_on_the_host(L):
    """Each bad argument returns SSD_ERR_INVALID_ARG (1) / UNSUPPORTED (2) /
    WORKSPACE (5) before any device work is enqueued."""
    inv = 1
    assert _verify(L, B=0) == inv
    assert _verify(L, K=0) == inv
    assert _verify(L, K=33, Kq=33) == inv
    assert _verify(L, Kq=6) == inv
    assert _verify(L, V=1) == inv
    assert _verify(L, V=1 << 24) == inv
    assert _verify(L, T=0.0) == 5                            # greedy: valid, no workspace
    assert _verify(L, T=-1.0) == inv
    assert _verify(L, T=float("inf")) == inv
    assert _verify(L, T=float("nan")) == inv
    assert _verify(L, C=0.0) == inv
    assert _verify(L, C=1.5) == inv
    assert _verify(L, C=float("nan")) == inv
    assert _verify(L, tok=None) == inv
    assert _verify(L, seeds=None) == inv
    assert _verify(L, acc=None) == inv
    assert _verify(L, bonus=None) == inv
    assert _verify(L, target=_fake(stride=31)) == inv
    assert _verify(L, target=_fake(ptr=0x10001)) == inv
    assert _verify(L, target=_fake(dtype=1)) == inv          # dtypes differ
    assert _verify(L, target=_fake(dtype=7), draft=_fake(dtype=7)) == inv
    assert _verify(L, target=_fake(ptr=0)) == inv
    assert _verify(L, V=100, target=_fake(stride=100), draft=_fake(stride=100),
                   fan=[3, 3, 2, 2, 40]) == 2                # F > SSD_MAX_F
    assert _verify(L, fan=[3, 3, 2, 2, -1]) == inv
    assert _verify(L, fan=[3, 3, 2, 2, 32]) == inv           # F + 1 > V
    # valid arguments but no workspace
    assert _verify(L, fan=[3, 3, 2, 2, 2]) == 5
    assert _verify(L, ws=0x1000 + 16, wsb=1 << 20) == 5      # misaligned
    assert _verify(L, ws=0x1000, wsb=16) == 5                # too small


def _verify_ck(L, Cv, K=4, Kq=5):
    C = None if Cv is None else np.asarray(Cv, dtype=np.float32)
    t, d = _fake(), _fake()
    return L.ssd_verify_ck(ctypes.byref(t), ctypes.byref(d), 1, K, Kq, 32, 1.0, 0x20000, 0x30000,
                           0, None, None if C is None else C.ctypes.data_as(ctypes.c_void_p),
                           0x40000, 0x50000, None, None, None, 1, None, 0, None, None)


def test_verify_ck_rejects_bad_factors_on_the_host(L):
    """Every per-position factor must lie in (0, 1]; a missing vector is an
    argument error.  Valid factors get as far as the (missing) workspace."""
    inv = 1
    assert _verify_ck(L, None) == inv
    assert _verify_ck(L, [0.5, 0.5, 0.0, 0.5]) == inv
    assert _verify_ck(L, [0.5, 1.5, 0.5, 0.5]) == inv
    assert _verify_ck(L, [0.5, 0.5, 0.5, float("nan")]) == inv
    assert _verify_ck(L, [0.5, 0.5, 0.5, 0.5], K=0, Kq=0) == inv
    assert _verify_ck(L, [0.3, 0.5, 1.0, 0.7]) == 5


def test_verify_ex_needs_its_temperatures(L):
    """ssd_verify_ex takes a device temperature per sequence (its values are
    checked on the device); a missing array or bad factors are argument
    errors, and valid arguments get as far as the (missing) workspace."""
    t, d = _fake(), _fake()
    C = np.array([0.5, 0.5, 0.0, 0.5], dtype=np.float32)

    def call(T_rows, Cp):
        return L.ssd_verify_ex(ctypes.byref(t), ctypes.byref(d), 1, 4, 5, 32, T_rows, 0x20000,
                               0x30000, 0, None, Cp, 0x40000, 0x50000, None, None, None, 1, None,
                               0, None, None)
    assert call(None, None) == 1
    assert call(0x60000, C.ctypes.data_as(ctypes.c_void_p)) == 1
    assert call(0x60000, None) == 5


def test_verify_round_checks_its_table(L):
    """ssd_verify_round needs the guesses, an output for the branches and a
    16-byte aligned table of at least ssd_cache_bytes(B*Kq*Fmax) bytes."""
    t, d = _fake(), _fake()
    F = np.array([3, 3, 2, 2, 2], dtype=np.int32)
    Fp = F.ctypes.data_as(ctypes.c_void_p)
    need = L.ssd_cache_bytes(1 * 5 * 3)

    def call(guesses=0x60000, table=0x70000, tb=None, branch=0x80000):
        return L.ssd_verify_round(ctypes.byref(t), ctypes.byref(d), 1, 4, 5, 32, 1.0, 0x20000,
                                  0x30000, 0, Fp, 0.5, 0x40000, 0x50000, None, guesses, None, 3,
                                  table, need if tb is None else tb, branch, None, None, 0, None,
                                  None)
    assert call(guesses=None) == 1
    assert call(branch=None) == 1
    assert call(table=None) == 1
    assert call(table=0x70008) == 1
    assert call(tb=need // 2) == 3
    assert call() == 5   # valid, but no workspace


def test_other_entry_points_reject_bad_arguments(L):
    d = _fake()
    F = np.array([1, 1], dtype=np.int32)
    Fp = F.ctypes.data_as(ctypes.c_void_p)
    assert L.ssd_topf_bonus(ctypes.byref(d), 0, 2, 32, 1.0, None, 0, Fp, 1, 0x1000, None, None,
                            0, None, None) == 1
    assert L.ssd_topf_bonus(ctypes.byref(d), 1, 2, 32, 1.0, None, 0, None, 1, 0x1000, None, None,
                            0, None, None) == 1
    assert L.ssd_topf_bonus(ctypes.byref(d), 1, 2, 32, 1.0, None, 0, Fp, 0, 0x1000, None, None,
                            0, None, None) == 1
    # (draft, R, V, T, C, F_row, Fmax, seeds, j, round, token, qprime, guess, ws, ws_bytes, ...)
    assert L.ssd_saguaro_sample(ctypes.byref(d), 4, 32, 1.0, 0.0, None, 2, 0x1000, 0, 0, 0x2000,
                                None, None, None, 0, None, None) == 1
    assert L.ssd_saguaro_sample(ctypes.byref(d), 4, 32, 1.0, 0.5, None, 32, 0x1000, 0, 0, 0x2000,
                                None, None, None, 0, None, None) == 1
    assert L.ssd_saguaro_sample(ctypes.byref(d), 4, 32, 1.0, 0.5, None, -1, 0x1000, 0, 0, 0x2000,
                                None, None, None, 0, None, None) == 1
    assert L.ssd_saguaro_sample(ctypes.byref(d), 4, 32, 1.0, 0.5, None, 16, 0x1000, 0, 0, 0x2000,
                                None, None, None, 0, None, None) == 2
    assert L.ssd_saguaro_sample(ctypes.byref(d), 4, 32, 1.0, 0.5, None, 2, 0x1000, 0, 0, 0x2000,
                                None, None, None, 0, None, None) == 5
    assert L.ssd_saguaro_sample(ctypes.byref(d), 4, 32, 1.0, 0.5, 0x3000, 2, 0x1000, 0, 0,
                                0x2000, None, None, None, 0, None, None) == 5
    assert L.ssd_cache_build(None, 4096, 1, 1, 1, 1, 4, None, None) == 1
    assert L.ssd_cache_build(0x1008, 4096, 1, 1, 1, 1, 4, None, None) == 1
    assert L.ssd_cache_build(0x1000, 64, 0x2000, 0x2000, 0x2000, 0x2000, 4, None, None) == 3
    assert L.ssd_cache_build_guesses(0x1000, 64, 0x2000, 2, 5, 3, None, None) == 3
    assert L.ssd_cache_lookup(None, 4096, 0x2000, 0x2000, 4, 0x3000, 0x4000, None) == 1
    assert L.ssd_cache_lookup(0x1000, 4096, 0x2000, 0x2000, 0, 0x3000, 0x4000, None) == 1
    # (workspace, bytes, B, K, Kq, V, dtype, out, stream)
    need = L.ssd_verify_workspace_size(4, 3, 4, 1000)
    assert L.ssd_verify_skipped_bytes(0x1000, need, 4, 3, 4, 1000, 0, None, None) == 1
    assert L.ssd_verify_skipped_bytes(0x1000, need, 4, 3, 5, 1000, 0, 0x2000, None) == 1
    assert L.ssd_verify_skipped_bytes(0x1000, need, 4, 3, 4, 1000, 7, 0x2000, None) == 1
    assert L.ssd_verify_skipped_bytes(None, need, 4, 3, 4, 1000, 0, 0x2000, None) == 5
    assert L.ssd_verify_skipped_bytes(0x1008, need, 4, 3, 4, 1000, 0, 0x2000, None) == 5
    assert L.ssd_verify_skipped_bytes(0x1000, need - 1, 4, 3, 4, 1000, 1, 0x2000, None) == 5


def test_binding_fails_loudly_without_a_gpu():
    """No CPU fallback: a CPU tensor is refused."""
    torch = pytest.importorskip("torch")
    t = torch.zeros((1, 5, 32))
    with pytest.raises(ssd.SSDError):
        ssd.verify(t, t, torch.zeros((1, 4), dtype=torch.int32), np.zeros(1, np.uint64), 0)


def test_uniform_fanout_allocation():
    """The ablation's uniform allocation spends the budget, differs by at most
    one between positions and gives the remainder to the lowest positions."""
    from sampling_ssd_verify_gb300.ablation import uniform_fanout

    for K in (1, 4, 8):
        for budget in (0, 5, 12, 24, 31):
            F = uniform_fanout(K, budget)
            assert len(F) == K + 1 and F.sum() == budget
            assert F.max() - F.min() <= 1
            assert np.all(np.diff(F) <= 0)
