"""ctypes front end of the CPU oracle (``ssd_oracle.cpp``).

TEST INFRASTRUCTURE ONLY: the correctness reference for the CUDA library and
the timed CPU baseline.  It is imported by ``tests/``, by the smoke check and
by the benchmark's CPU-baseline leg, never by the library itself.  It shares
no code with the CUDA path.

``build()`` compiles ``ssd_oracle.cpp`` with the host C++ compiler into
``oracle/_build/libssd_oracle.so`` (plain C++17, no architecture flags, so it
builds the same on x86-64 and aarch64).
"""

from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssd_oracle.cpp")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "libssd_oracle.so")
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i32p = ctypes.POINTER(ctypes.c_int32)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_u64p = ctypes.POINTER(ctypes.c_uint64)
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile the oracle shared library if missing or older than its source."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = [os.environ.get("CXX", "g++"), "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
           _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _configure(L):
    L.orc_philox4x32.argtypes = [_u32p, _u32p, _u32p]
    L.orc_philox4x64.argtypes = [_u64p, _u64p, _u64p]
    L.orc_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                              ctypes.c_uint32, ctypes.c_uint32]
    L.orc_uniform.restype = ctypes.c_double
    L.orc_uniform_batch.argtypes = [ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32,
                                    ctypes.c_uint32, ctypes.c_int, _dp]
    L.orc_softmax.argtypes = [_dp, ctypes.c_int, ctypes.c_double, _dp]
    L.orc_top_n.argtypes = [_dp, ctypes.c_int, ctypes.c_int, _i32p]
    L.orc_saguaro_dist.argtypes = [_dp, ctypes.c_int, ctypes.c_double, ctypes.c_int,
                                   ctypes.c_double, _dp]
    L.orc_accept_prob.argtypes = [ctypes.c_double, ctypes.c_double]
    L.orc_accept_prob.restype = ctypes.c_double
    L.orc_residual.argtypes = [_dp, _dp, ctypes.c_int, _dp]
    L.orc_residual.restype = ctypes.c_double
    L.orc_inverse_cdf.argtypes = [_dp, ctypes.c_int, ctypes.c_double, ctypes.c_double, _dp]
    L.orc_inverse_cdf.restype = ctypes.c_int
    L.orc_verify.argtypes = [_vp, _vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                             ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                             ctypes.c_double, _i32p, _u64p, ctypes.c_uint32, _i32p,
                             _dp, ctypes.c_int, _i32p, _i32p, _dp, _i32p, _dp,
                             _dp, _dp, ctypes.c_int, _i32p, _dp]
    L.orc_verify.restype = ctypes.c_int
    L.orc_topf_bonus.argtypes = [_vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_double, _i32p,
                                 ctypes.c_int, _i32p, ctypes.c_int, _i32p, _dp, ctypes.c_int]
    L.orc_saguaro_sample.argtypes = [_vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                     ctypes.c_int, _i32p, _u64p, ctypes.c_int, ctypes.c_uint32,
                                     _i32p, _dp, _i32p, _dp, ctypes.c_int, _i32p]
    L.orc_tree_verify.argtypes = [_vp, _vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                  _i32p, _i32p, _u64p, ctypes.c_uint32, _i32p, _i32p,
                                  ctypes.c_int, _i32p, _dp, _dp, _dp, ctypes.c_int]
    L.orc_tree_verify.restype = ctypes.c_int
    L.orc_tree_draft.argtypes = [_vp, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
                                 ctypes.c_int, ctypes.c_double, _i32p, _u64p, ctypes.c_uint32,
                                 _i32p, ctypes.c_int]
    L.orc_tree_draft.restype = ctypes.c_int
    L.orc_cache_lookup.argtypes = [_i32p, _i32p, _i32p, _i32p, ctypes.c_int, _i32p, _i32p,
                                   ctypes.c_int, _i32p, _i32p]
    L.orc_cache_lookup.restype = ctypes.c_int
    L.orc_fanout_real.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                  ctypes.c_double, _dp]
    L.orc_fanout_real.restype = ctypes.c_int
    L.orc_fanout.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                             _i32p]
    L.orc_fanout.restype = ctypes.c_int
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _configure(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def use_library(path):
    """Temporarily route every wrapper through another build of the oracle
    (the mutation tests compile copies with a planted mistake)."""
    global _lib
    saved = lib()
    _lib = _configure(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def build_variant(src_text: str, out_path: str) -> str:
    """Compile an edited copy of the oracle source (mutation tests)."""
    src = out_path + ".cpp"
    with open(src, "w") as f:
        f.write(src_text)
    subprocess.run([os.environ.get("CXX", "g++"), "-O1", "-std=c++17", "-shared", "-fPIC",
                    "-pthread", src, "-o", out_path], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _p(a, t):
    return a.ctypes.data_as(t) if a is not None else None


def _f64(a):
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a):
    return np.ascontiguousarray(a, dtype=np.int32)


# ---- Philox / uniforms -------------------------------------------------------
def philox4x32(ctr, key):
    c = np.asarray(ctr, dtype=np.uint32)
    k = np.asarray(key, dtype=np.uint32)
    o = np.zeros(4, dtype=np.uint32)
    lib().orc_philox4x32(_p(c, _u32p), _p(k, _u32p), _p(o, _u32p))
    return o


def philox4x64(ctr, key):
    c = np.asarray(ctr, dtype=np.uint64)
    k = np.asarray(key, dtype=np.uint64)
    o = np.zeros(4, dtype=np.uint64)
    lib().orc_philox4x64(_p(c, _u64p), _p(k, _u64p), _p(o, _u64p))
    return o


def uniform(seed, c0, c1, stream, round_):
    return lib().orc_uniform(int(seed), int(c0), int(c1), int(stream), int(round_))


def uniform_batch(seed, c1, stream, round_, n):
    out = np.zeros(n, dtype=np.float64)
    lib().orc_uniform_batch(int(seed), int(c1), int(stream), int(round_), int(n), _p(out, _dp))
    return out


# ---- single steps --------------------------------------------------------------
def softmax(z, T):
    z = _f64(z)
    p = np.zeros_like(z)
    lib().orc_softmax(_p(z, _dp), len(z), float(T), _p(p, _dp))
    return p


def top_n(z, n):
    z = _f64(z)
    idx = np.zeros(min(n, len(z)), dtype=np.int32)
    lib().orc_top_n(_p(z, _dp), len(z), int(n), _p(idx, _i32p))
    return idx


def saguaro_dist(z, T, F, C):
    z = _f64(z)
    q = np.zeros_like(z)
    lib().orc_saguaro_dist(_p(z, _dp), len(z), float(T), int(F), float(C), _p(q, _dp))
    return q


def accept_prob(px, qx):
    return lib().orc_accept_prob(float(px), float(qx))


def residual(p, q):
    p, q = _f64(p), _f64(q)
    w = np.zeros_like(p)
    Z = lib().orc_residual(_p(p, _dp), _p(q, _dp), len(p), _p(w, _dp))
    return w, Z


def inverse_cdf(w, Z, u):
    w = _f64(w)
    m = np.zeros(1)
    y = lib().orc_inverse_cdf(_p(w, _dp), len(w), float(Z), float(u), _p(m, _dp))
    return y, float(m[0])


# ---- batched entry points --------------------------------------------------------
def _dtype_code(arr):
    if arr.dtype == np.uint16:
        return 0
    if arr.dtype == np.float32:
        return 1
    raise TypeError(arr.dtype)


def per_position_C(C, K):
    """C as one Saguaro factor per draft position j = 0..K-1 (a scalar applies
    to every position)."""
    Cv = np.broadcast_to(np.asarray(C, dtype=np.float64), (K,)) if np.ndim(C) == 0 \
        else np.asarray(C, dtype=np.float64)
    if Cv.shape != (K,):
        raise ValueError("C must be a scalar or have one entry per draft position")
    return np.ascontiguousarray(Cv)


def verify(target, draft, tokens, seeds, round_, F, C, T, Fmax=None, nthreads=1,
           row_ids=None):
    """target [B,K+1,V], draft [B,Kq,V] (uint16 bf16 bits or float32); C a
    scalar or one factor per draft position; T a scalar or one temperature
    per sequence (0: the greedy limit)."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    B, K1, V = target.shape
    K = K1 - 1
    Kq = draft.shape[1]
    F = _i32(F)
    assert len(F) == Kq
    Fmax = int(max(1, F.max())) if Fmax is None else int(Fmax)
    tokens = _i32(tokens).reshape(B, K)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    acc = np.zeros(B, dtype=np.int32)
    bon = np.zeros(B, dtype=np.int32)
    Z = np.zeros(B)
    g = np.zeros((B, Kq, Fmax), dtype=np.int32)
    gq = np.zeros((B, Kq, Fmax))
    ma = np.zeros(B)
    mc = np.zeros(B)
    Cv = per_position_C(C, K)
    if np.ndim(T) == 0:
        T0, Tr = float(T), None
    else:
        Tr = np.ascontiguousarray(T, dtype=np.float64)
        if Tr.shape != (B,):
            raise ValueError("T must be a scalar or have one entry per sequence")
        T0 = 1.0
    rc = lib().orc_verify(target.ctypes.data, draft.ctypes.data, _dtype_code(target), V, V, B, K,
                          Kq, V, T0, _p(tokens, _i32p), _p(seeds, _u64p), int(round_),
                          _p(F, _i32p), _p(Cv, _dp), Fmax, _p(acc, _i32p), _p(bon, _i32p),
                          _p(Z, _dp), _p(g, _i32p), _p(gq, _dp), _p(ma, _dp), _p(mc, _dp),
                          int(nthreads), _p(None if row_ids is None else _i32(row_ids), _i32p),
                          _p(Tr, _dp))
    if rc:
        raise ValueError("draft token outside [0, V)")
    return dict(accept_len=acc, bonus=bon, resid_mass=Z, guesses=g, guess_q=gq,
                margin_accept=ma, margin_cdf=mc)


def topf_bonus(draft, F, T, tokens=None, K=0, Fmax=None, nthreads=1):
    draft = np.ascontiguousarray(draft)
    B, Kq, V = draft.shape
    F = _i32(F)
    Fmax = int(max(1, F.max())) if Fmax is None else int(Fmax)
    tok = None if tokens is None else _i32(tokens).reshape(B, K)
    g = np.zeros((B, Kq, Fmax), dtype=np.int32)
    gq = np.zeros((B, Kq, Fmax))
    lib().orc_topf_bonus(draft.ctypes.data, _dtype_code(draft), V, B, Kq, V, float(T),
                         _p(tok, _i32p), int(K), _p(F, _i32p), Fmax, _p(g, _i32p), _p(gq, _dp),
                         int(nthreads))
    return dict(guesses=g, guess_q=gq)


def saguaro_sample(rows, T, C, F, seeds, j, round_, nthreads=1, row_ids=None):
    """rows [R, V] (uint16 bf16 bits or float32); F one fan-out for every row
    or one per row (guesses then have max(F) columns, -1 padded)."""
    rows = np.ascontiguousarray(rows)
    R, V = rows.shape
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    if np.ndim(F) == 0:
        Fc, Fr = int(F), None
    else:
        Fr = _i32(F)
        if Fr.shape != (R,):
            raise ValueError("per-row F must have R entries")
        Fc = int(Fr.max()) if R else 0
    tok = np.zeros(R, dtype=np.int32)
    qp = np.zeros(R)
    g = np.zeros((R, max(Fc, 1)), dtype=np.int32)
    mc = np.zeros(R)
    lib().orc_saguaro_sample(rows.ctypes.data, _dtype_code(rows), V, R, V, float(T), float(C),
                             Fc, _p(Fr, _i32p), _p(seeds, _u64p), int(j), int(round_),
                             _p(tok, _i32p), _p(qp, _dp), _p(g, _i32p), _p(mc, _dp),
                             int(nthreads), _p(None if row_ids is None else _i32(row_ids), _i32p))
    return dict(token=tok, qprime=qp, guesses=g[:, :Fc], margin_cdf=mc)


def tree_depth(parent):
    """Depth of the deepest node of a tree given by parent[] (root 0)."""
    parent = _i32(parent)
    d = np.zeros(len(parent), dtype=np.int64)
    for u in range(1, len(parent)):
        d[u] = d[parent[u]] + 1
    return int(d.max()) if len(d) else 0


def tree_verify(target, draft, parent, tokens, seeds, round_, T, nthreads=1):
    """target, draft [B, N, V] (uint16 bf16 bits or float32): row u of a tree
    is p_u / q_u at node u; parent [N] (parent[0] = -1); tokens [B, N]."""
    target = np.ascontiguousarray(target)
    draft = np.ascontiguousarray(draft)
    B, N, V = target.shape
    parent = _i32(parent)
    tokens = _i32(tokens).reshape(B, N)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    Dmax = max(1, tree_depth(parent))
    acc = np.zeros(B, dtype=np.int32)
    path = np.zeros((B, Dmax), dtype=np.int32)
    bon = np.zeros(B, dtype=np.int32)
    Z = np.zeros(B)
    ma = np.zeros(B)
    mc = np.zeros(B)
    rc = lib().orc_tree_verify(target.ctypes.data, draft.ctypes.data, _dtype_code(target), V, V,
                               B, N, V, float(T), _p(parent, _i32p), _p(tokens, _i32p),
                               _p(seeds, _u64p), int(round_), _p(acc, _i32p), _p(path, _i32p),
                               Dmax, _p(bon, _i32p), _p(Z, _dp), _p(ma, _dp), _p(mc, _dp),
                               int(nthreads))
    if rc == 3:
        raise ValueError("parent[] is not a tree with parent[u] < u")
    if rc:
        raise ValueError("draft token outside [0, V)")
    return dict(accept_len=acc, path=path, bonus=bon, resid_mass=Z, margin_accept=ma,
                margin_cdf=mc)


def tree_draft(draft, parent, seeds, round_, T, nthreads=1):
    """Draft tokens [B, N] of a tree: x_v ~ q_{parent(v)} (entry 0 is -1)."""
    draft = np.ascontiguousarray(draft)
    B, N, V = draft.shape
    parent = _i32(parent)
    seeds = np.ascontiguousarray(seeds, dtype=np.uint64)
    tok = np.zeros((B, N), dtype=np.int32)
    if lib().orc_tree_draft(draft.ctypes.data, _dtype_code(draft), V, B, N, V, float(T),
                            _p(parent, _i32p), _p(seeds, _u64p), int(round_), _p(tok, _i32p),
                            int(nthreads)):
        raise ValueError("parent[] is not a tree with parent[u] < u")
    return tok


def cache_lookup(row, k, t, branch, accept_len, bonus):
    row, k, t, branch = _i32(row), _i32(k), _i32(t), _i32(branch)
    accept_len, bonus = _i32(accept_len), _i32(bonus)
    B = len(accept_len)
    out = np.zeros(B, dtype=np.int32)
    ah = np.zeros(1, dtype=np.int32)
    rc = lib().orc_cache_lookup(_p(row, _i32p), _p(k, _i32p), _p(t, _i32p), _p(branch, _i32p),
                                len(row), _p(accept_len, _i32p), _p(bonus, _i32p), B,
                                _p(out, _i32p), _p(ah, _i32p))
    if rc:
        raise KeyError("duplicate cache key")
    return out, int(ah[0])


def fanout_real(K, budget, a, r):
    x = np.zeros(K + 1)
    if lib().orc_fanout_real(int(K), int(budget), float(a), float(r), _p(x, _dp)):
        raise ValueError("bad fan-out arguments")
    return x


def fanout(K, budget, a, r):
    F = np.zeros(K + 1, dtype=np.int32)
    if lib().orc_fanout(int(K), int(budget), float(a), float(r), _p(F, _i32p)):
        raise ValueError("bad fan-out arguments")
    return F


def draft_tokens(draft, F, C, T, seeds, round_=0, K=None, nthreads=1):
    """Draw the drafts x_j ~ q'_j for every sequence (Saguaro sampling, stream 2).

    draft [B, Kq, V]; row (b, j) uses counter (b, j, 2, round) -- the same
    definition as the library's continuation sampler called once per position.
    C: a scalar or one factor per draft position.
    """
    draft = np.ascontiguousarray(draft)
    B, Kq, V = draft.shape
    K = Kq - 1 if K is None else K
    Cv = per_position_C(C, K)
    out = np.zeros((B, K), dtype=np.int32)
    for j in range(K):
        r = saguaro_sample(np.ascontiguousarray(draft[:, j, :]), T, Cv[j], int(F[j]), seeds, j,
                           round_, nthreads=nthreads)
        out[:, j] = r["token"]
    return out
