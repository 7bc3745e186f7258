"""GB300 (sm_103a) speculative-decoding sampling path: thin Python binding.

Every step of the path runs in the CUDA kernels of ``libssd.so`` (built from
``csrc/`` by :func:`build`); this module only marshals PyTorch tensors into
the C ABI declared in ``include/ssd.h`` (device pointers, the current CUDA
stream, workspace buffers) and raises on error codes.  There is no CPU
fallback: without the library, or without a GPU, every call raises.

Entry points (same names as the C ABI):
  verify, topf_bonus, saguaro_sample, cache_build, cache_build_guesses,
  cache_lookup, fanout, plus verify_host (host tensors in, host results out,
  copies included).

Sources (page title, section):
  [SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈"
  [SD-7.3]   "7.3 Speculative Decoding：投机采样加速"
"""

from __future__ import annotations

import ctypes
import os

import numpy as np

from . import _build

__all__ = [
    "SSDError", "build", "lib", "verify", "verify_round", "verify_host", "topf_bonus",
    "saguaro_sample", "tree_verify",
    "cache_bytes", "cache_build", "cache_build_guesses", "cache_lookup", "fanout",
    "DEV_BAD_TOKEN", "DEV_ZERO_RESIDUAL", "DEV_TIMEOUT", "DEV_TABLE_FULL", "DEV_DUPLICATE_KEY",
    "DEV_BAD_TEMPERATURE", "DEV_BAD_FANOUT",
]

DEV_BAD_TOKEN = 0x1
DEV_ZERO_RESIDUAL = 0x2
DEV_TIMEOUT = 0x4
DEV_TABLE_FULL = 0x8
DEV_DUPLICATE_KEY = 0x10
DEV_BAD_TEMPERATURE = 0x20
DEV_BAD_FANOUT = 0x40

SSD_BF16, SSD_F32 = 0, 1
_lib = None


class SSDError(RuntimeError):
    pass


class _Logits(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("pad_", ctypes.c_int32),
                ("row_stride", ctypes.c_int64)]


_vp = ctypes.c_void_p
_i = ctypes.c_int
_sz = ctypes.c_size_t
_LP = ctypes.POINTER(_Logits)

_SIGS = {
    "ssd_status_string": ([_i], ctypes.c_char_p),
    "ssd_version": ([], _i),
    "ssd_verify_workspace_size": ([_i, _i, _i, _i], _sz),
    "ssd_verify_skipped_bytes": ([_vp, _sz, _i, _i, _i, _i, _i, _vp, _vp], _i),
    "ssd_verify": ([_LP, _LP, _i, _i, _i, _i, ctypes.c_float, _vp, _vp, ctypes.c_uint32, _vp,
                    ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _i, _vp, _sz, _vp, _vp], _i),
    "ssd_verify_ck": ([_LP, _LP, _i, _i, _i, _i, ctypes.c_float, _vp, _vp, ctypes.c_uint32, _vp,
                       _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _sz, _vp, _vp], _i),
    "ssd_verify_ex": ([_LP, _LP, _i, _i, _i, _i, _vp, _vp, _vp, ctypes.c_uint32, _vp,
                       _vp, _vp, _vp, _vp, _vp, _vp, _i, _vp, _sz, _vp, _vp], _i),
    "ssd_verify_round": ([_LP, _LP, _i, _i, _i, _i, ctypes.c_float, _vp, _vp, ctypes.c_uint32,
                          _vp, ctypes.c_float, _vp, _vp, _vp, _vp, _vp, _i, _vp, _sz, _vp, _vp,
                          _vp, _sz, _vp, _vp], _i),
    "ssd_topf_workspace_size": ([_i, _i, _i], _sz),
    "ssd_topf_bonus": ([_LP, _i, _i, _i, ctypes.c_float, _vp, _i, _vp, _i, _vp, _vp, _vp, _sz,
                        _vp, _vp], _i),
    "ssd_saguaro_workspace_size": ([_i, _i], _sz),
    "ssd_saguaro_sample": ([_LP, _i, _i, ctypes.c_float, ctypes.c_float, _vp, _i, _vp, _i,
                            ctypes.c_uint32, _vp, _vp, _vp, _vp, _sz, _vp, _vp], _i),
    "ssd_tree_workspace_size": ([_i, _i, _i], _sz),
    "ssd_tree_verify": ([_LP, _LP, _i, _i, _i, ctypes.c_float, _vp, _vp, _vp, ctypes.c_uint32,
                         _vp, _vp, _i, _vp, _vp, _vp, _sz, _vp, _vp], _i),
    "ssd_cache_bytes": ([_i], _sz),
    "ssd_cache_build": ([_vp, _sz, _vp, _vp, _vp, _vp, _i, _vp, _vp], _i),
    "ssd_cache_build_guesses": ([_vp, _sz, _vp, _i, _i, _i, _vp, _vp], _i),
    "ssd_cache_lookup": ([_vp, _sz, _vp, _vp, _i, _vp, _vp, _vp], _i),
    "ssd_fanout": ([_i, _i, ctypes.c_double, ctypes.c_double, _vp], _i),
}


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libssd.so for sm_103a (see ``_build.py``)."""
    return _build.build(force=force, verbose=verbose)


def lib_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load libssd.so (it must have been built; nothing falls back)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB_PATH):
            raise SSDError(f"{_build.LIB_PATH} is missing: build it with "
                           "sampling_ssd_verify_gb300.build()")
        L = ctypes.CDLL(_build.LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def _check(status: int, what: str):
    if status != 0:
        msg = lib().ssd_status_string(status).decode()
        raise SSDError(f"{what}: {msg} (status {status})")


# ---- tensor marshalling ---------------------------------------------------------------
def _torch():
    import torch
    return torch


def _dev_ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise SSDError("expected a CUDA tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    torch = _torch()
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _logits(t, nrows_inner=None):
    """Describe a [..., R, V] tensor whose rows are evenly spaced."""
    torch = _torch()
    if not t.is_cuda:
        raise SSDError("logits must be on the GPU")
    if t.dtype == torch.bfloat16:
        dt = SSD_BF16
    elif t.dtype == torch.float32:
        dt = SSD_F32
    else:
        raise SSDError(f"unsupported logits dtype {t.dtype}")
    if t.stride(-1) != 1:
        raise SSDError("logit rows must be contiguous over the vocabulary")
    rs = t.stride(-2) if t.dim() >= 2 else t.shape[-1]
    for d in range(t.dim() - 2):
        if t.stride(d) != rs * int(np.prod(t.shape[d + 1:-1])):
            raise SSDError("logit rows must be evenly spaced")
    return _Logits(ctypes.c_void_p(t.data_ptr()), dt, 0, rs)


def _workspace(nbytes, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _i32(t):
    torch = _torch()
    if t.dtype != torch.int32 or not t.is_contiguous():
        raise SSDError("expected a contiguous int32 tensor")
    return t


def _u64_seeds(seeds, device):
    torch = _torch()
    if isinstance(seeds, np.ndarray):
        seeds = torch.from_numpy(seeds.astype(np.uint64).view(np.int64)).to(device)
    if seeds.dtype not in (torch.int64, getattr(torch, "uint64", torch.int64)):
        raise SSDError("seeds must be 64-bit")
    return seeds.contiguous()


# ---- entry points ------------------------------------------------------------------------
def verify(target, draft, draft_tokens, seeds, round_, fanout=None, C=1.0, T=1.0,
           guesses=True, guess_q=True, resid_mass=True, workspace=None, dev_status=None,
           stream=None, out=None):
    """ssd_verify on device tensors.

    target [B, K+1, V], draft [B, Kq, V] (bf16 or fp32, same dtype),
    draft_tokens int32 [B, K], seeds 64-bit [B], fanout: sequence of Kq ints.
    C: the Saguaro factor, or a sequence of K factors, one per draft position
    (ssd_verify_ck).  T: the temperature (0: greedy), or one per sequence --
    a device float32 tensor [B] or anything numpy reads (ssd_verify_ex).
    Returns a dict of device tensors: accept_len, bonus, resid_mass, guesses,
    guess_q (the optional ones only when requested).
    """
    torch = _torch()
    B, K1, V = target.shape
    K = K1 - 1
    Kq = draft.shape[-2]
    dev = target.device
    F = np.zeros(Kq, dtype=np.int32) if fanout is None else np.ascontiguousarray(fanout,
                                                                                  dtype=np.int32)
    if len(F) != Kq:
        raise SSDError("fanout must have Kq entries")
    Fmax = max(1, int(F.max()) if len(F) else 1)
    o = out if out is not None else {}
    if "accept_len" not in o:
        o["accept_len"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["bonus"] = torch.empty(B, dtype=torch.int32, device=dev)
        if resid_mass:
            o["resid_mass"] = torch.empty(B, dtype=torch.float32, device=dev)
        if guesses:
            o["guesses"] = torch.empty((B, Kq, Fmax), dtype=torch.int32, device=dev)
            if guess_q:
                o["guess_q"] = torch.empty((B, Kq, Fmax), dtype=torch.float32, device=dev)
    L = lib()
    wsb = L.ssd_verify_workspace_size(B, K, Kq, V)
    if wsb == 0:
        raise SSDError("invalid verify shape")
    ws = workspace if workspace is not None else _workspace(wsb, dev)
    tl, dl = _logits(target), _logits(draft)
    if np.ndim(T) > 0:
        Tr = T if hasattr(T, "is_cuda") else torch.as_tensor(np.asarray(T, dtype=np.float32),
                                                              device=dev)
        if Tr.shape != (B,) or Tr.dtype != torch.float32 or not Tr.is_cuda:
            raise SSDError("per-sequence T must be float32 [B] on the device")
        Tr = Tr.contiguous()
        Cv = None if np.ndim(C) == 0 and float(C) == 1.0 else \
            np.ascontiguousarray(np.broadcast_to(np.asarray(C, dtype=np.float32), (K,)))
        st = L.ssd_verify_ex(ctypes.byref(tl), ctypes.byref(dl), B, K, Kq, V, _dev_ptr(Tr),
                             _dev_ptr(_i32(draft_tokens)), _dev_ptr(_u64_seeds(seeds, dev)),
                             int(round_) & 0xFFFFFFFF, F.ctypes.data_as(ctypes.c_void_p),
                             None if Cv is None else Cv.ctypes.data_as(ctypes.c_void_p),
                             _dev_ptr(o["accept_len"]), _dev_ptr(o["bonus"]),
                             _dev_ptr(o.get("resid_mass")), _dev_ptr(o.get("guesses")),
                             _dev_ptr(o.get("guess_q")), Fmax, _dev_ptr(ws), ws.numel(),
                             _dev_ptr(dev_status), _stream(stream))
        _check(st, "ssd_verify_ex")
        return o
    if np.ndim(C) == 0:
        fn, c_arg, name = L.ssd_verify, float(C), "ssd_verify"
    else:
        Cv = np.ascontiguousarray(C, dtype=np.float32)
        if Cv.shape != (K,):
            raise SSDError("C must be a scalar or have one entry per draft position")
        fn, c_arg, name = L.ssd_verify_ck, Cv.ctypes.data_as(ctypes.c_void_p), "ssd_verify_ck"
    st = fn(ctypes.byref(tl), ctypes.byref(dl), B, K, Kq, V, float(T),
            _dev_ptr(_i32(draft_tokens)), _dev_ptr(_u64_seeds(seeds, dev)),
            int(round_) & 0xFFFFFFFF, F.ctypes.data_as(ctypes.c_void_p), c_arg,
            _dev_ptr(o["accept_len"]), _dev_ptr(o["bonus"]),
            _dev_ptr(o.get("resid_mass")), _dev_ptr(o.get("guesses")),
            _dev_ptr(o.get("guess_q")), Fmax, _dev_ptr(ws), ws.numel(),
            _dev_ptr(dev_status), _stream(stream))
    _check(st, name)
    return o


def verify_round(target, draft, draft_tokens, seeds, round_, fanout, C=1.0, T=1.0,
                 guess_q=True, resid_mass=True, table=None, workspace=None, dev_status=None,
                 stream=None, out=None):
    """ssd_verify_round: verify, the round's outcome cache and its lookup in
    one launch.  Returns verify's outputs (guesses always) plus ``branch``
    [B] and ``all_hit`` [1] (device tensors) and the ``table`` used."""
    torch = _torch()
    B, K1, V = target.shape
    K = K1 - 1
    Kq = draft.shape[-2]
    dev = target.device
    F = np.ascontiguousarray(fanout, dtype=np.int32)
    if len(F) != Kq:
        raise SSDError("fanout must have Kq entries")
    Fmax = max(1, int(F.max()))
    o = out if out is not None else {}
    if "accept_len" not in o:
        o["accept_len"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["bonus"] = torch.empty(B, dtype=torch.int32, device=dev)
        if resid_mass:
            o["resid_mass"] = torch.empty(B, dtype=torch.float32, device=dev)
        o["guesses"] = torch.empty((B, Kq, Fmax), dtype=torch.int32, device=dev)
        if guess_q:
            o["guess_q"] = torch.empty((B, Kq, Fmax), dtype=torch.float32, device=dev)
        o["branch"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["all_hit"] = torch.empty(1, dtype=torch.int32, device=dev)
    if table is None:
        table = o.get("table")
    if table is None:
        table = torch.empty(cache_bytes(B * Kq * Fmax), dtype=torch.uint8, device=dev)
    o["table"] = table
    L = lib()
    wsb = L.ssd_verify_workspace_size(B, K, Kq, V)
    if wsb == 0:
        raise SSDError("invalid verify shape")
    ws = workspace if workspace is not None else _workspace(wsb, dev)
    tl, dl = _logits(target), _logits(draft)
    st = L.ssd_verify_round(ctypes.byref(tl), ctypes.byref(dl), B, K, Kq, V, float(T),
                            _dev_ptr(_i32(draft_tokens)), _dev_ptr(_u64_seeds(seeds, dev)),
                            int(round_) & 0xFFFFFFFF, F.ctypes.data_as(ctypes.c_void_p), float(C),
                            _dev_ptr(o["accept_len"]), _dev_ptr(o["bonus"]),
                            _dev_ptr(o.get("resid_mass")), _dev_ptr(o["guesses"]),
                            _dev_ptr(o.get("guess_q")), Fmax, _dev_ptr(table), table.numel(),
                            _dev_ptr(o["branch"]), _dev_ptr(o["all_hit"]), _dev_ptr(ws), ws.numel(),
                            _dev_ptr(dev_status), _stream(stream))
    _check(st, "ssd_verify_round")
    return o


def verify_skipped_bytes(workspace, target, K, Kq, stream=None):
    """ssd_verify_skipped_bytes: the bytes of target rows the last verify
    call on `workspace` (target [B, K+1, V]) did not read, as a Python int
    (synchronises the stream)."""
    torch = _torch()
    B, V = target.shape[0], target.shape[-1]
    dt = SSD_BF16 if target.dtype == torch.bfloat16 else SSD_F32
    out = torch.zeros(1, dtype=torch.int64, device=workspace.device)
    st = lib().ssd_verify_skipped_bytes(_dev_ptr(workspace), workspace.numel(), B, K, Kq, V, dt,
                                        _dev_ptr(out), _stream(stream))
    _check(st, "ssd_verify_skipped_bytes")
    return int(out.item())


def verify_host(target, draft, draft_tokens, seeds, round_, fanout=None, C=1.0, T=1.0,
                device="cuda", guesses=True, workspace=None, dev_buffers=None):
    """End-to-end call with HOST tensors: copies the inputs to the GPU, runs
    ssd_verify and copies the results back (pinned host memory makes the
    copies asynchronous).  Returns a dict of CPU tensors."""
    torch = _torch()
    db = dev_buffers if dev_buffers is not None else {}
    for name, t in (("target", target), ("draft", draft), ("tokens", draft_tokens),
                    ("seeds", seeds)):
        if name not in db:
            db[name] = torch.empty(t.shape, dtype=t.dtype, device=device)
        db[name].copy_(t, non_blocking=True)
    o = verify(db["target"], db["draft"], db["tokens"], db["seeds"], round_, fanout, C, T,
               guesses=guesses, workspace=workspace, out=db.get("out"))
    db["out"] = o
    host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True) for k, v in o.items()}
    for k, v in o.items():
        host[k].copy_(v, non_blocking=True)
    torch.cuda.current_stream().synchronize()
    return host


def topf_bonus(draft, fanout, T=1.0, draft_tokens=None, K=None, Fmax=None, guess_q=True,
               workspace=None, dev_status=None, stream=None):
    """ssd_topf_bonus: guesses [B, Kq, Fmax] (+ guess_q) for draft [B, Kq, V]."""
    torch = _torch()
    B, Kq, V = draft.shape
    dev = draft.device
    F = np.ascontiguousarray(fanout, dtype=np.int32)
    Fmax = max(1, int(F.max())) if Fmax is None else int(Fmax)
    g = torch.empty((B, Kq, Fmax), dtype=torch.int32, device=dev)
    gq = torch.empty((B, Kq, Fmax), dtype=torch.float32, device=dev) if guess_q else None
    L = lib()
    ws = workspace if workspace is not None else _workspace(L.ssd_topf_workspace_size(B, Kq, V),
                                                            dev)
    Kt = 0 if draft_tokens is None else (draft_tokens.shape[-1] if K is None else int(K))
    dl = _logits(draft)
    st = L.ssd_topf_bonus(ctypes.byref(dl), B, Kq, V, float(T),
                          _dev_ptr(None if draft_tokens is None else _i32(draft_tokens)), Kt,
                          F.ctypes.data_as(ctypes.c_void_p), Fmax, _dev_ptr(g), _dev_ptr(gq),
                          _dev_ptr(ws), ws.numel(), _dev_ptr(dev_status), _stream(stream))
    _check(st, "ssd_topf_bonus")
    return {"guesses": g, "guess_q": gq}


def saguaro_sample(rows, T, C, F, seeds, j, round_, guesses=True, qprime=True, workspace=None,
                   dev_status=None, stream=None, out=None, Fmax=None):
    """ssd_saguaro_sample over branch rows [R, V]: token, qprime, guesses.

    F: one fan-out for every row (an int), or one per row -- a device int32
    tensor [R] (then Fmax, the largest, must be given) or anything numpy
    reads (uploaded here).  guesses are [R, Fmax], -1 padded."""
    torch = _torch()
    R, V = rows.shape[-2], rows.shape[-1]
    dev = rows.device
    F_row = None
    if np.ndim(F) == 0 and not hasattr(F, "is_cuda"):
        Fm = int(F)
    elif hasattr(F, "is_cuda"):
        if Fmax is None:
            raise SSDError("a device F tensor needs Fmax")
        F_row, Fm = _i32(F), int(Fmax)
    else:
        Fa = np.ascontiguousarray(F, dtype=np.int32)
        if Fa.shape != (R,):
            raise SSDError("per-row F must have R entries")
        Fm = int(Fa.max()) if Fmax is None else int(Fmax)
        F_row = torch.from_numpy(Fa).to(dev)
    if F_row is not None and F_row.shape != (R,):
        raise SSDError("per-row F must have R entries")
    o = out if out is not None else {}
    if "token" not in o:
        o["token"] = torch.empty(R, dtype=torch.int32, device=dev)
        if qprime:
            o["qprime"] = torch.empty(R, dtype=torch.float32, device=dev)
        if guesses and Fm > 0:
            o["guesses"] = torch.empty((R, Fm), dtype=torch.int32, device=dev)
    L = lib()
    ws = workspace if workspace is not None else _workspace(L.ssd_saguaro_workspace_size(R, V),
                                                            dev)
    rl = _logits(rows)
    st = L.ssd_saguaro_sample(ctypes.byref(rl), R, V, float(T), float(C), _dev_ptr(F_row), Fm,
                              _dev_ptr(_u64_seeds(seeds, dev)), int(j),
                              int(round_) & 0xFFFFFFFF, _dev_ptr(o["token"]),
                              _dev_ptr(o.get("qprime")), _dev_ptr(o.get("guesses")),
                              _dev_ptr(ws), ws.numel(), _dev_ptr(dev_status), _stream(stream))
    _check(st, "ssd_saguaro_sample")
    return o


def tree_verify(target, draft, parent, tokens, seeds, round_, T=1.0, workspace=None,
                dev_status=None, stream=None, out=None):
    """ssd_tree_verify: target, draft [B, N, V] (row u of a tree: p_u / q_u at
    node u), parent: N ints (parent[0] = -1, parent[u] < u), tokens int32
    [B, N] on the device.  Returns accept_len [B], path [B, depth], bonus
    [B] and resid_mass [B] (device tensors)."""
    torch = _torch()
    B, N, V = target.shape
    dev = target.device
    par = np.ascontiguousarray(parent, dtype=np.int32)
    if par.shape != (N,):
        raise SSDError("parent must have N entries")
    depth = np.zeros(N, dtype=np.int64)
    for u in range(1, N):
        if not 0 <= par[u] < u:
            raise SSDError("parent[u] must lie in [0, u)")
        depth[u] = depth[par[u]] + 1
    Dmax = max(1, int(depth.max()))
    o = out if out is not None else {}
    if "accept_len" not in o:
        o["accept_len"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["path"] = torch.empty((B, Dmax), dtype=torch.int32, device=dev)
        o["bonus"] = torch.empty(B, dtype=torch.int32, device=dev)
        o["resid_mass"] = torch.empty(B, dtype=torch.float32, device=dev)
    L = lib()
    wsb = L.ssd_tree_workspace_size(B, N, V)
    if wsb == 0:
        raise SSDError("invalid tree shape")
    ws = workspace if workspace is not None else _workspace(wsb, dev)
    tl, dl = _logits(target), _logits(draft)
    st = L.ssd_tree_verify(ctypes.byref(tl), ctypes.byref(dl), B, N, V, float(T),
                           par.ctypes.data_as(ctypes.c_void_p), _dev_ptr(_i32(tokens)),
                           _dev_ptr(_u64_seeds(seeds, dev)), int(round_) & 0xFFFFFFFF,
                           _dev_ptr(o["accept_len"]), _dev_ptr(o["path"]), Dmax,
                           _dev_ptr(o["bonus"]), _dev_ptr(o["resid_mass"]), _dev_ptr(ws),
                           ws.numel(), _dev_ptr(dev_status), _stream(stream))
    _check(st, "ssd_tree_verify")
    return o


def cache_bytes(n_keys: int) -> int:
    return int(lib().ssd_cache_bytes(int(n_keys)))


def cache_build(row, k, t, branch, table=None, dev_status=None, stream=None):
    torch = _torch()
    n = row.numel()
    if table is None:
        table = torch.empty(cache_bytes(n), dtype=torch.uint8, device=row.device)
    st = lib().ssd_cache_build(_dev_ptr(table), table.numel(), _dev_ptr(_i32(row)),
                               _dev_ptr(_i32(k)), _dev_ptr(_i32(t)), _dev_ptr(_i32(branch)), n,
                               _dev_ptr(dev_status), _stream(stream))
    _check(st, "ssd_cache_build")
    return table


def cache_build_guesses(guesses, table=None, dev_status=None, stream=None):
    torch = _torch()
    B, Kq, Fmax = guesses.shape
    if table is None:
        table = torch.empty(cache_bytes(B * Kq * Fmax), dtype=torch.uint8, device=guesses.device)
    st = lib().ssd_cache_build_guesses(_dev_ptr(table), table.numel(), _dev_ptr(_i32(guesses)),
                                       B, Kq, Fmax, _dev_ptr(dev_status), _stream(stream))
    _check(st, "ssd_cache_build_guesses")
    return table


def cache_lookup(table, accept_len, bonus, out=None, stream=None):
    torch = _torch()
    B = accept_len.numel()
    o = out if out is not None else {
        "branch": torch.empty(B, dtype=torch.int32, device=accept_len.device),
        "all_hit": torch.empty(1, dtype=torch.int32, device=accept_len.device)}
    st = lib().ssd_cache_lookup(_dev_ptr(table), table.numel(), _dev_ptr(_i32(accept_len)),
                                _dev_ptr(_i32(bonus)), B, _dev_ptr(o["branch"]),
                                _dev_ptr(o["all_hit"]), _stream(stream))
    _check(st, "ssd_cache_lookup")
    return o


def fanout(K: int, budget: int, a: float = 0.7, r: float = 1.0) -> np.ndarray:
    """Geometric fan-out F_0..F_K (host helper of the library)."""
    F = np.zeros(K + 1, dtype=np.int32)
    _check(lib().ssd_fanout(int(K), int(budget), float(a), float(r),
                            F.ctypes.data_as(ctypes.c_void_p)), "ssd_fanout")
    return F
