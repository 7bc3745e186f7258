"""Workload definitions and logit generators.

Generator "G" (Llama-3 / Qwen-3 sized vocabularies):
  per sequence b, a random permutation pi_b of the vocabulary; for target
  position i the logit of token pi_b(r-1) (rank r = 1..V) is
  ``-zipf * ln(r) + gumbel_scale * Gumbel(0,1)`` with a fresh Gumbel draw per
  (b, i, token), so the head is Zipf-sorted over a random vocab permutation;
  the draft row j is the target row j plus N(0, sigma_b^2) noise.
Generator "gauss" (the tiny exactness case): target ~ N(0, 2^2), draft =
  target + N(0, 1^2).

The vocabularies (128256, 151936), draft lengths K = 4..8, batch sizes 1..256
and the SSD two-level batch (outer batch x 12 branches) follow the workloads
the pages describe ([SSD-note] §"实现细节：缓存怎么建" / "两层 batch";
[SD-blog] §"四、三个工程坑" for K = 4..8).  Logits are produced in fp32 and,
for bf16 workloads, rounded to bf16 (round-to-nearest-even); both sides read
the same stored bytes.
"""

from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import os

import numpy as np


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    K: int
    V: int
    dtype: str            # "f32" | "bf16"
    T: float
    budget: int           # fan-out budget (sum of F over the K+1 positions)
    fanout: tuple         # F_0..F_K
    C: float              # Saguaro factor (1.0 = plain speculative decoding)
    gen: str              # "gauss" | "G"
    zipf: float = 1.1
    gumbel_scale: float = 0.5
    sigma: float = 0.8            # draft noise std
    sigma_range: tuple | None = None  # per-row U[lo, hi] noise std
    seed: int = 1000
    branches: int = 0     # SSD cache build: branch rows per outer row
    cont_positions: int = 0

    @property
    def Kq(self) -> int:
        # draft rows per sequence: K verified positions plus row K whose
        # distribution supplies the bonus guesses for the all-accepted outcome
        return self.K + 1

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def algorithmic_bytes(self, B: int | None = None) -> int:
        """One read of every target and draft logit of the verify call."""
        B = self.B if B is None else B
        return B * (self.K + 1 + self.Kq) * self.V * self.elem_bytes


# Fan-out vectors are the geometric allocation F_k ~ a^(k/(1+r)) with a=0.7,
# r=1, integerised by largest remainder (computed by the library's host helper
# and by the oracle; the values are restated here only as workload constants).
WORKLOADS = {
    "c1": Workload("tiny-exactness B=1 K=4 V=32 f32", B=1, K=4, V=32, dtype="f32", T=1.0,
                   budget=12, fanout=(3, 3, 2, 2, 2), C=0.5, gen="gauss", seed=1001),
    "c2": Workload("single-stream B=1 K=4 V=128256 bf16", B=1, K=4, V=128256, dtype="bf16",
                   T=0.7, budget=12, fanout=(3, 3, 2, 2, 2), C=0.5, gen="G", zipf=1.1,
                   sigma=0.8, seed=1002),
    "c3": Workload("batched B=64 K=8 V=128256 bf16", B=64, K=8, V=128256, dtype="bf16",
                   T=1.0, budget=16, fanout=(3, 3, 2, 2, 2, 1, 1, 1, 1), C=1.0, gen="G",
                   zipf=1.1, sigma_range=(0.3, 1.5), seed=1003),
    "c4": Workload("ssd-cache-build 32x12 K=4 V=151936 bf16", B=32, K=4, V=151936,
                   dtype="bf16", T=1.0, budget=12, fanout=(3, 3, 2, 2, 2), C=0.3, gen="G",
                   zipf=1.1, sigma=0.8, seed=1004, branches=12, cont_positions=4),
    "c5": Workload("large-batch B=256 K=8 V=151936 f32", B=256, K=8, V=151936, dtype="f32",
                   T=1.0, budget=24, fanout=(5, 4, 4, 3, 2, 2, 2, 1, 1), C=0.5, gen="G",
                   zipf=1.05, sigma=1.2, seed=1005),
}


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest even."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return ((u >> 16) & 0xFFFF).astype(np.uint16)


def bf16_to_f32(h: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> fp32 (exact)."""
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, b: int, stream: int = 0) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(key=(int(seed) << 64) | (int(stream) << 32) | int(b)))


def _gumbel_f32(rng: np.random.Generator, n: int) -> np.ndarray:
    u = rng.random(n, dtype=np.float32)
    u = np.clip(u, np.float32(2.0 ** -25), np.float32(1.0 - 2.0 ** -24))
    return -np.log(-np.log(u))


def sequence_logits(w: Workload, b: int, V: int | None = None, K: int | None = None,
                    seed: int | None = None):
    """fp32 logits of sequence b: (target [K+1, V], draft [K+1, V], sigma_b)."""
    V = w.V if V is None else V
    K = w.K if K is None else K
    seed = w.seed if seed is None else seed
    rng = _rng(seed, b)
    if w.sigma_range is not None:
        sigma = float(rng.uniform(w.sigma_range[0], w.sigma_range[1]))
    else:
        sigma = float(w.sigma)
    zp = np.empty((K + 1, V), dtype=np.float32)
    zq = np.empty((K + 1, V), dtype=np.float32)
    if w.gen == "gauss":
        for i in range(K + 1):
            zp[i] = rng.standard_normal(V, dtype=np.float32) * np.float32(2.0)
            zq[i] = zp[i] + rng.standard_normal(V, dtype=np.float32) * np.float32(1.0)
    elif w.gen == "G":
        perm = rng.permutation(V)
        base = np.empty(V, dtype=np.float32)
        base[perm] = (-w.zipf * np.log(np.arange(1, V + 1, dtype=np.float64))).astype(np.float32)
        for i in range(K + 1):
            zp[i] = base + np.float32(w.gumbel_scale) * _gumbel_f32(rng, V)
            zq[i] = zp[i] + rng.standard_normal(V, dtype=np.float32) * np.float32(sigma)
    else:
        raise ValueError(w.gen)
    return zp, zq, sigma


def _seq_bytes(w, b, V, K, seed, dtype):
    zp, zq, _ = sequence_logits(w, b, V=V, K=K, seed=seed)
    if dtype == "bf16":
        return bf16_bits(zp), bf16_bits(zq)
    return zp, zq


def make_batch(w: Workload, B: int | None = None, V: int | None = None, K: int | None = None,
               seed: int | None = None, dtype: str | None = None, rows=None,
               threads: int | None = None):
    """Generate a batch.

    Returns dict with ``target`` [B, K+1, V] and ``draft`` [B, K+1, V] (uint16
    bf16 bits or float32), ``seeds`` [B] uint64 (per-row Philox keys for the
    method's uniforms), and the workload scalars.  ``rows`` restricts the
    generation to a subset of sequence indices (the returned arrays then hold
    those rows only, in the given order).
    """
    B = w.B if B is None else B
    V = w.V if V is None else V
    K = w.K if K is None else K
    seed = w.seed if seed is None else seed
    dtype = w.dtype if dtype is None else dtype
    idx = list(range(B)) if rows is None else [int(r) for r in rows]
    npdt = np.uint16 if dtype == "bf16" else np.float32
    target = np.empty((len(idx), K + 1, V), dtype=npdt)
    draft = np.empty((len(idx), K + 1, V), dtype=npdt)
    nthr = threads or min(16, os.cpu_count() or 1)

    def work(n):
        t, d = _seq_bytes(w, idx[n], V, K, seed, dtype)
        target[n] = t
        draft[n] = d

    if nthr > 1 and len(idx) > 1:
        with _cf.ThreadPoolExecutor(nthr) as ex:
            list(ex.map(work, range(len(idx))))
    else:
        for n in range(len(idx)):
            work(n)
    seeds = row_seeds(seed, idx)
    return dict(target=target, draft=draft, seeds=seeds, rows=np.asarray(idx, dtype=np.int64),
                B=len(idx), K=K, Kq=K + 1, V=V, dtype=dtype, T=w.T, C=w.C,
                fanout=np.asarray(w.fanout, dtype=np.int32))


def row_seeds(seed: int, rows) -> np.ndarray:
    """Per-sequence 64-bit Philox keys for the method's uniforms."""
    out = np.empty(len(rows), dtype=np.uint64)
    for n, b in enumerate(rows):
        out[n] = _rng(seed, int(b), stream=7).integers(0, 2 ** 63, dtype=np.uint64)
    return out
