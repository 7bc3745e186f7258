"""Fan-out ablation: geometric against uniform allocation of the bonus guesses.

[SSD-note] "论文阅读：Speculative Speculative Decoding — 消除推测解码的最后一个顺序瓶颈"
§"最优扇出度分配" derives the geometric allocation F_k ~ a^(k/(1+r)) of a guess
budget over the K+1 verification outcomes, and §"消融实验" reports that it
beats a uniform allocation, most clearly at high temperature.  This module
measures that comparison on synthetic rounds with the library's own calls:
every round draws the drafts with ``saguaro_sample`` (one call per draft
position), verifies them with ``verify`` (which also returns the top-F
guesses of every position), builds the outcome cache from the guesses and
probes it with the round's outcome (k, t).  A row hits when its outcome was
guessed.

Everything runs on the GPU through the C ABI; the inputs are the seeded
synthetic workloads of ``ssd_inputs``.
"""

from __future__ import annotations

import dataclasses

import numpy as np

from . import cache_build_guesses, cache_bytes, cache_lookup, fanout, saguaro_sample, verify


def uniform_fanout(K: int, budget: int) -> np.ndarray:
    """The budget spread evenly over the K+1 outcomes, the remainder to the
    lowest positions (the same integerisation rule as the geometric one)."""
    F = np.full(K + 1, budget // (K + 1), dtype=np.int32)
    F[: budget - int(F.sum())] += 1
    return F


def _upload(bt, w, device):
    import torch

    if w.dtype == "bf16":
        tg = torch.from_numpy(bt["target"].view(np.int16)).to(device).view(torch.bfloat16)
        dg = torch.from_numpy(bt["draft"].view(np.int16)).to(device).view(torch.bfloat16)
    else:
        tg = torch.from_numpy(bt["target"]).to(device)
        dg = torch.from_numpy(bt["draft"]).to(device)
    seeds = torch.from_numpy(bt["seeds"].view(np.int64)).to(device)
    return tg, dg, seeds


def _round_on_device(tg, dg, seeds, K, F, C, T, rnd, device):
    """Drafts x_j ~ q'_j (Saguaro sampling), verification with the guesses of
    every position, the outcome cache of the guesses and its lookup."""
    import torch

    F = np.asarray(F, dtype=np.int32)
    Cv = np.broadcast_to(np.asarray(C, dtype=np.float32), (K,))
    B = tg.shape[0]
    tok = torch.empty((B, K), dtype=torch.int32, device=device)
    for j in range(K):
        tok[:, j] = saguaro_sample(dg[:, j, :], T, float(Cv[j]), int(F[j]), seeds, j, rnd,
                                   guesses=False, qprime=False)["token"]
    out = verify(tg, dg, tok.contiguous(), seeds, rnd, F, C if np.ndim(C) else float(C), T,
                 guess_q=False)
    table = torch.empty(cache_bytes(out["guesses"].numel()), dtype=torch.uint8, device=device)
    cache_build_guesses(out["guesses"], table=table)
    look = cache_lookup(table, out["accept_len"], out["bonus"])
    return tok, out, look


def round_hits(workload, F, C, T, seed, rnd, device="cuda"):
    """One synthetic round of B sequences: drafts x_j ~ q'_j, verification,
    cache of every position's guesses, lookup of (k, t).  Returns the host
    arrays accept_len, bonus, hit (bool per row) and the device outputs."""
    from ssd_inputs import make_batch

    w = workload
    bt = make_batch(w, seed=seed)
    tg, dg, seeds = _upload(bt, w, device)
    tok, out, look = _round_on_device(tg, dg, seeds, w.K, F, C, T, rnd, device)
    return dict(accept_len=out["accept_len"].cpu().numpy(), bonus=out["bonus"].cpu().numpy(),
                hit=look["branch"].cpu().numpy() >= 0, tokens=tok.cpu().numpy(),
                guesses=out["guesses"].cpu().numpy(), batch=bt)


def wilson(h, n, z=1.96):
    """Wilson score interval of a binomial proportion h / n."""
    if n == 0:
        return (0.0, 1.0)
    p = h / n
    d = 1 + z * z / n
    c = (p + z * z / (2 * n)) / d
    r = z * np.sqrt(p * (1 - p) / n + z * z / (4 * n * n)) / d
    return (max(0.0, c - r), min(1.0, c + r))


def fanout_ablation(workload, temperatures, budget, Cs=(1.0,), rounds=64, a=0.7, r=1.0,
                    B=None, V=None, seed=2024, device="cuda"):
    """Hit rate of the geometric allocation (a, r) and of the uniform one for
    every (C, T), over `rounds` seeded rounds of B sequences each.  Each
    round's logits are generated once and shared by every (C, T) and both
    allocations, so the two arms are compared on the same sequences and
    uniforms (paired).  Returns a list of dicts: C, T, F_geometric,
    F_uniform, hit_geometric, hit_uniform (with 95% Wilson intervals),
    diff = hit_geometric - hit_uniform with a 95% interval of the paired
    per-row differences, rows, accept_mean (geometric arm)."""
    from ssd_inputs import make_batch

    w = dataclasses.replace(workload, B=B or workload.B, V=V or workload.V)
    Fg = fanout(w.K, budget, a, r)
    Fu = uniform_fanout(w.K, budget)
    cells = {(C, T): {"geometric": [], "uniform": [], "acc": []} for C in Cs for T in temperatures}
    for i in range(rounds):
        bt = make_batch(w, seed=seed + i)
        tg, dg, seeds = _upload(bt, w, device)
        for C in Cs:
            for T in temperatures:
                cell = cells[(C, T)]
                for name, F in (("geometric", Fg), ("uniform", Fu)):
                    _, out, look = _round_on_device(tg, dg, seeds, w.K, F, C, float(T), i,
                                                    device)
                    cell[name].append(look["branch"].cpu().numpy() >= 0)
                    if name == "geometric":
                        cell["acc"].append(out["accept_len"].cpu().numpy())
    rows = []
    for (C, T), cell in cells.items():
        hg = np.concatenate(cell["geometric"])
        hu = np.concatenate(cell["uniform"])
        n = len(hg)
        d = hg.astype(np.float64) - hu.astype(np.float64)
        half = 1.96 * d.std(ddof=1) / np.sqrt(n) if n > 1 else 1.0
        rows.append(dict(C=float(C), T=float(T), F_geometric=Fg.tolist(), F_uniform=Fu.tolist(),
                         rows=n, hit_geometric=float(hg.mean()),
                         hit_geometric_ci=wilson(int(hg.sum()), n),
                         hit_uniform=float(hu.mean()), hit_uniform_ci=wilson(int(hu.sum()), n),
                         diff=float(d.mean()), diff_ci=(float(d.mean() - half),
                                                        float(d.mean() + half)),
                         accept_mean=float(np.concatenate(cell["acc"]).mean())))
    return rows
