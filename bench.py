#!/usr/bin/env python
"""Benchmark of the speculative-decoding verification round on GB300.

One step = one SSD verification round over one batch of synthetic logits
already resident in HBM:
  ssd_verify (online-softmax normalisers, fused top-F bonus guesses,
  Saguaro-biased q', accept test, residual bonus draw)
  -> ssd_cache_build_guesses (outcome cache from the guesses)
  -> ssd_cache_lookup (hit / all-rows-hit of the verified outcomes).

Default workload: large-batch stress, B=256, K=8, V=151936, fp32 logits,
Zipf(1.05) head, draft = target + N(0, 1.2^2), T=1, fan-out budget 24
(F = 5,4,4,3,2,2,2,1,1), C=0.5, cache of 256 x 24 keys.  The logits
(2.80 GB) are larger than L2 (no flush needed).

`--impl reference` times the CPU oracle on a bounded sample of the same
workload on the host cores.  Under torchrun each rank runs its own batch
(weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified rows/sec and logits GB/s (fraction of GB300 HBM peak) at V=128k-152k"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def csrc_hash():
    d = os.path.join(ROOT, "sampling_ssd_verify_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(d)):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def verify_roofline(alg, skipped, launch_ms, launch_ms_median, hbm_peak, peak_kind, traffic):
    """The roofline block of a verify round: `achieved` counts every logit once
    (the algorithmic bytes) over the mean launch time; the bytes the round
    actually streams (every logit minus the `skipped` target rows past a known
    rejection) and their rate go beside it."""
    read = alg - skipped
    achieved = alg / (launch_ms * 1e-3) / 1e9
    read_rate = read / (launch_ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
            "frac": achieved / hbm_peak, "traffic": traffic,
            "kernel": "ssd_verify_round (streaming pass, bonus draws, outcome cache)",
            "algorithmic_bytes_per_launch": alg,
            "bytes_read_per_launch": read,
            "skipped_target_bytes_per_launch": skipped,
            "gb_per_s_on_bytes_read": read_rate,
            "frac_on_bytes_read": read_rate / hbm_peak,
            "launch_ms": launch_ms,
            "launch_ms_median": launch_ms_median, "peak_kind": peak_kind}


def traffic_from_profile(workload):
    """Per-launch DRAM bytes recorded by an ncu capture, if the kernels have
    not changed since (profiles/<...>.md carries 'csrc_sha: <hash>' and
    'traffic_bytes_per_launch[<workload>]: <n>')."""
    pd = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pd):
        return None
    want = csrc_hash()
    for f in sorted(os.listdir(pd)):
        if not f.endswith(".md"):
            continue
        txt = open(os.path.join(pd, f)).read()
        if f"csrc_sha: {want}" not in txt:
            continue
        key = f"traffic_bytes_per_launch[{workload}]:"
        for line in txt.splitlines():
            if line.strip().startswith(key):
                return float(line.split(":", 1)[1].strip())
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)),
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# Multi-GPU runs are replicas: every rank verifies its own batch (independent
# sequences, so the path has no data exchange), the step time is the slowest
# rank's, and the throughput counts every rank's rows (weak scaling).
def rank_seed(w, rank):
    """Seed of rank `rank`'s synthetic batch (distinct per rank)."""
    return w.seed + 7919 * rank


def max_over_ranks(x, tdist, device=None):
    """The maximum of a per-rank float over all ranks (x itself on one rank)."""
    import torch
    if not (tdist.is_available() and tdist.is_initialized()) or tdist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    tdist.all_reduce(t, op=tdist.ReduceOp.MAX)
    return float(t.item())


def job_rows_per_s(rows_per_rank, world, seconds):
    """Whole-job throughput: rows verified by all ranks per second."""
    return rows_per_rank * world / seconds


# ------------------------------------------------------------------------------ ours
def bt_rows(bb, w):
    """The [R, V] branch logits of a K = 0 batch (uint16 bf16 bits or f32)."""
    rows = bb["target"][:, 0, :]
    return rows.view(np.int16) if w.dtype == "bf16" else rows


def side_workload(name, steps, warmup, rank, dev, tdist):
    """A further workload measured in the same process, after the headline
    one: its verify_round launches timed one by one with CUDA events (inputs
    resident), with their own roofline.  Inputs smaller than L2 (129 MB) are
    evicted before every launch by writing a 256 MB buffer, outside the
    launch's events; the step time is then the sum of the launches."""
    import torch

    import sampling_ssd_verify_gb300 as ssd
    from ssd_inputs import WORKLOADS, make_batch

    w = WORKLOADS[name]
    B, K, Kq, V = w.B, w.K, w.Kq, w.V
    F = np.asarray(w.fanout, dtype=np.int32)
    bt = make_batch(w, seed=rank_seed(w, rank))
    if w.dtype == "bf16":
        tg = torch.from_numpy(bt["target"].view(np.int16)).to(dev).view(torch.bfloat16)
        dg = torch.from_numpy(bt["draft"].view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        tg = torch.from_numpy(bt["target"]).to(dev)
        dg = torch.from_numpy(bt["draft"]).to(dev)
    seeds = torch.from_numpy(bt["seeds"].view(np.int64)).to(dev)
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    for j in range(K):
        tok[:, j] = ssd.saguaro_sample(dg[:, j, :], w.T, w.C, int(F[j]), seeds, j, 0,
                                       guesses=False, qprime=False)["token"]
    tok = tok.contiguous()
    ws = torch.empty(ssd.lib().ssd_verify_workspace_size(B, K, Kq, V), dtype=torch.uint8,
                     device=dev)
    table = torch.empty(ssd.cache_bytes(B * Kq * int(F.max())), dtype=torch.uint8, device=dev)
    out = {}
    alg = w.algorithmic_bytes()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev) if alg <= 129e6 else None
    stream = torch.cuda.current_stream()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(steps)]
    for s in range(warmup):
        ssd.verify_round(tg, dg, tok, seeds, 1 + s, F, w.C, w.T, table=table, workspace=ws, out=out)
    torch.cuda.synchronize()
    if tdist.is_available() and tdist.is_initialized():
        tdist.barrier()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    for s in range(steps):
        if flush is not None:
            flush.fill_(s & 0xFF)
        evs[s][0].record(stream)
        ssd.verify_round(tg, dg, tok, seeds, 1000 + s, F, w.C, w.T, table=table, workspace=ws,
                         out=out)
        evs[s][1].record(stream)
    t1.record(stream)
    torch.cuda.synchronize()
    launch = [a.elapsed_time(b) for a, b in evs]
    ms = max_over_ranks(t0.elapsed_time(t1) if flush is None else float(np.sum(launch)), tdist,
                        dev)
    # bytes of target rows past a known rejection, not read (untimed rounds)
    ns, skipped = 20, 0
    for s in range(ns):
        ssd.verify_round(tg, dg, tok, seeds, 5000 + s, F, w.C, w.T, table=table, workspace=ws,
                         out=out)
        skipped += ssd.verify_skipped_bytes(ws, tg, K, Kq)
    hbm_peak, peak_kind = peaks()
    world = tdist.get_world_size() if tdist.is_available() and tdist.is_initialized() else 1
    return {"workload": w.name, "B": B, "K": K, "Kq": Kq, "V": V, "dtype": w.dtype, "T": w.T,
            "C": w.C, "fanout": list(map(int, F)), "steps": steps, "warmup": warmup,
            "value": job_rows_per_s(B * steps, world, ms * 1e-3), "unit": "rows/s",
            "ms_per_step": ms / steps,
            "accept_mean": float(out["accept_len"].float().mean().item()),
            "roofline": verify_roofline(alg, skipped / ns, float(np.mean(launch)),
                                        float(np.median(launch)), hbm_peak, peak_kind,
                                        traffic_from_profile(name)),
            "l2": "inputs larger than L2 (no flush)" if flush is None else
                  "inputs smaller than L2: a 256 MB write before each launch, outside its events"}


def run_ours(args):
    import torch
    import torch.distributed as tdist

    import sampling_ssd_verify_gb300 as ssd
    from ssd_inputs import WORKLOADS, make_batch

    world, rank, local = dist_env()
    if world > 1:
        tdist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ssd.build()
    w = WORKLOADS[args.workload]
    if args.batch or args.vocab:
        w = dataclasses.replace(w, B=args.batch or w.B, V=args.vocab or w.V,
                                name=f"{w.name} [B={args.batch or w.B}, V={args.vocab or w.V}]")
    B, K, Kq, V = w.B, w.K, w.Kq, w.V
    F = np.asarray(w.fanout, dtype=np.int32)
    bt = make_batch(w, seed=rank_seed(w, rank))
    if w.dtype == "bf16":
        tg = torch.from_numpy(bt["target"].view(np.int16)).to(dev).view(torch.bfloat16)
        dg = torch.from_numpy(bt["draft"].view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        tg = torch.from_numpy(bt["target"]).to(dev)
        dg = torch.from_numpy(bt["draft"]).to(dev)
    seeds = torch.from_numpy(bt["seeds"].view(np.int64)).to(dev)
    # drafts x_j ~ q'_j from the library's Saguaro sampler (one call per position)
    tok = torch.empty((B, K), dtype=torch.int32, device=dev)
    for j in range(K):
        tok[:, j] = ssd.saguaro_sample(dg[:, j, :], w.T, w.C, int(F[j]), seeds, j, 0,
                                       guesses=False, qprime=False)["token"]
    tok = tok.contiguous()
    ws = torch.empty(ssd.lib().ssd_verify_workspace_size(B, K, Kq, V), dtype=torch.uint8,
                     device=dev)
    table = torch.empty(ssd.cache_bytes(B * Kq * int(F.max())), dtype=torch.uint8, device=dev)
    out = {}
    stream = torch.cuda.current_stream()
    ev_v = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)]

    # The SSD cache-build workload adds the drafter's side of the round: every
    # outer row's branches draw their next continuation token with Saguaro
    # sampling, one call per continuation position over fresh branch logits.
    branch = []
    if w.branches:
        R = B * w.branches
        for j in range(w.cont_positions):
            bb = make_batch(w, B=R, K=0, seed=w.seed + 100 + j)
            rows = torch.from_numpy(np.ascontiguousarray(bt_rows(bb, w))).to(dev)
            if w.dtype == "bf16":
                rows = rows.view(torch.bfloat16)
            bs = torch.from_numpy(bb["seeds"].view(np.int64)).to(dev)
            bws = torch.empty(ssd.lib().ssd_saguaro_workspace_size(R, V), dtype=torch.uint8,
                              device=dev)
            branch.append((rows, bs, int(F[j]), {}, bws))
    ev_s = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
            for _ in range(args.steps)] if branch else None

    def step(r, evs=None, evs_s=None):
        # one SSD round in one launch: verify, the outcome cache of the guesses
        # and the lookup of every sequence's outcome
        if evs is not None:
            evs[0].record(stream)
        ssd.verify_round(tg, dg, tok, seeds, r, F, w.C, w.T, table=table, workspace=ws, out=out)
        if evs is not None:
            evs[1].record(stream)
        if branch:
            if evs_s is not None:
                evs_s[0].record(stream)
            for j, (rows, bs, Fj, so, bws) in enumerate(branch):
                ssd.saguaro_sample(rows, w.T, w.C, Fj, bs, j, r, out=so, workspace=bws)
            if evs_s is not None:
                evs_s[1].record(stream)

    look = out

    for s in range(args.warmup):
        step(1 + s)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        tdist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    wall0 = time.perf_counter()
    t0.record(stream)
    for s in range(args.steps):
        step(1000 + s, ev_v[s], ev_s[s] if ev_s else None)
    t1.record(stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        tdist.barrier()
    ck = clocks.stop()
    ms = max_over_ranks(t0.elapsed_time(t1), tdist, dev)
    ms_step = ms / args.steps
    vts = [a.elapsed_time(b) for a, b in ev_v]
    verify_ms = float(np.mean(vts))
    verify_ms_median = float(np.median(vts))
    alg = w.algorithmic_bytes()
    hbm_peak, peak_kind = peaks()
    saguaro = None
    alg_step = alg
    if branch:
        s_ms = float(np.mean([a.elapsed_time(b) for a, b in ev_s])) / len(branch)
        s_alg = B * w.branches * V * w.elem_bytes
        alg_step = alg + len(branch) * s_alg
        saguaro = {"calls_per_step": len(branch), "rows": B * w.branches, "ms_per_call": s_ms,
                   "algorithmic_bytes_per_call": s_alg,
                   "gb_per_s": s_alg / (s_ms * 1e-3) / 1e9,
                   "frac": s_alg / (s_ms * 1e-3) / 1e9 / hbm_peak}

    # round statistics (untimed): acceptance, cache hit rate, all-rows-hit fraction
    # alpha: accepted over attempted draft positions (a row that stops at n < K
    # attempted n+1 of them); tail: the bonus draw's re-read, 2 rows (p and q')
    # after a rejection, 1 row (p_K) after a full acceptance
    acc_sum, hits, all_hits, nr = 0.0, 0, 0, 100
    att_sum, tail_rows, skipped = 0, 0, 0
    for r in range(nr):
        step(50_000 + r)
        skipped += ssd.verify_skipped_bytes(ws, tg, K, Kq)
        al = out["accept_len"].cpu().numpy().astype(np.int64)
        acc_sum += float(al.mean())
        att_sum += int(np.minimum(al + 1, K).sum())
        tail_rows += int(np.where(al < K, 2, 1).sum())
        hits += int((look["branch"] >= 0).sum().item())
        all_hits += int(look["all_hit"].item())
    h = hits / (nr * B)
    alpha = acc_sum * B / max(att_sum, 1)
    tail_bytes = tail_rows / nr * V * w.elem_bytes
    # target rows past a known rejection are not read: the round streams the
    # logits minus those (measured on the same rounds); the roofline's
    # algorithmic bytes stay every logit once, the bytes read go beside them
    streamed = alg - skipped / nr

    # end to end through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        ht = torch.from_numpy(bt["target"].view(np.int16) if w.dtype == "bf16" else bt["target"])
        hd = torch.from_numpy(bt["draft"].view(np.int16) if w.dtype == "bf16" else bt["draft"])
        ht, hd = ht.pin_memory(), hd.pin_memory()
        htok = tok.cpu().pin_memory()
        hseed = seeds.cpu().pin_memory()
        res_host = {k: torch.empty(v.shape, dtype=v.dtype, pin_memory=True)
                    for k, v in (("accept_len", out["accept_len"]), ("bonus", out["bonus"]),
                                 ("branch", look["branch"]), ("all_hit", look["all_hit"]))}
        tg_raw = tg.view(torch.int16) if w.dtype == "bf16" else tg
        dg_raw = dg.view(torch.int16) if w.dtype == "bf16" else dg
        ne = max(3, min(args.steps, args.e2e_steps))

        hbr = [(rows.view(torch.int16) if w.dtype == "bf16" else rows,
                rows.cpu().view(torch.int16 if w.dtype == "bf16" else torch.float32).pin_memory())
               for rows, *_ in branch]

        def e2e_step(r):
            tg_raw.copy_(ht, non_blocking=True)
            dg_raw.copy_(hd, non_blocking=True)
            for dev_rows, host_rows in hbr:
                dev_rows.copy_(host_rows, non_blocking=True)
            tok.copy_(htok, non_blocking=True)
            seeds.copy_(hseed, non_blocking=True)
            step(r)
            res_host["accept_len"].copy_(out["accept_len"], non_blocking=True)
            res_host["bonus"].copy_(out["bonus"], non_blocking=True)
            res_host["branch"].copy_(look["branch"], non_blocking=True)
            res_host["all_hit"].copy_(look["all_hit"], non_blocking=True)
            stream.synchronize()

        e2e_step(0)
        if world > 1:
            tdist.barrier()
        torch.cuda.synchronize()
        w0 = time.perf_counter()
        for s in range(ne):
            e2e_step(90_000 + s)
        e2e_s = max_over_ranks(time.perf_counter() - w0, tdist, dev)
        h2d = int(ht.numel() * ht.element_size() + hd.numel() * hd.element_size()
                  + htok.numel() * 4 + hseed.numel() * 8
                  + sum(h.numel() * h.element_size() for _, h in hbr))
        d2h = int(sum(v.numel() * v.element_size() for v in res_host.values()))
        e2e = {"value": job_rows_per_s(B * ne, world, e2e_s), "unit": "rows/s",
               "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": ne}

    # further workloads (the batched bf16 one, the small batches), measured in
    # the same process, each with its own roofline
    sides = {}
    if args.side and not (args.batch or args.vocab):
        for name in args.side.split(","):
            if name and name != args.workload:
                sides[name] = side_workload(name, args.steps, args.warmup, rank, dev, tdist)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)

    if rank == 0:
        traffic = traffic_from_profile(args.workload)
        line = {
            "metric": METRIC,
            "value": job_rows_per_s(B * args.steps, world, ms * 1e-3),
            "unit": "rows/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f32" if w.dtype == "f32" else "bf16",
            "data": "synthetic (seeded Zipf-head / Gumbel logits over a random vocab permutation; "
                    "drafts drawn by the library's Saguaro sampler)",
            "config": {"workload": w.name, "B": B, "K": K, "Kq": Kq, "V": V, "T": w.T,
                       "C": w.C, "fanout": list(map(int, F)), "global_batch": B * world,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "inputs larger than L2 (no flush)" if alg > 129e6 else
                             "inputs smaller than L2",
                       "positions_per_s": (K + 1) * B * world * args.steps / (ms * 1e-3),
                       "logits_gb_per_s": alg_step * world * args.steps / (ms * 1e-3) / 1e9,
                       "logits_read_gb_per_s": (alg_step - alg + streamed) * world * args.steps
                                               / (ms * 1e-3) / 1e9,
                       "saguaro_sampling": saguaro,
                       "accept_mean": acc_sum / nr, "alpha_measured": alpha, "hit_rate": h,
                       "all_hit_fraction": all_hits / nr, "h_pow_B": h ** B,
                       "wall_s_timed": wall},
            "roofline": dict(verify_roofline(alg, skipped / nr, verify_ms, verify_ms_median,
                                             hbm_peak, peak_kind, traffic),
                             tail_bytes_per_launch=tail_bytes),
            "e2e": e2e,
            "workloads": sides or None,
            "gpu_launches": args.steps,
            "clocks": ck,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line))
    if world > 1:
        tdist.destroy_process_group()


# ------------------------------------------------------------------------------ oracle
def oracle_round(orc, bt, tok, r, F, w, cores, rows):
    """One round by the oracle, as the GPU step does it: verify, then the
    outcome cache of the guesses probed with every sequence's outcome."""
    ref = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], r, F, w.C, w.T,
                     nthreads=cores, row_ids=rows)
    g = ref["guesses"]
    b, k, f = np.nonzero(g >= 0)
    branch = (b * g.shape[1] + k) * g.shape[2] + f
    return orc.cache_lookup(b, k, g[b, k, f], branch, ref["accept_len"], ref["bonus"])


def cpu_baseline(w, seconds, rows_per_call=None):
    """The CPU oracle, as it stands, on a bounded sample of the workload's
    rows (all host threads)."""
    from oracle import oracle as orc
    from ssd_inputs import make_batch

    cores = os.cpu_count() or 1
    n = rows_per_call or max(4, min(w.B, 2 * cores))
    rows = np.arange(n)
    bt = make_batch(w, rows=rows)
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=w.K, nthreads=cores)
    done, t0 = 0, time.perf_counter()
    while True:
        oracle_round(orc, bt, tok, done, F, w, cores, rows)
        done += 1
        el = time.perf_counter() - t0
        if el >= seconds or done >= 1000:
            break
    return {"value": n * done / el, "unit": "rows/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.B} rows x {done} rounds ({el:.1f} s), fp64 oracle verify "
                      f"and outcome-cache lookup, {cores} threads"}


def run_reference(args):
    from ssd_inputs import WORKLOADS

    world, rank, local = dist_env()
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    cores = os.cpu_count() or 1
    n = max(4, min(w.B, 2 * cores))
    from oracle import oracle as orc
    from ssd_inputs import make_batch

    rows = np.arange(n)
    bt = make_batch(w, rows=rows)
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=w.K, nthreads=cores)

    def step(r):
        oracle_round(orc, bt, tok, r, F, w, cores, rows)

    for s in range(args.warmup):
        step(s)
    t0 = time.perf_counter()
    for s in range(args.steps):
        step(1000 + s)
    el = time.perf_counter() - t0
    v = n * args.steps / el
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": v, "unit": "rows/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": el / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": w.name, "B": w.B, "K": w.K, "V": w.V},
        "cpu_baseline": {"value": v, "unit": "rows/s", "cores": cores, "kind": "oracle",
                         "sample": f"{n} of {w.B} rows per step"},
        "e2e": {"value": v, "unit": "rows/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def run_fanout_ablation(args):
    """Hit rate of the geometric and the uniform guess allocation against
    temperature, on the workload's shape (seeded synthetic rounds, library
    calls only).  Prints one JSON line."""
    from sampling_ssd_verify_gb300.ablation import fanout_ablation
    from ssd_inputs import WORKLOADS

    w = WORKLOADS[args.workload]
    budget = int(sum(w.fanout))
    rounds = args.rounds
    rows = fanout_ablation(w, (0.5, 0.7, 1.0, 1.3, 1.6), budget, Cs=sorted({1.0, w.C}),
                           rounds=rounds, B=args.batch or None, V=args.vocab or None)
    print(json.dumps({"ablation": "fanout", "workload": w.name, "budget": budget,
                      "B": args.batch or w.B, "V": args.vocab or w.V, "rounds": rounds,
                      "data": "synthetic", "rows": rows}))


TREES = {"chain-4": [-1, 0, 1, 2, 3], "binary-depth-3": [-1, 0, 0, 1, 1, 2, 2],
         "wide-3x2": [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3]}


def run_tree(args):
    """ssd_tree_verify on trees of the workload's rows (row u of a tree is
    the generator's position u; child v's token drawn from its parent's draft
    row by the library's sampler with C = 1, counter (b, v - 1, 2, round 0)),
    timed with CUDA events over back-to-back calls.  Prints one JSON line:
    trees/s and the roofline of the call's algorithmic bytes (every node's
    target and draft row read once)."""
    import torch

    import sampling_ssd_verify_gb300 as ssd
    from ssd_inputs import WORKLOADS, make_batch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    ssd.build()
    w = WORKLOADS[args.workload]
    parent = TREES[args.tree]
    N = len(parent)
    B = args.batch or w.B
    V = args.vocab or w.V
    bt = make_batch(w, B=B, V=V, K=N - 1, seed=w.seed)
    if w.dtype == "bf16":
        tg = torch.from_numpy(bt["target"].view(np.int16)).to(dev).view(torch.bfloat16)
        dg = torch.from_numpy(np.ascontiguousarray(bt["draft"][:, :N]).view(np.int16)).to(dev)
        dg = dg.view(torch.bfloat16)
    else:
        tg = torch.from_numpy(bt["target"]).to(dev)
        dg = torch.from_numpy(np.ascontiguousarray(bt["draft"][:, :N])).to(dev)
    seeds = torch.from_numpy(bt["seeds"].view(np.int64)).to(dev)
    tok = torch.full((B, N), -1, dtype=torch.int32, device=dev)
    for v in range(1, N):
        tok[:, v] = ssd.saguaro_sample(dg[:, parent[v], :], w.T, 1.0, 0, seeds, v - 1, 0,
                                       guesses=False, qprime=False)["token"]
    ws = torch.empty(ssd.lib().ssd_tree_workspace_size(B, N, V), dtype=torch.uint8, device=dev)
    out = {}
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    f = lambda i: ssd.tree_verify(tg, dg, parent, tok, seeds, i, w.T, workspace=ws, out=out,
                                  dev_status=status)
    for i in range(args.warmup):
        f(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(args.steps):
        f(1000 + i)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    es = 2 if w.dtype == "bf16" else 4
    alg = B * N * 2 * V * es
    hbm_peak, peak_kind = peaks()
    achieved = alg / (ms * 1e-3) / 1e9
    print(json.dumps({"metric": "tree drafts verified per second", "value": B / (ms * 1e-3),
                      "unit": "trees/s", "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": ms, "dtype": w.dtype, "data": "synthetic",
                      "config": {"workload": w.name, "tree": args.tree, "parent": parent,
                                 "B": B, "N": N, "V": V, "T": w.T,
                                 "accept_mean": float(out["accept_len"].float().mean().item()),
                                 "l2": "inputs larger than L2 (no flush)" if alg > 129e6 else
                                       "inputs smaller than L2"},
                      "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak,
                                   "unit": "GB/s", "frac": achieved / hbm_peak,
                                   "algorithmic_bytes_per_call": alg, "peak_kind": peak_kind,
                                   "launches_per_call": 2},
                      "status": int(status.item())}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=None)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="c5", choices=["c2", "c3", "c4", "c5"])
    ap.add_argument("--batch", type=int, default=0, help="override the workload's batch B")
    ap.add_argument("--vocab", type=int, default=0, help="override the workload's vocabulary V")
    ap.add_argument("--side", default="c3,c4,c2", help="further workloads measured in the same "
                    "run, comma-separated (empty: none)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--rounds", type=int, default=64, help="rounds per ablation cell")
    ap.add_argument("--ablation", choices=["fanout"], default=None,
                    help="instead of the benchmark: geometric vs uniform fan-out hit rates")
    ap.add_argument("--tree", choices=sorted(TREES), default=None,
                    help="instead of the benchmark: tree-draft verification of that shape")
    args = ap.parse_args()
    if args.ablation == "fanout":
        run_fanout_ablation(args)
        return
    if args.tree:
        args.steps = 100 if args.steps is None else args.steps
        args.warmup = 5 if args.warmup is None else max(3, args.warmup)
        run_tree(args)
        return
    if args.impl == "reference":
        args.steps = 3 if args.steps is None else args.steps
        args.warmup = 1 if args.warmup is None else args.warmup
        run_reference(args)
        return
    args.steps = 2000 if args.steps is None else args.steps
    args.warmup = 20 if args.warmup is None else max(3, args.warmup)
    run_ours(args)


if __name__ == "__main__":
    main()
