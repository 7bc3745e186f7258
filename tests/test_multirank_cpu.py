"""Multi-GPU runs are replicas: every rank verifies its own batch and only the
timing is combined.  These tests run the host side of that with two `gloo`
ranks on the CPU (the verification itself by the oracle, so no GPU is
needed): per-rank batches differ, each rank's results equal a single-process
run on the same batch, the step time is the maximum over ranks and the job
throughput counts both ranks' rows.
"""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as tdist

    import bench
    from oracle import oracle as orc
    from ssd_inputs import WORKLOADS, make_batch

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD))
    tdist.init_process_group("gloo", rank=rank, world_size=WORLD)
    w = WORKLOADS["c1"]
    bt = make_batch(w, B=64, seed=bench.rank_seed(w, rank))
    F = np.asarray(w.fanout, dtype=np.int32)
    tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=w.K)
    res = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 3, F, w.C, w.T)
    step_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(step_ms, tdist)
    rows_s = bench.job_rows_per_s(64 * 7, WORLD, ms * 1e-3)
    gathered = [None] * WORLD
    tdist.all_gather_object(gathered, {"accept_len": res["accept_len"].tolist(),
                                       "bonus": res["bonus"].tolist()})
    tdist.barrier()
    tdist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"ms": ms, "rows_s": rows_s, "gathered": gathered,
                   "first_logit": float(bt["target"].reshape(-1)[0])}, f)


def test_replicas_over_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp

    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, port, str(tmp_path))) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=300)
        assert p.exitcode == 0, "a rank failed"
    out = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(WORLD)]

    # timing: the slowest rank's step time everywhere, throughput over both ranks
    for o in out:
        assert o["ms"] == 15.0
        assert o["rows_s"] == pytest.approx(64 * 7 * WORLD / 15e-3)
    # the ranks verified different batches
    assert out[0]["first_logit"] != out[1]["first_logit"]
    assert out[0]["gathered"] == out[1]["gathered"]

    # each rank's results equal a single-process run on that rank's batch
    sys.path.insert(0, ROOT)
    import bench
    from oracle import oracle as orc
    from ssd_inputs import WORKLOADS, make_batch

    w = WORKLOADS["c1"]
    F = np.asarray(w.fanout, dtype=np.int32)
    for r in range(WORLD):
        bt = make_batch(w, B=64, seed=bench.rank_seed(w, r))
        tok = orc.draft_tokens(bt["draft"], F, w.C, w.T, bt["seeds"], K=w.K)
        ref = orc.verify(bt["target"], bt["draft"], tok, bt["seeds"], 3, F, w.C, w.T)
        assert out[0]["gathered"][r]["accept_len"] == ref["accept_len"].tolist()
        assert out[0]["gathered"][r]["bonus"] == ref["bonus"].tolist()


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "3", "--warmup", "3"], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
