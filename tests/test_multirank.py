"""The N > 1 path of bench.py on the CPU: two gloo ranks.

Every (b, h) head is independent, so the ranks share no data: each draws its
own batch (seed offset by its rank), runs the whole workload, and the job's
time is the slowest rank's (an all-reduce MAX).  The reference arm under
torchrun runs on rank 0 only and prints one line."""

import importlib.util
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        b = _bench()
        from io_aware_exact_05_gb300.inputs import make_inputs, workload

        ws, r, _ = b.dist_env()
        w = b.rank_workload(workload("tiny_f32"), r)
        q = make_inputs(w)["q"]
        # the slowest rank's time is the job's: rank r pretends to take 10 + 5 r ms
        t = b.max_over_ranks(10.0 + 5.0 * r, True, "cpu")
        dist.barrier()
        json.dump({"ws": ws, "rank": r, "seed": w.seed, "q0": float(q.flatten()[0]), "t": t},
                  open(os.path.join(out_dir, "rank%d.json" % r), "w"))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    res = [json.load(open(tmp_path / ("rank%d.json" % r))) for r in range(2)]
    assert [x["ws"] for x in res] == [2, 2] and [x["rank"] for x in res] == [0, 1]
    assert res[0]["seed"] != res[1]["seed"] and res[0]["q0"] != res[1]["q0"]   # own batches
    assert res[0]["t"] == res[1]["t"] == 15.0                                  # max over ranks


def test_whole_job_rate_and_single_rank_identity():
    b = _bench()
    assert b.max_over_ranks(3.5, False, "cpu") == 3.5
    # 2 ranks x 10 steps x 1e12 FLOPs in 2000 ms = 10 TFLOP/s
    assert b.whole_job_tflops(1e12, 2, 10, 2000.0) == pytest.approx(10.0)
    from io_aware_exact_05_gb300.inputs import workload

    w = workload("b2h16_n8k_d128")
    assert b.rank_workload(w, 0) == w
    assert b.rank_workload(w, 3).seed == w.seed + 3 * 7919
    assert b.rank_workload(w, 3).with_shape(seed=w.seed) == w


def test_dq_mode_default_follows_the_library_rule():
    b = _bench()
    from io_aware_exact_05_gb300.inputs import workload

    w = workload("b2h8_n4k_d256")
    assert b.dq_mode_used("auto", w.with_shape(d=64)) == b.dq_mode_used("auto", w.with_shape(d=128)) == "atomic"
    assert b.dq_mode_used("auto", w) == "spill"                          # non-causal, dense, 537 MB
    assert b.dq_mode_used("auto", w.with_shape(causal=True)) == "pass"
    assert b.dq_mode_used("auto", w.with_shape(H_kv=4)) == "pass"
    assert b.dq_mode_used("auto", w.with_shape(sparse=(1, 1, 1))) == "pass"
    assert b.dq_mode_used("auto", w.with_shape(B=16, n=32768)) == "pass"   # over 4 GiB
    assert b.dq_mode_used("pass", w) == "pass" and b.dq_mode_used("atomic", w) == "atomic"


def test_reference_arm_under_torchrun_prints_once():
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny_f32", "--steps", "2", "--warmup", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [l for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
