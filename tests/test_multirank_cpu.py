"""The bench's multi-rank host logic on CPU with two gloo ranks (no GPU).

The path has no collective of its own (replicas only): ranks rendezvous,
meet at barriers around the timed region, and take the maximum of their
times. The reference arm under torchrun runs on rank 0 alone; the other
ranks exit 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, port, out_dir):
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": "2", "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    sys.path.insert(0, ROOT)
    import bench
    ws, r, _ = bench.dist_setup("gloo")
    bench.dist_barrier(ws)
    mx = bench.dist_max(ws, 1.5 * (r + 1))
    bench.dist_barrier(ws)
    import torch.distributed as dist
    dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"ws": ws, "rank": r, "max": mx}, f)


def test_dist_helpers_two_gloo_ranks(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    for r in range(2):
        d = json.load(open(tmp_path / f"rank{r}.json"))
        assert d == {"ws": 2, "rank": r, "max": 3.0}


def test_reference_arm_under_torchrun_prints_once():
    pytest.importorskip("torch")
    env = dict(os.environ, TTS_BB_REF_BUDGET_S="5")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference", "--gpus", "2",
           "--steps", "1", "--warmup", "3"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


def test_clock_sampler_watches_this_ranks_gpu(monkeypatch):
    """Each rank samples the clocks of its own device (cuda:LOCAL_RANK), named as nvidia-smi names it."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "4,5,6,7")
    monkeypatch.setenv("LOCAL_RANK", "2")
    assert bench.this_rank_gpu() == "6"
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "GPU-aaa, GPU-bbb")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.this_rank_gpu() == "GPU-bbb"
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    monkeypatch.setenv("LOCAL_RANK", "3")
    assert bench.this_rank_gpu() == "3"
