"""bench.py's multi-rank plumbing on CPU (gloo, world size 2): the max-over-ranks
timing reduction and the barrier, and the reference arm printing one line
from rank 0 only.  Every rank is a separate process, as under torchrun."""
import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _launch(code_or_args, world=2, timeout=240):
    port = _free_port()
    procs = []
    for rank in range(world):
        env = {**os.environ, "RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
               "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "CUDA_VISIBLE_DEVICES": ""}
        cmd = [sys.executable, "-c", code_or_args] if isinstance(code_or_args, str) else [sys.executable, *code_or_args]
        procs.append(subprocess.Popen(cmd, cwd=ROOT, env=env, stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                      text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=timeout)
        outs.append((p.returncode, out, err))
    return outs


def test_max_over_ranks_and_barrier_with_gloo():
    code = (
        "import bench, json, os\n"
        "args = bench.parse_args([])\n"
        "rank, ws = bench.dist_setup(args)\n"
        "bench.barrier(ws)\n"
        "m = bench.reduce_max(10.0 * (rank + 1) + 0.25, ws)\n"
        "bench.barrier(ws)\n"
        "print(json.dumps({'rank': rank, 'ws': ws, 'max': m}))\n"
        "import torch.distributed as dist\n"
        "dist.destroy_process_group()\n"
    )
    outs = _launch(code)
    for rank, (rc, out, err) in enumerate(outs):
        assert rc == 0, err
        line = json.loads(out.strip().splitlines()[-1])
        assert line == {"rank": rank, "ws": 2, "max": 20.25}


def test_reference_arm_prints_one_line_from_rank_0_only():
    outs = _launch(["bench.py", "--impl", "reference", "--config", "llama31_8b_b1_4k", "--steps", "1",
                    "--warmup", "3", "--gpus", "2"])
    (rc0, out0, err0), (rc1, out1, err1) = outs
    assert rc0 == 0 and rc1 == 0, (err0, err1)
    assert out1.strip() == ""
    lines = [l for l in out0.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
