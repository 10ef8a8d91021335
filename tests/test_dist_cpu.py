"""bench.py's multi-process path on CPU: two gloo ranks, each timing its own
replica, must agree on the max over ranks and the aggregate rate, and the
reference arm must stay silent on every rank but 0."""
import json
import os
import socket
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


CHILD = textwrap.dedent("""
    import json, os, sys
    sys.path.insert(0, os.environ["KDA_ROOT"])
    import bench
    ws, rank, local = bench.dist_setup()
    assert ws == 2 and rank == int(os.environ["RANK"])
    ms = bench.reduce_max(1.5 + rank, ws)          # rank 1 is the slower one
    bench.barrier(ws)
    tokens = 65536
    value = ws * tokens / (ms * 1e-3) / 1e6
    print(json.dumps({"rank": rank, "ms": ms, "value": value}), flush=True)
    import torch.distributed as dist
    dist.destroy_process_group()
""")


def test_two_rank_gloo_max_and_aggregate():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), KDA_ROOT=ROOT,
                   CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, "-c", CHILD], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=120)
        assert p.returncode == 0, e
        outs.append(json.loads(o.strip().splitlines()[-1]))
    for o in outs:
        assert o["ms"] == 2.5                      # max over ranks, not the local time
        assert abs(o["value"] - 2 * 65536 / 2.5e-3 / 1e6) < 1e-9


def test_reference_arm_other_ranks_exit_silently(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class A:
        steps, warmup, gpus = 1, 3, 2

    assert bench.run_reference(A, 2, 1) is None
    assert capsys.readouterr().out == ""
