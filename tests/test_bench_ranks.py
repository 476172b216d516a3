"""The multi-rank host logic of bench.py on CPU: two gloo ranks on 127.0.0.1.

bench.py runs one process per GPU under torchrun; the ranks share no data, but the timed
region is bracketed by a barrier and the reported time is the maximum over ranks.  This
runs those helpers (dist_setup, barrier, max_over_ranks) in two real processes.
"""

import json
import os
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


RANK_SCRIPT = textwrap.dedent("""
    import json, sys, time
    sys.path.insert(0, {root!r})
    import bench
    rank, world, local = bench.dist_setup()
    # rank 1 arrives late: the barrier must hold rank 0 until it does
    if rank == 1:
        time.sleep(0.5)
    t0 = time.time()
    bench.barrier(world)
    waited = time.time() - t0
    worst = bench.max_over_ranks(10.0 * (rank + 1), world)
    import torch.distributed as dist
    dist.destroy_process_group()
    print(json.dumps({{"rank": rank, "world": world, "local": local, "waited": waited, "max": worst}}))
""")


@pytest.mark.timeout(180)
def test_two_ranks_barrier_and_max(tmp_path):
    script = tmp_path / "rank.py"
    script.write_text(RANK_SCRIPT.format(root=ROOT))
    port = _free_port()
    procs = []
    for r in range(2):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE="2",
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=170)
        assert p.returncode == 0, err
        outs.append(json.loads(out.strip().splitlines()[-1]))
    by_rank = {o["rank"]: o for o in outs}
    assert set(by_rank) == {0, 1}
    for r, o in by_rank.items():
        assert o["world"] == 2 and o["local"] == r
        assert o["max"] == 20.0          # the slowest rank's time is reported by every rank
    assert by_rank[0]["waited"] >= 0.3   # rank 0 was held at the barrier for the late rank


def test_single_process_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    env = {k: os.environ.get(k) for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    try:
        for k in env:
            os.environ.pop(k, None)
        assert bench.dist_setup() == (0, 1, 0)
        bench.barrier(1)
        assert bench.max_over_ranks(3.5, 1) == 3.5
    finally:
        for k, v in env.items():
            if v is not None:
                os.environ[k] = v
