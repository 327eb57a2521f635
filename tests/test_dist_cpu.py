"""The N > 1 plumbing of bench.py on CPU: two gloo ranks (127.0.0.1).

bench.py runs one replica of the hot path per GPU (weak scaling, no
data-path collective).  Its only cross-rank steps are a barrier around the
timed region and the max over ranks of the elapsed time; the reference arm
runs on rank 0 alone.  These are checked here with world_size 2 on gloo.
"""
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import os, sys, json
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
d.init("gloo")
d.barrier()
mx = d.max(1.5 + d.rank, "cpu")
d.barrier()
print(json.dumps({{"rank": d.rank, "world": d.world, "max": mx}}), flush=True)
d.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_barrier_and_max():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE="2", MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, "-c", WORKER.format(root=ROOT)], env=env,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        out, err = p.communicate(timeout=120)
        assert p.returncode == 0, err
        outs.append(out.strip().splitlines()[-1])
    import json

    res = sorted((json.loads(o) for o in outs), key=lambda r: r["rank"])
    assert [r["rank"] for r in res] == [0, 1]
    assert all(r["world"] == 2 and r["max"] == 2.5 for r in res)


def test_reference_arm_only_on_rank_zero():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
