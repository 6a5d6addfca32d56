"""bench.py's N > 1 path on the CPU (replicas only, one process per rank):
two gloo ranks launched the way torchrun sets them up (RANK, LOCAL_RANK,
WORLD_SIZE, MASTER_ADDR=127.0.0.1, MASTER_PORT).

* `_max_over_ranks` gives every rank the slowest rank's figure (the
  whole-job value divides all ranks' units by it);
* the reference arm runs and prints on rank 0 alone, with n_gpus = 2; rank 1
  exits 0 without output.
"""

import json
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, sys
sys.path.insert(0, sys.argv[1])
import bench
ws, rank, local = bench._dist()
dist = bench._dist_setup(ws)
x = bench._max_over_ranks(10.0 + 5.0 * rank, dist)
print(json.dumps({"rank": rank, "ws": ws, "backend": dist.get_backend(), "max": x}))
dist.destroy_process_group()
"""


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _launch(args, ws=2):
    port = _free_port()
    procs = []
    for r in range(ws):
        env = dict(os.environ, RANK=str(r), LOCAL_RANK=str(r), WORLD_SIZE=str(ws),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable] + args, env=env, cwd=ROOT, text=True,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE))
    out = []
    for p in procs:
        o, e = p.communicate(timeout=300)
        out.append((p.returncode, o, e))
    return out


def test_max_over_ranks_on_gloo():
    res = _launch(["-c", WORKER, ROOT])
    for rc, _, err in res:
        assert rc == 0, err
    lines = [json.loads(o.strip().splitlines()[-1]) for _, o, _ in res]
    assert sorted(l["rank"] for l in lines) == [0, 1]
    for l in lines:
        assert l["backend"] == "gloo" and l["ws"] == 2 and l["max"] == 15.0


def test_reference_arm_prints_on_rank0_only():
    res = _launch(["bench.py", "--impl", "reference", "--workload", "tiny-L4-d256",
                   "--steps", "2", "--warmup", "1"])
    (rc0, out0, err0), (rc1, out1, err1) = res
    assert rc0 == 0 and rc1 == 0, (err0, err1)
    line = json.loads(out0.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert out1.strip() == ""
