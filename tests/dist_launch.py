"""Launch a few ranks of tests/dist_rank_worker.py as child processes on
this machine (gloo rendezvous on 127.0.0.1) and collect their outputs."""
import dataclasses
import json
import os
import socket
import subprocess
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def run_ranks(w, ops: str, tmpdir, timeout: float = 600.0):
    """Run P = w.P ranks; returns one dict of arrays per rank."""
    port = _free_port()
    out = os.path.join(str(tmpdir), f"{w.name}-{ops}")
    wd = dataclasses.asdict(w)
    procs = []
    for r in range(w.P):
        env = dict(os.environ, RANK=str(r), WORLD_SIZE=str(w.P), LOCAL_RANK=str(r), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT=str(port), OMP_NUM_THREADS="1")
        procs.append(subprocess.Popen([sys.executable, os.path.join(HERE, "dist_rank_worker.py"), "--ops", ops,
                                       "--workload", json.dumps(wd), "--out", out], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True))
    logs = []
    try:
        for p in procs:
            logs.append(p.communicate(timeout=timeout)[0])
    finally:
        for p in procs:
            if p.poll() is None:
                p.kill()
    for r, p in enumerate(procs):
        assert p.returncode == 0, f"rank {r} failed:\n{logs[r][-4000:]}"
    return [dict(np.load(f"{out}.rank{r}.npz")) for r in range(w.P)]
