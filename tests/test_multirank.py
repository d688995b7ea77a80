"""The bench's multi-rank plumbing on two gloo ranks (CPU only).

Each rank runs its own batch (no data exchange); the only collectives are the
barrier and the max-over-ranks of the timed region.  The reference arm prints
on rank 0 only; the other ranks exit quietly.
"""

import os
import socket
import subprocess
import sys
import textwrap

from conftest import ROOT


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_rank_barrier_and_max_over_ranks(tmp_path):
    script = tmp_path / "ranks.py"
    script.write_text(textwrap.dedent(f"""
        import sys
        sys.path.insert(0, {ROOT!r})
        import bench
        rank, local, world = bench.init_dist("gloo")
        assert world == 2
        v = bench.max_over_ranks(float(10 * (rank + 1)))
        bench.barrier()
        if rank == 1:
            class Args:
                steps = 1
                warmup = 0
            bench.run_reference(Args())   # returns without work or output on rank 1
        print(f"rank{{rank}} max={{v}}", flush=True)
    """))
    env = dict(os.environ, PYTHONPATH=ROOT)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}", str(script)]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "rank0 max=20.0" in r.stdout and "rank1 max=20.0" in r.stdout, r.stdout
    assert '"impl": "reference"' not in r.stdout
