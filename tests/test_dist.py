"""The multi-rank host path of bench.py on CPU: two ranks under torchrun with the
gloo backend (replicas only: the ranks share nothing but the barrier around the
timed region and the maximum of their times)."""
import os
import re
import socket
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


SCRIPT = textwrap.dedent("""
    import os, sys, time
    sys.path.insert(0, {root!r})
    import bench
    d = bench.Dist(2)
    assert d.world == 2 and d.rank == int(os.environ["RANK"])
    t0 = time.perf_counter()
    if d.rank == 1:
        time.sleep(0.3)             # the slower rank sets the job's time
    d.barrier()
    waited = time.perf_counter() - t0
    m = d.max(float(d.rank + 1) * 10.0)
    print(f"rank {{d.rank}} max {{m}} waited {{waited:.2f}}", flush=True)
    d.close()
""")


def test_two_ranks_over_gloo_barrier_and_max(tmp_path):
    pytest.importorskip("torch")
    script = tmp_path / "ranks.py"
    script.write_text(SCRIPT.format(root=ROOT))
    env = dict(os.environ, FA_BENCH_BACKEND="gloo", OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), str(script)]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=240)
    assert out.returncode == 0, out.stderr[-2000:]
    # the two ranks print concurrently: their lines may interleave
    found = re.findall(r"rank (\d) max ([0-9.]+) waited ([0-9.]+)", out.stdout)
    assert sorted(r for r, _, _ in found) == ["0", "1"], out.stdout
    for rank, mx, waited in found:
        assert float(mx) == 20.0                      # the maximum over both ranks
        if rank == "0":
            assert float(waited) >= 0.25              # rank 0 waited at the barrier for rank 1
