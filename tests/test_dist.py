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


SHARD_SCRIPT = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, {root!r})
    import numpy as np
    import torch
    import torch.distributed as dist
    import fa_inputs
    import oracle
    from attention_forward_tma_gb300 import context

    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    B, Nq, Nk, H, Hkv, d, causal = 2, 96, 160, 4, 2, 64, {causal}
    q, k, v = fa_inputs.make_qkv(B, Nq, H, d, seed=55, Nkv=Nk, Hkv=Hkv)
    scale = 1 / np.sqrt(d)

    def partial(r):
        # stand-in for the GPU partial of rank r's key shard: the oracle over those keys
        # with the whole sequence's diagonal (query i sees global key j <= i + Nk - Nq)
        lo, hi = context.shard_range(Nk, r, world)
        o, l = oracle.attention(q, k[:, lo:hi], v[:, lo:hi], scale, causal, off=Nk - Nq - lo)
        return torch.from_numpy(o.astype(np.float32)), torch.from_numpy(l.astype(np.float32))

    o_part, lse_part = partial(rank)
    o_parts, lse_parts = context.gather_partials(o_part, lse_part, dst=0)
    if rank == 0:
        for r in range(world):
            o_r, l_r = partial(r)
            assert torch.equal(o_parts[r], o_r) and torch.equal(lse_parts[r], l_r), r
        o_all, l_all = oracle.attention(q, k, v, scale, causal)
        P = world
        om, lm = oracle.lse_combine(o_parts.numpy().reshape(P, -1, d),
                                    lse_parts.numpy().transpose(0, 1, 3, 2).reshape(P, -1))
        assert np.abs(om - o_all.reshape(-1, d)).max() < 1e-5
        fin = np.isfinite(l_all.transpose(0, 2, 1).reshape(-1))
        assert np.abs(lm[fin] - l_all.transpose(0, 2, 1).reshape(-1)[fin]).max() < 1e-5
        print("shards merged ok", flush=True)
    else:
        assert o_parts is None and lse_parts is None
    dist.destroy_process_group()
""")


@pytest.mark.parametrize("causal", [False, True])
def test_key_shards_gathered_to_the_owner_over_gloo(tmp_path, causal):
    """Two CPU ranks each hold half of a sequence's keys; their partial results (oracle
    stand-ins here) reach rank 0 unchanged through context.gather_partials, and merged
    through the LSE they equal the oracle over all keys."""
    pytest.importorskip("torch")
    script = tmp_path / "shards.py"
    script.write_text(SHARD_SCRIPT.format(root=ROOT, causal=causal))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()), str(script)]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=240)
    assert out.returncode == 0, out.stderr[-3000:]
    assert "shards merged ok" in out.stdout


def test_shard_ranges_cover_the_keys_once():
    from attention_forward_tma_gb300 import context
    for n, world in [(10, 3), (4096, 8), (7, 7), (1000, 1)]:
        ranges = [context.shard_range(n, r, world) for r in range(world)]
        assert ranges[0][0] == 0 and ranges[-1][1] == n
        assert all(a[1] == b[0] for a, b in zip(ranges, ranges[1:]))
        sizes = [hi - lo for lo, hi in ranges]
        assert max(sizes) - min(sizes) <= 1
