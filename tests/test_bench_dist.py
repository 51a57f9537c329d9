"""The multi-rank path of bench.py on CPU: two gloo ranks (torchrun-style env)
check the barrier, the max-over-ranks time and the summed rows that make up
the whole-job value.  No GPU and no data-path collective are involved."""
import os
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import os, sys
    sys.path.insert(0, {root!r})
    import bench
    rank, world = bench.dist_init()
    assert world == 2
    bench.dist_barrier(world)
    # rank r processes (r+1)*10 rows in (r+1)*2 ms: value = 30 rows / 4 ms
    value, ms_max, rows = bench.aggregate(float((rank + 1) * 10), float((rank + 1) * 2.0), world)
    assert ms_max == 4.0 and rows == 30.0, (ms_max, rows)
    assert abs(value - 30 / 4e-3) < 1e-6
    bench.dist_barrier(world)
    import torch.distributed as dist
    dist.destroy_process_group()
    print("rank", rank, "ok")
""")


def test_two_gloo_ranks(tmp_path):
    script = tmp_path / "child.py"
    script.write_text(CHILD.format(root=ROOT))
    procs = []
    for rank in range(2):
        env = dict(os.environ, WORLD_SIZE="2", RANK=str(rank), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                   MASTER_PORT="29731", SPV_BENCH_BACKEND="gloo", CUDA_VISIBLE_DEVICES="")
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.STDOUT, text=True))
    outs = [p.communicate(timeout=120)[0] for p in procs]
    for rank, (p, out) in enumerate(zip(procs, outs)):
        assert p.returncode == 0, out
        assert f"rank {rank} ok" in out
