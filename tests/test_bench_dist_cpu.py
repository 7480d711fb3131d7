"""The N > 1 path of bench.py on CPU: world_size-2 gloo ranks over 127.0.0.1.
The library's path does not shard (independent replicas), so what there is to
check is the bench's rendezvous, barrier and max-over-ranks timing, and that
the reference arm prints one line from rank 0 while the other rank exits 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.multiprocessing as tmp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w, _ = bench.dist_setup(world)
    bench.barrier(w)
    m = bench.max_over_ranks(10.0 + r, w)
    with open(os.path.join(out_dir, f"rank{r}.json"), "w") as f:
        json.dump({"rank": r, "world": w, "max": m}, f)
    import torch.distributed as dist
    dist.destroy_process_group()


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU gloo path")
def test_rendezvous_barrier_and_max_over_ranks(tmp_path):
    port = free_port()
    tmp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(2)]
    assert [x["rank"] for x in res] == [0, 1] and all(x["world"] == 2 for x in res)
    assert all(x["max"] == 11.0 for x in res)       # both ranks see the slowest rank's time


@pytest.mark.skipif(torch.cuda.is_available(), reason="CPU gloo path")
def test_reference_arm_under_torchrun_prints_once():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2", "--master-addr",
           "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "1"]
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(l) for l in p.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, p.stdout
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    # the same metric and workload as the product arm's headline, so the driver can divide them
    sys.path.insert(0, ROOT)
    import bench
    assert line["metric"] == bench.METRIC_DENSE and line["config"]["workload"] == bench.WORKLOAD_DENSE
    assert line["unit"] == "TFLOP/s" and line["higher_is_better"] is True
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
