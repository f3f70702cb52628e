"""The N > 1 bench path on CPU: two gloo ranks, each an independent replica;
the reported throughput is all ranks' work over the slowest rank's time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    secs = [1.0, 2.0][rank]                      # rank 1 is the slow one
    out[rank] = (bench.reduce_max(secs, dist), bench.replica_throughput(10.0, secs, world, dist))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_gloo():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    for rank in range(world):
        slowest, thr = res[rank]
        assert slowest == 2.0
        assert thr == pytest.approx(2 * 10.0 / 2.0)


def test_single_rank_identity():
    import bench
    assert bench.reduce_max(3.5) == 3.5
    assert bench.replica_throughput(8.0, 2.0, 1) == 4.0


def test_reference_arm_prints_one_json_line():
    """bench.py --impl reference times the fp64 oracle on the host (no GPU needed)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["unit"] == "TFLOP/s" and rec["value"] > 0
    assert rec["cpu_baseline"]["kind"] == "oracle" and rec["cpu_baseline"]["cores"] >= 1
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["e2e"]["d2h_bytes_per_step"] == 0


def test_roofline_bound_of_sweep_entries():
    """The roofline side of a call: causal N=8192 forward is tensor-bound, a
    256-key window and causal N=1024 are HBM-bound (B=1, H=32, d=128)."""
    import bench
    pk = {"bf16": 1927.9, "hbm_gbs": 6784.5}
    rows = 32 * 8192
    assert bench.attention_bytes(rows, 128, False) == rows * (4 * 256 + 4)
    assert bench.attention_bytes(rows, 128, True) == rows * (8 * 256 + 12)
    full = 4.0 * 32 * 8192 * 8192 * 128 / 2
    bound, frac = bench.roofline_of(full / 0.4e-3 / 1e12, 0.4, bench.attention_bytes(rows, 128, False), pk)
    assert bound == "tensor" and abs(frac - full / 1927.9e12 / 0.4e-3) < 1e-9
    win = 4.0 * 32 * (256 * 8192 - 256 * 255 / 2) * 128
    nbytes = bench.attention_bytes(rows, 128, False)
    bound, frac = bench.roofline_of(win / 0.12e-3 / 1e12, 0.12, nbytes, pk)
    assert bound == "hbm" and abs(frac - nbytes / 6784.5e9 / 0.12e-3) < 1e-9
    small = 4.0 * 32 * 1024 * 1024 * 128 / 2
    assert bench.roofline_of(small / 0.023e-3 / 1e12, 0.023, bench.attention_bytes(32 * 1024, 128, False), pk)[0] == "hbm"
