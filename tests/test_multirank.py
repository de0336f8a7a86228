"""The replica path across ranks, on CPU with gloo (world size 2).

Requests are independent, so replicas share nothing on the data path; the
only cross-rank step is the host-side reduction of the timing in bench.py
(max of the time, sum of the tokens).  Each rank also draws its own request
stream (the engine seeds it with the rank)."""
import os
import socket
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from demand_paged_kv_gqa_b300 import synth
    t_ms, tokens = bench.reduce_over_ranks(10.0 + 5.0 * rank, 100 * (rank + 1), torch.device("cpu"))
    # the rank's own seeded stream
    w = synth.WORKLOADS["tiny"]
    bs = synth.BatchStream(w, 2, [16, 16], device="cpu", seed=rank)
    q, _, _ = bs.next_step()
    with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
        f.write(f"{t_ms} {tokens} {float(q.float().sum())}\n")
    dist.barrier()
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_worker, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    rows = [open(tmp_path / f"r{r}.txt").read().split() for r in range(2)]
    for r in rows:
        assert float(r[0]) == 15.0            # max over ranks
        assert float(r[1]) == 300.0           # sum over ranks
    assert rows[0][2] != rows[1][2]           # different request streams per rank


def test_single_process_reduction_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(3.5, 7, torch.device("cpu")) == (3.5, 7.0)
