"""The N > 1 path on the CPU (gloo, two ranks): each rank holds its shard of
the rows, the shards together are exactly the global workload, results
gathered from the ranks equal the oracle on the whole batch, the cross
entropy's batch mean comes from the ranks' mean parts summed by the
binding's all-reduce (the path's one exchange step), and the bench's
max-over-ranks timing reduction gives every rank the slowest rank's time.
Every other step is independent per row."""
import os
import socket
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import bench
    import oracle
    import reduction_pointwise_row_gb300 as fr
    from synth import workloads

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.SHARD = (rank, world)
        o = oracle.get()
        results = {}
        for cfg, rows, cols in ((1, 40, 1000), (4, 30, 5000), (2, 12, 512)):
            w = bench.make_shard(workloads, cfg, rows=rows, cols=cols)
            assert w.params["row0"] == rank * rows and w.params["global_rows"] == world * rows
            if cfg == 1:
                local = o.softmax(w.arrays["x"])
            elif cfg == 4:
                local = o.xent(w.arrays["logits"], w.arrays["target"], -100)["loss"]
                # the exchange step: this rank's mean parts, laid out as an
                # fr_xent workspace holds them, summed over the ranks in place
                counted = w.arrays["target"] != -100
                ws = torch.zeros(fr.XENT_PARTS_OFFSET + 16 + 64, dtype=torch.uint8)
                parts = fr.xent_mean_parts(ws)
                parts[0] = float(np.sum(local[counted].astype(np.float64)))
                parts[1] = float(np.count_nonzero(counted))
                fr.allreduce_mean_parts(parts)
                results["mean"] = np.array([parts[0].item() / parts[1].item()])
            else:
                local = o.layernorm(w.arrays["x"], w.arrays["gamma"], w.arrays["beta"],
                                    float(np.float32(1e-5)))[0]
            parts = [torch.empty_like(torch.from_numpy(np.ascontiguousarray(local)))
                     for _ in range(world)]
            dist.all_gather(parts, torch.from_numpy(np.ascontiguousarray(local)))
            results[cfg] = torch.cat(parts).numpy()
        slowest = bench.max_over_ranks(1.0 + rank, world, torch.device("cpu"))
        dist.barrier()
        if rank == 0:
            np.savez(os.path.join(out_dir, "gathered.npz"), slowest=slowest,
                     **{str(k): v for k, v in results.items()})
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_and_reduce_timing(tmp_path):
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import oracle
    from synth import workloads

    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = np.load(tmp_path / "gathered.npz")
    assert float(got["slowest"]) == 2.0  # the slower rank's time, on every rank
    o = oracle.get()
    whole = workloads.make(1, rows=80, cols=1000)
    assert (got["1"] == o.softmax(whole.arrays["x"])).all()
    whole = workloads.make(4, rows=60, cols=5000)
    ref = o.xent(whole.arrays["logits"], whole.arrays["target"], -100)
    assert (got["4"] == ref["loss"]).all()
    # the batch mean from the ranks' summed parts is the oracle's mean over the batch
    assert abs(float(got["mean"][0]) - float(ref["mean"])) <= 1e-6 * abs(float(ref["mean"]))
    assert int((whole.arrays["target"] == -100).sum()) == 3  # 5 % of the global batch
    whole = workloads.make(2, rows=24, cols=512)
    assert (got["2"] == o.layernorm(whole.arrays["x"], whole.arrays["gamma"],
                                    whole.arrays["beta"], float(np.float32(1e-5)))[0]).all()


def test_bench_value_is_whole_job_throughput():
    """value = (ranks x bytes per rank) / the slowest rank's time."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.shard_rows(32768, 0, 1) == (0, 32768)
    assert bench.shard_rows(32768, 3, 4) == (98304, 131072)
    assert bench.max_over_ranks(5.0, 1, torch.device("cpu")) == 5.0
