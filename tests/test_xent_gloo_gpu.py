"""The cross entropy's batch mean over two ranks, end to end through the
library: two processes on one GPU each run fr_xent on their own rows (the
row shards of one batch) with group=, so the binding all-reduces the two fp64
mean parts the call left in its workspace (torch.distributed, gloo here; NCCL
on one GPU per rank) and fr_xent_mean_from_parts writes the batch mean.  Both
ranks must hold the same mean, equal to the oracle's mean over the whole
batch.  The ranks' kernels never wait on each other: the exchange runs on the
host between the two launches of each rank."""
import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ROWS, COLS = 300, 5003


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, out_dir: str):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import reduction_pointwise_row_gb300 as fr
    from synth import workloads
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        per = ROWS // world
        w = workloads.make(4, rows=per, cols=COLS, seed=4343, row0=rank * per, global_rows=ROWS)
        lg = torch.from_numpy(w.arrays["logits"].view(np.int16)).cuda().view(torch.bfloat16)
        tg = torch.from_numpy(w.arrays["target"]).cuda()
        ws = fr.fr_xent_workspace(per, COLS, "bf16")
        r = fr.fr_xent(lg, tg, -100, workspace=ws, group=dist.group.WORLD)
        parts = fr.xent_mean_parts(ws).cpu().numpy()
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.concatenate([r["mean"].cpu().numpy().astype(np.float64), parts,
                                r["loss"].cpu().numpy().astype(np.float64)]))
        assert fr.fr_check_device_error() == 0
    finally:
        dist.destroy_process_group()


def test_batch_mean_through_a_process_group(tmp_path):
    sys.path.insert(0, ROOT)
    import oracle
    from compare import assert_close
    from synth import workloads
    world = 2
    mp.start_processes(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    got = [np.load(str(tmp_path / f"rank{r}.npy")) for r in range(world)]
    w = workloads.make(4, rows=ROWS, cols=COLS, seed=4343)
    ref = oracle.get().xent(w.arrays["logits"], w.arrays["target"], -100)
    # both ranks: the same mean, bit for bit, and the summed parts
    assert got[0][0] == got[1][0]
    assert (got[0][1:3] == got[1][1:3]).all()
    assert got[0][2] == np.count_nonzero(w.arrays["target"] != -100)
    assert_close(np.float32(got[0][0]), ref["mean"], "loss", "batch mean over two ranks")
    loss = np.concatenate([g[3:] for g in got])
    assert_close(loss.astype(np.float32), ref["loss"], "loss", "per-row losses of the shards")
