"""Multi-GPU launch path of bench.py on CPU: two gloo ranks (replicas only — streams are
independent, there is no collective on the data path).  Each rank must get its own stream's
inputs, the barrier must hold both ranks, and the timing used for the aggregate must be the
maximum over ranks."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    import synth
    import torch.distributed as dist
    w, r, local = bench.dist_setup(None)
    assert (w, r, local) == (world, rank, rank)
    # each replica decodes its own stream: prompts and variates differ by rank
    prompt = synth.prompt("frame", stream=r)
    expo = synth.expo(100 + r, 0, 4)
    bench.barrier(w)
    t = bench.max_over_ranks(1.5 + r, w)     # this rank's time; the aggregate uses the slowest
    np.save(os.path.join(out_dir, f"r{r}.npy"), np.array([t, prompt[:, 0].sum(), expo.sum()]))
    dist.destroy_process_group()


def test_two_gloo_ranks_replicas(tmp_path):
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, str(tmp_path))) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    a, b = np.load(tmp_path / "r0.npy"), np.load(tmp_path / "r1.npy")
    assert a[0] == b[0] == 2.5                 # max over ranks reaches both
    assert a[1] != b[1] and a[2] != b[2]       # independent streams per replica
