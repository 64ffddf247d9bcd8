"""The N > 1 host logic of bench.py on two gloo ranks on the CPU: each rank
owns its own sequences (rank 0 keeps the single-rank streams, rank 1 draws
others from the same chain), weights are shared, and the job's time is the
maximum over ranks.  No data-path collective exists to test: the sequences are
independent."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from synth import configs as C


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = C.CHUNKED_FP32.replace(d=16, d_ff=32, vocab=64, chunk=8, B=2, T=32, n_prefix=1)
    inp = bench.rank_inputs(wl, rank)
    t = bench.max_over_ranks(10.0 + rank, world, "cpu")
    np.save(os.path.join(out_dir, f"tok{rank}.npy"), inp["tokens"])
    np.save(os.path.join(out_dir, f"w{rank}.npy"), inp["weights"]["U"])
    np.save(os.path.join(out_dir, f"t{rank}.npy"), np.array([t]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_own_sequences_and_report_the_slowest(tmp_path):
    import bench
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    wl = C.CHUNKED_FP32.replace(d=16, d_ff=32, vocab=64, chunk=8, B=2, T=32, n_prefix=1)
    single = bench.rank_inputs(wl, 0)
    tok0, tok1 = np.load(tmp_path / "tok0.npy"), np.load(tmp_path / "tok1.npy")
    np.testing.assert_array_equal(tok0, single["tokens"])
    assert tok1.shape == tok0.shape and not np.array_equal(tok0, tok1)
    assert (tok1[:, 0] == 0).all()                     # every stream starts at BOS
    np.testing.assert_array_equal(np.load(tmp_path / "w0.npy"), np.load(tmp_path / "w1.npy"))
    assert float(np.load(tmp_path / "t0.npy")[0]) == 11.0 == float(np.load(tmp_path / "t1.npy")[0])
