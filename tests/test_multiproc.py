"""N > 1 path on CPU (gloo, world size 2): rows shard across ranks with no
data-path exchange -- each rank's rows equal the same rows of the unsharded
batch -- and the timing reduction takes the maximum over ranks."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _workload():
    from paged_split_kv_gqa_gb300 import workloads as W
    lens = np.array([40, 33, 1025, 300, 17, 2048, 1, 999], dtype=np.int32)
    return W.Workload("sharding", lens, 16, W.Family("local", 8, 2, 256, 1024),
                      W.Family("global", 8, 2, 512, 0))


def _worker(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from oracle import oracle as O
    from paged_split_kv_gqa_gb300 import workloads as W
    wl = _workload()
    res = {}
    for fam in wl.families():
        fi = W.make_family_inputs(wl, fam, poison=True)
        rows = list(range(rank, wl.batch, world))            # this rank's shard
        out = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                       num_kv_heads=fam.num_kv_heads, window=fam.window,
                       scale=1 / math.sqrt(fam.head_dim), rows=rows, nthreads=2)
        t = torch.from_numpy(out)
        gathered = [torch.zeros_like(t) for _ in range(world)] if rank == 0 else None
        dist.gather(t, gathered, dst=0)
        if rank == 0:
            full = torch.zeros(wl.batch, *t.shape[1:], dtype=t.dtype)
            for r in range(world):
                full[r::world] = gathered[r]
            res[fam.name] = full.numpy()
    elapsed = torch.tensor([1.0 + rank])
    dist.all_reduce(elapsed, op=dist.ReduceOp.MAX)
    if rank == 0:
        np.savez(os.path.join(out_dir, "sharded.npz"), elapsed=elapsed.numpy(), **res)
    dist.barrier()
    dist.destroy_process_group()


def test_row_sharding_gloo_world2(tmp_path):
    port = _free_port()
    mp.start_processes(_worker, args=(2, port, str(tmp_path)), nprocs=2, start_method="spawn")
    from oracle import oracle as O
    from paged_split_kv_gqa_gb300 import workloads as W
    got = np.load(tmp_path / "sharded.npz")
    assert float(got["elapsed"][0]) == 2.0
    wl = _workload()
    for fam in wl.families():
        fi = W.make_family_inputs(wl, fam, poison=True)
        ref = O.decode(fi.q, fi.k_pool, fi.v_pool, fi.page_table, fi.seq_lens,
                       num_kv_heads=fam.num_kv_heads, window=fam.window,
                       scale=1 / math.sqrt(fam.head_dim))
        np.testing.assert_array_equal(got[fam.name], ref)
