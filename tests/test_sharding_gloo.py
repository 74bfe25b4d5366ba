"""Row sharding across ranks (CPU, gloo, world size 2): each rank computes
its contiguous share of a batch with the CPU oracle, the shares are
all-gathered, and the result equals the oracle on the whole batch."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sparse_attention_top_packed_b300.sharding import row_range, slice_args


def test_row_range_partitions_every_row():
    for n in [0, 1, 7, 8, 4096, 8191]:
        for world in [1, 2, 3, 8]:
            spans = [row_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
                assert a1 == b0
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        row_range(4, 2, 2)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from oracle import topk_packed_reference
        from sparse_attention_top_packed_b300.workloads import random_problem

        rng = np.random.default_rng(5)
        p = random_problem(rng, rows=37, max_len=3000, k=128, page_size=16, values="ties")
        rows = p.num_rows
        scores = torch.from_numpy(p.scores).reshape(rows, p.row_stride)
        seq = torch.from_numpy(p.seq_lens)
        st = torch.from_numpy(p.row_starts)
        rtb = torch.from_numpy(p.row_to_batch)
        out = torch.empty((rows, p.k), dtype=torch.int32)
        a, b = row_range(rows, rank, world)
        sc, sl, ss, sr, so, ident = slice_args(scores, p.row_stride, seq, st, rtb, out, a, b)
        assert ident is None
        mine = topk_packed_reference(sc.numpy().reshape(-1), p.row_stride, sl.numpy(), ss.numpy(),
                                     sr.numpy(), p.page_table, p.pt_stride, p.page_size, p.k)
        # gather the shares (sizes differ by one at most: pad to the largest)
        size = max(row_range(rows, r, world)[1] - row_range(rows, r, world)[0] for r in range(world))
        buf = torch.full((size, p.k), -9, dtype=torch.int32)
        buf[: b - a] = torch.from_numpy(mine)
        parts = [torch.empty_like(buf) for _ in range(world)]
        dist.all_gather(parts, buf)
        if rank == 0:
            got = np.concatenate([parts[r][: row_range(rows, r, world)[1] - row_range(rows, r, world)[0]].numpy()
                                  for r in range(world)])
            want = topk_packed_reference(p.scores, p.row_stride, p.seq_lens, p.row_starts, p.row_to_batch,
                                         p.page_table, p.pt_stride, p.page_size, p.k)
            np.save(result_path, np.array([np.array_equal(got, want)]))
    finally:
        dist.destroy_process_group()


def test_two_ranks_gather_the_whole_batch(tmp_path):
    world = 2
    path = str(tmp_path / "ok.npy")
    mp.start_processes(_worker, args=(world, _free_port(), path), nprocs=world, start_method="spawn")
    assert bool(np.load(path)[0])
