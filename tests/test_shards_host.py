"""Host side of vocabulary sharding (no GPU): the split into id ranges, and
the all-gather of per-shard lists between ranks, run as world-size-2 gloo
process groups on the CPU. The per-shard lists come from the oracle; the
check is that the gathered [rows][G][k] layout, with each shard's offset
added, holds the top k of the unsharded row."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from sampling_row_fp32_gb300 import shards, synth


def test_offsets_split_and_align():
    for V in (1, 4, 7, 1000, 1025, 151_936, 202_048, 248_320):
        for G in (1, 2, 3, 5, 8):
            try:
                offs = shards.shard_offsets(V, G)
            except ValueError:
                assert V < 4 * G  # only tiny rows cannot be split on 4-element boundaries
                continue
            assert offs[0] == 0 and offs[-1] == V and len(offs) == G + 1
            assert all(offs[g] < offs[g + 1] for g in range(G))
            assert all(o % 4 == 0 for o in offs[1:-1])
            sizes = np.diff(offs)
            assert sizes.max() - sizes.min() <= 4 + 3  # near-equal


def test_offsets_reject_too_small_shards():
    with pytest.raises(ValueError):
        shards.shard_offsets(100, 2, min_size=60)
    assert shards.shard_offsets(248_320, 2, min_size=84) == [0, 124_160, 248_320]
    with pytest.raises(ValueError):
        shards.shard_offsets(10, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, V, rows, k, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        orc = oracle.default()
        x = synth.normal_rows(21, rows, V, 2.0)
        lo, hi = shards.shard_range(V, world, rank, min_size=k)
        vals, ids = orc.topk(np.ascontiguousarray(x[:, lo:hi]), k)
        gv, gi = shards.gather_lists(torch.from_numpy(vals), torch.from_numpy(ids.view(np.int32)))
        np.save(os.path.join(out_dir, f"vals{rank}.npy"), gv.numpy())
        np.save(os.path.join(out_dir, f"ids{rank}.npy"), gi.numpy())
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("V,k", [(1000, 7), (248_320, 20)])
def test_gather_two_ranks_holds_the_row_top_k(tmp_path, V, k):
    world, rows = 2, 3
    mp.start_processes(_rank_main, args=(world, _free_port(), V, rows, k, str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    import oracle
    orc = oracle.default()
    x = synth.normal_rows(21, rows, V, 2.0)
    want_vals, want_ids = orc.topk(x, k)
    offs = shards.shard_offsets(V, world, min_size=k)
    for rank in range(world):  # every rank holds the same gathered lists
        gv = np.load(tmp_path / f"vals{rank}.npy")
        gi = np.load(tmp_path / f"ids{rank}.npy").view(np.uint32)
        assert gv.shape == (rows, world, k) and gi.shape == (rows, world, k)
        for r in range(rows):
            glob = np.concatenate([gi[r, g].astype(np.int64) + offs[g] for g in range(world)])
            v = gv[r].reshape(-1)
            order = np.lexsort((glob, -v.astype(np.float64)))[:k]
            assert np.array_equal(glob[order], want_ids[r].astype(np.int64))
            assert np.array_equal(v[order], want_vals[r])
