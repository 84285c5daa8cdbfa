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


def _rank_stats_main(rank, world, port, out_dir):
    """Each rank: a statistics record per row of its slice (packed as
    sel_row_stats), its survivor masses, and a draw output in which it holds
    the id of some rows; then the gathers and the combine."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rows, V = 4, 1000
        x = synth.normal_rows(22, rows, V, 2.0)
        lo, hi = shards.shard_range(V, world, rank)
        rec = np.zeros(rows, dtype=shards.ROW_STATS_DTYPE)
        xs = x[:, lo:hi].astype(np.float64)
        rec["max"] = x[:, lo:hi].max(axis=1)
        rec["x0"] = x[:, lo]
        rec["n"] = hi - lo
        rec["s1"] = (xs - xs[:, :1]).sum(axis=1)
        rec["z"] = np.exp(xs - xs.max(axis=1, keepdims=True)).sum(axis=1)
        st = torch.from_numpy(rec.view(np.uint8).reshape(rows, 48).copy())
        gs = shards.gather_stats(st)
        mass = torch.tensor([float(rank + 1), 0.5 * rank, 2.0, 0.0], dtype=torch.float64)
        gm = shards.gather_masses(mass)
        # row 0: rank 1 holds the draw; row 1: rank 0; row 2: failed everywhere;
        # row 3: rank 0 holds id 0 (the smallest id)
        ids = torch.tensor([shards.OTHER_SHARD if rank == 0 else 700, 5 if rank == 0 else shards.OTHER_SHARD,
                            0xFFFFFFFF, 0 if rank == 0 else shards.OTHER_SHARD], dtype=torch.int64)
        ids = torch.from_numpy(ids.numpy().astype(np.uint32).view(np.int32))
        probs = torch.tensor([0.0 if rank == 0 else 0.25, 0.125 if rank == 0 else 0.0, float("nan"),
                              1.0 if rank == 0 else 0.0], dtype=torch.float32)
        ci, cp = shards.combine_draws(ids, probs)
        np.save(os.path.join(out_dir, f"stats{rank}.npy"), gs.numpy())
        np.save(os.path.join(out_dir, f"mass{rank}.npy"), gm.numpy())
        np.save(os.path.join(out_dir, f"cid{rank}.npy"), ci.numpy())
        np.save(os.path.join(out_dir, f"cp{rank}.npy"), cp.numpy())
    finally:
        dist.destroy_process_group()


def test_stats_masses_and_draws_between_two_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_stats_main, args=(world, _free_port(), str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    x = synth.normal_rows(22, 4, 1000, 2.0)
    offs = shards.shard_offsets(1000, world)
    for rank in range(world):
        gs = np.load(tmp_path / f"stats{rank}.npy")
        assert gs.shape == (4, world, 48)
        rec = gs.view(shards.ROW_STATS_DTYPE)[..., 0]
        for g in range(world):  # shard order = rank order
            assert np.all(rec["n"][:, g] == offs[g + 1] - offs[g])
            assert np.array_equal(rec["x0"][:, g], x[:, offs[g]])
            assert np.array_equal(rec["max"][:, g], x[:, offs[g]:offs[g + 1]].max(axis=1))
        gm = np.load(tmp_path / f"mass{rank}.npy")
        assert np.array_equal(gm, np.array([[1.0, 2.0], [0.0, 0.5], [2.0, 2.0], [0.0, 0.0]]))
        ci = np.load(tmp_path / f"cid{rank}.npy")
        cp = np.load(tmp_path / f"cp{rank}.npy")
        assert list(ci) == [700, 5, 0xFFFFFFFF, 0]
        assert cp[0] == 0.25 and cp[1] == 0.125 and np.isnan(cp[2]) and cp[3] == 1.0


def test_full_row_list_len_and_local_combine():
    assert shards.full_row_list_len([0, 100, 200]) == 64
    assert shards.full_row_list_len([0, 40, 200]) == 40
    ids = [torch.tensor([-2, 3, -1], dtype=torch.int32), torch.tensor([9, -2, -1], dtype=torch.int32)]
    probs = [torch.tensor([0.0, 0.5, float("nan")]), torch.tensor([0.75, 0.0, float("nan")])]
    ci, cp = shards.combine_draws_local(ids, probs)
    assert ci.tolist() == [9, 3, 0xFFFFFFFF]
    assert cp[0] == 0.75 and cp[1] == 0.5 and torch.isnan(cp[2])


def _rank_spec_main(rank, world, port, out_dir):
    """Each rank: its spec parts (bytes that name the rank), its draw masses,
    and an emitted array in which it holds the drawn token of some
    sequences; then the gathers and the combine."""
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        S, K = 3, 2
        parts = torch.full((S, 2 * K + 1, 32), rank + 1, dtype=torch.uint8)
        gp = shards.gather_parts(parts)
        mass = torch.tensor([[0.25 * rank, 1.0], [0.0, 0.5 + rank], [3.0, 3.0]], dtype=torch.float64)
        gm = shards.gather_spec_masses(mass)
        # every rank wrote t_0..t_{n-1} the same way; the drawn slot (n) holds
        # the token on one rank and SEL_OTHER_SHARD on the others
        other = shards.OTHER_SHARD
        inv = 0xFFFFFFFF
        rows = [[11, 12, 900 if rank == 1 else other],
                [40 if rank == 0 else other, inv, inv],
                [inv, inv, inv]]
        em = torch.from_numpy(np.array(rows, dtype=np.uint32).view(np.int32))
        ce = shards.combine_emitted(em)
        np.save(os.path.join(out_dir, f"gp{rank}.npy"), gp.numpy())
        np.save(os.path.join(out_dir, f"gm{rank}.npy"), gm.numpy())
        np.save(os.path.join(out_dir, f"ce{rank}.npy"), ce.numpy())
    finally:
        dist.destroy_process_group()


def test_spec_parts_masses_and_emitted_between_two_ranks(tmp_path):
    world = 2
    mp.start_processes(_rank_spec_main, args=(world, _free_port(), str(tmp_path)),
                       nprocs=world, join=True, start_method="spawn")
    for rank in range(world):
        gp = np.load(tmp_path / f"gp{rank}.npy")
        assert gp.shape == (3, world, 5, 32)
        assert np.all(gp[:, 0] == 1) and np.all(gp[:, 1] == 2)  # shard order = rank order
        gm = np.load(tmp_path / f"gm{rank}.npy")
        assert gm.shape == (3, world, 2)
        assert np.array_equal(gm[0], [[0.0, 1.0], [0.25, 1.0]]) and np.array_equal(gm[1], [[0.0, 0.5], [0.0, 1.5]])
        ce = np.load(tmp_path / f"ce{rank}.npy")
        assert ce.tolist() == [[11, 12, 900], [40, 0xFFFFFFFF, 0xFFFFFFFF], [0xFFFFFFFF] * 3]
