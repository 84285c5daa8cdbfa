"""Vocabulary shards on one GPU: each row is split into G id ranges, each
range runs sel_topk on its own slice (shard-local ids), and the gathered
lists merge through sel_merge_shards / sel_sample_shards. The merged top k
must equal sel_topk on the whole row and the oracle bit for bit; the merged
sample must equal sel_sample on the whole row (same candidates, same
policy, same u) and match the oracle."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_fp32_gb300 import binding as B, shards, synth
from gpu_helpers import INVALID, assert_sample_matches, device, sample, to_dev, topk

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def shard_lists(x: np.ndarray, G: int, k: int):
    """Per-shard sel_topk over contiguous slices, stacked [rows][G][k]."""
    rows, V = x.shape
    offs = shards.shard_offsets(V, G, min_size=k)
    vals, ids = [], []
    for g in range(G):
        v, i = topk(np.ascontiguousarray(x[:, offs[g]:offs[g + 1]]), k)
        vals.append(v)
        ids.append(i)
    return offs, np.stack(vals, axis=1), np.stack(ids, axis=1)


def merge(vals, ids, offs):
    rows, G, k = vals.shape
    ov = torch.full((rows, k), -7.0, device=device())
    oi = torch.full((rows, k), -7, dtype=torch.int32, device=device())
    B.sel_merge_shards(to_dev(vals), to_dev(ids.view(np.int32)), offs, ov, oi)
    torch.cuda.synchronize()
    return ov.cpu().numpy(), B.ids_to_numpy(oi)


@pytest.mark.parametrize("rows,V,G,k", [(3, 248_320, 2, 84), (49, 248_320, 3, 20), (5, 202_048, 5, 40),
                                        (4, 10_007, 7, 1), (2, 4_100, 2, 1024), (1, 64, 16, 4)])
def test_merged_topk_equals_whole_row(orc, rows, V, G, k):
    x = synth.normal_rows(31 + G, rows, V, 2.0)
    x[:, ::997] = np.round(x[:, ::997])  # equal values across shard seams
    offs, vals, ids = shard_lists(x, G, k)
    mv, mi = merge(vals, ids, offs)
    ov, oi = orc.topk(x, k)
    assert np.array_equal(mi, oi)
    assert np.array_equal(mv, ov)
    wv, wi = topk(x, k)
    assert np.array_equal(mi, wi) and np.array_equal(mv, wv)


def test_ties_across_shards_go_to_the_lower_global_id(orc):
    V, G, k = 4_096, 4, 8
    x = np.full((2, V), -5.0, dtype=np.float32)
    x[0, [5, 1030, 2100, 4000]] = 3.0          # one maximum in each shard
    x[1, [4095, 0, 2048]] = 1.0
    offs, vals, ids = shard_lists(x, G, k)
    mv, mi = merge(vals, ids, offs)
    assert list(mi[0, :4]) == [5, 1030, 2100, 4000]
    assert list(mi[1, :3]) == [0, 2048, 4095]
    ov, oi = orc.topk(x, k)
    assert np.array_equal(mi, oi)


def test_argmax_is_the_k1_merge(orc):
    x, planted = synth.planted_argmax(seed=0)
    offs, vals, ids = shard_lists(x, 3, 1)
    _, mi = merge(vals, ids, offs)
    assert mi[0, 0] == planted.min() == orc.argmax(x)[0]


def test_a_nonfinite_shard_fails_the_row_closed():
    x = synth.normal_rows(41, 3, 30_000, 2.0)
    x[1, 25_000] = np.inf
    offs, vals, ids = shard_lists(x, 3, 10)
    assert np.all(ids[1, 2] == INVALID)
    mv, mi = merge(vals, ids, offs)
    assert np.all(mi[1] == INVALID) and np.all(np.isnan(mv[1]))
    assert np.all(mi[[0, 2]] != INVALID)


def test_malformed_lists_fail_the_row_closed():
    x = synth.normal_rows(42, 3, 8_192, 2.0)
    offs, vals, ids = shard_lists(x, 2, 6)
    ids = ids.copy()
    vals = vals.copy()
    ids[0, 1, 2] = offs[2] - offs[1]            # id outside its shard
    vals[2, 0, 1], vals[2, 0, 3] = vals[2, 0, 3], vals[2, 0, 1]  # list out of order
    mv, mi = merge(vals, ids, offs)
    assert np.all(mi[0] == INVALID) and np.all(mi[2] == INVALID)
    assert np.all(mi[1] != INVALID)


@pytest.mark.parametrize("G,temp_last", [(2, False), (3, True), (4, False)])
def test_merged_sample_equals_whole_row(orc, G, temp_last):
    rows, V = 64, 202_048
    x, u, pol = synth.workload_sample(rows, V)
    offs, vals, ids = shard_lists(x, G, pol.top_k)
    prm = B.SampleParams(pol.temperature, pol.top_k, pol.top_p, pol.min_p,
                         B.SEL_ORDER_TEMP_LAST if temp_last else B.SEL_ORDER_TEMP_FIRST)
    oi = torch.full((rows,), -7, dtype=torch.int32, device=device())
    op = torch.full((rows,), -7.0, device=device())
    B.sel_sample_shards(to_dev(vals), to_dev(ids.view(np.int32)), offs, prm, to_dev(u), oi, op)
    torch.cuda.synchronize()
    got_i, got_p = B.ids_to_numpy(oi), op.cpu().numpy()
    whole_i, whole_p = sample(x, u, pol.temperature, pol.top_k, pol.top_p, pol.min_p, temp_last)
    assert np.array_equal(got_i, whole_i)
    assert np.array_equal(got_p, whole_p)
    ref = orc.sample(x, u, pol.temperature, pol.top_k, pol.top_p, pol.min_p, temp_last)
    assert_sample_matches(got_i, got_p, ref)


def test_sample_shards_greedy_and_policy_check():
    rows, V, k = 4, 50_000, 5
    x = synth.normal_rows(43, rows, V, 2.0)
    offs, vals, ids = shard_lists(x, 2, k)
    u = synth.uniforms(44, rows)
    oi = torch.empty(rows, dtype=torch.int32, device=device())
    op = torch.empty(rows, device=device())
    B.sel_sample_shards(to_dev(vals), to_dev(ids.view(np.int32)), offs, B.SampleParams(0.0, 0, 1.0, 0.0, 0),
                        to_dev(u), oi, op)
    torch.cuda.synchronize()
    assert np.array_equal(B.ids_to_numpy(oi), np.argmax(x, axis=1).astype(np.uint32))
    assert np.all(op.cpu().numpy() == 1.0)
    with pytest.raises(B.SelError):  # top_k must equal the lists' k when T > 0
        B.sel_sample_shards(to_dev(vals), to_dev(ids.view(np.int32)), offs,
                            B.SampleParams(1.0, k + 1, 1.0, 0.0, 0), to_dev(u), oi, op)
