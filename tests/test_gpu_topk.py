"""sel_topk on the GPU against the CPU oracle (bit-exact values and ids)."""
import numpy as np
import pytest

import oracle
import gpu_helpers as G
from sampling_row_fp32_gb300 import binding as B
from sampling_row_fp32_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    return oracle.default()


def check(orc, x, k, misalign=False):
    gv, gi = G.topk(x, k, misalign)
    ov, oi = orc.topk(x, k)
    bad = np.nonzero((gi != oi).any(axis=1))[0]
    assert bad.size == 0, (bad[:5], gi[bad[0]][:10], oi[bad[0]][:10])
    np.testing.assert_array_equal(gv, ov)


@pytest.mark.parametrize("rows,V,k", [
    (1, 1, 1), (2, 5, 3), (3, 16, 16), (2, 1000, 20), (4, 1025, 84), (3, 8192, 84),
    (3, 8193, 20), (5, 20_000, 40), (2, 65_537, 256), (2, 65_537, 257), (2, 100_000, 1024),
    (3, 202_048, 84), (2, 248_320, 1), (4, 300_000, 20), (70, 5000, 7),
    (3, 248_320, 128), (3, 248_320, 129)])
@pytest.mark.parametrize("misalign", [False, True])
def test_random_rows(orc, rows, V, k, misalign):
    x = synth.normal_rows(rows + V + k, rows, V, 2.0)
    check(orc, x, k, misalign)


@pytest.mark.parametrize("V,k", [(500, 20), (9000, 84), (70_000, 84), (248_320, 20)])
def test_many_ties(orc, V, k):
    """Integer-valued rows: the k-th boundary falls inside a run of equal
    values, which must be filled by the lowest ids."""
    rng = np.random.default_rng(V + k)
    x = rng.integers(0, 30, size=(6, V)).astype(np.float32)
    check(orc, x, k)


@pytest.mark.parametrize("V,k", [(100, 7), (20_000, 84), (248_320, 20), (248_320, 128), (248_320, 129),
                                 (248_320, 1024)])
def test_adversarial_rows(orc, V, k):
    """All-equal, ascending and descending rows overflow the candidate
    buffer or defeat the filters; the fallback paths stay exact."""
    asc = np.arange(V, dtype=np.float32)[None] / np.float32(V)
    x = np.concatenate([np.full((1, V), 1.5, dtype=np.float32), asc, asc[:, ::-1].copy(),
                        np.tile(np.float32([0.0, -0.0]), (1, V // 2 + 1))[:, :V]])
    check(orc, x, k)


def test_nonfinite_rows(orc):
    x = synth.normal_rows(8, 6, 70_000, 1.0)
    x[1, 3] = np.nan
    x[2, 69_999] = -np.inf
    x[4, 40_000] = np.inf
    gv, gi = G.topk(x, 20)
    ov, oi = orc.topk(x, 20)
    assert np.array_equal(gi, oi)
    assert np.all(gi[[1, 2, 4]] == G.INVALID) and np.all(np.isnan(gv[[1, 2, 4]]))
    np.testing.assert_array_equal(gv[[0, 3, 5]], ov[[0, 3, 5]])


def test_k_one_is_argmax(orc):
    x = synth.normal_rows(4, 9, 248_320, 3.0)
    _, gi = G.topk(x, 1)
    assert np.array_equal(gi[:, 0], G.argmax(x))


def test_peaked_topk_workload(orc):
    """3 x 248,320 ~N(0, 4) with 0.1 % of ids boosted by +8; k = 84."""
    x, k = synth.workload_topk_peaked()
    check(orc, x, k)


def test_verify_batch_topk_workload(orc):
    """49 x 248,320 Gumbel-perturbed Zipf(1.1) rows; k = 20."""
    x, k = synth.workload_verify_batch()
    check(orc, x, k)


def test_workspace_reuse_and_determinism(orc):
    x, k = synth.workload_verify_batch()
    ws = B.workspace(B.SEL_OP_TOPK, 49, x.shape[1], 84, device=G.device())
    ov, oi = orc.topk(x, 84)
    for _ in range(4):
        gv, gi = G.topk(x, 84, ws=ws)
        assert np.array_equal(gi, oi) and np.array_equal(gv, ov)
    gv, gi = G.topk(x[:5], 20, ws=ws)     # smaller k and rows fit the same workspace
    assert np.array_equal(gi, oi[:5, :20])
