"""sel_argmax on the GPU against the CPU oracle (bit-exact ids)."""
import numpy as np
import pytest
import torch

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


SHAPES = [(1, 1), (1, 2), (3, 5), (2, 1023), (2, 1024), (2, 1025), (4, 8191), (3, 8193),
          (5, 65_537), (2, 202_047), (3, 202_048), (7, 248_320), (130, 3000)]


@pytest.mark.parametrize("rows,V", SHAPES)
@pytest.mark.parametrize("misalign", [False, True])
def test_random_rows(orc, rows, V, misalign):
    x = synth.normal_rows(rows * 7 + V, rows, V, 3.0)
    assert np.array_equal(G.argmax(x, misalign), orc.argmax(x))


@pytest.mark.parametrize("V", [7, 1000, 33_333, 248_320])
def test_ties_keep_the_lower_id(orc, V):
    rng = np.random.default_rng(V)
    x = rng.integers(0, 4, size=(9, V)).astype(np.float32)   # many equal maxima
    assert np.array_equal(G.argmax(x), orc.argmax(x))
    assert np.array_equal(G.argmax(x, misalign=True), orc.argmax(x))


def test_planted_argmax_workload(orc):
    """1 x 202,048 ~N(0, 9), maximum planted at 3 ids: the lowest wins."""
    x, ids = synth.workload_argmax_planted()
    got = G.argmax(x)
    assert got[0] == ids[0] == orc.argmax(x)[0]


def test_partition_edges(orc):
    """Maximum at each chunk edge of 202,048 = 197 x 1,024 + 320 and in the tail."""
    import oracle_pins
    g = oracle_pins.golden("argmax_partition.json")
    base = synth.normal_rows(0, 1, g["V"], 3.0)[0]
    x = np.tile(base, (len(g["positions"]), 1))
    for r, pos in enumerate(g["positions"]):
        x[r, pos] = base.max() + 1
    got = G.argmax(x)
    assert got.tolist() == g["positions"]
    assert np.array_equal(got, orc.argmax(x))


def test_nonfinite_rows_fail_closed(orc):
    x = synth.normal_rows(5, 8, 50_000, 1.0)
    x[1, 0] = np.nan
    x[2, 49_999] = np.inf
    x[3, 12_345] = -np.inf
    x[4, 30_000] = np.nan
    x[4, 30_001] = 1e30
    got = G.argmax(x)
    assert np.array_equal(got, orc.argmax(x))
    assert np.all(got[1:5] == G.INVALID) and np.all(got[[0, 5, 6, 7]] != G.INVALID)


def test_signed_zeros_tie():
    x = np.array([[-1.0, -0.0, 0.0, -2.0], [-3.0, 0.0, -0.0, -1.0]], dtype=np.float32)
    assert G.argmax(x).tolist() == [1, 1]


def test_extreme_values(orc):
    x = np.full((3, 9000), -3.4e38, dtype=np.float32)
    x[1, 8999] = -3.3e38
    x[2, 4500] = 3.4e38
    x[2, 4501] = 3.4e38
    assert np.array_equal(G.argmax(x), orc.argmax(x))
    assert G.argmax(x).tolist() == [0, 8999, 4500]


def test_verify_batch_full_size(orc):
    """49 x 248,320 Gumbel-perturbed Zipf(1.1) rows, every id exact."""
    x, _ = synth.workload_verify_batch()
    assert np.array_equal(G.argmax(x), orc.argmax(x))


def test_workspace_reuse_and_determinism(orc):
    """Counters reset themselves: one workspace serves repeated calls and
    smaller batches; results are identical launch after launch."""
    x = synth.normal_rows(9, 49, 248_320, 2.0)
    x[:, ::977] = x.max()            # equal maxima spread across chunks
    ws = B.workspace(B.SEL_OP_ARGMAX, 49, 248_320, device=G.device())
    want = orc.argmax(x)
    for _ in range(5):
        assert np.array_equal(G.argmax(x, ws=ws), want)
    assert np.array_equal(G.argmax(x[:13], ws=ws), want[:13])


def test_stream_argument(orc):
    x = synth.normal_rows(3, 4, 100_000, 1.0)
    xd = G.to_dev(x)
    out = torch.empty(4, dtype=torch.int32, device=G.device())
    ws = B.workspace(B.SEL_OP_ARGMAX, 4, 100_000, device=G.device())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    B.sel_argmax(xd, out, ws, stream=s)
    s.synchronize()
    assert np.array_equal(B.ids_to_numpy(out), orc.argmax(x))


def test_undersized_workspace_is_refused():
    x = G.to_dev(synth.normal_rows(1, 2, 100_000, 1.0))
    out = torch.empty(2, dtype=torch.int32, device=G.device())
    need = B.sel_workspace_bytes(B.SEL_OP_ARGMAX, 2, 100_000)
    ws = torch.zeros(need - 8, dtype=torch.uint8, device=G.device())
    with pytest.raises(B.SelError) as e:
        B.sel_argmax(x, out, ws)
    assert e.value.status == B.SEL_EWORKSPACE
