"""sel_sample on the GPU against the CPU oracle: ids bit-exact except where
u (or a top-p / min-p decision) lies within 1e-6 of its threshold,
probabilities within 1e-5 relative."""
import numpy as np
import pytest

import oracle
import gpu_helpers as G
from sampling_row_fp32_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    return oracle.default()


def check(orc, x, u, T, k, p, m, temp_last=False, misalign=False, max_mismatch=0):
    gi, gp = G.sample(x, u, T, k, p, m, temp_last, misalign)
    ref = orc.sample(x, u, T, k, p, m, temp_last)
    G.assert_sample_matches(gi, gp, ref, max_mismatch)
    return gi, gp, ref


def test_sampling_workload(orc):
    """64 x 202,048 ~N(0, 9), T 0.7, top_k 40, top_p 0.9, min_p 0.05."""
    x, u, pol = synth.workload_sample()
    check(orc, x, u, pol.temperature, pol.top_k, pol.top_p, pol.min_p)


def test_sampling_on_verify_batch(orc):
    """The same policy on the 49 x 248,320 Zipf/Gumbel verify batch."""
    x, _ = synth.workload_verify_batch()
    u = synth.uniforms(4, 49)
    check(orc, x, u, 0.7, 40, 0.9, 0.05)


@pytest.mark.parametrize("T,k,p,m,last", [
    (1.0, 40, 1.0, 0.0, False), (0.7, 40, 0.9, 0.05, True), (1.3, 84, 0.95, 0.0, False),
    (0.5, 20, 1.0, 0.1, False), (2.0, 300, 0.5, 0.02, False), (1.0, 1024, 0.99, 0.0, False),
    (0.9, 5, 0.3, 0.0, True)])
@pytest.mark.parametrize("misalign", [False, True])
def test_policies(orc, T, k, p, m, last, misalign):
    x = synth.normal_rows(17, 40, 30_001, 2.5)
    u = synth.uniforms(18, 40)
    check(orc, x, u, T, k, p, m, last, misalign)


def test_many_draws_on_one_row(orc):
    """2,000 uniforms against the same row sweep the CDF of the candidates."""
    row = synth.normal_rows(21, 1, 50_000, 2.0)
    x = np.tile(row, (2000, 1))
    u = synth.uniforms(22, 2000)
    gi, _, ref = check(orc, x, u, 0.8, 40, 0.95, 0.01)
    assert len(set(gi.tolist())) > 10


def test_greedy_and_top1(orc):
    x = synth.normal_rows(23, 12, 70_000, 2.0)
    x[3, [5, 60_000]] = x[3].max() + 1
    u = synth.uniforms(24, 12)
    want = orc.argmax(x)
    for T, k in ((0.0, 40), (0.0, 0), (0.7, 1)):
        gi, gp, _ = check(orc, x, u, T, k, 0.9, 0.05)
        assert np.array_equal(gi, want) and np.all(gp == 1.0)


def test_top_k_beyond_v(orc):
    x = synth.normal_rows(25, 3, 50, 1.0)
    u = synth.uniforms(26, 3)
    check(orc, x, u, 1.0, 500, 1.0, 0.0)


def test_invalid_rows(orc):
    x = synth.normal_rows(27, 6, 9000, 1.0)
    x[4, 100] = np.nan
    u = np.array([0.5, 1.0, -0.25, np.nan, 0.5, 0.999999], dtype=np.float32)
    gi, gp, ref = check(orc, x, u, 0.7, 40, 0.9, 0.05)
    assert np.all(gi[1:5] == G.INVALID) and gi[0] != G.INVALID and gi[5] != G.INVALID
