"""The two further filters of the sampler chain (Muser book, "Ch 21 --
Sampling, argmax, and grammar", 21.7) on the GPU against the CPU oracle:
top-n-sigma (a mask at max - n * sigma of the row's logits, before top-k)
and locally typical sampling (after top-k, before top-p). Ids bit-exact
except where a decision lies within 1e-6 of its threshold; probabilities
within 1e-5 relative."""
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


def check(orc, x, u, T, k, p, m, nsig=0.0, typ=0.0, temp_last=False, misalign=False, max_mismatch=0):
    gi, gp = G.sample(x, u, T, k, p, m, temp_last, misalign, nsig, typ)
    ref = orc.sample(x, u, T, k, p, m, temp_last, top_n_sigma=nsig, typical_p=typ if typ > 0 else 1.0)
    G.assert_sample_matches(gi, gp, ref, max_mismatch)
    return gi, gp, ref


@pytest.mark.parametrize("nsig", [0.25, 0.5, 1.0, 2.0, 50.0])
def test_top_n_sigma(orc, nsig):
    x = synth.normal_rows(41, 48, 60_001, 3.0)
    u = synth.uniforms(42, 48)
    gi, _, ref = check(orc, x, u, 0.8, 40, 1.0, 0.0, nsig=nsig)
    # every drawn logit reaches max - n * sigma of its row
    thr = x.max(axis=1) - nsig * x.std(axis=1)
    ok = gi != G.INVALID
    assert np.all(x[np.arange(48)[ok], gi[ok]] >= thr[ok] - 1e-4)


def test_top_n_sigma_tiny_keeps_the_max(orc):
    """n so small that only the maximum reaches the threshold: greedy, P = 1."""
    x = synth.normal_rows(43, 16, 20_000, 2.0)
    u = synth.uniforms(44, 16)
    gi, gp, _ = check(orc, x, u, 1.0, 40, 0.9, 0.0, nsig=1e-6)
    assert np.array_equal(gi, orc.argmax(x)) and np.all(gp == 1.0)


@pytest.mark.parametrize("typ", [0.05, 0.2, 0.5, 0.9, 0.99])
@pytest.mark.parametrize("last", [False, True])
def test_typical_p(orc, typ, last):
    x = synth.normal_rows(45, 48, 40_003, 2.5)
    u = synth.uniforms(46, 48)
    check(orc, x, u, 0.9, 40, 1.0, 0.0, typ=typ, temp_last=last)


@pytest.mark.parametrize("k", [2, 7, 40, 84, 300])
def test_typical_p_with_the_rest_of_the_chain(orc, k):
    x = synth.normal_rows(47, 40, 30_001, 2.0)
    u = synth.uniforms(48, 40)
    check(orc, x, u, 0.7, k, 0.9, 0.05, nsig=1.5, typ=0.6)


def test_typical_off_values_change_nothing(orc):
    x = synth.normal_rows(49, 20, 10_000, 2.0)
    u = synth.uniforms(50, 20)
    base = G.sample(x, u, 0.8, 40, 0.9, 0.05)
    for typ in (0.0, 1.0):
        got = G.sample(x, u, 0.8, 40, 0.9, 0.05, typical_p=typ)
        assert np.array_equal(got[0], base[0]) and np.array_equal(got[1], base[1])


def test_filters_on_verify_batch(orc):
    """The full chain on the 49 x 248,320 Zipf/Gumbel verify batch."""
    x, _ = synth.workload_verify_batch()
    u = synth.uniforms(51, 49)
    check(orc, x, u, 0.7, 40, 0.9, 0.05, nsig=1.0, typ=0.8)


@pytest.mark.parametrize("misalign", [False, True])
def test_filters_ragged_rows(orc, misalign):
    """Ragged V (the scalar path when misaligned) and a row shorter than k."""
    x = synth.normal_rows(52, 9, 8_195, 1.5)
    u = synth.uniforms(53, 9)
    check(orc, x, u, 1.1, 64, 0.95, 0.0, nsig=0.75, typ=0.7, misalign=misalign)
    y = synth.normal_rows(54, 5, 31, 1.0)
    check(orc, y, synth.uniforms(55, 5), 1.0, 40, 1.0, 0.0, nsig=1.0, typ=0.5)


def test_nonfinite_row_fails_closed(orc):
    x = synth.normal_rows(56, 4, 5_000, 1.0)
    x[2, 77] = np.inf
    u = synth.uniforms(57, 4)
    gi, _, _ = check(orc, x, u, 1.0, 20, 1.0, 0.0, nsig=1.0, typ=0.5)
    assert gi[2] == G.INVALID and np.all(gi[[0, 1, 3]] != G.INVALID)
