"""The seeded input generators against the recipes they state (no GPU):
shapes, dtypes, value ranges, the planted and boosted structure, the shared
Zipf permutation under per-row Gumbel noise, the draft noise level, and the
Gumbel-max draft tokens' law. Both the CUDA path and the oracle read these
bytes, so a wrong recipe would go unseen by parity alone."""
import math

import numpy as np
import pytest

import oracle_pins
from sampling_row_fp32_gb300 import synth


def test_uniforms_are_float32_in_the_half_open_unit_interval():
    u = synth.uniforms(4, 200_000)
    assert u.dtype == np.float32 and u.shape == (200_000,)
    assert float(u.min()) >= 0.0 and float(u.max()) < 1.0
    assert np.array_equal(u, synth.uniforms(4, 200_000))
    assert not np.array_equal(u, synth.uniforms(5, 200_000))
    assert abs(float(u.mean()) - 0.5) < 0.005


def test_planted_argmax_has_exactly_its_three_maxima():
    x, ids = synth.workload_argmax_planted()
    assert x.dtype == np.float32 and x.shape == (1, synth.V_MUSER)
    top = np.flatnonzero(x[0] == x.max())
    assert np.array_equal(top, ids) and ids.size == 3
    rest = np.delete(x[0], ids)
    # the plant is the row's original maximum plus 1, so at least 1 above the rest
    assert float(x.max()) >= float(rest.max()) + 1.0 - 1e-5
    assert abs(float(rest.std()) - 3.0) < 0.03


def test_peaked_rows_carry_the_boosted_head():
    x, k = synth.workload_topk_peaked()
    assert k == 84 and x.dtype == np.float32 and x.shape == (3, synth.V_QWEN)
    n_boost = int(0.001 * synth.V_QWEN)  # 248
    for row in x:
        # N(0, 2^2) reaches 8 about 8 times in 248,320 draws; the 248 ids
        # boosted by +8 put about half of themselves there
        above = int(np.sum(row > 8.0))
        assert n_boost // 4 < above < n_boost, above
        assert abs(float(np.median(row))) < 0.02
        assert abs(float(np.percentile(row, 84.13)) - 2.0) < 0.05


def test_verify_batch_shares_one_zipf_permutation_under_gumbel_noise():
    x, k = synth.workload_verify_batch()
    assert k == 20 and x.dtype == np.float32 and x.shape == (49, synth.V_QWEN)
    # two rows differ only by their noise: G1 - G2 has variance pi^2 / 3
    d = x[0].astype(np.float64) - x[1].astype(np.float64)
    assert abs(float(d.var()) - math.pi ** 2 / 3) < 0.05
    assert abs(float(d.mean())) < 0.02
    # the column means follow the shared Zipf log-probabilities: the head
    # sits where the permutation put rank 1, not at id 0
    head = int(np.argmax(x.mean(axis=0)))
    assert head != 0
    # Zipf(1.1): the head's log-probability exceeds the 10th rank's by
    # 1.1 ln 10; the column means keep that gap within the noise of 49 rows
    m = np.sort(x.mean(axis=0).astype(np.float64))[::-1]
    assert 1.1 * math.log(10) - 1.0 < m[0] - m[9] < 1.1 * math.log(10) + 1.0


def test_sample_workload_and_policy():
    x, u, pol = synth.workload_sample()
    assert x.dtype == np.float32 and x.shape == (64, synth.V_MUSER)
    assert u.dtype == np.float32 and u.shape == (64,) and float(u.max()) < 1.0
    assert (pol.temperature, pol.top_k, pol.top_p, pol.min_p, pol.temp_last) == (0.7, 40, 0.9, 0.05, False)
    assert abs(float(x.std()) - 3.0) < 0.01


def test_spec_workload_draft_noise_and_tokens():
    si = synth.workload_spec()
    S, K, V = 8, 8, synth.V_SPEC
    assert si.target.shape == (S, K + 1, V) and si.draft.shape == (S, K, V)
    assert si.draft_tokens.dtype == np.uint32 and si.draft_tokens.shape == (S, K)
    assert int(si.draft_tokens.max()) < V
    assert si.u_acc.shape == (S, K) and si.u_fin.shape == (S,)
    assert float(max(si.u_acc.max(), si.u_fin.max())) < 1.0 and float(min(si.u_acc.min(), si.u_fin.min())) >= 0.0
    noise = si.draft.astype(np.float64) - si.target[:, :K].astype(np.float64)
    assert abs(float(noise.std()) - 0.5) < 0.002
    assert abs(float(si.target.std()) - 2.0) < 0.005
    # the same seeds give the same bytes
    again = synth.workload_spec()
    assert np.array_equal(again.draft_tokens, si.draft_tokens) and np.array_equal(again.draft, si.draft)


def test_given_target_rows_are_used_as_they_are():
    t = np.arange(2 * 3 * 8, dtype=np.float32).reshape(2, 3, 8)
    si = synth.spec_inputs(S=2, K=2, V=8, target=t)
    assert np.array_equal(si.target, t)


@pytest.mark.parametrize("T", [1.0, 0.5])
def test_gumbel_max_draft_tokens_follow_the_softmax(T):
    """Argmax of logits / T plus standard Gumbel noise samples
    softmax(logits / T) exactly: 12,000 draws over 6 ids against it by the
    chi-square recipe (dof 5, reject above 25.7448)."""
    g = oracle_pins.golden("chi_square_recipe.json")
    logits = np.array([1.0, 0.0, -0.5, 2.0, 0.3, -1.0], dtype=np.float32)
    rows = np.broadcast_to(logits, (g["samples"], logits.size))
    draws = synth.gumbel_max_draws(11, rows, T)
    z = logits.astype(np.float64) / T
    p = np.exp(z - z.max())
    p /= p.sum()
    counts = np.bincount(draws.astype(np.int64), minlength=logits.size)
    assert oracle_pins.chi_square(counts, p) <= g["critical"]
