"""Full-row sampling (sel_sample with top_k = 0) on the GPU against the CPU
oracle. The filters act on softmax(x / T) over the whole vocabulary (the
sampler chain of the Muser book, "Ch 21 -- Sampling, argmax, and grammar",
21.1 and 21.7, without top-k); the draw walks the survivors in ascending id.

Temperature alone, min-p, top-n-sigma, top-p and locally typical sampling
are decided on every row: a cut inside the row's 64 most probable tokens is
decided from them, one past them by the cut search over the whole row (a
radix select weighted by probability mass, on the value key for top-p and
on the distance to the typical logit for the typical window, exact ties
going to the lower ids; under top-n-sigma the search first sums the
candidate set's mass and mean log-weight over the row)."""
import numpy as np
import pytest
import torch

import oracle
import gpu_helpers as G
from sampling_row_fp32_gb300 import binding as B
from sampling_row_fp32_gb300 import synth

pytestmark = pytest.mark.gpu
CAND = 64
ERR_BEYOND = 8


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    return oracle.default()


def run(x, u, T, top_p, min_p, nsig=0.0, typ=0.0, temp_last=False, misalign=False):
    rows, V = x.shape
    xd = G.to_dev(x, misalign)
    ud = G.to_dev(np.asarray(u, dtype=np.float32).reshape(rows))
    ids = torch.full((rows,), G.SENTINEL, dtype=torch.int32, device=G.device())
    probs = torch.full((rows,), -7.0, dtype=torch.float32, device=G.device())
    ws = B.workspace(B.SEL_OP_SAMPLE, rows, V, 0, device=G.device())
    prm = B.SampleParams(T, 0, top_p, min_p, B.SEL_ORDER_TEMP_LAST if temp_last else B.SEL_ORDER_TEMP_FIRST,
                         nsig, typ)
    B.sel_sample(xd, prm, ud, ids, probs, ws)
    torch.cuda.synchronize()
    return B.ids_to_numpy(ids), probs.cpu().numpy(), G.ws_error(ws)


def nucleus_sizes(x, T, top_p):
    """Tokens in each row's top-p nucleus (double precision)."""
    z = x.astype(np.float64) / T
    z -= z.max(axis=1, keepdims=True)
    w = np.exp(z)
    w /= w.sum(axis=1, keepdims=True)
    c = np.cumsum(-np.sort(-w, axis=1), axis=1)
    return (c < top_p).sum(axis=1) + 1


def check(orc, x, u, T, top_p, min_p, nsig=0.0, typ=0.0, temp_last=False, misalign=False, decided=None):
    gi, gp, err = run(x, u, T, top_p, min_p, nsig, typ, temp_last, misalign)
    ref = orc.sample(x, u, T, 0, top_p, min_p, temp_last, top_n_sigma=nsig, typical_p=typ if typ > 0 else 1.0)
    failed = (gi == G.INVALID) & (ref.ids != G.INVALID)
    if decided is not None:
        assert np.array_equal(~failed, decided), (np.nonzero(failed != ~decided)[0][:10])
    assert bool(err & ERR_BEYOND) == bool(failed.any()), (err, failed.sum())
    assert err & ~ERR_BEYOND == 0, err
    assert np.all(np.isnan(gp[failed]))
    keep = ~failed
    G.assert_sample_matches(gi[keep], gp[keep], type(ref)(ref.ids[keep], ref.probs[keep], ref.margin[keep]))
    return gi, gp, ref, failed


@pytest.mark.parametrize("T", [0.5, 1.0, 1.7])
@pytest.mark.parametrize("misalign", [False, True])
def test_temperature_alone(orc, T, misalign):
    """No filter: every row decided, the draw over all V in ascending id."""
    x = synth.normal_rows(61, 40, 30_001, 2.0)
    u = synth.uniforms(62, 40)
    check(orc, x, u, T, 1.0, 0.0, misalign=misalign, decided=np.ones(40, bool))


@pytest.mark.parametrize("min_p", [0.001, 0.05, 0.3])
def test_min_p(orc, min_p):
    x = synth.normal_rows(63, 40, 60_001, 3.0)
    u = synth.uniforms(64, 40)
    check(orc, x, u, 0.8, 1.0, min_p, decided=np.ones(40, bool))


@pytest.mark.parametrize("nsig", [0.5, 1.0, 3.0])
def test_top_n_sigma(orc, nsig):
    x = synth.normal_rows(65, 32, 50_003, 2.5)
    u = synth.uniforms(66, 32)
    check(orc, x, u, 1.0, 1.0, 0.0, nsig=nsig, decided=np.ones(32, bool))


def test_top_p_on_verify_batch(orc):
    """49 x 248,320 Zipf/Gumbel rows at T 0.7, top_p 0.9: the rows whose
    nucleus fits the 64 candidates and the rows whose nucleus does not (the
    cut search) are all decided."""
    x, _ = synth.workload_verify_batch()
    u = synth.uniforms(67, 49)
    sizes = nucleus_sizes(x, 0.7, 0.9)
    assert (sizes > CAND).any() and (sizes <= CAND).mean() > 0.6
    check(orc, x, u, 0.7, 0.9, 0.0, decided=np.ones(49, bool))


@pytest.mark.parametrize("T,top_p", [(0.5, 0.9), (1.0, 0.5), (1.0, 0.95), (2.0, 0.3)])
@pytest.mark.parametrize("misalign", [False, True])
def test_top_p_past_the_candidates(orc, T, top_p, misalign):
    """Flat rows (N(0, 1.5^2)): every nucleus holds hundreds to thousands
    of tokens, so the cut search decides it; every row matches the oracle."""
    x = synth.normal_rows(68, 40, 30_001, 1.5)
    u = synth.uniforms(69, 40)
    assert (nucleus_sizes(x, T, top_p) > CAND).mean() > 0.5
    check(orc, x, u, T, top_p, 0.0, misalign=misalign, decided=np.ones(40, bool))


@pytest.mark.parametrize("nsig,min_p,temp_last", [(2.0, 0.0, False), (0.0, 0.01, False), (1.5, 0.02, True),
                                                  (0.0, 0.0, True)])
def test_top_p_search_with_the_other_filters(orc, nsig, min_p, temp_last):
    """The cut search under top-n-sigma (the candidates are the ids above
    max - n sigma), followed by min-p, and in the temperature-last order."""
    x = synth.normal_rows(76, 24, 50_000, 3.0)
    u = synth.uniforms(77, 24)
    check(orc, x, u, 1.3, 0.8, min_p, nsig=nsig, temp_last=temp_last, decided=np.ones(24, bool))


@pytest.mark.parametrize("top_p", [0.3, 0.5, 0.77])
def test_top_p_cut_inside_a_run_of_equal_logits(orc, top_p):
    """Integer-valued rows: thousands of ids share each value, so the cut
    falls inside a run of equal logits and takes its lowest ids only (the
    tie order of the chain)."""
    rng = np.random.default_rng(int(top_p * 100))
    x = rng.integers(0, 6, size=(12, 20_000)).astype(np.float32)
    u = synth.uniforms(78, 12)
    check(orc, x, u, 1.0, top_p, 0.0, decided=np.ones(12, bool))


def test_top_p_search_on_a_large_row(orc):
    """One flat row of 2,000,003 logits (a ragged tail, eight segments of a
    cluster that are not all equal)."""
    x = synth.normal_rows(79, 2, 2_000_003, 5.0)
    u = synth.uniforms(80, 2)
    check(orc, x, u, 1.0, 0.9, 0.0, decided=np.ones(2, bool))


def test_typical_search_on_a_large_row(orc):
    """Two flat rows of 2,000,003 logits: the typical window (then top-p
    inside it) found by the search on segments too long to stage in shared
    memory, so every pass reads the row from global memory."""
    x = synth.normal_rows(91, 2, 2_000_003, 4.0)
    u = synth.uniforms(92, 2)
    check(orc, x, u, 1.0, 0.9, 0.0, typ=0.6, decided=np.ones(2, bool))


def test_whole_chain_on_short_rows(orc):
    """V <= 64: the candidates hold the whole row, so every filter of the
    chain is decided, in both temperature orders."""
    x = synth.normal_rows(70, 30, 60, 2.0)
    u = synth.uniforms(71, 30)
    for last in (False, True):
        check(orc, x, u, 0.8, 0.9, 0.02, nsig=2.0, typ=0.7, temp_last=last, decided=np.ones(30, bool))


def test_typical_and_top_p_together(orc):
    x = synth.normal_rows(72, 30, 20_000, 3.0)
    u = synth.uniforms(73, 30)
    check(orc, x, u, 0.6, 0.9, 0.0, nsig=1.0, typ=0.8, decided=np.ones(30, bool))


@pytest.mark.parametrize("nsig,typ,top_p,temp_last", [(3.0, 0.6, 1.0, False), (2.0, 0.8, 0.7, False),
                                                      (4.0, 0.5, 0.9, True)])
def test_typical_under_top_n_sigma_past_the_candidates(orc, nsig, typ, top_p, temp_last):
    """Top-n-sigma keeps thousands of ids (a loose n), so the candidate set
    C runs past the 64: the search sums C's mass and mean log-weight over the
    row for the typical logit, then finds the window inside C."""
    x = synth.normal_rows(89, 24, 30_000, 1.5)
    u = synth.uniforms(90, 24)
    check(orc, x, u, 1.0, top_p, 0.0, nsig=nsig, typ=typ, temp_last=temp_last, decided=np.ones(24, bool))


def test_invalid_rows(orc):
    x = synth.normal_rows(74, 5, 9_000, 1.0)
    x[3, 10] = np.nan
    u = np.array([0.5, 1.0, -0.1, 0.5, 0.25], dtype=np.float32)
    gi, gp, _, _ = check(orc, x, u, 1.0, 1.0, 0.0, decided=np.ones(5, bool))
    assert np.all(gi[1:4] == G.INVALID) and gi[0] != G.INVALID and gi[4] != G.INVALID


def test_draw_walks_ascending_ids(orc):
    """Many uniforms against one row: the drawn id rises with u."""
    row = synth.normal_rows(75, 1, 5_000, 1.5)
    n = 2000
    x = np.tile(row, (n, 1))
    u = ((np.arange(n) + 0.5) / n).astype(np.float32)
    gi, _, _, _ = check(orc, x, u, 1.0, 1.0, 0.0, decided=np.ones(n, bool))
    assert np.all(np.diff(gi.astype(np.int64)) >= 0)


@pytest.mark.parametrize("V,misalign", [(20_001, False), (20_000, True), (16_671, True)])
def test_typical_on_scalar_path_rows(orc, V, misalign):
    """A locally typical cut needs the row's mean log-weight; rows that take
    the scalar loads (V % 4 != 0, or misaligned) end in a chunk where some
    threads hold only fill values, which must add nothing to it. Rows whose
    window lies inside the 64 candidates and rows whose window runs past them
    (the cut search) are all decided."""
    x = synth.normal_rows(81, 30, V, 3.0)
    u = synth.uniforms(82, 30)
    reach = typical_window_reach(x, 0.6, 0.8)
    assert (reach < CAND - 8).sum() >= 20 and (reach >= CAND).any()
    check(orc, x, u, 0.6, 1.0, 0.0, typ=0.8, misalign=misalign, decided=np.ones(30, bool))


@pytest.mark.parametrize("T,typ", [(1.0, 0.5), (0.7, 0.9), (1.5, 0.3), (1.0, 0.95)])
@pytest.mark.parametrize("misalign", [False, True])
def test_typical_past_the_candidates(orc, T, typ, misalign):
    """Flat rows (N(0, 1.5^2)): the typical window holds thousands of ids,
    so the cut search finds it over the row (a radix select on the distance
    to the typical logit, weighted by mass); every row matches the oracle."""
    x = synth.normal_rows(83, 32, 30_001, 1.5)
    u = synth.uniforms(84, 32)
    assert (typical_window_reach(x[:4], T, typ) >= CAND).all()
    check(orc, x, u, T, 1.0, 0.0, typ=typ, misalign=misalign, decided=np.ones(32, bool))


@pytest.mark.parametrize("top_p,min_p,temp_last", [(0.8, 0.0, False), (1.0, 0.05, False), (0.6, 0.01, True),
                                                   (0.9, 0.2, True)])
def test_typical_search_then_top_p_and_min_p(orc, top_p, min_p, temp_last):
    """After the window, top-p keeps the shortest prefix of the window (a
    second search inside it) and min-p compares with the window's most
    probable id; in both temperature orders."""
    x = synth.normal_rows(85, 24, 40_000, 2.0)
    u = synth.uniforms(86, 24)
    check(orc, x, u, 1.2, top_p, min_p, typ=0.7, temp_last=temp_last, decided=np.ones(24, bool))


@pytest.mark.parametrize("typ,top_p", [(0.4, 1.0), (0.65, 0.5), (0.9, 1.0)])
def test_typical_window_inside_a_run_of_equal_logits(orc, typ, top_p):
    """Integer-valued rows: thousands of ids share each value, so the
    window's edge falls inside a run of equal logits (one side of the
    typical logit), of which the lowest ids are kept: the chain's order
    among ids of equal score."""
    rng = np.random.default_rng(int(typ * 1000))
    x = rng.integers(0, 7, size=(12, 24_000)).astype(np.float32)
    u = synth.uniforms(87, 12)
    check(orc, x, u, 1.0, top_p, 0.0, typ=typ, decided=np.ones(12, bool))


def test_typical_on_verify_batch(orc):
    """The 49 verify rows at T 0.7 with typical_p 0.9: windows inside and
    past the 64 candidates, all decided."""
    x, _ = synth.workload_verify_batch()
    u = synth.uniforms(88, 49)
    check(orc, x, u, 0.7, 1.0, 0.0, typ=0.9, decided=np.ones(49, bool))


def typical_window_reach(x, T, typ):
    """Per row, the largest probability rank (0 = most probable) inside the
    locally typical window (double precision, ties by id)."""
    out = np.zeros(x.shape[0], dtype=np.int64)
    for r in range(x.shape[0]):
        z = x[r].astype(np.float64) / T
        z -= z.max()
        p = np.exp(z)
        p /= p.sum()
        lp = np.log(p)
        score = np.abs(-lp - (-(p * lp).sum()))
        order = np.lexsort((np.arange(p.size), score))
        n = int(np.searchsorted(np.cumsum(p[order]), typ) + 1)
        rank = np.empty(p.size, dtype=np.int64)
        rank[np.lexsort((np.arange(p.size), -p))] = np.arange(p.size)
        out[r] = rank[order[:n]].max()
    return out
