"""spec_accept on the GPU against the CPU oracle, plus the statistical laws
of the rejection rule measured on the GPU's own output stream."""
import math

import numpy as np
import pytest

import oracle
import oracle_pins
import gpu_helpers as G
from sampling_row_fp32_gb300 import binding as B
from sampling_row_fp32_gb300 import synth

pytestmark = pytest.mark.gpu
REJ, ARG = B.SPEC_MODE_REJECTION, B.SPEC_MODE_ARGMAX


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    return oracle.default()


def run_both(orc, si, mode, misalign=False, max_mismatch=0):
    acc, emi = G.spec(si.target, si.draft, si.draft_tokens, si.u_acc, si.u_fin,
                      si.temperature, mode, misalign)
    ref = orc.spec_accept(si.target, si.draft, si.draft_tokens, si.temperature, mode,
                          si.u_acc, si.u_fin)
    G.assert_spec_matches(acc, emi, ref, max_mismatch)
    return acc, emi, ref


@pytest.mark.parametrize("mode", [REJ, ARG])
def test_spec_workload(orc, mode):
    """8 sequences x 8 drafts, V = 151,936, draft = target + N(0, 0.25)."""
    run_both(orc, synth.workload_spec(), mode)


@pytest.mark.parametrize("S,K,V,T", [(3, 1, 5, 1.0), (4, 3, 1000, 0.8), (5, 4, 8191, 1.0),
                                     (2, 8, 33_333, 1.3), (6, 2, 248_320, 1.0), (9, 0, 4096, 1.0),
                                     (3, 3, 100_000, 1.0), (4, 2, 50_000, 0.9), (2, 2, 300_000, 1.0)])
@pytest.mark.parametrize("misalign", [False, True])
@pytest.mark.parametrize("mode", [REJ, ARG])
def test_shapes(orc, S, K, V, T, misalign, mode):
    si = synth.spec_inputs(S=S, K=K, V=V, temperature=T, seed_target=S + K, seed_draft=V,
                           seed_u=int(T * 10) + 3, sigma_noise=0.7)
    run_both(orc, si, mode, misalign)


def _head(si, n, start=0):
    """Sequences start .. start + n - 1 of a SpecInputs."""
    sl = slice(start, start + n)
    return synth.SpecInputs(si.target[sl], si.draft[sl], si.draft_tokens[sl], si.u_acc[sl], si.u_fin[sl],
                            si.temperature)


def test_both_draw_paths_agree(orc):
    """Twelve sequences over V = 248,320 take the two-launch draw (twelve
    clusters of 16 CTAs do not fit on the GPU at once); the first seven
    alone take the one-launch cluster draw. Both match the oracle, and so
    each other."""
    si = synth.spec_inputs(S=12, K=3, V=248_320, seed_target=5, seed_draft=6, seed_u=7, sigma_noise=0.7)
    acc, emi, ref = run_both(orc, si, REJ)
    assert np.any(acc < 3) and np.any(acc == 3)  # residual and bonus draws both occur
    acc7, emi7, _ = run_both(orc, _head(si, 7), REJ)
    np.testing.assert_array_equal(acc7, acc[:7])
    np.testing.assert_array_equal(emi7, emi[:7])


def test_bench_workload(orc):
    """7 sequences x 6 drafts over the 49 x 248,320 verify batch as targets."""
    x, _ = synth.workload_verify_batch()
    si = synth.spec_inputs(S=7, K=6, V=x.shape[1], target=x.reshape(7, 7, -1))
    run_both(orc, si, REJ)
    run_both(orc, si, ARG)


@pytest.mark.parametrize("S,K,V,equal_upto", [(2, 70, 3000, 66), (3, 66, 1000, 66), (1, 1, 8_400_001, 0)])
def test_separate_decision_launch(orc, S, K, V, equal_upto):
    """Shapes past the fused decision launch's limits (more than 64 drafts,
    or more than 1,024 phase-1 chunks per row) take the separate merge
    launch. Drafts equal to the target up to position 66 are accepted
    whatever u is, so those chains pass position 64 and read their logits
    past the prefetched ones; the residual or bonus draw then reads rows
    past position 64."""
    si = synth.spec_inputs(S=S, K=K, V=V, seed_target=K + 1, seed_draft=V, seed_u=S + 11, sigma_noise=0.7)
    if equal_upto:
        si.draft[:, :equal_upto] = si.target[:, :equal_upto]
    acc, _, _ = run_both(orc, si, REJ)
    if equal_upto:
        assert np.all(acc >= equal_upto)
    run_both(orc, si, ARG)


@pytest.mark.parametrize("K", [1, 31, 32, 40])
def test_argmax_rule_long_chains(orc, K):
    """Drafts that match the targets' argmax for a prefix of every length
    (0 .. K, so some sequences accept all K and emit the bonus argmax):
    the one-warp decision up to K = 31 and the block decision above it."""
    S, V = K + 1, 5000
    si = synth.spec_inputs(S=S, K=K, V=V, seed_target=K + 40, seed_draft=K + 41, seed_u=K + 42)
    best = si.target.argmax(axis=2).astype(np.uint32)   # first maximum, as the rule's argmax
    for s_ in range(S):
        si.draft_tokens[s_, :s_] = best[s_, :s_]
        if s_ < K:
            si.draft_tokens[s_, s_] = (best[s_, s_] + 1) % V
    acc, emi, ref = run_both(orc, si, ARG)
    assert np.array_equal(acc, np.arange(S))


def test_temperature_zero_is_the_argmax_rule(orc):
    si = synth.spec_inputs(S=6, K=4, V=9000, temperature=1.0, sigma_noise=0.1)
    a0, e0 = G.spec(si.target, si.draft, si.draft_tokens, si.u_acc, si.u_fin, 0.0, REJ)
    a1, e1 = G.spec(si.target, None, si.draft_tokens, None, None, 1.0, ARG)
    assert np.array_equal(a0, a1) and np.array_equal(e0, e1)
    ref = orc.spec_accept(si.target, None, si.draft_tokens, 1.0, ARG)
    assert np.array_equal(a1, ref.accepted) and np.array_equal(e1, ref.emitted)


def test_invalid_sequences(orc):
    si = synth.spec_inputs(S=6, K=3, V=5000)
    si.target[1, 2, 17] = np.nan
    si.draft[2, 0, 4999] = np.inf
    si.draft_tokens[3, 1] = 5000           # token >= V
    si.u_acc[4, 2] = 1.0                   # uniform outside [0, 1)
    si.u_fin[5] = -0.5
    acc, emi, ref = run_both(orc, si, REJ)
    assert np.all(acc[1:] == G.INVALID) and np.all(emi[1:] == G.INVALID) and acc[0] != G.INVALID
    acc, emi, ref = run_both(orc, si, ARG)   # the argmax rule reads no draft row or uniform
    assert acc[1] == G.INVALID and acc[3] == G.INVALID and acc[2] != G.INVALID


def _rounds(p, q, n, seed, K=1, bonus=None):
    rng = np.random.default_rng(seed)
    V = p.size
    lp, lq = oracle_pins._logits_from(p), oracle_pins._logits_from(q)
    lb = oracle_pins._logits_from(p if bonus is None else bonus)
    target = np.empty((n, K + 1, V), dtype=np.float32)
    target[:, :K] = lp
    target[:, K] = lb
    draft = np.empty((n, K, V), dtype=np.float32)
    draft[:] = lq
    tokens = rng.choice(V, size=(n, K), p=q / q.sum()).astype(np.uint32)
    return synth.SpecInputs(target, draft, tokens, rng.random((n, K), dtype=np.float32),
                            rng.random(n, dtype=np.float32), 1.0)


def test_stream_matches_target_by_chi_square(orc):
    """The GPU's emitted stream against the exact categorical p: 12,000
    tokens, dof 5, reject above 25.7448 (the mlxcel regression guard)."""
    g = oracle_pins.golden("chi_square_recipe.json")
    rng = np.random.default_rng(61)
    p = rng.dirichlet(np.ones(6) * 2)
    q = rng.dirichlet(np.ones(6) * 2)
    si = _rounds(p, q, g["samples"], 62)
    acc, emi, _ = run_both(orc, si, REJ)
    counts = np.bincount(emi[:, 0].astype(np.int64), minlength=6)
    assert oracle_pins.chi_square(counts, p) <= g["critical"]
    rate = float(np.mean(acc == 1))
    smin = float(np.minimum(p, q).sum())
    assert abs(rate - smin) < 5 * math.sqrt(smin * (1 - smin) / acc.size)


def test_chi_square_on_the_cluster_draw(orc):
    """The same recipe with the vocabulary padded to 8 ids (two of mass 0,
    so rows are whole 16-byte quads) in batches of 150 sequences: every
    batch takes the one-launch cluster draw. The padding is never emitted."""
    g = oracle_pins.golden("chi_square_recipe.json")
    rng = np.random.default_rng(61)
    p = rng.dirichlet(np.ones(6) * 2)
    q = rng.dirichlet(np.ones(6) * 2)
    pad = np.zeros(2)
    si = _rounds(np.concatenate([p, pad]), np.concatenate([q, pad]), g["samples"], 62)
    first = []
    for b0 in range(0, g["samples"], 150):
        _, emi, _ = run_both(orc, _head(si, 150, b0), REJ)
        first.append(emi[:, 0])
    counts = np.bincount(np.concatenate(first).astype(np.int64), minlength=8)
    assert counts[6:].sum() == 0
    assert oracle_pins.chi_square(counts[:6], p) <= g["critical"]


def test_ceiling_example(orc):
    """p(a) = 0.3, q(a) = 0.95: argmax rule 0.95, rejection rule ~0.30."""
    g = oracle_pins.golden("spec_ceiling_example.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    si = _rounds(p, q, 20_000, 33)
    for mode, want in ((REJ, g["accept_rejection_rule"]), (ARG, g["accept_argmax_rule"])):
        acc, _, _ = run_both(orc, si, mode)
        rate = float(np.mean(acc == 1))
        assert abs(rate - want) < 5 * math.sqrt(want * (1 - want) / acc.size), (mode, rate)


def test_support_is_never_violated(orc):
    rng = np.random.default_rng(71)
    p = np.array([0.0, 0.6, 0.0, 0.4, 0.0, 0.0])
    q = rng.dirichlet(np.ones(6))
    si = _rounds(p, q, 5000, 72, bonus=p)
    acc, emi, _ = run_both(orc, si, REJ)
    assert set(emi[:, 0].tolist()) <= {1, 3}
    assert set(emi[acc == 1, 1].tolist()) <= {1, 3}


def test_regimes(orc):
    """q = p accepts everything; disjoint supports reject at position 0."""
    rng = np.random.default_rng(81)
    p = rng.dirichlet(np.ones(5))
    si = _rounds(p, p, 2000, 82, K=3, bonus=rng.dirichlet(np.ones(5)))
    acc, _, _ = run_both(orc, si, REJ)
    assert np.all(acc == 3)
    si = _rounds(np.array([0.5, 0.5, 0, 0, 0]), np.array([0, 0, 0.2, 0.3, 0.5]), 2000, 83, K=2)
    acc, emi, _ = run_both(orc, si, REJ)
    assert np.all(acc == 0) and set(emi[:, 0].tolist()) <= {0, 1}


def test_workspace_reuse(orc):
    si = synth.workload_spec()
    S, K, V = si.draft_tokens.shape[0], si.draft_tokens.shape[1], si.target.shape[2]
    ws = B.workspace(B.SEL_OP_SPEC, S, V, K, device=G.device())
    ref = orc.spec_accept(si.target, si.draft, si.draft_tokens, 1.0, REJ, si.u_acc, si.u_fin)
    t = G.to_dev(si.target)
    d = G.to_dev(si.draft)
    tok = G.to_dev(si.draft_tokens.view(np.int32))
    ua, uf = G.to_dev(si.u_acc), G.to_dev(si.u_fin)
    import torch
    acc = torch.empty(S, dtype=torch.int32, device=G.device())
    emi = torch.empty(S, K + 1, dtype=torch.int32, device=G.device())
    for mode in (REJ, ARG, REJ, REJ, ARG):
        B.spec_accept(t, d, tok, B.SpecParams(1.0, mode), ua, uf, acc, emi, ws)
        r = ref if mode == REJ else orc.spec_accept(si.target, None, si.draft_tokens, 1.0, ARG)
        G.assert_spec_matches(B.ids_to_numpy(acc), B.ids_to_numpy(emi), r)
