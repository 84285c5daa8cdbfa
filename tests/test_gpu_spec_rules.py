"""Sampler-match acceptance (spec_accept_sampler) and the closed-form
diagnostics (spec_diagnostics) against the oracle, on the spec workload's
shapes and on hand-made rows."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_fp32_gb300 import binding as B, synth
from gpu_helpers import INVALID, PROB_RTOL, SENTINEL, assert_spec_matches, device, to_dev, ws_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def sampler(target, tokens, u, T, top_k, top_p, min_p, temp_last=False, misalign=False):
    S, K1, V = target.shape
    t = to_dev(target, misalign)
    tok = to_dev(np.ascontiguousarray(tokens, dtype=np.uint32).reshape(S, K1 - 1).view(np.int32))
    ud = to_dev(np.asarray(u, dtype=np.float32).reshape(S, K1))
    acc = torch.full((S,), SENTINEL, dtype=torch.int32, device=device())
    emi = torch.full((S, K1), SENTINEL, dtype=torch.int32, device=device())
    ws = B.workspace(B.SEL_OP_SPEC_SAMPLER, S * K1, V, top_k, device=device())
    prm = B.SampleParams(T, top_k, top_p, min_p, B.SEL_ORDER_TEMP_LAST if temp_last else B.SEL_ORDER_TEMP_FIRST)
    B.spec_accept_sampler(t, tok, prm, ud, acc, emi, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    return B.ids_to_numpy(acc), B.ids_to_numpy(emi)


def diagnostics(target, draft, T, misalign=False):
    S, K1, V = target.shape
    smin = torch.full((S, K1 - 1), -7.0, device=device())
    sprod = torch.full((S, K1 - 1), -7.0, device=device())
    ws = B.workspace(B.SEL_OP_SPEC_DIAG, S, V, K1 - 1, device=device())
    B.spec_diagnostics(to_dev(target, misalign), to_dev(np.ascontiguousarray(draft), misalign), T, smin, sprod, ws)
    torch.cuda.synchronize()
    assert ws_error(ws) == 0
    return smin.cpu().numpy(), sprod.cpu().numpy()


def drafts_near_target(target, seed, share=0.6):
    """Draft tokens: the target row's argmax with probability `share`, else a
    random id, so that chains of several acceptances occur."""
    rng = np.random.default_rng(seed)
    S, K1, V = target.shape
    a = np.argmax(target[:, :K1 - 1], axis=2)
    return np.where(rng.random((S, K1 - 1)) < share, a, rng.integers(0, V, size=(S, K1 - 1))).astype(np.uint32)


@pytest.mark.parametrize("T,top_k,top_p,min_p,temp_last", [(1.0, 40, 0.9, 0.05, False), (0.7, 8, 1.0, 0.0, False),
                                                           (1.3, 20, 0.8, 0.02, True), (0.0, 0, 1.0, 0.0, False)])
def test_sampler_match_on_the_spec_workload(orc, T, top_k, top_p, min_p, temp_last):
    si = synth.workload_spec()
    tgt = (si.target * 3.0).astype(np.float32)  # peaked enough for multi-token chains
    tok = drafts_near_target(tgt, 70)
    S, K1, _ = tgt.shape
    u = synth.uniforms(71, S * K1).reshape(S, K1)
    acc, emi = sampler(tgt, tok, u, T, top_k, top_p, min_p, temp_last)
    ref = orc.spec_sampler(tgt, tok, T, top_k, top_p, min_p, u, temp_last)
    assert_spec_matches(acc, emi, ref)
    if T == 0.0:  # greedy sampler = the argmax rule
        a = np.argmax(tgt, axis=2)
        for s in range(S):
            n = int(acc[s])
            assert emi[s, n] == a[s, n] and all(tok[s, :n] == a[s, :n])


@pytest.mark.parametrize("T,top_p,min_p,temp_last", [(1.0, 1.0, 0.0, False), (0.8, 1.0, 0.05, False),
                                                     (1.0, 0.9, 0.0, False), (1.2, 0.95, 0.02, True)])
@pytest.mark.parametrize("misalign", [False, True])
def test_sampler_match_full_row(orc, T, top_p, min_p, temp_last, misalign):
    """top_k = 0: each position draws from its whole target row (sel_sample's
    full-row sampling). The rows are peaked enough (the spec workload's
    logits times 6: every nucleus of these policies holds at most 32 ids)
    that every top-p cut lies within the 64 candidates the draw is decided
    on, so no row fails closed."""
    si = synth.workload_spec()
    tgt = (si.target * 6.0).astype(np.float32)
    tok = drafts_near_target(tgt, 76)
    S, K1, _ = tgt.shape
    u = synth.uniforms(77, S * K1).reshape(S, K1)
    acc, emi = sampler(tgt, tok, u, T, 0, top_p, min_p, temp_last, misalign)
    ref = orc.spec_sampler(tgt, tok, T, 0, top_p, min_p, u, temp_last)
    assert np.all(acc != INVALID)
    assert_spec_matches(acc, emi, ref)


@pytest.mark.parametrize("S,K,V,misalign", [(1, 0, 1000, False), (5, 1, 4097, True), (33, 3, 2048, False)])
def test_sampler_match_shapes(orc, S, K, V, misalign):
    rng = np.random.default_rng(72 + K)
    tgt = (rng.normal(0, 3, size=(S, K + 1, V))).astype(np.float32)
    tok = drafts_near_target(tgt, 73)
    u = rng.random((S, K + 1), dtype=np.float32)
    acc, emi = sampler(tgt, tok, u, 1.0, 16, 0.95, 0.0, misalign=misalign)
    ref = orc.spec_sampler(tgt, tok, 1.0, 16, 0.95, 0.0, u)
    assert_spec_matches(acc, emi, ref)


def test_sampler_match_fails_closed(orc):
    rng = np.random.default_rng(74)
    S, K, V = 6, 3, 3000
    tgt = rng.normal(0, 2, size=(S, K + 1, V)).astype(np.float32)
    tok = drafts_near_target(tgt, 75)
    u = rng.random((S, K + 1), dtype=np.float32)
    u[0, K] = 1.0            # a bad uniform at a position the chain may not reach
    tok[1, 1] = V            # a draft token past the vocabulary
    tgt[2, 3, 17] = np.nan   # a nonfinite bonus row
    u[3, 0] = -0.5
    acc, emi = sampler(tgt, tok, u, 1.0, 10, 1.0, 0.0)
    for s in range(4):
        assert acc[s] == INVALID and np.all(emi[s] == INVALID)
    ref = orc.spec_sampler(tgt, tok, 1.0, 10, 1.0, 0.0, u)
    assert_spec_matches(acc, emi, ref)


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_diagnostics_on_the_spec_workload(orc, T):
    si = synth.workload_spec()
    smin, sprod = diagnostics(si.target, si.draft, T)
    rmin, rprod = orc.spec_diagnostics(si.target, si.draft, T)
    np.testing.assert_allclose(smin, rmin, rtol=PROB_RTOL, atol=1e-7)
    np.testing.assert_allclose(sprod, rprod, rtol=PROB_RTOL, atol=1e-9)
    assert np.all(smin >= sprod)


def test_diagnostics_closed_forms_and_nonfinite(orc):
    from oracle_pins import _logits_from, golden
    cases = golden("spec_diagnostics_closed_forms.json")["cases"]
    for c in cases:
        lp, lq = _logits_from(c["p"]), _logits_from(c["q"])
        t = np.stack([lp, lp])[None]
        d = lq[None, None]
        smin, sprod = diagnostics(t, d, 1.0)
        assert abs(smin[0, 0] - c["sum_min"]) < 1e-5 and abs(sprod[0, 0] - c["sum_prod"]) < 1e-5, c["name"]
    rng = np.random.default_rng(76)
    t = rng.normal(0, 1, size=(3, 3, 5000)).astype(np.float32)
    d = (t[:, :2] + rng.normal(0, 0.3, size=(3, 2, 5000))).astype(np.float32)
    t[1, 0, 4] = np.inf
    d[2, 1, 9] = np.nan
    smin, sprod = diagnostics(t, d, 1.0, misalign=True)
    assert np.isnan(smin[1, 0]) and np.isnan(sprod[2, 1]) and not np.isnan(smin[1, 1])
    rmin, rprod = orc.spec_diagnostics(t, d, 1.0)
    ok = ~np.isnan(rmin)
    np.testing.assert_allclose(smin[ok], rmin[ok], rtol=PROB_RTOL, atol=1e-7)
