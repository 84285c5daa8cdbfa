"""Pins for the CPU oracle: checks that tie the oracle to what the pages and
the mathematics fix, independently of the oracle's own code.

Each ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
on a violation. The test files run every pin on the real oracle; the mutant
test compiles copies of the oracle with a planted mistake and requires that
at least one pin fails for each copy.

Kinds of pin used here:
  * values the pages print (the tie rule, the 202,048 partition, the
    p(a)=0.3 / q(a)=0.95 ceiling example, the chi-square recipe);
  * closed forms derived by hand (tests/golden/*.json);
  * brute force on tiny inputs (rank counting for top-k, a characterisation
    of the first maximum);
  * library routines for special cases (numpy's first-occurrence argmax,
    numpy's lexsort ordering);
  * statistical laws: acceptance -> sum min(p, q), emitted stream -> p.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
INVALID = 0xFFFFFFFF
NEG = -1e30  # a finite logit whose probability is exactly 0 in double


def golden(name: str):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _logits_from(case_or_probs) -> np.ndarray:
    if isinstance(case_or_probs, dict):
        if "logits" in case_or_probs:
            return np.asarray(case_or_probs["logits"], dtype=np.float32)
        case_or_probs = case_or_probs["probs"]
    p = np.asarray(case_or_probs, dtype=np.float64)
    with np.errstate(divide="ignore"):
        lg = np.where(p > 0, np.log(np.where(p > 0, p, 1.0)), NEG)
    return lg.astype(np.float32)


# ---------------------------------------------------------------------------
# argmax
# ---------------------------------------------------------------------------

def _is_first_max(x: np.ndarray, i: int) -> bool:
    """i attains the maximum and no earlier index does."""
    return bool(np.all(x[i] >= x) and np.all(x[:i] < x[i]))


def pin_argmax_ties(orc):
    """Ch 21, 21.3: strict '>' keeps the lower index on ties. Planted equal
    maxima (the planted-argmax workload's recipe) -> lowest planted id."""
    rng = np.random.default_rng(123)
    for V in (7, 1000, 202048):
        x = rng.normal(0, 3, size=V).astype(np.float32)
        ids = np.sort(rng.choice(V, size=3, replace=False))
        x[ids] = x.max() + np.float32(1.0)
        got = int(orc.argmax(x[None])[0])
        assert got == ids[0], (V, got, ids)
    # -0.0 and +0.0 compare equal: the lower index wins
    x = np.array([-1.0, -0.0, 0.0, -2.0], dtype=np.float32)
    assert int(orc.argmax(x[None])[0]) == 1
    x = np.array([-1.0, 0.0, -0.0], dtype=np.float32)
    assert int(orc.argmax(x[None])[0]) == 1


def pin_argmax_bruteforce(orc):
    """Every row over the alphabet {0, 1, 2} up to length 6: the result is the
    unique first maximum (characterised, not recomputed by a scan)."""
    for V in range(1, 7):
        rows = np.array(list(itertools.product((0.0, 1.0, 2.0), repeat=V)),
                        dtype=np.float32)
        got = orc.argmax(rows)
        for r in range(rows.shape[0]):
            assert _is_first_max(rows[r], int(got[r])), (rows[r], got[r])


def pin_argmax_numpy(orc):
    """numpy.argmax documents first-occurrence; on finite rows it must agree.
    Rows drawn from a small integer set so ties are frequent."""
    rng = np.random.default_rng(7)
    x = rng.integers(0, 5, size=(64, 333)).astype(np.float32)
    assert np.array_equal(orc.argmax(x), np.argmax(x, axis=1).astype(np.uint32))
    x = rng.normal(size=(16, 5000)).astype(np.float32)
    assert np.array_equal(orc.argmax(x), np.argmax(x, axis=1).astype(np.uint32))


def pin_argmax_partition(orc):
    """Ch 21, Figure 21.1: V = 202,048 = 197 x 1,024 + 320. The maximum placed
    at each chunk edge and in the ragged tail is found."""
    g = golden("argmax_partition.json")
    V, chunk = g["V"], g["chunk"]
    assert g["full_chunks"] * chunk + g["tail"] == V
    assert math.ceil(V / chunk) == g["chunks"]
    base = np.random.default_rng(0).normal(0, 3, size=V).astype(np.float32)
    for pos in g["positions"]:
        x = base.copy()
        x[pos] = x.max() + np.float32(1.0)
        assert int(orc.argmax(x[None])[0]) == pos, pos
    for V in (1, 2, 3, 5, 1023, 1024, 1025, 202047):
        x = np.random.default_rng(V).normal(size=V).astype(np.float32)
        for pos in {0, V // 2, V - 1}:
            y = x.copy()
            y[pos] = 100.0
            assert int(orc.argmax(y[None])[0]) == pos, (V, pos)


def pin_argmax_nonfinite(orc):
    """Ch 21, 21.4 / 21.6: any NaN or +-Inf makes the row fail closed."""
    for bad in (np.nan, np.inf, -np.inf):
        for pos in (0, 17, 99):
            x = np.zeros((1, 100), dtype=np.float32)
            x[0, pos] = bad
            assert int(orc.argmax(x)[0]) == INVALID, (bad, pos)


def pin_eog_bruteforce(orc):
    """Ch 21, 21.4 (greedy serving variant, EOG exclusion): every row over
    {0, 1, 2} up to length 5 with every excluded subset. The answer is a
    non-excluded id holding the largest non-excluded value, the lowest such
    id; with every id excluded there is none (0xFFFFFFFF)."""
    for V in range(1, 6):
        rows = np.array(list(itertools.product((0.0, 1.0, 2.0), repeat=V)), dtype=np.float32)
        for mask in range(1 << V):
            ex = [i for i in range(V) if mask >> i & 1]
            got = orc.argmax_excluding(rows, ex)
            keep = [i for i in range(V) if i not in ex]
            for r in range(rows.shape[0]):
                g = int(got[r])
                if not keep:
                    assert g == INVALID, (rows[r], ex, g)
                    continue
                assert g in keep, (rows[r], ex, g)
                kv = rows[r][keep]
                assert rows[r][g] == kv.max(), (rows[r], ex, g)
                assert all(rows[r][i] < rows[r][g] for i in keep if i < g), (rows[r], ex, g)


def pin_eog_reduces_to_argmax(orc):
    """An empty set, or ids past the row, changes nothing; excluding the
    argmax gives numpy's first maximum of the row with that id masked (an
    independent library route); duplicates in the set do not matter."""
    rng = np.random.default_rng(17)
    x = rng.integers(0, 6, size=(32, 500)).astype(np.float32)
    assert np.array_equal(orc.argmax_excluding(x, []), orc.argmax(x))
    assert np.array_equal(orc.argmax_excluding(x, [500, 777, 0xFFFFFFF0]), orc.argmax(x))
    for r in range(8):
        a = int(np.argmax(x[r]))
        ex = [a, a, 3, 499]
        masked = x[r].astype(np.float64).copy()
        masked[[a, 3, 499]] = -np.inf
        assert int(orc.argmax_excluding(x[r:r + 1], ex)[0]) == int(np.argmax(masked))


def pin_eog_nonfinite(orc):
    """The latch covers excluded ids too: a NaN or Inf anywhere fails the
    row, and masking never turns a finite row invalid."""
    x = np.zeros((1, 50), dtype=np.float32)
    x[0, 7] = 1.0
    for bad in (np.nan, np.inf, -np.inf):
        y = x.copy()
        y[0, 20] = bad
        assert int(orc.argmax_excluding(y, [20])[0]) == INVALID
    assert int(orc.argmax_excluding(x, [7])[0]) == 0


# ---------------------------------------------------------------------------
# top-k
# ---------------------------------------------------------------------------

def _rank_topk(x: np.ndarray, k: int):
    """O(V^2) rank counting: rank_i = #{j : x_j > x_i or (x_j == x_i, j < i)}."""
    V = x.size
    rank = np.array([sum(1 for j in range(V)
                         if x[j] > x[i] or (x[j] == x[i] and j < i))
                     for i in range(V)])
    ids = np.argsort(rank)[:k]
    return ids


def pin_topk_bruteforce(orc):
    rng = np.random.default_rng(11)
    for V in range(1, 17):
        for _ in range(6):
            x = rng.integers(-3, 4, size=V).astype(np.float32)
            for k in sorted({1, (V + 1) // 2, V}):
                vals, ids = orc.topk(x[None], k)
                want = _rank_topk(x, k)
                assert np.array_equal(ids[0], want.astype(np.uint32)), (x, k, ids, want)
                assert np.array_equal(vals[0], x[want]), (x, k)


def pin_topk_lexsort(orc):
    """numpy.lexsort orders by (-value, id): an independent library route."""
    rng = np.random.default_rng(12)
    x = rng.integers(0, 50, size=(8, 3000)).astype(np.float32)
    vals, ids = orc.topk(x, 84)
    for r in range(x.shape[0]):
        order = np.lexsort((np.arange(x.shape[1]), -x[r].astype(np.float64)))
        assert np.array_equal(ids[r], order[:84].astype(np.uint32))


def pin_topk_special(orc):
    rng = np.random.default_rng(13)
    x = rng.normal(size=(5, 999)).astype(np.float32)
    _, ids1 = orc.topk(x, 1)
    assert np.array_equal(ids1[:, 0], orc.argmax(x))      # k = 1 is argmax
    eq = np.full((1, 50), 2.5, dtype=np.float32)           # all equal: ids 0..k-1
    _, ids = orc.topk(eq, 7)
    assert np.array_equal(ids[0], np.arange(7, dtype=np.uint32))
    vals, ids = orc.topk(x, 999)                            # k = V: full order
    assert np.all(np.diff(vals, axis=1) <= 0)
    assert np.array_equal(np.sort(ids, axis=1),
                          np.tile(np.arange(999, dtype=np.uint32), (5, 1)))
    bad = x.copy()
    bad[2, 500] = np.nan
    vals, ids = orc.topk(bad, 3)
    assert np.all(ids[2] == INVALID) and np.all(np.isnan(vals[2]))
    assert np.all(ids[[0, 1, 3, 4]] != INVALID)


# ---------------------------------------------------------------------------
# filtered sampling
# ---------------------------------------------------------------------------

def pin_sample_closed_forms(orc):
    g = golden("sample_closed_forms.json")
    for case in g["cases"]:
        x = _logits_from(case)[None]
        for u, want_id, want_p in case["draws"]:
            r = orc.sample(x, [u], case["T"], case["top_k"], case["top_p"],
                           case["min_p"], case["temp_last"])
            assert int(r.ids[0]) == want_id, (case["name"], u, r.ids[0])
            assert abs(r.probs[0] - want_p) <= 1e-6 * max(1.0, want_p), \
                (case["name"], u, r.probs[0], want_p)


def pin_sample_cdf_grid(orc):
    """Sweep u over a 10^5-point grid on a row with hand-chosen probabilities:
    the share of grid points mapped to each id equals its probability, and
    the map is monotone in u along the draw order: (P desc, id asc) for the
    top-k candidates (top_k = V here), ascending id for full-row sampling
    (top_k = 0)."""
    P = np.array([0.05, 0.4, 0.15, 0.1, 0.3])  # order by P: ids 1, 4, 2, 3, 0
    x = np.tile(_logits_from(P), (100_000, 1))
    u = ((np.arange(100_000) + 0.5) / 100_000).astype(np.float32)
    for top_k, rank_of in ((5, {1: 0, 4: 1, 2: 2, 3: 3, 0: 4}), (0, {i: i for i in range(5)})):
        r = orc.sample(x, u, 1.0, top_k, 1.0, 0.0)
        share = np.bincount(r.ids.astype(np.int64), minlength=5) / 100_000
        assert np.allclose(share, P, atol=2e-5), (top_k, share)
        ranks = np.array([rank_of[int(i)] for i in r.ids])
        assert np.all(np.diff(ranks) >= 0), top_k
        # each drawn id's reported probability is its own
        assert np.allclose(r.probs, P[r.ids.astype(np.int64)], rtol=1e-6)


def pin_sample_support(orc):
    """Zero tolerance on support: every draw lies in the top_k set, and with
    top_p = 1, min_p = 0 every top_k id is reachable."""
    rng = np.random.default_rng(21)
    x = np.tile(rng.normal(0, 2, size=300).astype(np.float32), (4000, 1))
    u = rng.random(4000, dtype=np.float32)
    _, top = orc.topk(x[:1], 8)
    r = orc.sample(x, u, 0.8, 8, 1.0, 0.0)
    assert set(r.ids.tolist()) <= set(top[0].tolist())
    assert set(r.ids.tolist()) == set(top[0].tolist())


def pin_sample_invalid(orc):
    x = np.zeros((4, 10), dtype=np.float32)
    x[3, 2] = np.inf
    r = orc.sample(x, np.array([1.0, -0.25, np.nan, 0.5], dtype=np.float32),
                   1.0, 0, 1.0, 0.0)
    assert np.all(r.ids == INVALID) and np.all(np.isnan(r.probs))


def pin_sample_margins(orc):
    """The decision margins of filtered sampling, hand-derived
    (golden margins_closed_forms.json): distance of u to the nearest CDF step
    (neither 0 nor the final step counts), of each top-p prefix to top_p, of
    each min-p ratio to min_p, of the typical cut (with its score gap) and of
    the ids around the top-n-sigma threshold. These margins decide which GPU
    rows are exempt from bit-exact comparison."""
    g = golden("margins_closed_forms.json")
    for case in g["sample"]:
        x = _logits_from(case)[None]
        r = orc.sample(x, [case["u"]], case["T"], case["top_k"], case["top_p"], case["min_p"],
                       False, case.get("top_n_sigma", 0.0), case.get("typical_p", 1.0))
        assert int(r.ids[0]) == case["id"], (case["name"], r.ids[0])
        assert abs(r.probs[0] - case["prob"]) <= 1e-6, (case["name"], r.probs[0])
        assert abs(r.margin[0] - case["margin"]) <= 1e-6, (case["name"], r.margin[0], case["margin"])


def pin_spec_margins(orc):
    """The rejection test's margin |u q - p| / max(p, q) and the residual and
    bonus draws' CDF margins in ascending id, hand-derived (golden
    margins_closed_forms.json)."""
    g = golden("margins_closed_forms.json")
    rows = {k: _logits_from(v) for k, v in g["spec_rows"].items()}
    for case in g["spec"]:
        target = np.stack([rows[n] for n in case["target"]])[None]
        draft = np.stack([rows[n] for n in case["draft"]])[None]
        tok = np.asarray(case["tokens"], dtype=np.uint32)[None]
        r = orc.spec_accept(target, draft, tok, 1.0, 0, np.asarray(case["u_acc"], np.float32)[None],
                            np.asarray([case["u_fin"]], np.float32))
        assert int(r.accepted[0]) == case["accepted"], (case["name"], r.accepted[0])
        assert [int(e) for e in r.emitted[0]] == case["emitted"], (case["name"], r.emitted[0])
        assert abs(r.margin_accept[0] - case["margin_accept"]) <= 1e-6, (case["name"], r.margin_accept[0])
        assert abs(r.margin_draw[0] - case["margin_draw"]) <= 1e-6, (case["name"], r.margin_draw[0])
    rows = {k: _logits_from(v) for k, v in g["sampler_rows"].items()}
    for case in g["sampler"]:
        target = np.stack([rows[n] for n in case["target"]])[None]
        tok = np.asarray(case["tokens"], dtype=np.uint32)[None]
        u = np.asarray(case["u"], dtype=np.float32)[None]
        r = orc.spec_sampler(target, tok, case["T"], case["top_k"], 1.0, 0.0, u)
        assert int(r.accepted[0]) == case["accepted"], (case["name"], r.accepted[0])
        assert [int(e) for e in r.emitted[0]] == case["emitted"], (case["name"], r.emitted[0])
        assert abs(r.margin_draw[0] - case["margin"]) <= 1e-6, (case["name"], r.margin_draw[0])


# ---------------------------------------------------------------------------
# speculative acceptance
# ---------------------------------------------------------------------------

def _spec_case_arrays(g, case):
    rows = {k: _logits_from(v) for k, v in g["rows"].items()}
    target = np.stack([rows[n] for n in case["target"]])[None]
    draft = None if case["draft"] is None else np.stack([rows[n] for n in case["draft"]])[None]
    return target, draft


def pin_spec_closed_forms(orc):
    g = golden("spec_closed_forms.json")
    for case in g["cases"]:
        target, draft = _spec_case_arrays(g, case)
        mode = 0 if case["mode"] == "rejection" else 1
        K = len(case["tokens"])
        r = orc.spec_accept(target, draft, np.array([case["tokens"]]),
                            case.get("T", 1.0), mode,
                            np.array([case.get("u_acc", [0.0] * K)], dtype=np.float32),
                            np.array([case.get("u_fin", 0.0)], dtype=np.float32))
        want = [INVALID if e is None else e for e in case["emitted"]]
        assert int(r.accepted[0]) == case["accepted"], (case["name"], r.accepted)
        assert r.emitted[0].tolist() == want, (case["name"], r.emitted[0])


def _draws_from(rng, P, n):
    return rng.choice(P.size, size=n, p=P / P.sum())


def _spec_rounds(orc, p, q, n, seed, mode=0, K=1, bonus=None):
    """n independent single-sequence rounds with draft tokens drawn from q."""
    rng = np.random.default_rng(seed)
    V = p.size
    lp, lq = _logits_from(p), _logits_from(q)
    lb = _logits_from(p if bonus is None else bonus)
    target = np.empty((n, K + 1, V), dtype=np.float32)
    target[:, :K] = lp
    target[:, K] = lb
    draft = np.empty((n, K, V), dtype=np.float32)
    draft[:] = lq
    tokens = _draws_from(rng, q, n * K).reshape(n, K)
    u_acc = rng.random((n, K), dtype=np.float32)
    u_fin = rng.random(n, dtype=np.float32)
    return orc.spec_accept(target, draft, tokens, 1.0, mode, u_acc, u_fin)


def pin_spec_ceiling_example(orc):
    """mlxcel, The acceptance ceiling: argmax rule 0.95 vs ceiling 0.30."""
    g = golden("spec_ceiling_example.json")
    p, q = np.array(g["p"]), np.array(g["q"])
    n = 20_000
    assert abs(np.minimum(p, q).sum() - g["accept_rejection_rule"]) < 1e-12
    assert abs(q[np.argmax(p)] - g["accept_argmax_rule"]) < 1e-12
    for mode, want in ((0, g["accept_rejection_rule"]), (1, g["accept_argmax_rule"])):
        r = _spec_rounds(orc, p, q, n, seed=31 + mode, mode=mode)
        rate = float(np.mean(r.accepted == 1))
        sd = math.sqrt(want * (1 - want) / n)
        assert abs(rate - want) < 5 * sd, (mode, rate, want)


def pin_spec_acceptance_law(orc):
    """Per-position acceptance converges to sum_x min(p, q) (the rule's
    closed form) and not to sum_x p q (sampler-match)."""
    rng = np.random.default_rng(41)
    for trial in range(3):
        p = rng.dirichlet(np.ones(6))
        q = rng.dirichlet(np.ones(6))
        n = 20_000
        r = _spec_rounds(orc, p, q, n, seed=50 + trial)
        rate = float(np.mean(r.accepted == 1))
        smin = float(np.minimum(p, q).sum())
        sd = math.sqrt(smin * (1 - smin) / n)
        assert abs(rate - smin) < 5 * sd, (rate, smin)


def chi_square(counts: np.ndarray, probs: np.ndarray) -> float:
    expected = probs * counts.sum()
    return float(np.sum((counts - expected) ** 2 / expected))


def pin_spec_stream_is_target(orc):
    """mlxcel, Regression guards: the emitted stream matches the target's
    exact categorical by chi-square (12000 tokens, dof 5, reject > 25.7448)."""
    g = golden("chi_square_recipe.json")
    rng = np.random.default_rng(61)
    p = rng.dirichlet(np.ones(6) * 2)
    q = rng.dirichlet(np.ones(6) * 2)
    r = _spec_rounds(orc, p, q, g["samples"], seed=62)
    counts = np.bincount(r.emitted[:, 0].astype(np.int64), minlength=6)
    stat = chi_square(counts, p)
    assert stat <= g["critical"], stat


def pin_spec_chi_square_power(orc):
    """mlxcel, Regression guards: the stream statistic has power. On the
    same rounds as the stream pin it rejects two known-wrong rules: argmax
    against argmax (the oracle's other mode), and the rejection rule's own
    decisions followed by a redraw from p instead of the residual (built
    here from the same draft tokens and uniforms; its accept decisions must
    equal the oracle's)."""
    g = golden("chi_square_recipe.json")
    rng = np.random.default_rng(61)
    p = rng.dirichlet(np.ones(6) * 2)
    q = rng.dirichlet(np.ones(6) * 2)
    n = g["samples"]
    r = _spec_rounds(orc, p, q, n, seed=62, mode=1)
    counts = np.bincount(r.emitted[:, 0].astype(np.int64), minlength=6)
    assert chi_square(counts, p) > g["critical"]
    # the same uniforms and tokens _spec_rounds draws (K = 1)
    ref = _spec_rounds(orc, p, q, n, seed=62)
    rng = np.random.default_rng(62)
    t = _draws_from(rng, q, n)
    u_acc = rng.random((n, 1), dtype=np.float32)[:, 0].astype(np.float64)
    u_fin = rng.random(n, dtype=np.float32).astype(np.float64)
    accept = u_acc * q[t] <= p[t]
    assert np.array_equal(accept, ref.accepted == 1)
    redraw = np.searchsorted(np.cumsum(p) / p.sum(), u_fin, side="right")
    wrong = np.where(accept, t, redraw)
    assert chi_square(np.bincount(wrong, minlength=6), p) > g["critical"]


def pin_spec_support(orc):
    """mlxcel, Regression guards: with a top_k = 2 target no emitted token
    ever lies outside the target's support (accepted drafts, residual draws
    and bonus draws alike)."""
    rng = np.random.default_rng(71)
    p = np.array([0.0, 0.6, 0.0, 0.4, 0.0, 0.0])
    q = rng.dirichlet(np.ones(6))
    r = _spec_rounds(orc, p, q, 5000, seed=72, bonus=p)
    first = r.emitted[:, 0]
    bonus = r.emitted[:, 1][r.accepted == 1]
    assert set(first.tolist()) <= {1, 3}, set(first.tolist())
    assert set(bonus.tolist()) <= {1, 3}, set(bonus.tolist())
    assert bonus.size > 0 and np.any(r.accepted == 0)


def pin_spec_regimes(orc):
    """q = p accepts every draft (u < 1) and draws the bonus from p_K;
    disjoint supports reject at position 0 and draw the residual = p."""
    rng = np.random.default_rng(81)
    p = rng.dirichlet(np.ones(5))
    pb = rng.dirichlet(np.ones(5))
    n = 3000
    r = _spec_rounds(orc, p, p, n, seed=82, K=3, bonus=pb)
    assert np.all(r.accepted == 3)
    counts = np.bincount(r.emitted[:, 3].astype(np.int64), minlength=5)
    assert chi_square(counts, pb) < 25.0
    pd = np.array([0.5, 0.5, 0.0, 0.0, 0.0])
    qd = np.array([0.0, 0.0, 0.2, 0.3, 0.5])
    r = _spec_rounds(orc, pd, qd, n, seed=83, K=2)
    assert np.all(r.accepted == 0)
    assert set(r.emitted[:, 0].tolist()) <= {0, 1}
    share0 = float(np.mean(r.emitted[:, 0] == 0))
    assert abs(share0 - 0.5) < 5 * math.sqrt(0.25 / n)


def pin_spec_greedy(orc):
    """mlxcel, RNG dependency / Regression guards: temperature 0 is the argmax
    rule, byte-identical to greedy target decoding, whatever the uniforms."""
    rng = np.random.default_rng(91)
    S, K, V = 50, 4, 40
    target = rng.normal(size=(S, K + 1, V)).astype(np.float32)
    draft = rng.normal(size=(S, K, V)).astype(np.float32)
    greedy = np.argmax(target, axis=2)
    tokens = np.where(rng.random((S, K)) < 0.7, greedy[:, :K],
                      rng.integers(0, V, size=(S, K)))
    r0 = orc.spec_accept(target, draft, tokens, 0.0, 0,
                         rng.random((S, K), dtype=np.float32),
                         rng.random(S, dtype=np.float32))
    r1 = orc.spec_accept(target, None, tokens, 1.0, 1)
    assert np.array_equal(r0.accepted, r1.accepted)
    assert np.array_equal(r0.emitted, r1.emitted)
    for s in range(S):
        n = int(r1.accepted[s])
        assert np.array_equal(r1.emitted[s, :n + 1], greedy[s, :n + 1])


def pin_spec_invalid(orc):
    rng = np.random.default_rng(95)
    target = rng.normal(size=(3, 3, 8)).astype(np.float32)
    draft = rng.normal(size=(3, 2, 8)).astype(np.float32)
    tokens = np.array([[1, 2], [8, 0], [0, 1]])
    target[2, 2, 5] = np.nan
    r = orc.spec_accept(target, draft, tokens, 1.0, 0,
                        np.full((3, 2), 0.5, dtype=np.float32),
                        np.full(3, 0.5, dtype=np.float32))
    assert r.accepted[0] != INVALID
    assert r.accepted[1] == INVALID and np.all(r.emitted[1] == INVALID)
    assert r.accepted[2] == INVALID and np.all(r.emitted[2] == INVALID)


def pin_filters_closed_forms(orc):
    """Ch 21, 21.7 (top_n_sigma, typical_p in the chain): survivors and draw
    probabilities from golden sample_filters_closed_forms.json. A grid of u
    over [0, 1) must map onto exactly the kept ids with frequencies Q, and
    each draw reports its Q."""
    n = 20000
    u = ((np.arange(n) + 0.5) / n).astype(np.float32)
    for c in golden("sample_filters_closed_forms.json")["cases"]:
        x = np.tile(np.asarray(c["logits"], dtype=np.float32), (n, 1))
        r = orc.sample(x, u, 1.0, 0, c["top_p"], 0.0, top_n_sigma=c["top_n_sigma"], typical_p=c["typical_p"])
        kept, Q = c["kept"], np.asarray(c["Q"])
        assert set(np.unique(r.ids).tolist()) <= set(kept), (c["name"], np.unique(r.ids))
        freq = np.array([np.mean(r.ids == i) for i in kept])
        assert np.allclose(freq, Q, atol=2e-4), (c["name"], freq, Q)
        for i, q in zip(kept, Q):
            got = r.probs[r.ids == i]
            assert got.size and np.allclose(got, q, rtol=1e-9), (c["name"], i)


def pin_filters_reduce(orc):
    """top_n_sigma <= 0 and typical_p >= 1 change nothing; the sigma mask is
    the same at every temperature (it compares logits against the max) and
    keeps the ids numpy's population std (an independent library routine)
    puts at or above max - n sigma."""
    rng = np.random.default_rng(41)
    x = rng.normal(0, 2, size=(24, 400)).astype(np.float32)
    u = rng.random(24, dtype=np.float32)
    base = orc.sample(x, u, 0.8, 50, 0.9, 0.02)
    for a, b in ((0.0, 1.0), (-1.0, 1.0), (0.0, 1.5)):
        r = orc.sample(x, u, 0.8, 50, 0.9, 0.02, top_n_sigma=a, typical_p=b)
        assert np.array_equal(r.ids, base.ids) and np.allclose(r.probs, base.probs, rtol=1e-12)
    n = 1.5
    xd = x.astype(np.float64)
    thr = xd.max(axis=1) - n * xd.std(axis=1)
    uu = ((np.arange(400) + 0.5) / 400).astype(np.float32)
    for T in (0.5, 2.0):
        for rr in range(4):
            r = orc.sample(np.tile(x[rr], (400, 1)), uu, T, 0, 1.0, 0.0, top_n_sigma=n)
            assert np.all(x[rr][r.ids] >= thr[rr]), (T, rr)
            assert np.any(x[rr][r.ids] == x[rr].max())


# ---------------------------------------------------------------------------
# sampler-match acceptance and the closed-form diagnostics
# ---------------------------------------------------------------------------

def _pair_rows(p, q):
    """target [1, 2, V] (positions 0 and the bonus row both p) and draft [1, 1, V]."""
    lp, lq = _logits_from(p), _logits_from(q)
    return np.stack([lp, lp])[None], lq[None, None]


def pin_diag_closed_forms(orc):
    """mlxcel rules, "Verifying the gain": hand-computed sum min(p, q) and
    sum p q (golden spec_diagnostics_closed_forms.json). The rows are fp32
    logits log(p), so p comes back within ~1e-7."""
    for c in golden("spec_diagnostics_closed_forms.json")["cases"]:
        t, d = _pair_rows(c["p"], c["q"])
        smin, sprod = orc.spec_diagnostics(t, d, 1.0)
        assert abs(smin[0, 0] - c["sum_min"]) < 1e-6, (c["name"], smin)
        assert abs(sprod[0, 0] - c["sum_prod"]) < 1e-6, (c["name"], sprod)
        # the same distributions as logits 2 log p at temperature 2
        smin2, sprod2 = orc.spec_diagnostics(2 * t, 2 * d, 2.0)
        assert abs(smin2[0, 0] - c["sum_min"]) < 1e-6 and abs(sprod2[0, 0] - c["sum_prod"]) < 1e-6


def pin_diag_inequality(orc):
    """sum_min >= sum_prod always (min(a, b) >= a b on [0, 1]); both lie in
    [0, 1]; p = q gives sum_min = 1; temperature scales both rows."""
    rng = np.random.default_rng(31)
    t = rng.normal(0, 2, size=(3, 5, 300)).astype(np.float32)
    d = (t[:, :4] + rng.normal(0, 1, size=(3, 4, 300))).astype(np.float32)
    for T in (0.5, 1.0, 2.0):
        smin, sprod = orc.spec_diagnostics(t, d, T)
        assert np.all(smin >= sprod - 1e-15) and np.all((sprod >= 0) & (smin <= 1 + 1e-12))
    smin, _ = orc.spec_diagnostics(t, t[:, :4].copy(), 1.0)
    assert np.allclose(smin, 1.0, atol=1e-12)
    bad = d.copy()
    bad[1, 2, 7] = np.nan
    smin, sprod = orc.spec_diagnostics(t, bad, 1.0)
    assert np.isnan(smin[1, 2]) and np.isnan(sprod[1, 2]) and not np.isnan(smin[1, 1])


def _draw(rng, probs, n):
    return rng.choice(len(probs), size=n, p=np.asarray(probs) / np.sum(probs))


def pin_diag_is_the_rejection_acceptance(orc):
    """The rejection rule's empirical acceptance at a position, over drafts
    drawn from q, converges to the oracle's sum_min (5 sigma binomial)."""
    c = golden("spec_diagnostics_closed_forms.json")["cases"][3]
    t, d = _pair_rows(c["p"], c["q"])
    smin, _ = orc.spec_diagnostics(t, d, 1.0)
    n = 20000
    rng = np.random.default_rng(32)
    tok = _draw(rng, c["q"], n).astype(np.uint32).reshape(n, 1)
    res = orc.spec_accept(np.repeat(t, n, 0), np.repeat(d, n, 0), tok, 1.0, 0,
                          rng.random((n, 1), dtype=np.float32), rng.random(n, dtype=np.float32))
    rate = float(np.mean(res.accepted == 1))
    sd = math.sqrt(smin[0, 0] * (1 - smin[0, 0]) / n)
    assert abs(rate - smin[0, 0]) < 5 * sd, (rate, smin)


def _sampler(orc, t, tok, u, T=1.0, top_k=0):
    return orc.spec_sampler(t, tok, T, top_k, 1.0, 0.0, u)


def pin_sampler_acceptance_law(orc):
    """mlxcel rules, "Sampler-match": acceptance probability sum_x p(x) q(x)
    for drafts drawn from q and a fresh draw from p (5 sigma binomial), with
    sum p q computed here from the two distributions."""
    for c in golden("spec_diagnostics_closed_forms.json")["cases"][:4:3]:
        p, q = np.asarray(c["p"]), np.asarray(c["q"])
        t, _ = _pair_rows(p, q)
        n = 20000
        rng = np.random.default_rng(33)
        tok = _draw(rng, q, n).astype(np.uint32).reshape(n, 1)
        res = _sampler(orc, np.repeat(t, n, 0), tok, rng.random((n, 2), dtype=np.float32))
        want = float(np.sum(p * q))
        rate = float(np.mean(res.accepted == 1))
        sd = math.sqrt(want * (1 - want) / n)
        assert abs(rate - want) < 5 * sd + 1e-12, (c["name"], rate, want)


def pin_sampler_stream_is_target(orc):
    """Lossless: the token emitted at the first position is distributed as p
    whatever q is (chi-square, the recipe of golden chi_square_recipe.json)."""
    rec = golden("chi_square_recipe.json")
    V, n = rec["dof"] + 1, rec["samples"]
    p = np.array([0.30, 0.22, 0.18, 0.12, 0.10, 0.08])
    q = np.array([0.02, 0.03, 0.05, 0.10, 0.30, 0.50])
    assert V == p.size
    t, _ = _pair_rows(p, q)
    rng = np.random.default_rng(34)
    tok = _draw(rng, q, n).astype(np.uint32).reshape(n, 1)
    res = _sampler(orc, np.repeat(t, n, 0), tok, rng.random((n, 2), dtype=np.float32))
    first = res.emitted[:, 0]
    counts = np.bincount(first.astype(np.int64), minlength=V)
    chi2 = float(np.sum((counts - n * p) ** 2 / (n * p)))
    assert chi2 < rec["critical"], chi2
    # power: emitting the draft token itself would fail
    counts_q = np.bincount(tok[:, 0].astype(np.int64), minlength=V)
    assert float(np.sum((counts_q - n * p) ** 2 / (n * p))) > rec["critical"]


def pin_sampler_greedy_and_support(orc):
    """T = 0: every draw is the row's first maximum (numpy.argmax), so the
    chain is the first-mismatch rule on argmaxes; with top_k = 2 every emitted
    draw lies in its row's top two."""
    rng = np.random.default_rng(35)
    S, K, V = 40, 4, 9
    t = rng.integers(0, 4, size=(S, K + 1, V)).astype(np.float32)
    a = np.argmax(t, axis=2)
    tok = np.where(rng.random((S, K)) < 0.7, a[:, :K], rng.integers(0, V, size=(S, K))).astype(np.uint32)
    res = orc.spec_sampler(t, tok, 0.0, 1, 1.0, 0.0, rng.random((S, K + 1), dtype=np.float32))
    for s in range(S):
        n = 0
        while n < K and tok[s, n] == a[s, n]:
            n += 1
        assert res.accepted[s] == n
        assert list(res.emitted[s, :n]) == list(tok[s, :n]) and res.emitted[s, n] == a[s, n]
        assert np.all(res.emitted[s, n + 1:] == INVALID)
    t2 = rng.normal(0, 1, size=(S, K + 1, V)).astype(np.float32)
    res = orc.spec_sampler(t2, tok, 1.0, 2, 1.0, 0.0, rng.random((S, K + 1), dtype=np.float32))
    for s in range(S):
        n = int(res.accepted[s])
        top2 = set(np.argsort(-t2[s, n], kind="stable")[:2])
        assert int(res.emitted[s, n]) in top2


def pin_sampler_invalid(orc):
    """Fail closed: a bad uniform at any position (used or not), a draft token
    >= V or a nonfinite target row makes every id of the sequence invalid."""
    rng = np.random.default_rng(36)
    S, K, V = 4, 3, 20
    t = rng.normal(size=(S, K + 1, V)).astype(np.float32)
    tok = rng.integers(0, V, size=(S, K)).astype(np.uint32)
    u = rng.random((S, K + 1), dtype=np.float32)
    u[0, K] = 1.0
    tok[1, 2] = V
    t[2, 1, 5] = np.inf
    res = orc.spec_sampler(t, tok, 1.0, 5, 0.9, 0.0, u)
    for s in range(3):
        assert res.accepted[s] == INVALID and np.all(res.emitted[s] == INVALID)
    assert res.accepted[3] != INVALID


ALL_PINS = [
    pin_argmax_ties, pin_argmax_bruteforce, pin_argmax_numpy,
    pin_argmax_partition, pin_argmax_nonfinite,
    pin_eog_bruteforce, pin_eog_reduces_to_argmax, pin_eog_nonfinite,
    pin_topk_bruteforce, pin_topk_lexsort, pin_topk_special,
    pin_sample_closed_forms, pin_sample_cdf_grid, pin_sample_support,
    pin_sample_invalid, pin_sample_margins, pin_filters_closed_forms, pin_filters_reduce,
    pin_spec_closed_forms, pin_spec_ceiling_example, pin_spec_acceptance_law,
    pin_spec_stream_is_target, pin_spec_chi_square_power, pin_spec_support, pin_spec_regimes,
    pin_spec_greedy, pin_spec_invalid, pin_spec_margins,
    pin_diag_closed_forms, pin_diag_inequality, pin_diag_is_the_rejection_acceptance,
    pin_sampler_acceptance_law, pin_sampler_stream_is_target, pin_sampler_greedy_and_support,
    pin_sampler_invalid,
]


def _main(argv):
    """Run the pins against the oracle library at argv[1]; print the first
    failing pin's name and exit 1, or exit 0 if every pin holds. Used by the
    mutant test in a child process, so a planted mistake that crashes the
    library cannot take the test runner down."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(GOLDEN)))
    import oracle
    orc = oracle.load(argv[1])
    for pin in ALL_PINS:
        try:
            pin(orc)
        except AssertionError:
            print("FAIL", pin.__name__, flush=True)
            return 1
    return 0


if __name__ == "__main__":
    import sys
    sys.exit(_main(sys.argv))
