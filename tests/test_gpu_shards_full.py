"""Filters over the whole row on vocabulary shards, on one GPU: each row is
split into G id ranges, each range runs sel_topk_stats on its own slice (its
top list and its sel_row_stats record), and the gathered lists and records
drive sel_sample_shards. Top-n-sigma with top_k > 0 is decided there; with
top_k = 0 the call writes a plan per row and the draw runs on the slices
(sel_shard_draw_mass, a gather of the masses, sel_shard_draw, a min/sum
combine), as G ranks would run it. Results must match the oracle on the
unsharded row (the sampler chain of the Muser book, "Ch 21 -- Sampling,
argmax, and grammar", 21.1 and 21.7; full-row draws walk the survivors in
ascending id); a row whose top-p cut or typical window lies past the merged
64 candidates fails closed with error bit 8."""
import numpy as np
import pytest
import torch

import oracle
import gpu_helpers as G_
from sampling_row_fp32_gb300 import binding as B, shards, synth

pytestmark = pytest.mark.gpu
ERR_BEYOND = 8


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    return oracle.default()


def policy(T, top_k, top_p=1.0, min_p=0.0, nsig=0.0, typ=0.0, temp_last=False):
    return B.SampleParams(T, top_k, top_p, min_p, B.SEL_ORDER_TEMP_LAST if temp_last else B.SEL_ORDER_TEMP_FIRST,
                          nsig, typ)


def slice_stats(x, offs, k, prm, misalign=False):
    """sel_topk_stats on every shard's slice: the device slices, the gathered
    [rows][G][k] lists and the gathered [rows][G][48] statistics."""
    rows = x.shape[0]
    G = len(offs) - 1
    slices, vals, ids, stats = [], [], [], []
    for g in range(G):
        xs = G_.to_dev(np.ascontiguousarray(x[:, offs[g]:offs[g + 1]]), misalign)
        V_g = offs[g + 1] - offs[g]
        v = torch.full((rows, k), -7.0, device=G_.device())
        i = torch.full((rows, k), -7, dtype=torch.int32, device=G_.device())
        st = torch.zeros((rows, B.ROW_STATS_BYTES), dtype=torch.uint8, device=G_.device())
        ws = B.workspace(B.SEL_OP_TOPK, rows, V_g, k, device=G_.device())
        B.sel_topk_stats(xs, k, prm, v, i, st, ws)
        torch.cuda.synchronize()
        assert G_.ws_error(ws) == 0
        slices.append(xs)
        vals.append(v)
        ids.append(i)
        stats.append(st)
    return slices, torch.stack(vals, 1).contiguous(), torch.stack(ids, 1).contiguous(), torch.stack(stats, 1).contiguous()


def run_full_row(x, u, prm, G, misalign=False):
    """Full-row sampling (top_k = 0) on G shards: returns ids (uint32), probs
    and the OR of the shards' error words."""
    rows, V = x.shape
    offs = shards.shard_offsets(V, G)
    k = shards.full_row_list_len(offs)
    slices, vals, ids, stats = slice_stats(x, offs, k, prm, misalign)
    ud = G_.to_dev(np.asarray(u, dtype=np.float32).reshape(rows))
    plan = torch.zeros((rows, B.SHARD_PLAN_BYTES), dtype=torch.uint8, device=G_.device())
    B.sel_sample_shards(vals, ids, offs, prm, ud, stats=stats, plan=plan)
    wss, masses = [], []
    for g in range(G):
        ws = B.workspace(B.SEL_OP_SHARD_DRAW, rows, offs[g + 1] - offs[g], device=G_.device())
        m = torch.full((rows,), -1.0, dtype=torch.float64, device=G_.device())
        B.sel_shard_draw_mass(slices[g], offs[g], plan, m, ws)
        wss.append(ws)
        masses.append(m)
    gathered = torch.stack(masses, 1).contiguous()  # the all-gather
    outs_i, outs_p = [], []
    for g in range(G):
        oi = torch.full((rows,), -7, dtype=torch.int32, device=G_.device())
        op = torch.full((rows,), -7.0, device=G_.device())
        B.sel_shard_draw(slices[g], offs[g], g, G, plan, gathered, oi, op, wss[g])
        outs_i.append(oi)
        outs_p.append(op)
    torch.cuda.synchronize()
    # exactly one shard writes a real id for a decided row
    per = np.stack([B.ids_to_numpy(t) for t in outs_i])
    real = per < shards.OTHER_SHARD
    assert np.all(real.sum(axis=0) <= 1)
    assert np.all((real.sum(axis=0) == 1) | np.all(per == G_.INVALID, axis=0))
    ci, cp = shards.combine_draws_local(outs_i, outs_p)
    err = 0
    for ws in wss:
        err |= G_.ws_error(ws)
    return ci.cpu().numpy().astype(np.uint32), cp.cpu().numpy(), err, gathered.cpu().numpy()


def nucleus_sizes(x, T, top_p):
    z = x.astype(np.float64) / T
    z -= z.max(axis=1, keepdims=True)
    w = np.exp(z)
    w /= w.sum(axis=1, keepdims=True)
    c = np.cumsum(-np.sort(-w, axis=1), axis=1)
    return (c < top_p).sum(axis=1) + 1


def check_full(orc, x, u, prm, G, misalign=False, decided=None):
    gi, gp, err, _ = run_full_row(x, u, prm, G, misalign)
    ref = orc.sample(x, u, prm.temperature, 0, prm.top_p, prm.min_p, prm.order == B.SEL_ORDER_TEMP_LAST,
                     top_n_sigma=prm.top_n_sigma, typical_p=prm.typical_p if prm.typical_p > 0 else 1.0)
    failed = (gi == G_.INVALID) & (ref.ids != G_.INVALID)
    if decided is not None:
        assert np.array_equal(~failed, decided), np.nonzero(failed != ~decided)[0][:10]
    assert bool(err & ERR_BEYOND) == bool(failed.any()), (err, int(failed.sum()))
    assert err & ~ERR_BEYOND == 0, err
    assert np.all(np.isnan(gp[failed]))
    keep = ~failed
    G_.assert_sample_matches(gi[keep], gp[keep], type(ref)(ref.ids[keep], ref.probs[keep], ref.margin[keep]))
    return gi, gp, ref, failed


def test_stats_records_describe_each_slice():
    """Each record holds its slice's max, width, first logit, shifted moments
    and exponent sums (double-precision sums of the fp32 logits)."""
    rows, V, G, T = 5, 50_003, 3, 0.8
    x = synth.normal_rows(90, rows, V, 2.5)
    offs = shards.shard_offsets(V, G)
    prm = policy(T, 0, typ=0.7)
    _, _, _, stats = slice_stats(x, offs, 16, prm)
    rec = shards.stats_records(stats)
    assert rec.shape == (rows, G)
    for g in range(G):
        xs = x[:, offs[g]:offs[g + 1]].astype(np.float64)
        m = xs.max(axis=1)
        d = xs - xs[:, :1]
        w = np.exp((xs - m[:, None]) / T)
        gl = (xs - m[:, None]) / T
        r = rec[:, g]
        assert np.array_equal(r["max"], m.astype(np.float32))
        assert np.all(r["flags"] == 0) and np.all(r["n"] == offs[g + 1] - offs[g])
        assert np.array_equal(r["x0"], x[:, offs[g]])
        np.testing.assert_allclose(r["s1"], d.sum(axis=1), rtol=1e-6, atol=1e-3 * np.sqrt(xs.shape[1]))
        np.testing.assert_allclose(r["s2"], (d * d).sum(axis=1), rtol=1e-6)
        np.testing.assert_allclose(r["z"], w.sum(axis=1), rtol=1e-5)
        np.testing.assert_allclose(r["h"], (w * gl).sum(axis=1), rtol=1e-5)


def test_stats_flag_a_nonfinite_slice():
    x = synth.normal_rows(91, 3, 9_000, 1.0)
    x[1, 7_000] = np.nan
    offs = shards.shard_offsets(9_000, 2)
    _, _, ids, stats = slice_stats(x, offs, 8, policy(1.0, 0))
    rec = shards.stats_records(stats)
    assert rec["flags"][1, 1] == 1 and rec["flags"][1, 0] == 0 and np.all(rec["flags"][[0, 2]] == 0)
    assert np.all(B.ids_to_numpy(ids)[1, 1] == G_.INVALID)


@pytest.mark.parametrize("G,nsig,temp_last", [(2, 1.0, False), (3, 0.5, True), (5, 0.75, False)])
def test_top_n_sigma_with_top_k_on_shards(orc, G, nsig, temp_last):
    """top_k > 0 with top-n-sigma: the merged standard deviation sets the
    threshold over the merged candidates; the result matches the oracle."""
    rows, V, k = 48, 100_003, 40
    x = synth.normal_rows(92 + G, rows, V, 2.0)
    u = synth.uniforms(93, rows)
    offs = shards.shard_offsets(V, G, min_size=k)
    prm = policy(1.0, k, 0.95, 0.0, nsig=nsig, temp_last=temp_last)
    _, vals, ids, stats = slice_stats(x, offs, k, prm)
    oi = torch.full((rows,), -7, dtype=torch.int32, device=G_.device())
    op = torch.full((rows,), -7.0, device=G_.device())
    B.sel_sample_shards(vals, ids, offs, prm, G_.to_dev(u), oi, op, stats=stats)
    torch.cuda.synchronize()
    ref = orc.sample(x, u, 1.0, k, 0.95, 0.0, temp_last, top_n_sigma=nsig)
    G_.assert_sample_matches(B.ids_to_numpy(oi), op.cpu().numpy(), ref)
    # the filter is active: fewer than k candidates survive on most rows
    sigma = x.astype(np.float64).std(axis=1)
    top = np.sort(x, axis=1)[:, -k:]
    assert (top < (x.max(axis=1) - nsig * sigma)[:, None]).any()


@pytest.mark.parametrize("G", [2, 3, 5])
@pytest.mark.parametrize("misalign", [False, True])
def test_full_row_temperature_alone(orc, G, misalign):
    """No filter: every id survives; the draw falls in any shard."""
    rows = 40
    x = synth.normal_rows(94, rows, 30_001, 2.0)
    u = synth.uniforms(95, rows)
    gi, _, _, _ = check_full(orc, x, u, policy(0.9, 0), G, misalign, decided=np.ones(rows, bool))
    offs = shards.shard_offsets(30_001, G)
    owner = np.searchsorted(offs, gi.astype(np.int64), side="right") - 1
    assert len(set(owner.tolist())) == G  # draws landed in every shard


@pytest.mark.parametrize("min_p,T", [(0.05, 0.8), (0.001, 1.0), (0.3, 1.5)])
def test_full_row_min_p(orc, min_p, T):
    x = synth.normal_rows(96, 40, 60_001, 3.0)
    u = synth.uniforms(97, 40)
    check_full(orc, x, u, policy(T, 0, min_p=min_p), 3, decided=np.ones(40, bool))


@pytest.mark.parametrize("nsig", [0.5, 1.0, 3.0])
def test_full_row_top_n_sigma(orc, nsig):
    x = synth.normal_rows(98, 32, 50_003, 2.5)
    u = synth.uniforms(99, 32)
    check_full(orc, x, u, policy(1.0, 0, nsig=nsig), 4, decided=np.ones(32, bool))


@pytest.mark.parametrize("temp_last", [False, True])
def test_full_row_top_p_on_verify_batch(orc, temp_last):
    """Zipf/Gumbel rows at T 0.7, top_p 0.9: rows whose nucleus fits the 64
    merged candidates are decided and match the oracle; the others fail
    closed with bit 8 (the cut search runs unsharded only)."""
    x, _ = synth.workload_verify_batch()
    u = synth.uniforms(100, 49)
    T = 0.7
    Tf = 1.0 if temp_last else T
    sizes = nucleus_sizes(x, Tf, 0.9)
    _, _, _, failed = check_full(orc, x, u, policy(T, 0, 0.9, temp_last=temp_last), 2)
    assert np.array_equal(failed, sizes > shards.FULL_ROW_CANDIDATES)
    if not temp_last:
        assert failed.any() and (~failed).sum() > 20


def test_full_row_typical_and_filters_on_short_rows(orc):
    """V = 200 on two shards: the 64 merged candidates and a row of 200; a
    typical window, min-p and top-n-sigma, in both temperature orders."""
    x = synth.normal_rows(101, 30, 200, 2.0)
    u = synth.uniforms(102, 30)
    for last in (False, True):
        _, _, _, failed = check_full(orc, x, u, policy(0.8, 0, 0.95, 0.02, nsig=1.0, typ=0.9, temp_last=last), 2)
        assert failed.mean() < 0.5


def test_full_row_matches_unsharded_call(orc):
    """The same policy through sel_sample on the whole row and through the
    shards: the same draws (the two sum the row's mass in different orders,
    so only rows on a decision margin could differ)."""
    rows, V = 64, 202_048
    x = synth.normal_rows(103, rows, V, 3.0)
    u = synth.uniforms(104, rows)
    prm = policy(0.7, 0, 1.0, 0.05)
    gi, gp, _, _ = check_full(orc, x, u, prm, 3, decided=np.ones(rows, bool))
    wi, wp = G_.sample(x, u, 0.7, 0, 1.0, 0.05)
    ref = orc.sample(x, u, 0.7, 0, 1.0, 0.05, False)
    differ = gi != wi
    assert np.all(ref.margin[differ] <= G_.MARGIN)
    np.testing.assert_allclose(gp[~differ], wp[~differ], rtol=G_.PROB_RTOL)


def test_full_row_masses_add_up_to_the_row():
    """Temperature alone: the shards' masses sum to the row's softmax
    normaliser relative to its maximum."""
    rows, V, T = 6, 40_000, 1.3
    x = synth.normal_rows(105, rows, V, 2.0)
    u = synth.uniforms(106, rows)
    _, _, _, masses = run_full_row(x, u, policy(T, 0), 4)
    xd = x.astype(np.float64)
    want = np.exp((xd - xd.max(axis=1, keepdims=True)) / T).sum(axis=1)
    np.testing.assert_allclose(masses.sum(axis=1), want, rtol=1e-5)


def test_full_row_fails_closed_on_bad_rows(orc):
    x = synth.normal_rows(107, 5, 9_000, 1.0)
    x[3, 8_500] = np.inf          # in the last shard
    u = np.array([0.5, 1.0, -0.1, 0.5, 0.25], dtype=np.float32)
    gi, gp, _, _ = check_full(orc, x, u, policy(1.0, 0), 3, decided=np.ones(5, bool))
    assert np.all(gi[1:4] == G_.INVALID) and np.all(np.isnan(gp[1:4]))
    assert gi[0] != G_.INVALID and gi[4] != G_.INVALID


def test_full_row_draw_walks_ascending_global_ids(orc):
    """Many uniforms against one row: the drawn global id rises with u across
    the shard seams."""
    row = synth.normal_rows(108, 1, 5_000, 1.5)
    n = 600
    x = np.tile(row, (n, 1))
    u = ((np.arange(n) + 0.5) / n).astype(np.float32)
    gi, _, _, _ = check_full(orc, x, u, policy(1.0, 0), 3, decided=np.ones(n, bool))
    assert np.all(np.diff(gi.astype(np.int64)) >= 0)
    offs = shards.shard_offsets(5_000, 3)
    assert gi.min() < offs[1] and gi.max() >= offs[2]
