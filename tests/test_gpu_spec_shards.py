"""Speculative acceptance on vocabulary shards, on one GPU: every target and
draft row is split into G id ranges; each range runs spec_shard_stats on its
slices, the gathered parts drive spec_accept_shards, and in the rejection
rule the residual draw runs on the slices (spec_shard_draw_mass, a gather of
the masses, spec_shard_draw on each shard, a minimum over the shards'
emitted arrays), as G ranks would run it. Accepted counts and emitted tokens
must match the oracle on the unsharded rows ("Speculative-decoding
acceptance rules": modified rejection sampling, steps 1-3, and
argmax-against-argmax; draws in ascending token id)."""
import numpy as np
import pytest
import torch

import oracle
import gpu_helpers as G_
from sampling_row_fp32_gb300 import binding as B, shards, synth

pytestmark = pytest.mark.gpu
REJ, ARG = B.SPEC_MODE_REJECTION, B.SPEC_MODE_ARGMAX


@pytest.fixture(scope="module")
def orc():
    import __graft_entry__
    __graft_entry__.build()
    return oracle.default()


def run_spec_shards(target, draft, tokens, u_acc, u_fin, T, mode, G, misalign=False):
    S, K1, V = target.shape
    K = K1 - 1
    offs = shards.shard_offsets(V, G)
    rej = mode == REJ and T > 0.0
    prm = B.SpecParams(T, mode)
    tok = G_.to_dev(np.ascontiguousarray(tokens, dtype=np.uint32).reshape(S, K).view(np.int32))
    ts_, ds_, parts = [], [], []
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        ts = G_.to_dev(np.ascontiguousarray(target[:, :, lo:hi]), misalign)
        ds = G_.to_dev(np.ascontiguousarray(draft[:, :, lo:hi]), misalign) if rej and K > 0 else None
        pt = torch.zeros((S, 2 * K + 1, B.SPEC_SHARD_PART_BYTES), dtype=torch.uint8, device=G_.device())
        ws = B.workspace(B.SEL_OP_SPEC, S, hi - lo, K, device=G_.device())
        B.spec_shard_stats(ts, ds, tok, lo, prm, pt, ws)
        torch.cuda.synchronize()
        assert G_.ws_error(ws) == 0
        ts_.append(ts)
        ds_.append(ds)
        parts.append(pt)
    gathered = torch.stack(parts, 1).contiguous()
    ua = G_.to_dev(np.asarray(u_acc, dtype=np.float32).reshape(S, K)) if rej else None
    uf = G_.to_dev(np.asarray(u_fin, dtype=np.float32).reshape(S)) if rej else None
    acc = torch.full((S,), G_.SENTINEL, dtype=torch.int32, device=G_.device())
    emi = torch.full((S, K + 1), G_.SENTINEL, dtype=torch.int32, device=G_.device())
    plan = torch.zeros((S, B.SPEC_SHARD_PLAN_BYTES), dtype=torch.uint8, device=G_.device()) if rej else None
    B.spec_accept_shards(gathered, tok, offs, prm, ua, uf, acc, emi, plan)
    torch.cuda.synchronize()
    if not rej:
        return B.ids_to_numpy(acc), B.ids_to_numpy(emi)
    wss, masses = [], []
    for g in range(G):
        ws = B.workspace(B.SEL_OP_SPEC_SHARD_DRAW, S, offs[g + 1] - offs[g], device=G_.device())
        m = torch.full((S, 2), -1.0, dtype=torch.float64, device=G_.device())
        B.spec_shard_draw_mass(ts_[g], ds_[g], plan, m, ws)
        wss.append(ws)
        masses.append(m)
    gm = torch.stack(masses, 1).contiguous()  # the all-gather
    ems = []
    for g in range(G):
        e = emi.clone()  # this rank's own copy of spec_accept_shards' output
        B.spec_shard_draw(ts_[g], ds_[g], offs[g], g, G, plan, gm, e, wss[g])
        ems.append(e)
    torch.cuda.synchronize()
    # one shard writes the drawn token; the others mark the slot theirs not
    acc_np = B.ids_to_numpy(acc)
    per = np.stack([B.ids_to_numpy(e) for e in ems])
    for s in range(S):
        n = acc_np[s]
        if n != G_.INVALID:
            col = per[:, s, n]
            assert (col < shards.OTHER_SHARD).sum() == 1, col
            assert np.all((col < shards.OTHER_SHARD) | (col == shards.OTHER_SHARD))
    for ws in wss:
        assert G_.ws_error(ws) == 0
    combined = shards.combine_emitted_local(ems).cpu().numpy().astype(np.uint32)
    return acc_np, combined


def check(orc, si, mode, G, misalign=False):
    acc, emi = run_spec_shards(si.target, si.draft, si.draft_tokens, si.u_acc, si.u_fin, si.temperature, mode, G,
                               misalign)
    ref = orc.spec_accept(si.target, si.draft, si.draft_tokens, si.temperature, mode, si.u_acc, si.u_fin)
    G_.assert_spec_matches(acc, emi, ref)
    return acc, emi, ref


@pytest.mark.parametrize("mode", [REJ, ARG])
@pytest.mark.parametrize("G", [2, 3])
def test_spec_workload_on_shards(orc, mode, G):
    """8 sequences x 8 drafts, V = 151,936, draft = target + N(0, 0.25)."""
    check(orc, synth.workload_spec(), mode, G)


@pytest.mark.parametrize("S,K,V,T,G", [(4, 3, 1000, 0.8, 2), (5, 4, 8191, 1.0, 3), (2, 8, 33_333, 1.3, 5),
                                       (9, 0, 4096, 1.0, 2), (3, 64, 2_000, 1.0, 4)])
@pytest.mark.parametrize("misalign", [False, True])
@pytest.mark.parametrize("mode", [REJ, ARG])
def test_shapes_on_shards(orc, S, K, V, T, G, misalign, mode):
    si = synth.spec_inputs(S=S, K=K, V=V, temperature=T, seed_target=S + K, seed_draft=V,
                           seed_u=int(T * 10) + 3, sigma_noise=0.7)
    check(orc, si, mode, G, misalign)


def test_all_accepted_draws_the_bonus_across_shards(orc):
    """Draft = target: every position accepts and the bonus token comes from
    p_K, whichever shard it lies in."""
    si = synth.spec_inputs(S=24, K=3, V=20_000, temperature=1.0, seed_target=5, seed_draft=6, seed_u=7,
                           sigma_noise=0.5)
    si.draft[:] = si.target[:, :3]
    acc, emi, _ = check(orc, si, REJ, 4)
    assert np.all(acc == 3)
    owners = np.searchsorted(shards.shard_offsets(20_000, 4), emi[:, 3].astype(np.int64), side="right") - 1
    assert len(set(owners.tolist())) > 1


def test_disjoint_supports_reject_at_once(orc):
    """Draft mass far from the target's: position 0 rejects and the residual
    is (almost) p itself."""
    si = synth.spec_inputs(S=12, K=4, V=9_000, temperature=1.0, seed_target=8, seed_draft=9, seed_u=10,
                           sigma_noise=0.5)
    si.draft[:] = -si.target[:, :4]
    si.draft_tokens[:] = np.argmax(si.draft, axis=2).astype(np.uint32)  # likely under q, not under p
    acc, _, _ = check(orc, si, REJ, 3)
    assert np.mean(acc == 0) > 0.5


def test_tokens_on_shard_seams(orc):
    """Draft tokens at the first and last id of each shard: their logits
    come from exactly one shard."""
    S, K, V, G = 6, 4, 12_000, 3
    si = synth.spec_inputs(S=S, K=K, V=V, temperature=1.0, seed_target=11, seed_draft=12, seed_u=13,
                           sigma_noise=0.3)
    offs = shards.shard_offsets(V, G)
    seam = np.array([offs[1] - 1, offs[1], offs[2] - 1, offs[2], 0, V - 1], dtype=np.uint32)
    rng = np.random.default_rng(14)
    si.draft_tokens[:] = rng.choice(seam, size=(S, K))
    # make those tokens likely under both distributions
    for s in range(S):
        for j in range(K):
            t = si.draft_tokens[s, j]
            si.target[s, j, t] += 6.0
            si.draft[s, j, t] += 6.0
    check(orc, si, REJ, G)
    check(orc, si, ARG, G)


def test_a_nonfinite_shard_invalidates_the_sequence(orc):
    si = synth.spec_inputs(S=4, K=3, V=8_000, temperature=1.0, seed_target=15, seed_draft=16, seed_u=17)
    si.target[1, 2, 7_900] = np.nan   # last shard of a target row
    si.draft[2, 0, 10] = np.inf       # first shard of a draft row
    acc, emi, _ = check(orc, si, REJ, 3)
    assert acc[1] == G_.INVALID and acc[2] == G_.INVALID and np.all(emi[[1, 2]] == G_.INVALID)
    assert acc[0] != G_.INVALID and acc[3] != G_.INVALID


def test_shards_agree_with_the_unsharded_call(orc):
    si = synth.workload_spec()
    acc, emi, ref = check(orc, si, REJ, 2)
    a1, e1 = G_.spec(si.target, si.draft, si.draft_tokens, si.u_acc, si.u_fin, si.temperature, REJ)
    exempt = (ref.margin_accept <= G_.MARGIN) | (ref.margin_draw <= G_.MARGIN)
    differ = (acc != a1) | (emi != e1).any(axis=1)
    assert not (differ & ~exempt).any()
