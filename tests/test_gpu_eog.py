"""sel_argmax_excluding (the greedy serving variant with an EOG set) against
the oracle: bit-exact ids on the full verify batch, ragged and misaligned
rows, sets that hit unit and segment seams, the row's own maxima, ids past
the row, duplicates, an all-excluded row and nonfinite excluded logits."""
import numpy as np
import pytest
import torch

import oracle
from sampling_row_fp32_gb300 import binding as B, synth
from gpu_helpers import INVALID, SENTINEL, device, to_dev, ws_error

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def orc():
    return oracle.default()


def run(x, ex, misalign=False):
    rows, V = x.shape
    xd = to_dev(x, misalign)
    exd = to_dev(np.asarray(ex, dtype=np.uint32).view(np.int32)) if len(ex) else None
    out = torch.full((rows,), SENTINEL, dtype=torch.int32, device=device())
    ws = B.workspace(B.SEL_OP_ARGMAX, rows, V, device=device())
    B.sel_argmax_excluding(xd, exd, out, ws)
    torch.cuda.synchronize()
    if ws is not None:
        assert ws_error(ws) == 0
    return B.ids_to_numpy(out)


def test_verify_batch_excluding_the_maxima(orc):
    x, _ = synth.workload_verify_batch()
    top = np.argmax(x, axis=1)
    rng = np.random.default_rng(5)
    ex = list(np.unique(top[:20])) + list(rng.choice(x.shape[1], 30, replace=False)) + [0, 4095, 4096, 248_319]
    got = run(x, ex)
    want = orc.argmax_excluding(x, ex)
    assert np.array_equal(got, want)
    assert np.any(got != orc.argmax(x))  # the set changed some rows


@pytest.mark.parametrize("V", [1, 2, 5, 1023, 1025, 4097, 202_047, 202_048])
@pytest.mark.parametrize("misalign", [False, True])
def test_ragged_rows_and_tail_ids(orc, V, misalign):
    x = synth.normal_rows(60 + V % 97, 4, V, 2.0)
    x[:, V - 1] = 50.0          # the maximum in the ragged tail ...
    x[1, 0] = 50.0              # ... tied with id 0 in one row
    ex = sorted({V - 1, min(2, V - 1), V, V + 7, V - 1})  # tail, a low id, ids past the row, a duplicate
    got = run(x, ex, misalign)
    assert np.array_equal(got, orc.argmax_excluding(x, ex))


def test_segment_seams_and_duplicates(orc):
    rows, V = 7, 100_000
    x = synth.normal_rows(61, rows, V, 1.0)
    seams = [1023, 1024, 4095, 4096, 8191, 8192, 16383, 16384, 49_999, 50_000]
    for r in range(rows):
        x[r, seams] = 9.0 + r   # equal maxima at every seam
    ex = seams[: 2 * 3] + seams[:2] * 4
    got = run(x, ex)
    want = orc.argmax_excluding(x, ex)
    assert np.array_equal(got, want)
    assert np.all(got == 16383)  # the lowest seam left


def test_full_set_size_and_no_set(orc):
    x = synth.normal_rows(62, 9, 30_000, 3.0)
    ex = list(np.argsort(-x[0])[: B.SEL_MAX_EXCLUDED])  # the 256 largest of row 0
    got = run(x, ex)
    assert np.array_equal(got, orc.argmax_excluding(x, ex))
    assert np.array_equal(run(x, []), orc.argmax(x))


def test_all_excluded_and_nonfinite(orc):
    x = synth.normal_rows(63, 3, 40, 1.0)
    assert np.all(run(x, list(range(40))) == INVALID)
    y = x.copy()
    y[1, 13] = np.nan
    y[2, 30] = -np.inf
    got = run(y, [13, 30])
    assert got[1] == INVALID and got[2] == INVALID and got[0] != INVALID
    assert np.array_equal(got, orc.argmax_excluding(y, [13, 30]))


def test_too_many_ids_is_rejected():
    x = torch.zeros(1, 64, device=device())
    ex = torch.zeros(B.SEL_MAX_EXCLUDED + 1, dtype=torch.int32, device=device())
    out = torch.empty(1, dtype=torch.int32, device=device())
    ws = B.workspace(B.SEL_OP_ARGMAX, 1, 64, device=device())
    with pytest.raises(B.SelError):
        B.sel_argmax_excluding(x, ex, out, ws)
