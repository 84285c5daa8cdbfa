"""sel_argmax_noalloc: the argmax entry point for callers that cannot
allocate device memory (it takes no workspace and uses scratch the library
reserved at load). Its ids must equal sel_argmax's, bit for bit, on two
calls in a row; requests too large for the reserved scratch are refused.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import ctypes

import numpy as np
import pytest
import torch

from sampling_row_fp32_gb300 import binding as B
from sampling_row_fp32_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    return B.load()


def regular_argmax(x):
    rows, V = x.shape
    out = torch.full((rows,), -7, dtype=torch.int32, device="cuda")
    ws = B.workspace(B.SEL_OP_ARGMAX, rows, V, device="cuda")
    B.sel_argmax(x, out, ws)
    return out


def noalloc_argmax(x):
    out = torch.full((x.shape[0],), -7, dtype=torch.int32, device="cuda")
    B.sel_argmax_noalloc(x, out)
    return out


def test_matches_sel_argmax_on_two_calls_in_a_row(lib):
    a = torch.from_numpy(synth.zipf_gumbel_rows(seed=31, rows=49, V=248_320)).cuda()
    b = torch.from_numpy(synth.normal_rows(32, 64, 202_048, 3.0)).cuda()
    b[5, [17, 90_000]] = b[5].max() + 1           # a planted tie
    b[9, 1234] = float("nan")                      # a row that fails closed
    want_a, want_b = regular_argmax(a), regular_argmax(b)
    got_a = noalloc_argmax(a)                      # first call
    got_b = noalloc_argmax(b)                      # second call, other shape
    torch.cuda.synchronize()
    assert torch.equal(got_a, want_a)
    assert torch.equal(got_b, want_b)
    assert int(got_b[5]) == 17 and B.ids_to_numpy(got_b)[9] == B.SEL_INVALID_ID
    # and again on the first input, after the second call left its state
    assert torch.equal(noalloc_argmax(a), want_a)


def test_rejects_requests_beyond_the_reserved_scratch(lib):
    rows, V = 200_000, 248_320
    need = B.sel_workspace_bytes(B.SEL_OP_ARGMAX, rows, V)
    assert need > B.SEL_NOALLOC_SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: the size check comes first
    assert lib.sel_argmax_noalloc(fake, rows, V, fake, None) == B.SEL_EWORKSPACE
    # 8 bytes per row after a 256-byte header, in 256-byte steps
    assert B.sel_workspace_bytes(B.SEL_OP_ARGMAX, 131_040, V) <= B.SEL_NOALLOC_SCRATCH_BYTES
    assert B.sel_workspace_bytes(B.SEL_OP_ARGMAX, 131_041, V) > B.SEL_NOALLOC_SCRATCH_BYTES


def test_largest_request_that_fits(lib):
    """131,040 rows need the whole reserved scratch (8 bytes a row after the
    header): the largest call the entry point accepts, on short rows."""
    rows, V = 131_040, 8
    assert B.sel_workspace_bytes(B.SEL_OP_ARGMAX, rows, V) <= B.SEL_NOALLOC_SCRATCH_BYTES
    x = torch.from_numpy(synth.normal_rows(33, rows, V, 3.0)).cuda()
    x[7, [2, 5]] = x[7].max() + 1                  # a tie inside one row
    want = regular_argmax(x)
    for _ in range(2):
        got = noalloc_argmax(x)
        torch.cuda.synchronize()
        assert torch.equal(got, want)
    assert int(got[7]) == 2


def test_calls_on_two_streams_ordered_by_an_event(lib):
    """The calls share one scratch array, so calls on different streams must
    be ordered: here the second stream waits on an event recorded after the
    first call. Both results equal sel_argmax's."""
    a = torch.from_numpy(synth.normal_rows(34, 49, 248_320, 3.0)).cuda()
    b = torch.from_numpy(synth.normal_rows(35, 64, 202_048, 3.0)).cuda()
    want_a, want_b = regular_argmax(a), regular_argmax(b)
    out_a = torch.full((49,), -7, dtype=torch.int32, device="cuda")
    out_b = torch.full((64,), -7, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()  # inputs and pre-filled outputs are ready for both streams
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    done = torch.cuda.Event()
    with torch.cuda.stream(s1):
        B.sel_argmax_noalloc(a, out_a, stream=s1)
        done.record(s1)
    s2.wait_event(done)
    with torch.cuda.stream(s2):
        B.sel_argmax_noalloc(b, out_b, stream=s2)
    torch.cuda.synchronize()
    assert torch.equal(out_a, want_a)
    assert torch.equal(out_b, want_b)
