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
