"""The C-ABI library builds, loads and exports what include/sel.h declares;
host-side argument checks answer without touching a GPU (no GPU needed)."""
import ctypes
import os
import re
import shutil

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sel.h")

pytestmark = pytest.mark.skipif(shutil.which("nvcc") is None and
                                not os.path.exists("/usr/local/cuda/bin/nvcc"),
                                reason="nvcc is needed to build the library")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:sel_status|size_t|const char\s*\*)\s*(\w+)\s*\(",
                                 text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from sampling_row_fp32_gb300 import binding, build
    build.build()
    return binding.load()


def test_header_declares_the_four_operations():
    names = declared_functions()
    for n in ("sel_argmax", "sel_topk", "sel_sample", "spec_accept",
              "sel_workspace_bytes", "sel_workspace_init", "sel_status_string"):
        assert n in names, names


def test_every_declared_symbol_is_exported(lib):
    raw = ctypes.CDLL(lib._name)
    for name in declared_functions():
        assert hasattr(raw, name), name
    from sampling_row_fp32_gb300 import binding
    assert sorted(binding.EXPORTED) == declared_functions()


def test_status_strings(lib):
    from sampling_row_fp32_gb300 import binding as B
    for s in range(5):
        assert B.status_string(s).startswith("SEL_")


def test_workspace_sizes_are_host_only_and_monotone(lib):
    from sampling_row_fp32_gb300 import binding as B
    a = B.sel_workspace_bytes(B.SEL_OP_ARGMAX, 49, 248_320)
    assert a > 0 and a % 8 == 0
    assert B.sel_workspace_bytes(B.SEL_OP_ARGMAX, 98, 248_320) > a
    assert 256 <= B.sel_workspace_bytes(B.SEL_OP_ARGMAX, 4, 1000) <= 4096  # header + counters
    t20 = B.sel_workspace_bytes(B.SEL_OP_TOPK, 49, 248_320, 20)
    t84 = B.sel_workspace_bytes(B.SEL_OP_TOPK, 49, 248_320, 84)
    assert 0 < t20 < t84
    assert B.sel_workspace_bytes(B.SEL_OP_TOPK, 49, 248_320, 0) == 0  # invalid k
    assert B.sel_workspace_bytes(B.SEL_OP_TOPK, 1, 10, 11) == 0       # k > V
    assert B.sel_workspace_bytes(B.SEL_OP_SAMPLE, 64, 202_048, 40) == \
        B.sel_workspace_bytes(B.SEL_OP_TOPK, 64, 202_048, 40)
    assert B.sel_workspace_bytes(8, 1, 10, 1) == 0                    # unknown op


def test_host_validation_needs_no_gpu(lib):
    """Arguments the host can reject are rejected before any CUDA call."""
    from sampling_row_fp32_gb300 import binding as B
    vp = ctypes.c_void_p
    fake = vp(0x10000)   # never dereferenced: every call below fails validation first
    assert lib.sel_argmax(fake, 1, 0, fake, None, 0, None) == B.SEL_EINVAL          # V = 0
    assert lib.sel_argmax(fake, 1, 0x80000000, fake, None, 0, None) == B.SEL_EINVAL  # V >= 2^31
    assert lib.sel_argmax(None, 1, 10, fake, None, 0, None) == B.SEL_EINVAL          # null logits
    assert lib.sel_argmax(vp(0x10002), 1, 10, fake, None, 0, None) == B.SEL_EINVAL   # misaligned
    assert lib.sel_argmax(None, 0, 10, None, None, 0, None) == B.SEL_OK              # rows = 0
    assert lib.sel_argmax(fake, 3, 300_000, fake, None, 0, None) == B.SEL_EINVAL     # ws missing
    assert lib.sel_argmax(fake, 3, 300_000, fake, fake, 16, None) == B.SEL_EWORKSPACE
    assert lib.sel_argmax(fake, 3, 300_000, fake, vp(0x10010), 1 << 30, None) == B.SEL_EINVAL
    assert lib.sel_topk(fake, 1, 10, 11, fake, fake, None, 0, None) == B.SEL_EINVAL  # k > V
    assert lib.sel_topk(fake, 1, 10, 0, fake, fake, None, 0, None) == B.SEL_EINVAL   # k = 0
    assert lib.sel_topk(fake, 1, 5000, 1025, fake, fake, None, 0, None) == B.SEL_EUNSUPPORTED

    def sample(T, k, p, m, order=0, nsig=0.0, typ=0.0):
        prm = B.SampleParams(T, k, p, m, order, nsig, typ)
        return lib.sel_sample(fake, 1, 10, ctypes.byref(prm), fake, fake, fake, None, 0, None)
    # top-n-sigma: finite and >= 0; typical_p in [0, 1] (0 and 1 are off)
    assert sample(1.0, 5, 1.0, 0.0, nsig=-0.5) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, 0.0, nsig=float("nan")) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, 0.0, nsig=float("inf")) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, 0.0, typ=-0.1) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, 0.0, typ=1.5) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, 0.0, typ=float("nan")) == B.SEL_EINVAL
    assert sample(float("nan"), 5, 1.0, 0.0) == B.SEL_EINVAL
    assert sample(-1.0, 5, 1.0, 0.0) == B.SEL_EINVAL
    assert sample(1.0, 5, 0.0, 0.0) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.5, 0.0) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, 1.0) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, -0.1) == B.SEL_EINVAL
    assert sample(1.0, 5, 1.0, 0.0, order=2) == B.SEL_EINVAL
    assert sample(1.0, 0, 1.0, 0.0) == B.SEL_EINVAL          # full-row sampling: needs its workspace
    assert B.sel_workspace_bytes(B.SEL_OP_SAMPLE, 4, 248_320, 0) >= B.sel_workspace_bytes(B.SEL_OP_SAMPLE, 4, 248_320, 64)
    prm = B.SampleParams(1.0, 5, 1.0, 0.0, 0)
    assert lib.sel_sample(fake, 1, 10, None, fake, fake, fake, None, 0, None) == B.SEL_EINVAL
    assert lib.sel_sample(fake, 0, 10, ctypes.byref(prm), None, None, None, None, 0, None) == B.SEL_OK


def test_shard_merge_validation_needs_no_gpu(lib):
    from sampling_row_fp32_gb300 import binding as B
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    U = ctypes.c_uint32

    def offs(*o):
        return ctypes.cast((U * len(o))(*o), vp)

    good = offs(0, 100, 200)
    m = lib.sel_merge_shards
    assert m(fake, fake, 0, 2, 5, good, fake, fake, None) == B.SEL_OK                # rows = 0
    assert m(fake, fake, 1, 0, 5, good, fake, fake, None) == B.SEL_EINVAL            # G = 0
    assert m(fake, fake, 1, 65, 5, offs(*range(0, 66 * 10, 10)), fake, fake, None) == B.SEL_EINVAL
    assert m(fake, fake, 1, 2, 0, good, fake, fake, None) == B.SEL_EINVAL            # k = 0
    assert m(fake, fake, 1, 2, 1025, offs(0, 2000, 4000), fake, fake, None) == B.SEL_EINVAL
    assert m(fake, fake, 1, 2, 5, offs(0, 3, 200), fake, fake, None) == B.SEL_EINVAL  # shard < k
    assert m(fake, fake, 1, 2, 5, offs(0, 100, 90), fake, fake, None) == B.SEL_EINVAL  # not increasing
    assert m(fake, fake, 1, 2, 5, offs(0, 100, 0x80000000), fake, fake, None) == B.SEL_EINVAL
    assert m(fake, fake, 1, 2, 5, None, fake, fake, None) == B.SEL_EINVAL             # no offsets
    assert m(None, fake, 1, 2, 5, good, fake, fake, None) == B.SEL_EINVAL
    assert m(fake, fake, 1, 2, 5, good, None, fake, None) == B.SEL_EINVAL
    assert m(vp(0x10002), fake, 1, 2, 5, good, fake, fake, None) == B.SEL_EINVAL      # misaligned
    s = lib.sel_sample_shards
    p = B.SampleParams(0.7, 5, 0.9, 0.05, 0)
    # (vals, ids, stats, rows, G, k, offsets, params, uniforms, out_ids, out_probs, plan, stream)
    assert s(fake, fake, None, 1, 2, 5, good, None, fake, fake, fake, None, None) == B.SEL_EINVAL
    assert s(fake, fake, None, 1, 2, 5, good, ctypes.byref(B.SampleParams(0.7, 6, 0.9, 0.05, 0)),
             fake, fake, fake, None, None) == B.SEL_EINVAL                             # top_k != k
    assert s(fake, fake, None, 1, 2, 5, good, ctypes.byref(B.SampleParams(float("nan"), 5, 0.9, 0.05, 0)),
             fake, fake, fake, None, None) == B.SEL_EINVAL
    assert s(fake, fake, None, 1, 2, 5, good, ctypes.byref(B.SampleParams(0.7, 5, 1.5, 0.05, 0)),
             fake, fake, fake, None, None) == B.SEL_EINVAL
    assert s(fake, fake, None, 1, 2, 5, good, ctypes.byref(p), None, fake, fake, None, None) == B.SEL_EINVAL
    # top-n-sigma needs the whole row's standard deviation: the shards' statistics
    nsig = ctypes.byref(B.SampleParams(0.7, 5, 0.9, 0.05, 0, 1.0, 0.0))
    assert s(fake, fake, None, 1, 2, 5, good, nsig, fake, fake, fake, None, None) == B.SEL_EINVAL
    assert s(fake, fake, vp(0x10004), 1, 2, 5, good, nsig, fake, fake, fake, None, None) == B.SEL_EINVAL
    # full-row sampling: statistics, a plan, and at most 64 candidates per list
    full = ctypes.byref(B.SampleParams(0.7, 0, 0.9, 0.0, 0))
    assert s(fake, fake, None, 1, 2, 5, good, full, fake, None, None, fake, None) == B.SEL_EINVAL
    assert s(fake, fake, fake, 1, 2, 5, good, full, fake, None, None, None, None) == B.SEL_EINVAL
    assert s(fake, fake, fake, 1, 2, 65, offs(0, 100, 200), full, fake, None, None, fake,
             None) == B.SEL_EINVAL
    assert s(fake, fake, fake, 1, 2, 5, good, full, fake, None, None, vp(0x10008), None) == B.SEL_EINVAL
    assert s(fake, fake, None, 0, 2, 5, good, ctypes.byref(p), None, None, None, None, None) == B.SEL_OK


def test_shard_stats_and_draw_validation_needs_no_gpu(lib):
    from sampling_row_fp32_gb300 import binding as B
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    p = B.SampleParams(1.0, 0, 0.9, 0.0, 0)
    st = lib.sel_topk_stats
    assert st(fake, 0, 100, 5, ctypes.byref(p), None, None, None, None, 0, None) == B.SEL_OK    # rows = 0
    assert st(fake, 1, 100, 5, None, fake, fake, fake, fake, 1 << 20, None) == B.SEL_EINVAL     # no policy
    assert st(fake, 1, 100, 5, ctypes.byref(p), fake, fake, None, fake, 1 << 20, None) == B.SEL_EINVAL
    assert st(fake, 1, 100, 5, ctypes.byref(p), fake, fake, vp(0x10004), fake, 1 << 20, None) == B.SEL_EINVAL
    assert st(fake, 1, 100, 0, ctypes.byref(p), fake, fake, fake, fake, 1 << 20, None) == B.SEL_EINVAL
    assert st(fake, 1, 4, 5, ctypes.byref(p), fake, fake, fake, fake, 1 << 20, None) == B.SEL_EINVAL  # k > V
    n = B.sel_workspace_bytes(B.SEL_OP_SHARD_DRAW, 3, 100_000, 0)
    assert n > 0 and n == B.sel_workspace_bytes(B.SEL_OP_SHARD_DRAW, 3, 100_000, 7)
    assert B.sel_workspace_bytes(B.SEL_OP_SHARD_DRAW, 3, 0, 0) == 0
    m = lib.sel_shard_draw_mass
    # (logits, rows, V, offset, plan, mass, ws, ws_bytes, stream)
    assert m(None, 0, 100, 0, None, None, None, 0, None) == B.SEL_OK                            # rows = 0
    assert m(fake, 3, 0, 0, fake, fake, fake, n, None) == B.SEL_EINVAL                          # V = 0
    assert m(fake, 3, 100_000, 0x7FFFFFFF, fake, fake, fake, n, None) == B.SEL_EINVAL           # ids past 2^31
    assert m(fake, 3, 100_000, 0, None, fake, fake, n, None) == B.SEL_EINVAL                    # no plan
    assert m(fake, 3, 100_000, 0, vp(0x10008), fake, fake, n, None) == B.SEL_EINVAL             # plan alignment
    assert m(fake, 3, 100_000, 0, fake, None, fake, n, None) == B.SEL_EINVAL                    # no mass
    assert m(fake, 3, 100_000, 0, fake, fake, fake, n - 1, None) == B.SEL_EWORKSPACE
    assert m(fake, 3, 100_000, 0, fake, fake, vp(0x10080), n, None) == B.SEL_EINVAL             # ws alignment
    d = lib.sel_shard_draw
    # (logits, rows, V, offset, g, G, plan, masses, out_ids, out_probs, ws, ws_bytes, stream)
    assert d(fake, 3, 100_000, 0, 2, 2, fake, fake, fake, fake, fake, n, None) == B.SEL_EINVAL  # g >= G
    assert d(fake, 3, 100_000, 0, 0, 65, fake, fake, fake, fake, fake, n, None) == B.SEL_EINVAL
    assert d(fake, 3, 100_000, 0, 0, 2, fake, None, fake, fake, fake, n, None) == B.SEL_EINVAL  # no masses
    assert d(fake, 3, 100_000, 0, 0, 2, fake, vp(0x10004), fake, fake, fake, n, None) == B.SEL_EINVAL
    assert d(fake, 3, 100_000, 0, 0, 2, fake, fake, fake, fake, fake, 16, None) == B.SEL_EWORKSPACE
    assert d(fake, 0, 100_000, 0, 0, 2, None, None, None, None, None, 0, None) == B.SEL_OK


def test_spec_shard_validation_needs_no_gpu(lib):
    from sampling_row_fp32_gb300 import binding as B
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    U = ctypes.c_uint32
    rej = ctypes.byref(B.SpecParams(1.0, B.SPEC_MODE_REJECTION))
    arg = ctypes.byref(B.SpecParams(1.0, B.SPEC_MODE_ARGMAX))
    n = B.sel_workspace_bytes(B.SEL_OP_SPEC, 4, 1000, 3)
    st = lib.spec_shard_stats
    # (target, draft, tokens, S, K, V, offset, params, parts, ws, ws_bytes, stream)
    assert st(fake, fake, fake, 0, 3, 1000, 0, rej, fake, fake, n, None) == B.SEL_OK             # S = 0
    assert st(fake, fake, fake, 4, 65, 1000, 0, rej, fake, fake, n, None) == B.SEL_EUNSUPPORTED  # K > 64
    assert st(fake, fake, fake, 4, 3, 0, 0, rej, fake, fake, n, None) == B.SEL_EINVAL            # V = 0
    assert st(fake, fake, fake, 4, 3, 1000, 0x7FFFFFFF, rej, fake, fake, n, None) == B.SEL_EINVAL
    assert st(fake, None, fake, 4, 3, 1000, 0, rej, fake, fake, n, None) == B.SEL_EINVAL         # no draft
    assert st(fake, fake, fake, 4, 3, 1000, 0, rej, None, fake, n, None) == B.SEL_EINVAL         # no parts
    assert st(fake, fake, fake, 4, 3, 1000, 0, rej, vp(0x10004), fake, n, None) == B.SEL_EINVAL
    assert st(fake, fake, fake, 4, 3, 1000, 0, rej, fake, fake, n - 1, None) == B.SEL_EWORKSPACE
    assert st(fake, fake, fake, 4, 3, 1000, 0, None, fake, fake, n, None) == B.SEL_EINVAL
    acc = lib.spec_accept_shards
    offs = ctypes.cast((U * 3)(0, 500, 1000), vp)
    # (parts, tokens, S, K, G, offsets, params, u_acc, u_fin, accepted, emitted, plan, stream)
    assert acc(fake, fake, 0, 3, 2, offs, rej, fake, fake, fake, fake, fake, None) == B.SEL_OK
    assert acc(fake, fake, 4, 3, 0, offs, rej, fake, fake, fake, fake, fake, None) == B.SEL_EINVAL
    assert acc(fake, fake, 4, 3, 2, ctypes.cast((U * 3)(1, 500, 1000), vp), rej, fake, fake, fake, fake, fake,
               None) == B.SEL_EINVAL                                                            # not from 0
    assert acc(fake, fake, 4, 3, 2, ctypes.cast((U * 3)(0, 500, 500), vp), rej, fake, fake, fake, fake, fake,
               None) == B.SEL_EINVAL                                                            # empty shard
    assert acc(fake, fake, 4, 65, 2, offs, rej, fake, fake, fake, fake, fake, None) == B.SEL_EUNSUPPORTED
    assert acc(fake, fake, 4, 3, 2, offs, rej, fake, fake, fake, fake, None, None) == B.SEL_EINVAL  # no plan
    assert acc(fake, fake, 4, 3, 2, offs, rej, fake, None, fake, fake, fake, None) == B.SEL_EINVAL  # no u_fin
    assert acc(fake, fake, 4, 3, 2, offs, rej, fake, fake, fake, fake, vp(0x10008), None) == B.SEL_EINVAL
    n2 = B.sel_workspace_bytes(B.SEL_OP_SPEC_SHARD_DRAW, 4, 500, 0)
    assert n2 > 0
    m = lib.spec_shard_draw_mass
    # (target, draft, S, K, V, plan, mass, ws, ws_bytes, stream)
    assert m(fake, fake, 0, 3, 500, fake, fake, fake, n2, None) == B.SEL_OK
    assert m(fake, fake, 4, 3, 500, None, fake, fake, n2, None) == B.SEL_EINVAL
    assert m(fake, fake, 4, 3, 500, fake, None, fake, n2, None) == B.SEL_EINVAL
    assert m(fake, fake, 4, 3, 500, fake, fake, fake, n2 - 1, None) == B.SEL_EWORKSPACE
    assert m(fake, fake, 4, 65, 500, fake, fake, fake, n2, None) == B.SEL_EINVAL
    d = lib.spec_shard_draw
    # (target, draft, S, K, V, offset, g, G, plan, masses, emitted, ws, ws_bytes, stream)
    assert d(fake, fake, 4, 3, 500, 500, 2, 2, fake, fake, fake, fake, n2, None) == B.SEL_EINVAL  # g >= G
    assert d(fake, fake, 4, 3, 500, 500, 1, 2, fake, None, fake, fake, n2, None) == B.SEL_EINVAL
    assert d(fake, fake, 4, 3, 500, 500, 1, 2, fake, fake, None, fake, n2, None) == B.SEL_EINVAL
    assert d(fake, fake, 4, 3, 500, 500, 1, 2, fake, fake, fake, fake, 16, None) == B.SEL_EWORKSPACE
    assert d(fake, fake, 0, 3, 500, 500, 1, 2, None, None, None, None, 0, None) == B.SEL_OK


def test_eog_validation_needs_no_gpu(lib):
    from sampling_row_fp32_gb300 import binding as B
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    f = lib.sel_argmax_excluding
    assert f(fake, 1, 10, fake, 257, fake, fake, 4096, None) == B.SEL_EINVAL   # too many ids
    assert f(fake, 1, 10, None, 3, fake, fake, 4096, None) == B.SEL_EINVAL     # no id array
    assert f(fake, 1, 10, vp(0x10002), 3, fake, fake, 4096, None) == B.SEL_EINVAL
    assert f(fake, 1, 0, fake, 3, fake, fake, 4096, None) == B.SEL_EINVAL      # V = 0
    assert f(None, 0, 10, fake, 3, None, None, 0, None) == B.SEL_OK            # rows = 0
    assert f(fake, 3, 300_000, fake, 3, fake, fake, 16, None) == B.SEL_EWORKSPACE


def test_spec_rules_validation_needs_no_gpu(lib):
    from sampling_row_fp32_gb300 import binding as B
    vp = ctypes.c_void_p
    fake = vp(0x10000)
    p = B.SampleParams(1.0, 10, 0.9, 0.0, 0)
    f = lib.spec_accept_sampler
    assert f(fake, fake, 0, 3, 100, ctypes.byref(p), fake, fake, fake, fake, 4096, None) == B.SEL_OK  # S = 0
    assert f(fake, fake, 2, 3, 100, None, fake, fake, fake, fake, 4096, None) == B.SEL_EINVAL
    assert f(fake, fake, 2, 3, 100, ctypes.byref(B.SampleParams(1.0, 0, 0.9, 0.0, 0)), fake, fake, fake,
             fake, 16, None) == B.SEL_EWORKSPACE                                              # top_k = 0: full row
    assert (B.sel_workspace_bytes(B.SEL_OP_SPEC_SAMPLER, 8, 151_936, 0)
            == B.sel_workspace_bytes(B.SEL_OP_SPEC_SAMPLER, 8, 151_936, 64))
    assert f(fake, fake, 2, 3, 100, ctypes.byref(p), None, fake, fake, fake, 4096, None) == B.SEL_EINVAL
    assert f(fake, fake, 2, 3, 300_000, ctypes.byref(p), fake, fake, fake, fake, 16, None) == B.SEL_EWORKSPACE
    g = lib.spec_diagnostics
    assert g(fake, fake, 2, 3, 100, ctypes.c_float(0.0), fake, fake, fake, 4096, None) == B.SEL_EINVAL  # T = 0
    assert g(fake, fake, 2, 0, 100, ctypes.c_float(1.0), fake, fake, fake, 4096, None) == B.SEL_OK      # K = 0
    assert g(fake, None, 2, 3, 100, ctypes.c_float(1.0), fake, fake, fake, 4096, None) == B.SEL_EINVAL
    assert g(fake, fake, 2, 3, 300_000, ctypes.c_float(1.0), fake, fake, fake, 16, None) == B.SEL_EWORKSPACE
    assert B.sel_workspace_bytes(B.SEL_OP_SPEC_DIAG, 8, 151_936, 8) > B.sel_workspace_bytes(B.SEL_OP_SPEC, 8, 151_936, 8)
    assert B.sel_workspace_bytes(B.SEL_OP_SPEC_SAMPLER, 72, 151_936, 40) > B.sel_workspace_bytes(B.SEL_OP_SAMPLE, 72, 151_936, 40)
