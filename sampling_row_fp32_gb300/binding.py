"""Python binding of the C-ABI library (``include/sel.h``).

Argument marshalling only: torch CUDA tensors supply device pointers and the
current (or given) CUDA stream; every step of the selection path runs in the
library's kernels. The functions carry the C names. A missing or unloadable
library raises immediately -- there is no fallback implementation.

Ids are 32-bit unsigned on the device; torch tensors of dtype int32 or
uint32 are accepted for them (SEL_INVALID_ID reads as -1 through int32).
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

from . import build as _build

SEL_OK, SEL_EINVAL, SEL_EWORKSPACE, SEL_ECUDA, SEL_EUNSUPPORTED = range(5)
SEL_INVALID_ID = 0xFFFFFFFF
SEL_MAX_K = 1024
(SEL_OP_ARGMAX, SEL_OP_TOPK, SEL_OP_SAMPLE, SEL_OP_SPEC, SEL_OP_SPEC_SAMPLER, SEL_OP_SPEC_DIAG,
 SEL_OP_SHARD_DRAW, SEL_OP_SPEC_SHARD_DRAW) = range(8)
SEL_ORDER_TEMP_FIRST, SEL_ORDER_TEMP_LAST = 0, 1
SPEC_MODE_REJECTION, SPEC_MODE_ARGMAX = 0, 1

EXPORTED = ("sel_workspace_bytes", "sel_workspace_init", "sel_argmax", "sel_topk",
            "sel_sample", "spec_accept", "sel_status_string", "sel_argmax_noalloc",
            "sel_merge_shards", "sel_sample_shards", "sel_argmax_excluding",
            "spec_accept_sampler", "spec_diagnostics", "sel_topk_stats", "sel_shard_draw_mass",
            "sel_shard_draw", "spec_shard_stats", "spec_accept_shards", "spec_shard_draw_mass",
            "spec_shard_draw")
SEL_NOALLOC_SCRATCH_BYTES = 1 << 20
SEL_MAX_SHARDS = 64
SEL_MAX_EXCLUDED = 256
SEL_OTHER_SHARD = 0xFFFFFFFE
ROW_STATS_BYTES = 48   # struct sel_row_stats
SHARD_PLAN_BYTES = 48  # struct sel_shard_plan
FULL_ROW_CANDIDATES = 64
SPEC_SHARD_PART_BYTES = 32  # struct spec_shard_part
SPEC_SHARD_PLAN_BYTES = 32  # struct spec_shard_plan
SPEC_SHARD_MAX_K = 64


class SelError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class SampleParams(ctypes.Structure):
    """struct sel_sample_params (top_n_sigma and typical_p default to off)"""
    _fields_ = [("temperature", ctypes.c_float), ("top_k", ctypes.c_uint32),
                ("top_p", ctypes.c_float), ("min_p", ctypes.c_float),
                ("order", ctypes.c_int32), ("top_n_sigma", ctypes.c_float),
                ("typical_p", ctypes.c_float)]


class SpecParams(ctypes.Structure):
    """struct spec_params"""
    _fields_ = [("temperature", ctypes.c_float), ("mode", ctypes.c_int32)]


_vp = ctypes.c_void_p
_u32 = ctypes.c_uint32
_sz = ctypes.c_size_t
_lib: ctypes.CDLL | None = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None) -> ctypes.CDLL:
    """Load libsel.so (once). Raises if it has not been built."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or library_path()
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is not built: run `python -m sampling_row_fp32_gb300.build` "
                           "(or __graft_entry__.build()) first")
    lib = ctypes.CDLL(p)
    lib.sel_workspace_bytes.argtypes = [ctypes.c_int, _u32, _u32, _u32]
    lib.sel_workspace_bytes.restype = _sz
    lib.sel_workspace_init.argtypes = [_vp, _sz, _vp]
    lib.sel_workspace_init.restype = ctypes.c_int
    lib.sel_argmax.argtypes = [_vp, _u32, _u32, _vp, _vp, _sz, _vp]
    lib.sel_argmax.restype = ctypes.c_int
    lib.sel_topk.argtypes = [_vp, _u32, _u32, _u32, _vp, _vp, _vp, _sz, _vp]
    lib.sel_topk.restype = ctypes.c_int
    lib.sel_sample.argtypes = [_vp, _u32, _u32, ctypes.POINTER(SampleParams), _vp, _vp, _vp,
                               _vp, _sz, _vp]
    lib.sel_sample.restype = ctypes.c_int
    lib.spec_accept.argtypes = [_vp, _vp, _vp, _u32, _u32, _u32, ctypes.POINTER(SpecParams),
                                _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.spec_accept.restype = ctypes.c_int
    lib.sel_argmax_noalloc.argtypes = [_vp, _u32, _u32, _vp, _vp]
    lib.sel_argmax_noalloc.restype = ctypes.c_int
    lib.spec_accept_sampler.argtypes = [_vp, _vp, _u32, _u32, _u32, ctypes.POINTER(SampleParams), _vp,
                                        _vp, _vp, _vp, _sz, _vp]
    lib.spec_accept_sampler.restype = ctypes.c_int
    lib.spec_diagnostics.argtypes = [_vp, _vp, _u32, _u32, _u32, ctypes.c_float, _vp, _vp, _vp, _sz, _vp]
    lib.spec_diagnostics.restype = ctypes.c_int
    lib.sel_argmax_excluding.argtypes = [_vp, _u32, _u32, _vp, _u32, _vp, _vp, _sz, _vp]
    lib.sel_argmax_excluding.restype = ctypes.c_int
    lib.sel_merge_shards.argtypes = [_vp, _vp, _u32, _u32, _u32, _vp, _vp, _vp, _vp]
    lib.sel_merge_shards.restype = ctypes.c_int
    lib.sel_sample_shards.argtypes = [_vp, _vp, _vp, _u32, _u32, _u32, _vp, ctypes.POINTER(SampleParams),
                                      _vp, _vp, _vp, _vp, _vp]
    lib.sel_topk_stats.argtypes = [_vp, _u32, _u32, _u32, ctypes.POINTER(SampleParams), _vp, _vp, _vp, _vp,
                                   _sz, _vp]
    lib.sel_topk_stats.restype = ctypes.c_int
    lib.sel_shard_draw_mass.argtypes = [_vp, _u32, _u32, _u32, _vp, _vp, _vp, _sz, _vp]
    lib.sel_shard_draw_mass.restype = ctypes.c_int
    lib.sel_shard_draw.argtypes = [_vp, _u32, _u32, _u32, _u32, _u32, _vp, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.sel_shard_draw.restype = ctypes.c_int
    lib.spec_shard_stats.argtypes = [_vp, _vp, _vp, _u32, _u32, _u32, _u32, ctypes.POINTER(SpecParams), _vp, _vp,
                                     _sz, _vp]
    lib.spec_shard_stats.restype = ctypes.c_int
    lib.spec_accept_shards.argtypes = [_vp, _vp, _u32, _u32, _u32, _vp, ctypes.POINTER(SpecParams), _vp, _vp, _vp,
                                       _vp, _vp, _vp]
    lib.spec_accept_shards.restype = ctypes.c_int
    lib.spec_shard_draw_mass.argtypes = [_vp, _vp, _u32, _u32, _u32, _vp, _vp, _vp, _sz, _vp]
    lib.spec_shard_draw_mass.restype = ctypes.c_int
    lib.spec_shard_draw.argtypes = [_vp, _vp, _u32, _u32, _u32, _u32, _u32, _u32, _vp, _vp, _vp, _vp, _sz, _vp]
    lib.spec_shard_draw.restype = ctypes.c_int
    lib.sel_sample_shards.restype = ctypes.c_int
    lib.sel_status_string.argtypes = [ctypes.c_int]
    lib.sel_status_string.restype = ctypes.c_char_p
    if path is None:
        _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().sel_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != SEL_OK:
        raise SelError(status, what)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("tensors passed to the selection library must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("tensors passed to the selection library must be contiguous")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check_f32(t, name):
    if t is not None and not isinstance(t, int) and t.dtype != torch.float32:
        raise ValueError(f"{name} must be float32")


def _check_ids(t, name):
    if t is not None and not isinstance(t, int) and t.dtype not in (torch.int32, torch.uint32):
        raise ValueError(f"{name} must be int32 or uint32")


def _nbytes(ws) -> int:
    return 0 if ws is None else ws.numel() * ws.element_size()


# ---------------------------------------------------------------------------
# entry points (C names)
# ---------------------------------------------------------------------------

def sel_workspace_bytes(op: int, rows: int, V: int, k: int = 0) -> int:
    return int(load().sel_workspace_bytes(op, rows, V, k))


def sel_workspace_init(ws, stream=None) -> None:
    _check(load().sel_workspace_init(_ptr(ws), _nbytes(ws), _stream(stream)), "sel_workspace_init")


def sel_argmax(logits, out_ids, ws=None, stream=None) -> None:
    _check_f32(logits, "logits")
    _check_ids(out_ids, "out_ids")
    rows, V = logits.shape
    _check(load().sel_argmax(_ptr(logits), rows, V, _ptr(out_ids), _ptr(ws), _nbytes(ws),
                             _stream(stream)), "sel_argmax")


def sel_argmax_excluding(logits, excluded, out_ids, ws=None, stream=None) -> None:
    """sel_argmax with the ids of `excluded` (a device id tensor, one set for
    every row) masked out of the reduction."""
    _check_f32(logits, "logits")
    _check_ids(out_ids, "out_ids")
    if excluded is not None and not isinstance(excluded, int):
        _check_ids(excluded, "excluded")
    rows, V = logits.shape
    n = 0 if excluded is None else excluded.numel()
    _check(load().sel_argmax_excluding(_ptr(logits), rows, V, _ptr(excluded) if n else None, n,
                                       _ptr(out_ids), _ptr(ws), _nbytes(ws), _stream(stream)),
           "sel_argmax_excluding")


def sel_argmax_noalloc(logits, out_ids, stream=None) -> None:
    """sel_argmax on the library's reserved scratch (no workspace argument)."""
    _check_f32(logits, "logits")
    _check_ids(out_ids, "out_ids")
    rows, V = logits.shape
    _check(load().sel_argmax_noalloc(_ptr(logits), rows, V, _ptr(out_ids), _stream(stream)),
           "sel_argmax_noalloc")


def sel_topk(logits, k: int, out_vals, out_ids, ws=None, stream=None) -> None:
    _check_f32(logits, "logits")
    _check_f32(out_vals, "out_vals")
    _check_ids(out_ids, "out_ids")
    rows, V = logits.shape
    _check(load().sel_topk(_ptr(logits), rows, V, k, _ptr(out_vals), _ptr(out_ids), _ptr(ws),
                           _nbytes(ws), _stream(stream)), "sel_topk")


def sel_sample(logits, params: SampleParams, uniforms, out_ids, out_probs, ws=None,
               stream=None) -> None:
    _check_f32(logits, "logits")
    _check_f32(uniforms, "uniforms")
    _check_f32(out_probs, "out_probs")
    _check_ids(out_ids, "out_ids")
    rows, V = logits.shape
    _check(load().sel_sample(_ptr(logits), rows, V, ctypes.byref(params), _ptr(uniforms),
                             _ptr(out_ids), _ptr(out_probs), _ptr(ws), _nbytes(ws),
                             _stream(stream)), "sel_sample")


def spec_accept(target, draft, draft_tokens, params: SpecParams, u_acc, u_fin, accepted,
                emitted, ws=None, stream=None) -> None:
    """target [S, K+1, V], draft [S, K, V] (or None), draft_tokens [S, K]."""
    _check_f32(target, "target")
    _check_f32(draft, "draft")
    _check_ids(draft_tokens, "draft_tokens")
    S, K1, V = target.shape
    _check(load().spec_accept(_ptr(target), _ptr(draft), _ptr(draft_tokens), S, K1 - 1, V,
                              ctypes.byref(params), _ptr(u_acc), _ptr(u_fin), _ptr(accepted),
                              _ptr(emitted), _ptr(ws), _nbytes(ws), _stream(stream)),
           "spec_accept")


def spec_accept_sampler(target, draft_tokens, params: SampleParams, u, accepted, emitted, ws=None,
                        stream=None) -> None:
    """target [S, K+1, V], draft_tokens [S, K], u [S, K+1]."""
    _check_f32(target, "target")
    _check_f32(u, "u")
    _check_ids(draft_tokens, "draft_tokens")
    S, K1, V = target.shape
    _check(load().spec_accept_sampler(_ptr(target), _ptr(draft_tokens), S, K1 - 1, V, ctypes.byref(params),
                                      _ptr(u), _ptr(accepted), _ptr(emitted), _ptr(ws), _nbytes(ws),
                                      _stream(stream)), "spec_accept_sampler")


def spec_diagnostics(target, draft, temperature: float, sum_min, sum_prod, ws=None, stream=None) -> None:
    """target [S, K+1, V], draft [S, K, V] -> sum_min, sum_prod [S, K]."""
    _check_f32(target, "target")
    _check_f32(draft, "draft")
    _check_f32(sum_min, "sum_min")
    _check_f32(sum_prod, "sum_prod")
    S, K1, V = target.shape
    _check(load().spec_diagnostics(_ptr(target), _ptr(draft), S, K1 - 1, V, float(temperature), _ptr(sum_min),
                                   _ptr(sum_prod), _ptr(ws), _nbytes(ws), _stream(stream)), "spec_diagnostics")


def _host_offsets(offsets):
    """Shard offsets (G + 1 ints) as a host uint32 array kept alive by the caller."""
    arr = (ctypes.c_uint32 * len(offsets))(*[int(o) for o in offsets])
    return arr


def sel_merge_shards(vals, ids, offsets, out_vals, out_ids, stream=None) -> None:
    """vals/ids [rows, G, k] (shard-local ids), offsets G + 1 host ints."""
    _check_f32(vals, "vals")
    _check_f32(out_vals, "out_vals")
    _check_ids(ids, "ids")
    _check_ids(out_ids, "out_ids")
    rows, G, k = vals.shape
    if len(offsets) != G + 1:
        raise ValueError("offsets must hold G + 1 entries")
    off = _host_offsets(offsets)
    _check(load().sel_merge_shards(_ptr(vals), _ptr(ids), rows, G, k, ctypes.cast(off, _vp),
                                   _ptr(out_vals), _ptr(out_ids), _stream(stream)), "sel_merge_shards")


def sel_sample_shards(vals, ids, offsets, params: SampleParams, uniforms, out_ids=None, out_probs=None,
                      stats=None, plan=None, stream=None) -> None:
    """vals/ids [rows, G, k] gathered lists; stats [rows, G, 48] uint8 gathered
    sel_row_stats (top-n-sigma, top_k = 0); plan [rows, 48] uint8 (top_k = 0)."""
    _check_f32(vals, "vals")
    _check_f32(uniforms, "uniforms")
    _check_f32(out_probs, "out_probs")
    _check_ids(ids, "ids")
    _check_ids(out_ids, "out_ids")
    rows, G, k = vals.shape
    if len(offsets) != G + 1:
        raise ValueError("offsets must hold G + 1 entries")
    if stats is not None and tuple(stats.shape) != (rows, G, ROW_STATS_BYTES):
        raise ValueError("stats must be [rows, G, 48] bytes")
    if plan is not None and tuple(plan.shape) != (rows, SHARD_PLAN_BYTES):
        raise ValueError("plan must be [rows, 48] bytes")
    off = _host_offsets(offsets)
    _check(load().sel_sample_shards(_ptr(vals), _ptr(ids), _ptr(stats), rows, G, k, ctypes.cast(off, _vp),
                                    ctypes.byref(params), _ptr(uniforms), _ptr(out_ids),
                                    _ptr(out_probs), _ptr(plan), _stream(stream)), "sel_sample_shards")


def sel_topk_stats(logits, k: int, params: SampleParams, out_vals, out_ids, stats, ws=None, stream=None) -> None:
    """logits [rows, V] (a shard's slice) -> top k [rows, k] and stats [rows, 48] uint8."""
    _check_f32(logits, "logits")
    _check_f32(out_vals, "out_vals")
    _check_ids(out_ids, "out_ids")
    rows, V = logits.shape
    if tuple(stats.shape) != (rows, ROW_STATS_BYTES):
        raise ValueError("stats must be [rows, 48] bytes")
    _check(load().sel_topk_stats(_ptr(logits), rows, V, k, ctypes.byref(params), _ptr(out_vals), _ptr(out_ids),
                                 _ptr(stats), _ptr(ws), _nbytes(ws), _stream(stream)), "sel_topk_stats")


def sel_shard_draw_mass(logits, offset: int, plan, mass, ws=None, stream=None) -> None:
    """logits [rows, V] (a shard's slice), plan [rows, 48] -> mass [rows] float64."""
    _check_f32(logits, "logits")
    if mass.dtype != torch.float64:
        raise ValueError("mass must be float64")
    rows, V = logits.shape
    _check(load().sel_shard_draw_mass(_ptr(logits), rows, V, int(offset), _ptr(plan), _ptr(mass), _ptr(ws),
                                      _nbytes(ws), _stream(stream)), "sel_shard_draw_mass")


def sel_shard_draw(logits, offset: int, g: int, G: int, plan, masses, out_ids, out_probs, ws=None,
                   stream=None) -> None:
    """logits [rows, V] (shard g's slice), masses [rows, G] float64 -> out_ids,
    out_probs [rows] (SEL_OTHER_SHARD / 0 where the draw is another shard's)."""
    _check_f32(logits, "logits")
    _check_f32(out_probs, "out_probs")
    _check_ids(out_ids, "out_ids")
    if masses.dtype != torch.float64:
        raise ValueError("masses must be float64")
    rows, V = logits.shape
    _check(load().sel_shard_draw(_ptr(logits), rows, V, int(offset), int(g), int(G), _ptr(plan), _ptr(masses),
                                 _ptr(out_ids), _ptr(out_probs), _ptr(ws), _nbytes(ws), _stream(stream)),
           "sel_shard_draw")


def _spec_dims(target, draft):
    S, K1, V = target.shape
    if draft is not None and tuple(draft.shape) != (S, K1 - 1, V):
        raise ValueError("draft must be [S, K, V] with target [S, K+1, V]")
    return S, K1 - 1, V


def spec_shard_stats(target, draft, draft_tokens, offset: int, params: SpecParams, parts, ws=None,
                     stream=None) -> None:
    """A shard's slices target [S, K+1, V], draft [S, K, V] (global draft
    token ids) -> parts [S, 2K+1, 32] uint8 (spec_shard_part records)."""
    _check_f32(target, "target")
    _check_f32(draft, "draft")
    _check_ids(draft_tokens, "draft_tokens")
    S, K, V = _spec_dims(target, draft)
    if tuple(parts.shape) != (S, 2 * K + 1, SPEC_SHARD_PART_BYTES):
        raise ValueError("parts must be [S, 2K+1, 32] bytes")
    _check(load().spec_shard_stats(_ptr(target), _ptr(draft), _ptr(draft_tokens), S, K, V, int(offset),
                                   ctypes.byref(params), _ptr(parts), _ptr(ws), _nbytes(ws), _stream(stream)),
           "spec_shard_stats")


def spec_accept_shards(parts, draft_tokens, offsets, params: SpecParams, u_acc, u_fin, accepted, emitted,
                       plan=None, stream=None) -> None:
    """Gathered parts [S, G, 2K+1, 32] -> accepted [S], emitted [S, K+1] and
    (rejection rule) plan [S, 32] uint8."""
    _check_ids(draft_tokens, "draft_tokens")
    _check_f32(u_acc, "u_acc")
    _check_f32(u_fin, "u_fin")
    _check_ids(accepted, "accepted")
    _check_ids(emitted, "emitted")
    S, G, R, nb = parts.shape
    if nb != SPEC_SHARD_PART_BYTES or R % 2 != 1 or len(offsets) != G + 1:
        raise ValueError("parts must be [S, G, 2K+1, 32] bytes and offsets G + 1 ints")
    K = (R - 1) // 2
    off = _host_offsets(offsets)
    _check(load().spec_accept_shards(_ptr(parts), _ptr(draft_tokens), S, K, G, ctypes.cast(off, _vp),
                                     ctypes.byref(params), _ptr(u_acc), _ptr(u_fin), _ptr(accepted), _ptr(emitted),
                                     _ptr(plan), _stream(stream)), "spec_accept_shards")


def spec_shard_draw_mass(target, draft, plan, mass, ws=None, stream=None) -> None:
    """A shard's slices and the plans -> mass [S, 2] float64 (residual, target)."""
    _check_f32(target, "target")
    _check_f32(draft, "draft")
    if mass.dtype != torch.float64:
        raise ValueError("mass must be float64")
    S, K, V = _spec_dims(target, draft)
    _check(load().spec_shard_draw_mass(_ptr(target), _ptr(draft), S, K, V, _ptr(plan), _ptr(mass), _ptr(ws),
                                       _nbytes(ws), _stream(stream)), "spec_shard_draw_mass")


def spec_shard_draw(target, draft, offset: int, g: int, G: int, plan, masses, emitted, ws=None,
                    stream=None) -> None:
    """Shard g's slices, gathered masses [S, G, 2] -> emitted[s][accepted]."""
    _check_f32(target, "target")
    _check_f32(draft, "draft")
    _check_ids(emitted, "emitted")
    if masses.dtype != torch.float64:
        raise ValueError("masses must be float64")
    S, K, V = _spec_dims(target, draft)
    _check(load().spec_shard_draw(_ptr(target), _ptr(draft), S, K, V, int(offset), int(g), int(G), _ptr(plan),
                                  _ptr(masses), _ptr(emitted), _ptr(ws), _nbytes(ws), _stream(stream)),
           "spec_shard_draw")


# ---------------------------------------------------------------------------
# allocation helpers (torch owns the memory)
# ---------------------------------------------------------------------------

def workspace(op: int, rows: int, V: int, k: int = 0, device="cuda", stream=None):
    """A zeroed workspace tensor sized for (op, rows, V, k), or None if the
    operation needs none. torch's allocator returns 512-byte aligned blocks."""
    n = sel_workspace_bytes(op, rows, V, k)
    if n == 0:
        return None
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    sel_workspace_init(ws, stream)
    return ws


def ids_to_numpy(t):
    """Device ids (int32/uint32) as a numpy uint32 array."""
    import numpy as np
    return t.detach().cpu().contiguous().view(torch.int32).numpy().view(np.uint32)
