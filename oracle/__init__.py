"""CPU oracle for decode-step token selection -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package. The product path (the CUDA library and its
Python binding) never imports it, and the two share no code.

The arithmetic lives in ``sel_oracle.c`` (plain C, double precision). This
module compiles it with gcc on first use, loads it with ctypes and converts
numpy arrays. See the C file's header for the definitions and the page
passages each routine follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import tempfile
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sel_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libsel_oracle.so")

INVALID_ID = 0xFFFFFFFF

# -ffp-contract=off: no fused multiply-add, so x86 and Arm hosts round alike.
CFLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared"]


def compile_oracle(src: str = _SRC, out: str = _LIB_PATH,
                   extra_flags: tuple[str, ...] = ()) -> str:
    """Compile ``src`` into the shared library ``out`` (atomic replace)."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(out))
    os.close(fd)
    try:
        subprocess.run(["gcc", *CFLAGS, *extra_flags, "-o", tmp, src, "-lm"],
                       check=True, capture_output=True, text=True)
        os.replace(tmp, out)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return out


def build() -> str:
    """Compile the oracle if the library is missing or older than its source."""
    if (not os.path.exists(_LIB_PATH)
            or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        compile_oracle()
    return _LIB_PATH


_f32p = ctypes.POINTER(ctypes.c_float)
_u32p = ctypes.POINTER(ctypes.c_uint32)
_f64p = ctypes.POINTER(ctypes.c_double)
_u32 = ctypes.c_uint32


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    lib.orc_argmax_row.argtypes = [_f32p, _u32]
    lib.orc_argmax_row.restype = _u32
    lib.orc_argmax.argtypes = [_f32p, _u32, _u32, _u32p]
    lib.orc_argmax.restype = None
    lib.orc_argmax_excluding.argtypes = [_f32p, _u32, _u32, _u32p, _u32, _u32p]
    lib.orc_argmax_excluding.restype = None
    lib.orc_sample_ex.argtypes = [_f32p, _u32, _u32, ctypes.c_double, _u32, ctypes.c_double,
                                  ctypes.c_double, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                                  _f32p, _u32p, _f64p, _f64p]
    lib.orc_sample_ex.restype = ctypes.c_int
    lib.orc_spec_sampler.argtypes = [_f32p, _u32p, _u32, _u32, _u32, ctypes.c_double, _u32,
                                     ctypes.c_double, ctypes.c_double, ctypes.c_int, _f32p,
                                     _u32p, _u32p, _f64p]
    lib.orc_spec_sampler.restype = ctypes.c_int
    lib.orc_spec_diagnostics.argtypes = [_f32p, _f32p, _u32, _u32, _u32, ctypes.c_double,
                                         _f64p, _f64p]
    lib.orc_spec_diagnostics.restype = None
    lib.orc_topk.argtypes = [_f32p, _u32, _u32, _u32, _f32p, _u32p]
    lib.orc_topk.restype = None
    lib.orc_sample.argtypes = [_f32p, _u32, _u32, ctypes.c_double, _u32,
                               ctypes.c_double, ctypes.c_double, ctypes.c_int,
                               _f32p, _u32p, _f64p, _f64p]
    lib.orc_sample.restype = ctypes.c_int
    lib.orc_spec_accept.argtypes = [_f32p, _f32p, _u32p, _u32, _u32, _u32,
                                    ctypes.c_double, ctypes.c_int, _f32p,
                                    _f32p, _u32p, _u32p, _f64p, _f64p]
    lib.orc_spec_accept.restype = ctypes.c_int
    lib.orc_softmax_row.argtypes = [_f32p, _u32, ctypes.c_double, _f64p]
    lib.orc_softmax_row.restype = None
    return lib


def load(path: str | None = None) -> "Oracle":
    """Load the oracle library (building it first when ``path`` is None)."""
    return Oracle(_declare(ctypes.CDLL(path or build())))


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctype)


@dataclass
class SampleResult:
    ids: np.ndarray      # uint32 [rows]
    probs: np.ndarray    # float64 [rows], probability of the drawn id
    margin: np.ndarray   # float64 [rows], nearest decision's distance to its threshold


@dataclass
class SpecResult:
    accepted: np.ndarray       # uint32 [S]
    emitted: np.ndarray        # uint32 [S, K+1]
    margin_accept: np.ndarray  # float64 [S], min |u q - p| / max(p, q) over tested positions
    margin_draw: np.ndarray    # float64 [S], min |u - C_i| of the final draw


class Oracle:
    """Thin numpy wrapper over the C oracle. ctypes calls release the GIL,
    so rows can be spread over Python threads."""

    def __init__(self, lib: ctypes.CDLL):
        self.lib = lib

    def argmax(self, logits) -> np.ndarray:
        x = _f32(logits)
        rows, V = x.shape
        out = np.empty(rows, dtype=np.uint32)
        self.lib.orc_argmax(_ptr(x, _f32p), rows, V, _ptr(out, _u32p))
        return out

    def argmax_excluding(self, logits, excluded) -> np.ndarray:
        """Greedy serving variant: first maximum over the ids not in
        `excluded` (one set for every row)."""
        x = _f32(logits)
        rows, V = x.shape
        ex = np.ascontiguousarray(np.asarray(excluded, dtype=np.uint32).reshape(-1))
        out = np.empty(rows, dtype=np.uint32)
        self.lib.orc_argmax_excluding(_ptr(x, _f32p), rows, V, _ptr(ex, _u32p), ex.size,
                                      _ptr(out, _u32p))
        return out

    def spec_sampler(self, target, draft_tokens, temperature: float, top_k: int, top_p: float,
                     min_p: float, u, temp_last: bool = False) -> SpecResult:
        """Sampler-match acceptance: target [S, K+1, V], draft_tokens [S, K],
        u [S, K+1] (one uniform per verified position). margin_draw holds the
        smallest sampling margin of the draws each chain used."""
        t = _f32(target)
        S, K1, V = t.shape
        K = K1 - 1
        tok = np.ascontiguousarray(np.asarray(draft_tokens, dtype=np.uint32).reshape(S, K))
        uu = _f32(u).reshape(S, K1)
        acc = np.empty(S, dtype=np.uint32)
        emi = np.empty((S, K1), dtype=np.uint32)
        margin = np.empty(S, dtype=np.float64)
        self.lib.orc_spec_sampler(_ptr(t, _f32p), _ptr(tok, _u32p), S, K, V, float(temperature),
                                  int(top_k), float(top_p), float(min_p), int(bool(temp_last)),
                                  _ptr(uu, _f32p), _ptr(acc, _u32p), _ptr(emi, _u32p),
                                  _ptr(margin, _f64p))
        return SpecResult(acc, emi, np.full(S, np.inf), margin)

    def spec_diagnostics(self, target, draft, temperature: float):
        """(sum_min, sum_prod), each [S, K]: sum_x min(p, q) and sum_x p q per
        verified position."""
        t = _f32(target)
        d = _f32(draft)
        S, K1, V = t.shape
        K = K1 - 1
        smin = np.empty((S, K), dtype=np.float64)
        sprod = np.empty((S, K), dtype=np.float64)
        self.lib.orc_spec_diagnostics(_ptr(t, _f32p), _ptr(d, _f32p), S, K, V, float(temperature),
                                      _ptr(smin, _f64p), _ptr(sprod, _f64p))
        return smin, sprod

    def topk(self, logits, k: int) -> tuple[np.ndarray, np.ndarray]:
        x = _f32(logits)
        rows, V = x.shape
        vals = np.empty((rows, k), dtype=np.float32)
        ids = np.empty((rows, k), dtype=np.uint32)
        self.lib.orc_topk(_ptr(x, _f32p), rows, V, k, _ptr(vals, _f32p),
                          _ptr(ids, _u32p))
        return vals, ids

    def sample(self, logits, uniforms, temperature: float, top_k: int,
               top_p: float, min_p: float, temp_last: bool = False,
               top_n_sigma: float = 0.0, typical_p: float = 1.0) -> SampleResult:
        x = _f32(logits)
        rows, V = x.shape
        u = _f32(uniforms).reshape(rows)
        ids = np.empty(rows, dtype=np.uint32)
        probs = np.empty(rows, dtype=np.float64)
        margin = np.empty(rows, dtype=np.float64)
        self.lib.orc_sample_ex(_ptr(x, _f32p), rows, V, float(temperature),
                               int(top_k), float(top_p), float(min_p),
                               int(bool(temp_last)), float(top_n_sigma), float(typical_p),
                               _ptr(u, _f32p), _ptr(ids, _u32p), _ptr(probs, _f64p),
                               _ptr(margin, _f64p))
        return SampleResult(ids, probs, margin)

    def spec_accept(self, target, draft, draft_tokens, temperature: float,
                    mode: int, u_acc=None, u_fin=None) -> SpecResult:
        """target [S, K+1, V], draft [S, K, V] (None allowed for mode 1),
        draft_tokens [S, K]; mode 0 = rejection sampling, 1 = argmax rule."""
        t = _f32(target)
        S, K1, V = t.shape
        K = K1 - 1
        tok = np.ascontiguousarray(draft_tokens, dtype=np.uint32).reshape(S, K)
        d = None if draft is None else _f32(draft).reshape(S, K, V)
        if mode == 0 and d is None:
            raise ValueError("rejection mode needs draft logits")
        ua = None if u_acc is None else _f32(u_acc).reshape(S, K)
        uf = None if u_fin is None else _f32(u_fin).reshape(S)
        if mode == 0 and temperature != 0.0 and (ua is None or uf is None):
            raise ValueError("rejection mode needs u_acc and u_fin")
        acc = np.empty(S, dtype=np.uint32)
        emi = np.empty((S, K + 1), dtype=np.uint32)
        ma = np.empty(S, dtype=np.float64)
        md = np.empty(S, dtype=np.float64)
        self.lib.orc_spec_accept(
            _ptr(t, _f32p), None if d is None else _ptr(d, _f32p),
            _ptr(tok, _u32p), S, K, V, float(temperature), int(mode),
            None if ua is None else _ptr(ua, _f32p),
            None if uf is None else _ptr(uf, _f32p),
            _ptr(acc, _u32p), _ptr(emi, _u32p), _ptr(ma, _f64p),
            _ptr(md, _f64p))
        return SpecResult(acc, emi, ma, md)

    def softmax_row(self, x, temperature: float = 1.0) -> np.ndarray:
        x = _f32(x).reshape(-1)
        p = np.empty(x.size, dtype=np.float64)
        self.lib.orc_softmax_row(_ptr(x, _f32p), x.size, float(temperature),
                                 _ptr(p, _f64p))
        return p


_default: Oracle | None = None


def default() -> Oracle:
    global _default
    if _default is None:
        _default = load()
    return _default
