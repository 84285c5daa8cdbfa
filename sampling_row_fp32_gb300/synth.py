"""Seeded synthetic inputs for the selection path.

Shared by the tests, the smoke check and the benchmark. This module only
draws random numbers and arranges them into logits, uniforms and draft
tokens; it holds none of the selection arithmetic (no softmax, no filtering,
no acceptance test). Every generator uses numpy's PCG64 ``default_rng`` with
a fixed seed, so the CUDA path and the CPU oracle read identical bytes.

Shapes and distributions follow the workloads the pages describe:
  * greedy argmax over 1 x 202,048 logits with the maximum planted at three
    ids (the vocabulary of the Muser chapter, "21.3 The reduction problem");
  * top-k k=84 over 3 x 248,320 logits with a peaked head (the on-device
    top-k of the llama.cpp pull 49, "Change": 20 + 64 = 84 candidates);
  * a 49-row verify batch of Gumbel-perturbed Zipf(1.1) log-probabilities
    (the 49-token verify of the same pull request, "Problem");
  * filtered sampling over 64 x 202,048 logits;
  * speculative acceptance over 8 sequences x 8 drafts at V = 151,936.
Draft tokens are the drafter's proposals, an input to acceptance: they are
drawn from q = softmax(draft / T) with the Gumbel-max trick (argmax of the
scaled logits plus independent Gumbel noise), which samples q exactly.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

F32 = np.float32

V_MUSER = 202_048
V_QWEN = 248_320
V_SPEC = 151_936


def uniforms(seed: int, n, dtype=F32) -> np.ndarray:
    """U[0,1) draws made directly in float32 (never rounded up to 1.0)."""
    return np.random.default_rng(seed).random(n, dtype=dtype)


def normal_rows(seed: int, rows: int, V: int, sigma: float) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.normal(0.0, sigma, size=(rows, V)).astype(F32)


def planted_argmax(seed: int = 0, V: int = V_MUSER, n_plant: int = 3,
                   sigma: float = 3.0):
    """One row ~N(0, sigma^2); the value max(row) + 1 is written at
    ``n_plant`` distinct random ids. Returns (logits[1, V], planted ids)."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, sigma, size=(1, V)).astype(F32)
    ids = rng.choice(V, size=n_plant, replace=False)
    x[0, ids] = x.max() + F32(1.0)
    return x, np.sort(ids)


def peaked_rows(seed: int = 1, rows: int = 3, V: int = V_QWEN,
                sigma: float = 2.0, frac: float = 0.001,
                boost: float = 8.0) -> np.ndarray:
    """Rows ~N(0, sigma^2) with floor(frac * V) ids per row (drawn without
    replacement) raised by ``boost``."""
    rng = np.random.default_rng(seed)
    x = rng.normal(0.0, sigma, size=(rows, V)).astype(F32)
    n = int(frac * V)
    for r in range(rows):
        ids = rng.choice(V, size=n, replace=False)
        x[r, ids] += F32(boost)
    return x


def zipf_gumbel_rows(seed: int = 2, rows: int = 49, V: int = V_QWEN,
                     s: float = 1.1) -> np.ndarray:
    """Gumbel-perturbed Zipf(s) log-probabilities. A random permutation (one
    per call, shared by all rows) gives each id a rank r in 1..V; the row is
    -s ln r - ln H_{V,s} plus independent standard Gumbel noise."""
    rng = np.random.default_rng(seed)
    rank = rng.permutation(V).astype(np.float64) + 1.0
    log_h = np.log(np.sum(np.arange(1, V + 1, dtype=np.float64) ** -s))
    logp = -s * np.log(rank) - log_h
    out = np.empty((rows, V), dtype=F32)
    for r in range(rows):
        out[r] = (logp + rng.gumbel(size=V)).astype(F32)
    return out


def gumbel_max_draws(seed: int, logits: np.ndarray, temperature: float) -> np.ndarray:
    """One draw per row from softmax(logits / T): argmax(logits / T + G) with
    G i.i.d. standard Gumbel (the Gumbel-max trick), in float64."""
    rng = np.random.default_rng(seed)
    flat = np.asarray(logits, dtype=np.float64).reshape(-1, logits.shape[-1])
    out = np.empty(flat.shape[0], dtype=np.uint32)
    for i in range(flat.shape[0]):
        out[i] = np.argmax(flat[i] / temperature + rng.gumbel(size=flat.shape[1]))
    return out.reshape(logits.shape[:-1])


@dataclass
class SpecInputs:
    target: np.ndarray        # f32 [S, K+1, V]
    draft: np.ndarray         # f32 [S, K, V]
    draft_tokens: np.ndarray  # u32 [S, K]
    u_acc: np.ndarray         # f32 [S, K]
    u_fin: np.ndarray         # f32 [S]
    temperature: float = 1.0
    meta: dict = field(default_factory=dict)


def spec_inputs(S: int = 8, K: int = 8, V: int = V_SPEC, temperature: float = 1.0,
                seed_target: int = 5, seed_draft: int = 6, seed_u: int = 7,
                sigma_target: float = 2.0, sigma_noise: float = 0.5,
                target: np.ndarray | None = None) -> SpecInputs:
    """Target rows ~N(0, sigma_target^2) (or the given [S, K+1, V] array),
    draft rows = target rows 0..K-1 + N(0, sigma_noise^2), uniforms u_acc
    [S, K] then u_fin [S] from ``seed_u``, and draft tokens drawn from
    q = softmax(draft / T) by Gumbel-max with seed ``seed_u + 1000``."""
    if target is None:
        rng_t = np.random.default_rng(seed_target)
        target = rng_t.normal(0.0, sigma_target, size=(S, K + 1, V)).astype(F32)
    else:
        target = np.ascontiguousarray(target, dtype=F32).reshape(S, K + 1, V)
    rng_d = np.random.default_rng(seed_draft)
    draft = (target[:, :K, :].astype(np.float64)
             + rng_d.normal(0.0, sigma_noise, size=(S, K, V))).astype(F32)
    rng_u = np.random.default_rng(seed_u)
    u_acc = rng_u.random((S, K), dtype=F32)
    u_fin = rng_u.random(S, dtype=F32)
    tokens = gumbel_max_draws(seed_u + 1000, draft, temperature if temperature > 0 else 1.0)
    return SpecInputs(target, draft, tokens.astype(np.uint32), u_acc, u_fin, temperature)


# ---------------------------------------------------------------------------
# The five named workloads
# ---------------------------------------------------------------------------

@dataclass
class SamplePolicy:
    temperature: float = 0.7
    top_k: int = 40
    top_p: float = 0.9
    min_p: float = 0.05
    temp_last: bool = False


def workload_argmax_planted():
    """1 x 202,048 ~N(0, 9), max planted at 3 ids (seed 0)."""
    return planted_argmax(seed=0, V=V_MUSER)


def workload_topk_peaked():
    """3 x 248,320 ~N(0, 4) with 0.1 % of ids boosted by +8 (seed 1); k = 84."""
    return peaked_rows(seed=1, rows=3, V=V_QWEN), 84


def workload_verify_batch(rows: int = 49, V: int = V_QWEN):
    """49 x 248,320 Gumbel-perturbed Zipf(1.1) log-probs (seed 2); k = 20."""
    return zipf_gumbel_rows(seed=2, rows=rows, V=V), 20


def workload_sample(rows: int = 64, V: int = V_MUSER):
    """64 x 202,048 ~N(0, 9) (seed 3), uniforms from seed 4, policy
    T 0.7, top_k 40, top_p 0.9, min_p 0.05."""
    return normal_rows(3, rows, V, 3.0), uniforms(4, rows), SamplePolicy()


def workload_spec():
    """8 sequences x 8 drafts, V = 151,936, target ~N(0, 4) (seed 5), draft =
    target + N(0, 0.25) (seed 6), T = 1, uniforms seed 7."""
    return spec_inputs(S=8, K=8, V=V_SPEC, temperature=1.0)
