"""Seeded synthetic inputs for the ReplaySSM hot path.

This module is shared plumbing: it draws random numbers and rounds them onto the
grid of a storage dtype. It holds none of the gated delta rule's arithmetic.
Both the fp64 oracle and the CUDA path consume the arrays it returns, so both
sides see bit-identical quantised inputs.

Distributions (the tiny GDN decode workload of the pages' standard-decode
validation, reused for every workload):

* q, k ~ N(0, 1), L2-normalised per token and key head (in fp64), then rounded;
* v ~ N(0, 1);
* beta = sigmoid(N(0, 1)), one per token and value head;
* g = -softplus(N(0, 1)): one log-decay per token and value head (GDN), or one
  per token, value head and key channel (KDA);
* S0 ~ 0.1 * N(0, 1).

Every array is float64 holding values that are exactly representable in the
requested storage dtype ("f32", "bf16" or "f16"); the caller casts them to the
device dtype without further rounding.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "quantize",
    "seed_for",
    "window_inputs",
    "initial_state",
    "null_rows",
    "accept_lengths",
    "poison_rejected",
    "force_flags",
]

_NONFINITE = (np.nan, np.inf, -np.inf)


def seed_for(config_id: int, step: int, layer: int) -> int:
    """Per-(workload, step, layer) seed: 1000*config + 17*step + layer."""
    return 1000 * int(config_id) + 17 * int(step) + int(layer)


def _round_f32_to_bf16(x32: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest, ties to even)."""
    bits = x32.view(np.uint32).astype(np.uint64)
    lsb = (bits >> 16) & 1
    rounded = (bits + 0x7FFF + lsb) & 0xFFFF0000
    out = rounded.astype(np.uint32).view(np.float32)
    # NaN payloads must stay NaN (rounding could carry into the exponent).
    return np.where(np.isnan(x32), np.float32(np.nan), out)


def quantize(x: np.ndarray, dtype: str) -> np.ndarray:
    """Return float64 values on the grid of ``dtype`` (RNE), keeping NaN/Inf."""
    x = np.asarray(x, dtype=np.float64)
    if dtype == "f64":
        return x.copy()
    with np.errstate(over="ignore", invalid="ignore"):
        x32 = x.astype(np.float32)
        if dtype == "f32":
            return x32.astype(np.float64)
        if dtype == "f16":
            return x.astype(np.float16).astype(np.float64)
        if dtype == "bf16":
            return _round_f32_to_bf16(x32).astype(np.float64)
    raise ValueError(f"unknown dtype {dtype!r}")


def _l2_normalise(x: np.ndarray) -> np.ndarray:
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _sigmoid(x: np.ndarray) -> np.ndarray:
    return 1.0 / (1.0 + np.exp(-x))


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(0.0, x)


def window_inputs(seed: int, B: int, T: int, HK: int, HV: int, dk: int, dv: int,
                  algo: str = "gdn", in_dtype: str = "f32") -> dict:
    """Draw one window of T tokens for B request rows.

    Token-major layouts (row r's token i is index r*T + i):
    q, k: [B*T, HK, dk]; v: [B*T, HV, dv]; beta: [B*T, HV];
    g: [B*T, HV] (gdn) or [B*T, HV, dk] (kda). beta and g are fp32 values.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    n = B * T
    q = _l2_normalise(rng.standard_normal((n, HK, dk)))
    k = _l2_normalise(rng.standard_normal((n, HK, dk)))
    v = rng.standard_normal((n, HV, dv))
    beta = _sigmoid(rng.standard_normal((n, HV)))
    gshape = (n, HV) if algo == "gdn" else (n, HV, dk)
    g = -_softplus(rng.standard_normal(gshape))
    return {
        "q": quantize(q, in_dtype),
        "k": quantize(k, in_dtype),
        "v": quantize(v, in_dtype),
        "beta": quantize(beta, "f32"),
        "g": quantize(g, "f32"),
    }


def initial_state(seed: int, n_slots: int, HV: int, dk: int, dv: int,
                  state_dtype: str = "f32") -> np.ndarray:
    """Checkpoint S0 ~ 0.1*N(0,1), [n_slots, HV, dk, dv]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return quantize(0.1 * rng.standard_normal((n_slots, HV, dk, dv)), state_dtype)


def null_rows(seed: int, B: int, n_null: int) -> np.ndarray:
    """Indices of the rows whose state slot is the null slot (-1)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return np.sort(rng.choice(B, size=n_null, replace=False))


def accept_lengths(seed: int, B: int, T: int) -> np.ndarray:
    """Accepted draft length per row, uniform in [0, T]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(0, T + 1, size=B).astype(np.int32)


def ragged_lengths(seed: int, B: int, max_T: int) -> np.ndarray:
    """Window length per row, uniform in [0, max_T], with at least one idle
    row (0) and one full row (max_T) when B >= 2; returns cu_seqlens [B + 1]."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = rng.integers(0, max_T + 1, size=B)
    if B >= 2:
        i, j = rng.choice(B, size=2, replace=False)
        n[i], n[j] = 0, max_T
    return np.concatenate([[0], np.cumsum(n)]).astype(np.int32)


def ragged_accept(seed: int, cu_seqlens: np.ndarray) -> np.ndarray:
    """Accepted length per row, uniform in [0, T_r] for row r's window."""
    rng = np.random.Generator(np.random.PCG64(seed))
    n = np.diff(np.asarray(cu_seqlens, dtype=np.int64))
    return np.array([rng.integers(0, t + 1) for t in n], dtype=np.int32)


def force_flags(seed: int, B: int, p: float) -> np.ndarray:
    """Per-row forced-fold flags, each set with probability p."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.random(B) < p).astype(np.uint8)


def poison_rejected(inputs: dict, accept: np.ndarray, T: int, frac: float,
                    seed: int) -> tuple[dict, np.ndarray]:
    """Overwrite rejected draft positions of some rows with NaN/+Inf/-Inf.

    Among the rows with accept[r] < T, a seeded fraction ``frac`` (at least one
    when any such row exists) gets q, k, v, beta and g set, at every position
    i >= accept[r], to one non-finite value drawn from {NaN, +Inf, -Inf}.
    Returns the poisoned copy and the indices of the poisoned rows.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    cand = np.nonzero(accept < T)[0]
    out = {key: val.copy() for key, val in inputs.items()}
    if cand.size == 0:
        return out, cand
    n = max(1, int(round(frac * cand.size)))
    rows = np.sort(rng.choice(cand, size=n, replace=False))
    for r in rows:
        val = _NONFINITE[int(rng.integers(0, 3))]
        lo, hi = r * T + int(accept[r]), (r + 1) * T
        for key in ("q", "k", "v", "beta", "g"):
            out[key][lo:hi] = val
    return out, rows
