"""Seeded synthetic inputs, shared by the tests, the benchmark and the oracle.

This module draws random numbers and rounds them to the storage type; it holds
none of the attention method's arithmetic.  Generation is counter-based per
block so that any slice can be regenerated independently and in parallel:
block `i` of tensor `t` draws from numpy's PCG64 seeded with
SeedSequence([seed, t, i]).

Tensor ids follow the order q, k, v, joint_k, joint_v (0..4); other ids are
free for auxiliary tensors (partials, relayout payloads).
"""
from __future__ import annotations

from concurrent.futures import ThreadPoolExecutor
import os

import numpy as np

BLOCK = 1 << 22  # elements per independently seeded block

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "jk": 3, "jv": 4}


def normal_f32(seed: int, tensor_id: int, n: int, std: float = 1.0, mean: float = 0.0) -> np.ndarray:
    """n samples of N(mean, std^2) as float32, deterministic in (seed, tensor_id)."""
    out = np.empty(n, np.float32)
    nblk = (n + BLOCK - 1) // BLOCK

    def fill(i):
        lo, hi = i * BLOCK, min(n, (i + 1) * BLOCK)
        rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, tensor_id, i])))
        rng.standard_normal(hi - lo, dtype=np.float32, out=out[lo:hi])
        if std != 1.0:
            out[lo:hi] *= np.float32(std)
        if mean != 0.0:
            out[lo:hi] += np.float32(mean)

    if nblk <= 1:
        for i in range(nblk):
            fill(i)
    else:
        with ThreadPoolExecutor(max_workers=min(nblk, os.cpu_count() or 4)) as ex:
            list(ex.map(fill, range(nblk)))
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16, round-to-nearest-even; returns the bit patterns (uint16)."""
    u = np.ascontiguousarray(x, np.float32).view(np.uint32)
    rounded = u + (np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1)))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    return (np.ascontiguousarray(bits, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _e4m3_value(code: int) -> float:
    """Value of a non-negative e4m3 code (1 sign, 4 exponent bits of bias 7, 3 mantissa bits;
    exponent 0 is subnormal, m * 2^-9; code 127 is NaN, there is no infinity)."""
    e, m = (code >> 3) & 0xF, code & 7
    if e == 0:
        return m * 2.0**-9
    return (1.0 + m / 8.0) * 2.0 ** (e - 7)


_E4M3_POS = np.array([_e4m3_value(c) for c in range(127)], np.float64)  # codes 0..126, ascending; 448 = max


def e4m3_bits(x: np.ndarray) -> np.ndarray:
    """Round to e4m3, nearest with ties to the even code, saturating at +-448; the bit patterns (uint8)."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), 448.0)
    i = np.clip(np.searchsorted(_E4M3_POS, a), 1, 126)
    lo, hi = _E4M3_POS[i - 1], _E4M3_POS[i]
    pick_hi = (hi - a < a - lo) | ((hi - a == a - lo) & (i % 2 == 0))
    code = np.where(pick_hi, i, i - 1).astype(np.uint8)
    return code | (np.signbit(x).astype(np.uint8) << 7)


def e4m3_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of e4m3 bit patterns (no NaN codes expected) to float32."""
    b = np.asarray(bits, np.uint8)
    v = _E4M3_POS[np.minimum(b & 0x7F, 126)].astype(np.float32)
    return np.where(b & 0x80, -v, v).astype(np.float32)


def tensor(seed: int, tensor_id: int, shape, dtype: str, std: float = 1.0) -> np.ndarray:
    """A seeded N(0, std^2) tensor stored as float32, as bf16 bits (uint16) or as e4m3 bits (uint8)."""
    n = int(np.prod(shape))
    x = normal_f32(seed, tensor_id, n, std)
    if dtype == "bf16":
        return bf16_bits(x).reshape(shape)
    if dtype == "f32":
        return x.reshape(shape)
    if dtype == "e4m3":
        return e4m3_bits(x).reshape(shape)
    raise ValueError(dtype)


def make_inputs(w, seed: int = 42, qk_scale: float = 1.0, B: int | None = None) -> dict:
    """q [B][Nv+Nj][H][d], k/v [B][Nv][H][d], jk/jv [B][Nj][H][d] for a Workload.

    qk_scale multiplies the Q and K std (the "peaked" variant uses 4).
    """
    B = w.B if B is None else B
    S, Nv, Nj, H, d = w.S, w.Nv, w.Nj, w.H, w.d
    qs = w.qk_std * qk_scale
    return {
        "q": tensor(seed, 0, (B, S, H, d), w.dtype, qs),
        "k": tensor(seed, 1, (B, Nv, H, d), w.dtype, qs),
        "v": tensor(seed, 2, (B, Nv, H, d), w.dtype, w.v_std),
        "jk": tensor(seed, 3, (B, Nj, H, d), w.dtype, qs),
        "jv": tensor(seed, 4, (B, Nj, H, d), w.dtype, w.v_std),
    }


def sample_rows(S: int, Nv: int, chunk_len: int, count: int = 1024, seed: int = 42, tile: int = 128) -> np.ndarray:
    """Query rows for sampled parity at full size: first/last video rows, up to
    64 joint rows, rows around chunk and tile boundaries, and seeded random rows."""
    rows = {0, 1, Nv - 1, Nv - 2, S - 1}
    rows.update(range(Nv, min(S, Nv + 64)))
    for b in range(0, S, chunk_len):
        rows.update(r for r in (b - 1, b, b + 1) if 0 <= r < S)
    for b in range(tile, S, tile * 37):
        rows.update(r for r in (b - 1, b) if 0 <= r < S)
    rows.update(range(S - ((S % tile) or tile), S))  # the last (possibly ragged) query tile
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 99])))
    while len(rows) < count:
        rows.add(int(rng.integers(0, S)))
    return np.array(sorted(rows), np.int64)
