"""Shared test helpers: numpy <-> torch marshalling and the parity metrics."""
from __future__ import annotations

import numpy as np

from oracle import oracle as O

# Tolerances: bf16 inputs (fp32 accumulate) and fp32 inputs, as the workload
# definition states them, plus a relative-L2 bound on bf16 outputs that an
# all-zero output cannot meet when attention is near uniform.
BF16_MAX_ABS = 2e-2
BF16_MEAN_ABS = 2e-3
BF16_REL_L2 = 1e-2
F32_MAX_ABS = 1e-4
LSE_MAX_ABS = 1e-3


def geom(w, B=None) -> O.Geom:
    return O.Geom(w.B if B is None else B, w.H, w.d, w.grid, w.Nj, w.axis_dim, w.theta, w.joint_rope)


def to_dev(a: np.ndarray, dtype: str):
    import torch
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def to_host(t) -> np.ndarray:
    import torch
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy().astype(np.float64)
    return t.cpu().numpy().astype(np.float64)


def compare(out, ref, lse=None, ref_lse=None, dtype="bf16"):
    """Return the metrics dict and assert the bounds."""
    err = np.abs(out - ref)
    m = {"max_abs": float(err.max()), "mean_abs": float(err.mean()),
         "rel_l2": float(np.linalg.norm(out - ref) / max(np.linalg.norm(ref), 1e-300))}
    if lse is not None:
        m["lse_max_abs"] = float(np.abs(lse - ref_lse).max())
    if dtype == "bf16":
        assert m["max_abs"] <= BF16_MAX_ABS, m
        assert m["mean_abs"] <= BF16_MEAN_ABS, m
        assert m["rel_l2"] <= BF16_REL_L2, m
    else:
        assert m["max_abs"] <= F32_MAX_ABS, m
    if lse is not None:
        assert m["lse_max_abs"] <= LSE_MAX_ABS, m
    return m


_ORACLE_ROWS = {}


def oracle_sampled(w, x, rows):
    """Oracle output and LSE of the workload's inputs `x` on query `rows` (all
    heads, all keys), cached per (workload, rows): the full-size workloads cost
    seconds of CPU per call and several tests check the same sample."""
    key = (w.name, w.B, np.asarray(rows, np.int64).tobytes())
    if key not in _ORACLE_ROWS:
        _ORACLE_ROWS[key] = O.attention(geom(w), x["q"], x["k"], x["v"], x["jk"] if w.Nj else None,
                                        x["jv"] if w.Nj else None, rows=rows)
    return _ORACLE_ROWS[key]
