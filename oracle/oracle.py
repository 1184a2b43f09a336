"""ctypes wrapper of the fp64 CPU oracle (k6_oracle.c).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.  It shares no code
with the CUDA library; both sides only read inputs made by the seeded
generators.

Every function returns float64 numpy arrays.  Inputs are numpy arrays of
float64, float32, or bf16 bit patterns stored as uint16 (widened exactly).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "k6_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libk6oracle.so")

F32, BF16, F64 = 0, 1, 2


def build(force: bool = False, mutant: int = 0) -> str:
    """Compile the oracle with gcc (-O2, OpenMP, no fast-math).

    mutant > 0 builds a copy with one planted mistake (see K6O_MUTANT in the
    source), used only by the test that checks the pins catch it."""
    os.makedirs(_BUILD, exist_ok=True)
    path = _LIB_PATH if mutant == 0 else os.path.join(_BUILD, f"libk6oracle_mutant{mutant}.so")
    if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
        tmp = path + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", f"-DK6O_MUTANT={int(mutant)}",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, path)
    return path


class _Geom(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("d", ctypes.c_int),
                ("Nv", ctypes.c_long), ("Nj", ctypes.c_long),
                ("grid_t", ctypes.c_int), ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int),
                ("axis_dim", ctypes.c_int * 3), ("theta", ctypes.c_double),
                ("joint_rope", ctypes.c_int)]


@dataclass(frozen=True)
class Geom:
    """Problem geometry: batch, heads, head dim, video grid, joint tokens, RoPE."""
    B: int
    H: int
    d: int
    grid: tuple  # (t, h, w)
    Nj: int
    axis_dim: tuple = None  # dims of the t, h, w axes
    theta: float = 10000.0
    joint_rope: int = 0

    @property
    def Nv(self) -> int:
        return self.grid[0] * self.grid[1] * self.grid[2]

    @property
    def S(self) -> int:
        return self.Nv + self.Nj

    def c(self) -> _Geom:
        ad = self.axis_dim if self.axis_dim is not None else (self.d, 0, 0)
        return _Geom(self.B, self.H, self.d, self.Nv, self.Nj, self.grid[0], self.grid[1], self.grid[2],
                     (ctypes.c_int * 3)(*ad), float(self.theta), int(self.joint_rope))


_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


def use_mutant(mutant: int):
    """Point this module at a planted-mistake build (0 restores the oracle)."""
    global _lib
    _lib = _declare(ctypes.CDLL(build(mutant=mutant)))


def _declare(L):
    """Declare the argument and result types of every oracle entry point."""
    P = ctypes.c_void_p
    L.k6o_rope.argtypes = [ctypes.POINTER(_Geom), P, ctypes.c_int, P]
    L.k6o_rope_vec.argtypes = [ctypes.POINTER(_Geom), ctypes.c_long, P]
    L.k6o_rope_vec.restype = None
    L.k6o_attention.argtypes = [ctypes.POINTER(_Geom), ctypes.c_int, P, P, P, P, P, ctypes.c_int,
                                   ctypes.c_long, ctypes.c_long, P, ctypes.c_long, P, P]
    L.k6o_cross_attention.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_long,
                                         ctypes.c_long, P, P, P, ctypes.c_int, ctypes.c_long, ctypes.c_long, P, P]
    L.k6o_attention_backward.argtypes = [ctypes.POINTER(_Geom), ctypes.c_int, P, P, P, P, P, ctypes.c_int, P,
                                         P, P, P, P, P]
    L.k6o_row_bounds.argtypes = [ctypes.POINTER(_Geom), ctypes.c_int, P, P, P, ctypes.c_int, P]
    L.k6o_rms_norm.argtypes = [P, ctypes.c_int, ctypes.c_long, ctypes.c_long, P, ctypes.c_double, P]
    L.k6o_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                   P, P, ctypes.c_int, P, P]
    L.k6o_relayout.argtypes = [P, P, ctypes.c_int, ctypes.c_long, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.k6o_latent_grid.argtypes = [ctypes.c_int] * 3 + [ctypes.POINTER(ctypes.c_int)] * 3
    L.k6o_latent_grid.restype = None
    L.k6o_num_threads.restype = ctypes.c_int
    L.k6o_set_num_threads.argtypes = [ctypes.c_int]
    L.k6o_set_num_threads.restype = None
    return L


def num_threads() -> int:
    return lib().k6o_num_threads()


def set_num_threads(n: int) -> None:
    lib().k6o_set_num_threads(int(n))


def _typed(a: np.ndarray):
    a = np.ascontiguousarray(a)
    if a.dtype == np.float64:
        return a, F64
    if a.dtype == np.float32:
        return a, F32
    if a.dtype == np.uint16:
        return a, BF16
    raise TypeError(f"oracle input dtype {a.dtype} (want float64, float32 or bf16 bits as uint16)")


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def rope(g: Geom, x: np.ndarray) -> np.ndarray:
    """Rotary embedding of a [B][S][H][d] tensor (Q or K of the joint sequence)."""
    x, t = _typed(x)
    assert x.size == g.B * g.S * g.H * g.d
    y = np.empty((g.B, g.S, g.H, g.d), np.float64)
    rc = lib().k6o_rope(ctypes.byref(g.c()), _ptr(x), t, _ptr(y))
    if rc:
        raise ValueError(f"k6o_rope: {rc}")
    return y


def row_bounds(g: Geom, q, k, jk=None, *, rope: bool = True) -> np.ndarray:
    """Constant-max row bounds [B][H][S]: |q~_i| * max_j |k~_j| / sqrt(d) over all keys."""
    (q_, t), (k_, t2) = _typed(q), _typed(k)
    jk_ = _typed(jk)[0] if g.Nj > 0 else None
    out = np.empty((g.B, g.H, g.S), np.float64)
    rc = lib().k6o_row_bounds(ctypes.byref(g.c()), int(bool(rope)), _ptr(q_), _ptr(k_),
                              _ptr(jk_) if jk_ is not None else ctypes.c_void_p(0), t, _ptr(out))
    if rc:
        raise ValueError(f"k6o_row_bounds: {rc}")
    return out


def rms_norm(x: np.ndarray, w: np.ndarray, eps: float) -> np.ndarray:
    """RMSNorm over the last dim of x (a token's H*d hidden row for QK-norm)."""
    x_, t = _typed(x)
    n = x_.shape[-1]
    w_ = np.ascontiguousarray(w, np.float64)
    assert w_.shape == (n,)
    y = np.empty(x_.shape, np.float64)
    rc = lib().k6o_rms_norm(_ptr(x_), t, x_.size // n, n, _ptr(w_), float(eps), _ptr(y))
    if rc:
        raise ValueError(f"k6o_rms_norm: {rc}")
    return y


def rope_vec(g: Geom, n: int, x: np.ndarray) -> np.ndarray:
    """Rotary embedding of one head vector of token n."""
    y = np.array(x, np.float64, copy=True)
    lib().k6o_rope_vec(ctypes.byref(g.c()), int(n), _ptr(y))
    return y


def attention(g: Geom, q, k, v, jk=None, jv=None, *, rope: bool = True, kv_range=None, rows=None):
    """Attention of query rows over a K/V range of concat(k, joint_k).

    Returns (out [B][nrows][H][d], lse [B][H][nrows]), float64.
    """
    arrs = [q, k, v]
    if g.Nj > 0:
        arrs += [jk, jv]
    typed = [_typed(a) for a in arrs]
    types = {t for _, t in typed}
    if len(types) != 1:
        raise TypeError("q, k, v, joint_k, joint_v must share one dtype")
    t = types.pop()
    q_, k_, v_ = typed[0][0], typed[1][0], typed[2][0]
    jk_ = typed[3][0] if g.Nj > 0 else None
    jv_ = typed[4][0] if g.Nj > 0 else None
    kb, ke = (0, g.S) if kv_range is None else kv_range
    if rows is None:
        rows = np.arange(g.S, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = len(rows)
    out = np.empty((g.B, n, g.H, g.d), np.float64)
    lse = np.empty((g.B, g.H, n), np.float64)
    nullp = ctypes.c_void_p(0)
    rc = lib().k6o_attention(ctypes.byref(g.c()), int(bool(rope)), _ptr(q_), _ptr(k_), _ptr(v_),
                             _ptr(jk_) if jk_ is not None else nullp, _ptr(jv_) if jv_ is not None else nullp,
                             t, int(kb), int(ke), _ptr(rows), n, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"k6o_attention: {rc}")
    return out, lse


def attention_backward(g: Geom, q, k, v, jk, jv, dout, *, rope: bool = True):
    """Gradients (dq, dk, dv, djk, djv) of sum(out * dout) over the full joint sequence,
    with respect to the rotated q, k (rope=True) or the given ones (rope=False)."""
    arrs = [q, k, v] + ([jk, jv] if g.Nj > 0 else [])
    typed = [_typed(a) for a in arrs]
    t = typed[0][1]
    assert all(tt == t for _, tt in typed)
    do = np.ascontiguousarray(dout, np.float64)
    dq = np.empty((g.B, g.S, g.H, g.d))
    dk = np.empty((g.B, g.Nv, g.H, g.d))
    dv = np.empty((g.B, g.Nv, g.H, g.d))
    djk = np.empty((g.B, max(g.Nj, 0), g.H, g.d))
    djv = np.empty((g.B, max(g.Nj, 0), g.H, g.d))
    nullp = ctypes.c_void_p(0)
    j0 = _ptr(typed[3][0]) if g.Nj > 0 else nullp
    j1 = _ptr(typed[4][0]) if g.Nj > 0 else nullp
    rc = lib().k6o_attention_backward(ctypes.byref(g.c()), int(bool(rope)), _ptr(typed[0][0]), _ptr(typed[1][0]),
                                      _ptr(typed[2][0]), j0, j1, t, _ptr(do), _ptr(dq), _ptr(dk), _ptr(dv),
                                      _ptr(djk), _ptr(djv))
    if rc:
        raise ValueError(f"k6o_attention_backward: {rc}")
    return dq, dk, dv, djk, djv


def cross_attention(q, k, v, *, kv_range=None):
    """Cross-attention (no rotary) of q [B][Sq][H][d] over k, v [B][Sk][H][d].

    Returns (out [B][Sq][H][d], lse [B][H][Sq]), float64.
    """
    (q_, t1), (k_, t2), (v_, t3) = _typed(q), _typed(k), _typed(v)
    if len({t1, t2, t3}) != 1:
        raise TypeError("q, k, v must share one dtype")
    B, Sq, H, d = q_.shape
    Sk = k_.shape[1]
    assert k_.shape == (B, Sk, H, d) and v_.shape == (B, Sk, H, d)
    kb, ke = (0, Sk) if kv_range is None else kv_range
    out = np.empty((B, Sq, H, d), np.float64)
    lse = np.empty((B, H, Sq), np.float64)
    rc = lib().k6o_cross_attention(B, H, d, Sq, Sk, _ptr(q_), _ptr(k_), _ptr(v_), t1, int(kb), int(ke), _ptr(out),
                                   _ptr(lse))
    if rc:
        raise ValueError(f"k6o_cross_attention: {rc}")
    return out, lse


def chunk_bounds(S: int, n: int):
    """Equal contiguous K/V chunks [c*S/n, (c+1)*S/n), as ring ranks hold them."""
    if S % n:
        raise ValueError(f"{n} equal chunks cannot cover {S} keys")
    L = S // n
    return [(c * L, (c + 1) * L) for c in range(n)]


def lse_merge(part_o: np.ndarray, part_lse: np.ndarray):
    """Merge per-chunk partials. part_o [n][B][Sq][H][d], part_lse [n][B][H][Sq]."""
    po, t1 = _typed(part_o)
    pl, t2 = _typed(part_lse)
    if t1 != t2:
        raise TypeError("part_o and part_lse must share one dtype")
    n, B, Sq, H, d = po.shape
    assert pl.shape == (n, B, H, Sq)
    out = np.empty((B, Sq, H, d), np.float64)
    lse = np.empty((B, H, Sq), np.float64)
    rc = lib().k6o_lse_merge(n, B, Sq, H, d, _ptr(po), _ptr(pl), t1, _ptr(out), _ptr(lse))
    if rc:
        raise ValueError(f"k6o_lse_merge: {rc}")
    return out, lse


def relayout(src: np.ndarray, B: int, S: int, H: int, d: int, P: int, direction: int) -> np.ndarray:
    """seq [P][B][S/P][H][d] <-> head [P][B][S][H/P][d]; byte copy of any element type."""
    src = np.ascontiguousarray(src)
    dst = np.empty_like(src)
    rc = lib().k6o_relayout(_ptr(src), _ptr(dst), B, S, H, d, src.itemsize, P, direction)
    if rc:
        raise ValueError(f"k6o_relayout: {rc}")
    return dst


def latent_grid(height: int, width: int, frames: int):
    t, h, w = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    lib().k6o_latent_grid(height, width, frames, ctypes.byref(t), ctypes.byref(h), ctypes.byref(w))
    return t.value, h.value, w.value
