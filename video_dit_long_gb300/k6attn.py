"""Thin ctypes binding of libk6attn (argument marshalling only).

Every function mirrors a C entry point of include/k6attn.h under the same
name without the `k6attn_` prefix.  Tensors are torch CUDA tensors; their
device pointers are passed straight through, and the current torch stream is
used unless one is given.  All compute runs in the library's CUDA kernels;
there is no fallback: if the library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE, ERR_RANGE = range(7)
BF16, F32, F16, E4M3 = 0, 1, 2, 3
OPT_WAIT_LIMIT_NS, OPT_STRICT_MMA_ORDER, OPT_ROTATE_BF16 = 0, 1, 2

# every symbol the header declares
SYMBOLS = ["k6attn_create", "k6attn_destroy", "k6attn_rope_tables", "k6attn_rope_tables_bytes",
           "k6attn_workspace_bytes", "k6attn_rope_qk", "k6attn_forward", "k6attn_attention_chunks", "k6attn_lse_merge",
           "k6attn_seq2head_relayout", "k6attn_sync", "k6attn_set_option", "k6attn_status_string",
           "k6attn_last_error", "k6attn_forward_static_scratch", "k6attn_cross_workspace_bytes",
           "k6attn_cross_forward", "k6attn_norm_rope_qk", "k6attn_row_bounds_bytes", "k6attn_row_bounds",
           "k6attn_attention_chunks_bounded", "k6attn_backward_workspace_bytes", "k6attn_backward",
           "k6attn_chunk_group", "k6attn_attention_chunk_groups", "k6attn_rope_split_heads",
           "k6attn_lse_merge_heads", "k6attn_attention_chunk_groups_bounded"]


class K6Error(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"k6attn status {status}: {msg}")
        self.status = status


class Desc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("d", ctypes.c_int), ("dtype", ctypes.c_int),
                ("grid_t", ctypes.c_int), ("grid_h", ctypes.c_int), ("grid_w", ctypes.c_int),
                ("axis_dim", ctypes.c_int * 3), ("theta", ctypes.c_double), ("n_joint", ctypes.c_int),
                ("joint_rope", ctypes.c_int)]


_lib = None


def lib_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load libk6attn.so (building it first if asked and absent)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path):
        if not build_if_missing:
            raise OSError(f"libk6attn.so not built ({path})")
        _build.build()
    L = ctypes.CDLL(path)
    P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    L.k6attn_create.argtypes = [ctypes.POINTER(Desc), ctypes.POINTER(P)]
    L.k6attn_destroy.argtypes = [P]
    L.k6attn_destroy.restype = None
    L.k6attn_rope_tables.argtypes = [P]
    L.k6attn_rope_tables.restype = P
    L.k6attn_rope_tables_bytes.argtypes = [P]
    L.k6attn_rope_tables_bytes.restype = Z
    L.k6attn_workspace_bytes.argtypes = [P, I, I]
    L.k6attn_workspace_bytes.restype = Z
    L.k6attn_rope_qk.argtypes = [P, P, P, P, P, P, P, P, I, P]
    L.k6attn_forward.argtypes = [P, P, P, P, P, P, P, I, P, P, P, Z, P]
    L.k6attn_forward_static_scratch.argtypes = [P, P, P, P, P, P, P, I, P, P, P]
    L.k6attn_row_bounds_bytes.argtypes = [P]
    L.k6attn_row_bounds_bytes.restype = Z
    L.k6attn_row_bounds.argtypes = [P, P, P, P, I, P, P]
    L.k6attn_attention_chunks_bounded.argtypes = [P, P, P, P, P, P, I, P, I, P, P, P]
    L.k6attn_norm_rope_qk.argtypes = [P, P, P, P, P, P, P, P, ctypes.c_float, P, P, P, P, I, P]
    L.k6attn_cross_workspace_bytes.argtypes = [P, ctypes.c_long, I]
    L.k6attn_cross_workspace_bytes.restype = Z
    L.k6attn_cross_forward.argtypes = [P, P, ctypes.c_long, P, P, ctypes.c_long, I, P, P, P, Z, P]
    L.k6attn_attention_chunks.argtypes = [P, P, P, P, P, P, I, I, P, P, P]
    L.k6attn_backward_workspace_bytes.argtypes = [P]
    L.k6attn_backward_workspace_bytes.restype = Z
    L.k6attn_backward.argtypes = [P, P, P, P, P, P, I, P, P, P, P, P, P, P, P, P, Z, P]
    L.k6attn_lse_merge.argtypes = [P, P, P, I, P, P, P]
    L.k6attn_chunk_group.argtypes = [P, I]
    L.k6attn_chunk_group.restype = I
    L.k6attn_attention_chunk_groups.argtypes = [P, P, P, P, P, P, I, I, I, P, P, P]
    L.k6attn_rope_split_heads.argtypes = [P, P, P, P, P, P, P, I, I, P, P, P, P, P, P]
    L.k6attn_lse_merge_heads.argtypes = [P, P, P, I, I, P, P, P]
    L.k6attn_attention_chunk_groups_bounded.argtypes = [P, P, P, P, P, P, I, P, I, I, P, P, P]
    L.k6attn_seq2head_relayout.argtypes = [P, P, I, ctypes.c_long, I, I, I, I, I, P]
    L.k6attn_sync.argtypes = [P, P]
    L.k6attn_set_option.argtypes = [P, I, ctypes.c_longlong]
    L.k6attn_status_string.argtypes = [I]
    L.k6attn_status_string.restype = ctypes.c_char_p
    L.k6attn_last_error.argtypes = []
    L.k6attn_last_error.restype = ctypes.c_char_p
    for name in ("k6attn_create", "k6attn_rope_qk", "k6attn_forward", "k6attn_forward_static_scratch",
                 "k6attn_attention_chunks", "k6attn_lse_merge", "k6attn_cross_forward", "k6attn_norm_rope_qk",
                 "k6attn_row_bounds", "k6attn_attention_chunks_bounded", "k6attn_attention_chunk_groups",
                 "k6attn_rope_split_heads", "k6attn_lse_merge_heads", "k6attn_attention_chunk_groups_bounded",
                 "k6attn_seq2head_relayout", "k6attn_sync", "k6attn_set_option"):
        getattr(L, name).restype = I
    _lib = L
    return L


def _check(status: int):
    if status != OK:
        L = load()
        raise K6Error(status, (L.k6attn_last_error() or b"").decode() or L.k6attn_status_string(status).decode())


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        import torch
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(getattr(stream, "cuda_stream", stream))


class Handle:
    """Owns a k6attn handle (rotary tables + device error word)."""

    def __init__(self, B, H, d, dtype, grid, n_joint, axis_dim, theta=10000.0, joint_rope=0):
        L = load()
        self._desc = Desc(B, H, d, BF16 if dtype in ("bf16", BF16) else F32, grid[0], grid[1], grid[2],
                          (ctypes.c_int * 3)(*axis_dim), float(theta), n_joint, joint_rope)
        h = ctypes.c_void_p()
        _check(L.k6attn_create(ctypes.byref(self._desc), ctypes.byref(h)))
        self.h = h
        self.dtype = dtype

    @classmethod
    def for_workload(cls, w, B=None):
        return cls(w.B if B is None else B, w.H, w.d, w.dtype, w.grid, w.Nj, w.axis_dim, w.theta, w.joint_rope)

    def close(self):
        if getattr(self, "h", None):
            load().k6attn_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- ABI wrappers
    def rope_tables(self) -> int:
        return load().k6attn_rope_tables(self.h) or 0

    def rope_tables_bytes(self) -> int:
        return load().k6attn_rope_tables_bytes(self.h)

    def workspace_bytes(self, n_chunks: int, with_rope: bool) -> int:
        return load().k6attn_workspace_bytes(self.h, n_chunks, int(bool(with_rope)))

    def set_option(self, opt: int, value: int):
        _check(load().k6attn_set_option(self.h, opt, int(value)))

    def rope_qk(self, q, k, joint_k, tables=None, q_out=None, k_out=None, joint_k_out=None, out_dtype=None,
                stream=None):
        """Rotate q/k/joint_k; in place unless outputs are given (out_dtype F16 for fp16 copies)."""
        tab = ctypes.c_void_p(self.rope_tables() if tables is None else tables)
        qo = q if q_out is None else q_out
        ko = k if k_out is None else k_out
        jo = joint_k if joint_k_out is None else joint_k_out
        od = self._desc.dtype if out_dtype is None else out_dtype
        _check(load().k6attn_rope_qk(self.h, _ptr(q), _ptr(k), _ptr(joint_k), tab, _ptr(qo), _ptr(ko), _ptr(jo),
                                     int(od), _stream(stream)))

    def norm_rope_qk(self, q, k, joint_k, q_weight, k_weight, eps, joint_q_weight=None, joint_k_weight=None,
                     tables=None, q_out=None, k_out=None, joint_k_out=None, out_dtype=None, stream=None):
        """QK RMSNorm over each token's H*d row, then rotary; in place unless outputs are given."""
        tab = ctypes.c_void_p(self.rope_tables() if tables is None else tables)
        qo = q if q_out is None else q_out
        ko = k if k_out is None else k_out
        jo = joint_k if joint_k_out is None else joint_k_out
        od = self._desc.dtype if out_dtype is None else out_dtype
        _check(load().k6attn_norm_rope_qk(self.h, _ptr(q), _ptr(k), _ptr(joint_k), _ptr(q_weight), _ptr(k_weight),
                                          _ptr(joint_q_weight), _ptr(joint_k_weight), float(eps), tab, _ptr(qo),
                                          _ptr(ko), _ptr(jo), int(od), _stream(stream)))

    def forward(self, q, k, v, joint_k, joint_v, out, lse=None, *, rope=True, n_chunks=1, workspace=None,
                tables=None, stream=None):
        tab = None
        if rope:
            tab = ctypes.c_void_p(self.rope_tables() if tables is None else tables)
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(load().k6attn_forward(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k), _ptr(joint_v), tab,
                                     int(n_chunks), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                     _stream(stream)))

    def forward_static_scratch(self, q, k, v, joint_k, joint_v, out, lse=None, *, rope=True, n_chunks=1,
                               tables=None, stream=None):
        """k6attn_forward with the library's static scratch array (no allocation, no workspace)."""
        tab = None
        if rope:
            tab = ctypes.c_void_p(self.rope_tables() if tables is None else tables)
        _check(load().k6attn_forward_static_scratch(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k), _ptr(joint_v),
                                                    tab, int(n_chunks), _ptr(out), _ptr(lse), _stream(stream)))

    def attention_chunks(self, q, k, v, joint_k, joint_v, n_chunks, out, lse=None, qk_dtype=None, stream=None):
        qd = self._desc.dtype if qk_dtype is None else qk_dtype
        _check(load().k6attn_attention_chunks(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k), _ptr(joint_v),
                                              int(qd), int(n_chunks), _ptr(out), _ptr(lse), _stream(stream)))

    def chunk_group(self, n_chunks: int) -> int:
        return load().k6attn_chunk_group(self.h, int(n_chunks))

    def attention_chunk_groups(self, q, k, v, joint_k, joint_v, n_chunks, group, out, lse=None, qk_dtype=None,
                               stream=None):
        """Attention over n_chunks chunks, each group of `group` merged in the kernel (n_chunks/group partials)."""
        qd = self._desc.dtype if qk_dtype is None else qk_dtype
        _check(load().k6attn_attention_chunk_groups(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k), _ptr(joint_v),
                                                    int(qd), int(n_chunks), int(group), _ptr(out), _ptr(lse),
                                                    _stream(stream)))

    def rope_split_heads(self, q, k, v, joint_k, joint_v, P, q_out, k_out, v_out, joint_k_out=None,
                         joint_v_out=None, *, qk_out_dtype=F16, tables=None, stream=None):
        """Rotary of q/k/joint_k and the P-way seq->head split of all five tensors, one launch."""
        tab = ctypes.c_void_p(self.rope_tables() if tables is None else tables)
        _check(load().k6attn_rope_split_heads(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k), _ptr(joint_v), tab,
                                              int(P), int(qk_out_dtype), _ptr(q_out), _ptr(k_out), _ptr(v_out),
                                              _ptr(joint_k_out), _ptr(joint_v_out), _stream(stream)))

    def lse_merge_heads(self, part_o, part_lse, n_parts, P, out, lse=None, stream=None):
        """Merge of head-partitioned partials, written to the sequence layout [B][S][H][d]."""
        _check(load().k6attn_lse_merge_heads(self.h, _ptr(part_o), _ptr(part_lse), int(n_parts), int(P), _ptr(out),
                                             _ptr(lse), _stream(stream)))

    def backward_workspace_bytes(self) -> int:
        return load().k6attn_backward_workspace_bytes(self.h)

    def backward(self, q, k, v, joint_k, joint_v, out, dout, lse, dq, dk, dv, djoint_k=None, djoint_v=None, *,
                 workspace, qk_dtype=None, stream=None):
        """Gradients of the joint attention (fp32 dq, dk, dv, djoint_k, djoint_v) for the rotated q, k."""
        qd = self._desc.dtype if qk_dtype is None else qk_dtype
        ws_bytes = workspace.numel() * workspace.element_size()
        _check(load().k6attn_backward(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k), _ptr(joint_v), int(qd),
                                      _ptr(out), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv),
                                      _ptr(djoint_k), _ptr(djoint_v), _ptr(workspace), ws_bytes, _stream(stream)))

    def cross_workspace_bytes(self, Sq: int, n_chunks: int) -> int:
        return load().k6attn_cross_workspace_bytes(self.h, int(Sq), int(n_chunks))

    def cross_forward(self, q, k, v, out, lse=None, *, n_chunks=1, workspace=None, stream=None):
        """Cross-attention of q [B][Sq][H][d] over k, v [B][Sk][H][d] (no rotary)."""
        ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
        _check(load().k6attn_cross_forward(self.h, _ptr(q), int(q.shape[1]), _ptr(k), _ptr(v), int(k.shape[1]),
                                           int(n_chunks), _ptr(out), _ptr(lse), _ptr(workspace), ws_bytes,
                                           _stream(stream)))

    def row_bounds_bytes(self) -> int:
        return load().k6attn_row_bounds_bytes(self.h)

    def row_bounds(self, q, k, joint_k, bounds, qk_dtype=None, stream=None):
        qd = self._desc.dtype if qk_dtype is None else qk_dtype
        _check(load().k6attn_row_bounds(self.h, _ptr(q), _ptr(k), _ptr(joint_k), int(qd), _ptr(bounds),
                                        _stream(stream)))

    def attention_chunks_bounded(self, q, k, v, joint_k, joint_v, bounds, n_chunks, out, lse=None, qk_dtype=None,
                                 stream=None):
        qd = self._desc.dtype if qk_dtype is None else qk_dtype
        _check(load().k6attn_attention_chunks_bounded(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k),
                                                      _ptr(joint_v), int(qd), _ptr(bounds), int(n_chunks), _ptr(out),
                                                      _ptr(lse), _stream(stream)))

    def attention_chunk_groups_bounded(self, q, k, v, joint_k, joint_v, bounds, n_chunks, group, out, lse=None,
                                       qk_dtype=None, stream=None):
        qd = self._desc.dtype if qk_dtype is None else qk_dtype
        _check(load().k6attn_attention_chunk_groups_bounded(self.h, _ptr(q), _ptr(k), _ptr(v), _ptr(joint_k),
                                                            _ptr(joint_v), int(qd), _ptr(bounds), int(n_chunks),
                                                            int(group), _ptr(out), _ptr(lse), _stream(stream)))

    def lse_merge(self, part_o, part_lse, n_chunks, out, lse=None, stream=None):
        _check(load().k6attn_lse_merge(self.h, _ptr(part_o), _ptr(part_lse), int(n_chunks), _ptr(out), _ptr(lse),
                                       _stream(stream)))

    def sync(self, stream=None):
        _check(load().k6attn_sync(self.h, _stream(stream)))


def seq2head_relayout(src, dst, B, S, H, d, P, direction, stream=None):
    _check(load().k6attn_seq2head_relayout(_ptr(src), _ptr(dst), B, S, H, d, src.element_size(), P, direction,
                                           _stream(stream)))
