"""The attention step of a Ulysses-parallel video DiT layer, on one GPU.

Each row of the hot path is one C-ABI call of libk6attn, in the order the
pages give it ("Context Parallelism in vLLM Omni Neuron", "Self-Attention
with Context Parallelism": rotary on the local tokens, then attention;
"Comparison with Other CP Strategies" and xDiT PR #586, USP dispatch listing:
an all-to-all from the sequence-partitioned to the head-partitioned layout
before attention and back after it; "Ring attention (current
implementation)": attention per K/V chunk, partials merged by their
log-sum-exp):

  1. k6attn_rope_split_heads: rotary embeddings of q, k, joint_k (into fp16)
     and the P-way seq->head relayout of q, k, joint_k, v, joint_v, one pass;
  2. k6attn_attention_chunk_groups: attention over the n K/V chunks on the
     head-partitioned layout (P*B independent problems of H/P heads); each
     CTA's group of consecutive chunks is merged in the kernel, leaving
     n / group fp32 partials and their LSE;
  3. k6attn_lse_merge_heads: the LSE merge of those partials, written straight
     back to the sequence layout [B][S][H][d] (the head->seq relayout).

This module only holds the buffers and sequences the calls (marshalling); all
arithmetic runs in the library's kernels.  The benchmark times `step()`, and
the composed-step parity test checks what it produces against the oracle.
"""
from __future__ import annotations

import numpy as np

from . import k6attn as K


class UlyssesStep:
    """Device buffers and handles for one workload; `step()` runs the path once."""

    # rows of the hot path as timed by step(ev): names of the intervals between its events
    intervals = ("rope_split_heads", "attention_chunk_groups", "lse_merge_heads")

    def __init__(self, w, n_chunks: int, P: int, x: dict, qk: str = "f16"):
        """qk: the type of the rotated q/k copies, "f16" (the default path) or "e4m3" (the FP8 mode:
        Q.K^T on 8-bit operands)."""
        import torch
        self.torch = torch
        self.w, self.n, self.P = w, n_chunks, P
        B, S, H, d, Nv, Nj = w.B, w.S, w.H, w.d, w.Nv, w.Nj
        if H % P:
            raise ValueError(f"{H} heads are not divisible by {P}")
        if n_chunks < 2 or S % n_chunks:
            raise ValueError(f"the step merges chunk partials: n_chunks must be >= 2 and divide {S}")
        self.Hl = H // P
        bf, f16, f32 = torch.bfloat16, torch.float16, torch.float32

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(bf).cuda()

        self.seq = {k: dev(v) for k, v in x.items()}
        # the full problem (B, H heads): rotary tables, prologue and epilogue
        self.hs = K.Handle(B, H, d, "bf16", w.grid, Nj, w.axis_dim, w.theta, w.joint_rope)
        # attention runs on the head-partitioned layout: P*B independent problems of H/P heads
        self.h = K.Handle(P * B, self.Hl, d, "bf16", w.grid, Nj, w.axis_dim, w.theta, w.joint_rope)
        rows = {"q": S, "k": Nv, "v": Nv, "jk": Nj, "jv": Nj}
        if qk not in ("f16", "e4m3"):
            raise ValueError(qk)
        self.qk_code = K.F16 if qk == "f16" else K.E4M3
        qk_t = f16 if qk == "f16" else torch.uint8
        self.head = {k: torch.empty((P * B, r, self.Hl, d), dtype=qk_t if k in ("q", "k", "jk") else bf,
                                    device="cuda") for k, r in rows.items()}
        # chunks per CTA: the library's choice, kept below n so that the merge has partials to combine
        g = self.h.chunk_group(n_chunks)
        while n_chunks // g < 2:
            g = max(c for c in range(1, g) if n_chunks % c == 0)
        self.group, self.parts = g, n_chunks // g
        self.part_o = torch.empty((self.parts, P * B, S, self.Hl, d), dtype=f32, device="cuda")
        self.part_lse = torch.empty((self.parts, P * B, self.Hl, S), dtype=f32, device="cuda")
        self.out = torch.empty((B, S, H, d), dtype=bf, device="cuda")
        self.lse = torch.empty((B, H, S), dtype=f32, device="cuda")
        self.launches_per_step = 3

    def run(self, seq: dict, out, lse, ev=None):
        """One pass of the path from the sequence-layout inputs `seq` into out [B][S][H][d]
        and lse [B][H][S]; `ev` (4 CUDA events, or None in place of one) brackets its rows."""
        w, hd = self.w, self.head
        j = w.Nj > 0

        def mark(i):
            if ev and ev[i] is not None:
                ev[i].record()

        mark(0)
        self.hs.rope_split_heads(seq["q"], seq["k"], seq["v"], seq["jk"] if j else None, seq["jv"] if j else None,
                                 self.P, hd["q"], hd["k"], hd["v"], hd["jk"] if j else None,
                                 hd["jv"] if j else None, qk_out_dtype=self.qk_code)
        mark(1)
        self.h.attention_chunk_groups(hd["q"], hd["k"], hd["v"], hd["jk"] if j else None, hd["jv"] if j else None,
                                      self.n, self.group, self.part_o, self.part_lse, qk_dtype=self.qk_code)
        mark(2)
        self.hs.lse_merge_heads(self.part_o, self.part_lse, self.parts, self.P, out, lse)
        mark(3)

    def step(self, ev=None):
        self.run(self.seq, self.out, self.lse, ev)

    def sync(self):
        self.hs.sync()
        self.h.sync()
