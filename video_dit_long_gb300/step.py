"""The attention step of a Ulysses-parallel video DiT layer, on one GPU.

Each row of the hot path is one C-ABI call of libk6attn, in the order the
pages give it ("Context Parallelism in vLLM Omni Neuron", "Self-Attention
with Context Parallelism": rotary on the local tokens, then attention;
"Comparison with Other CP Strategies" and xDiT PR #586, USP dispatch listing:
an all-to-all from the sequence-partitioned to the head-partitioned layout
before attention and back after it):

  1. rotary embeddings of q, k and joint_k on the sequence layout (full head
     rows), into fp16 copies;
  2. seq->head relayout (P-way) of the rotated q, k, joint_k and of v, joint_v;
  3. attention over n K/V chunks on the head-partitioned layout (P*B
     independent problems of H/P heads), fp32 partials and their LSE;
  4. LSE merge of the partials (head layout);
  5. head->seq relayout of the output.

This module only holds the buffers and sequences the calls (marshalling); all
arithmetic runs in the library's kernels.  The benchmark times `step()`, and
the composed-step parity test checks what it produces against the oracle.
"""
from __future__ import annotations

import numpy as np

from . import k6attn as K


class UlyssesStep:
    """Device buffers and handles for one workload; `step()` runs the path once."""

    def __init__(self, w, n_chunks: int, P: int, x: dict):
        import torch
        self.torch = torch
        self.w, self.n, self.P = w, n_chunks, P
        B, S, H, d, Nj = w.B, w.S, w.H, w.d, w.Nj
        if H % P or S % P or w.Nv % P or Nj % P:
            raise ValueError(f"{P}-way relayout needs H, S, Nv and Nj divisible by {P}")
        self.Hl = H // P
        bf, f16 = torch.bfloat16, torch.float16

        def dev(a):
            return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(bf).cuda()

        self.seq = {k: dev(v) for k, v in x.items()}
        self.rows = {"q": S, "k": w.Nv, "v": w.Nv, "jk": Nj, "jv": Nj}
        # rotary on the sequence-partitioned tensors (full head rows), into fp16 copies
        self.hs = K.Handle(B, H, d, "bf16", w.grid, Nj, w.axis_dim, w.theta, w.joint_rope)
        self.rot = {k: torch.empty(self.seq[k].shape, dtype=f16, device="cuda") for k in ("q", "k", "jk")}
        # head-partitioned copies: rotated q/k/joint_k (fp16), v/joint_v (bf16)
        self.head = {k: torch.empty_like(self.rot[k]) for k in ("q", "k", "jk")}
        self.head.update({k: torch.empty_like(self.seq[k]) for k in ("v", "jv")})
        # attention runs on the head-partitioned layout: P*B independent problems of H/P heads
        self.h = K.Handle(P * B, self.Hl, d, "bf16", w.grid, Nj, w.axis_dim, w.theta, w.joint_rope)
        self.part_o = torch.empty((n_chunks, P * B, S, self.Hl, d), dtype=torch.float32, device="cuda")
        self.part_lse = torch.empty((n_chunks, P * B, self.Hl, S), dtype=torch.float32, device="cuda")
        self.out_h = torch.empty((P * B, S, self.Hl, d), dtype=bf, device="cuda")
        self.lse = torch.empty((P * B, self.Hl, S), dtype=torch.float32, device="cuda")
        self.out = torch.empty((B, S, H, d), dtype=bf, device="cuda")
        self.launches_per_step = 1 + sum(1 for r in self.rows.values() if r) + 1 + 1 + 1
        # rows of the hot path as timed by step(ev): names of the intervals between its events
        self.intervals = ("rope_qk", "relayout_seq2head_qkv", "attention_chunks", "lse_merge",
                          "relayout_head2seq_out")

    def relayout_in(self, src: dict, dst: dict):
        w = self.w
        for name in ("q", "k", "v", "jk", "jv"):
            if self.rows[name]:
                K.seq2head_relayout(src[name], dst[name], w.B, self.rows[name], w.H, w.d, self.P, 0)

    def step(self, ev=None):
        """One pass of the path; `ev` (6 CUDA events) brackets its rows."""
        w, hd, rt = self.w, self.head, self.rot
        if ev:
            ev[0].record()
        self.hs.rope_qk(self.seq["q"], self.seq["k"], self.seq["jk"] if w.Nj else None, q_out=rt["q"],
                        k_out=rt["k"], joint_k_out=rt["jk"] if w.Nj else None, out_dtype=K.F16)
        if ev:
            ev[1].record()
        self.relayout_in({"q": rt["q"], "k": rt["k"], "jk": rt["jk"], "v": self.seq["v"], "jv": self.seq["jv"]},
                         hd)
        if ev:
            ev[2].record()
        jk, jv = (hd["jk"], hd["jv"]) if w.Nj else (None, None)
        self.h.attention_chunks(hd["q"], hd["k"], hd["v"], jk, jv, self.n, self.part_o, self.part_lse,
                                qk_dtype=K.F16)
        if ev:
            ev[3].record()
        self.h.lse_merge(self.part_o, self.part_lse, self.n, self.out_h, self.lse)
        if ev:
            ev[4].record()
        K.seq2head_relayout(self.out_h, self.out, w.B, w.S, w.H, w.d, self.P, 1)
        if ev:
            ev[5].record()

    def lse_bhs(self):
        """The step's LSE as [B][H][S] (the merge leaves it in the head layout [P][B][H/P][S])."""
        w = self.w
        return self.lse.view(self.P, w.B, self.Hl, w.S).permute(1, 0, 2, 3).reshape(w.B, w.H, w.S)

    def sync(self):
        self.hs.sync()
        self.h.sync()
