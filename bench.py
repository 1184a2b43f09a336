#!/usr/bin/env python
"""Throughput of the joint-sequence attention path on one GB300.

One step = the whole hot path over one batch of synthetic input
(video_dit_long_gb300.step.UlyssesStep), each row a C-ABI call with CUDA
events between them:
  k6attn_rope_split_heads (rotary on q/k/joint_k into fp16 and the 8-way
  seq->head relayout of q, k, joint_k, v, joint_v, one pass) ->
  k6attn_attention_chunk_groups (attention over n K/V chunks on the head
  layout, each CTA's chunk group merged in the kernel: n/group fp32 partials
  + LSE) -> k6attn_lse_merge_heads (LSE merge written to the sequence layout).
The headline metric is attention TFLOP/s (4*B*H*S^2*d per step) over the whole
step; the attention kernel alone gives the roofline fraction against the
measured dense-bf16 peak (burst: it runs inside a step of tens of ms).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--config pro|long|lite|image] [--chunks n] [--no-secondary]

`--impl reference` times the fp64 CPU oracle on bounded row samples of the
same workload (rank 0 only).  Under torchrun (N > 1) every rank runs an
independent replica of the workload (the path does not shard across GPUs);
`value` counts the work of all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from video_dit_long_gb300 import configs, inputs  # noqa: E402
from video_dit_long_gb300 import k6attn as K  # noqa: E402  (loads the library lazily)
from video_dit_long_gb300.step import UlyssesStep  # noqa: E402

METRIC = "attention TFLOP/s & % of GB300 BF16 tensor peak at 52K/119K-token video DiT shapes"
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        out = {}
        for k in FALLBACK:
            v = d.get(k)
            if isinstance(v, dict):
                v = v.get("value")
            out[k] = float(v) if v is not None else None
        if all(out[k] for k in FALLBACK):
            out["source"] = "measured"
            return out
    return dict(FALLBACK, source="fallback")


# the sources each profiled kernel is built from: a traffic record counts only
# while these files are unchanged since the ncu capture
KERNEL_SOURCES = {
    "attn_tc_single_kernel": ("k6_attn_single.cu", "k6_attn_common.cuh", "k6_device.cuh"),
}
# the attention kernel of the step (and of every other attention line)
STEP_KERNEL = "attn_tc_single_kernel"


def strip_comments(src: str) -> str:
    """C/C++ source without its comments (string and character literals kept
    as they are), so that a comment edit leaves the digest of the code alone."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return "".join(out)


def source_digest(kernel: str, read=None) -> str:
    """sha256 (first 16 hex digits) of the kernel's sources with comments,
    blank lines and trailing blanks removed.  `read(name)` returns a file's
    text (default: the working tree)."""
    csrc = os.path.join(ROOT, "video_dit_long_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name), encoding="utf-8") as f:
                return f.read()
    digest = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        code = "\n".join(ln.rstrip() for ln in strip_comments(read(name)).splitlines() if ln.strip())
        digest.update(code.encode("utf-8"))
    return digest.hexdigest()[:16]


def traffic_record(kernel: str, workload: str):
    """DRAM bytes per launch of `kernel` on `workload` from the committed ncu
    summary, if it was taken on the kernel's current sources (their sha256 is
    recorded beside the figure); None otherwise."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path) or kernel not in KERNEL_SOURCES:
        return None
    sha = source_digest(kernel)
    with open(path) as f:
        for line in f:
            parts = dict(kv.split("=", 1) for kv in line.split() if "=" in kv)
            if (parts.get("kernel") == kernel and parts.get("workload") == workload
                    and parts.get("source_sha256") == sha):  # workload = <name>_n<chunks>
                return float(parts["dram_bytes_per_launch"])
    return None


class Clocks:
    """nvidia-smi sampler (200 ms) running while the timed region runs."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": float(np.median(sm)) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


# ------------------------------------------------------------------ our path


class Path(UlyssesStep):
    """The benchmarked step (`UlyssesStep.step`) plus the end-to-end loop from
    pinned host buffers, and the secondary rows on the same buffers: the merge
    of one partial per chunk and the constant-max variant."""

    E2E_BUFS = 3  # input and output buffer sets of the end-to-end loop (uploads run two steps ahead)

    def __init__(self, w, n_chunks, P, x):
        super().__init__(w, n_chunks, P, x)
        torch = self.torch
        bf = torch.bfloat16
        self.host = {k: torch.from_numpy(v.view(np.int16)).view(bf).pin_memory() for k, v in x.items()}
        self.e2e_in = [{k: torch.empty_like(self.seq[k]) for k in self.seq} for _ in range(self.E2E_BUFS)]
        self.e2e_out = [{"out": torch.empty_like(self.out), "lse": torch.empty_like(self.lse)}
                        for _ in range(self.E2E_BUFS)]
        self.h2d_stream = torch.cuda.Stream()
        self.d2h_stream = torch.cuda.Stream()
        self.out_host = torch.empty(self.out.shape, dtype=bf).pin_memory()
        self.lse_host = torch.empty(self.lse.shape, dtype=torch.float32).pin_memory()

    def chunk_partials(self):
        """One fp32 partial per chunk (the workload's n) on the head layout, from
        k6attn_attention_chunks, for the secondary rows."""
        torch, w, hd = self.torch, self.w, self.head
        if not hasattr(self, "pc_o"):
            f32 = torch.float32
            self.pc_o = torch.empty((self.n, self.P * w.B, w.S, self.Hl, w.d), dtype=f32, device="cuda")
            self.pc_lse = torch.empty((self.n, self.P * w.B, self.Hl, w.S), dtype=f32, device="cuda")
            self.out2 = torch.empty_like(self.out)
            self.lse2 = torch.empty_like(self.lse)
            jk, jv = (hd["jk"], hd["jv"]) if w.Nj else (None, None)
            self.h.attention_chunks(hd["q"], hd["k"], hd["v"], jk, jv, self.n, self.pc_o, self.pc_lse,
                                    qk_dtype=K.F16)
        return self.pc_o, self.pc_lse

    def standalone_rows(self, steps):
        """The unfused a1 and a4 rows alone, each one launch on the Pro buffers: rotary of q/k/joint_k into
        fp16 copies (sequence layout), the seq->head relayout of q, k, v, joint_k, joint_v (bf16) and the
        head->seq relayout of one output-sized tensor.  Returns ms per call of each."""
        torch, w, P = self.torch, self.w, self.P
        rows = {"q": w.S, "k": w.Nv, "v": w.Nv, "jk": w.Nj, "jv": w.Nj}
        rot = {n: torch.empty(self.seq[n].shape, dtype=torch.float16, device="cuda") for n in ("q", "k", "jk")}
        head = {n: torch.empty_like(self.seq[n]) for n in rows}
        j = w.Nj > 0

        def rope():
            self.hs.rope_qk(self.seq["q"], self.seq["k"], self.seq["jk"] if j else None, q_out=rot["q"],
                            k_out=rot["k"], joint_k_out=rot["jk"] if j else None, out_dtype=K.F16)

        def relayout_in():
            for n, r in rows.items():
                if r:
                    K.seq2head_relayout(self.seq[n], head[n], w.B, r, w.H, w.d, P, 0)

        def relayout_out():  # an output-sized bf16 tensor, head -> seq (into the fp16 buffer of the same size)
            K.seq2head_relayout(head["q"], rot["q"], w.B, w.S, w.H, w.d, P, 1)

        res = {"rope_qk": time_calls(rope, steps), "relayout_seq2head_qkv": time_calls(relayout_in, steps),
               "relayout_head2seq_out": time_calls(relayout_out, steps)}
        self.hs.sync()
        del rot, head
        return res

    def merge_per_chunk(self):
        """The LSE merge of one partial per chunk (n of them) into the sequence layout."""
        po, pl = self.chunk_partials()
        self.hs.lse_merge_heads(po, pl, self.n, self.P, self.out2, self.lse2)

    def const_max_step(self):
        """Constant-max variant of the attention + merge rows on the head-layout buffers
        that step() filled: row bounds, bounded attention over the chunks in the step's
        chunk groups (merged in the kernel), merge of the group partials."""
        w, hd = self.w, self.head
        if not hasattr(self, "bounds"):
            self.bounds = self.torch.empty(self.h.row_bounds_bytes() // 4, dtype=self.torch.float32, device="cuda")
            self.out2 = self.torch.empty_like(self.out)
            self.lse2 = self.torch.empty_like(self.lse)
        jk, jv = (hd["jk"], hd["jv"]) if w.Nj else (None, None)
        self.h.row_bounds(hd["q"], hd["k"], jk, self.bounds, qk_dtype=K.F16)
        self.h.attention_chunk_groups_bounded(hd["q"], hd["k"], hd["v"], jk, jv, self.bounds, self.n, self.group,
                                              self.part_o, self.part_lse, qk_dtype=K.F16)
        self.hs.lse_merge_heads(self.part_o, self.part_lse, self.parts, self.P, self.out2, self.lse2)

    def bounded_attention(self):
        """The bounded attention launch of const_max_step alone (bounds from its last call)."""
        w, hd = self.w, self.head
        jk, jv = (hd["jk"], hd["jv"]) if w.Nj else (None, None)
        self.h.attention_chunk_groups_bounded(hd["q"], hd["k"], hd["v"], jk, jv, self.bounds, self.n, self.group,
                                              self.part_o, self.part_lse, qk_dtype=K.F16)

    def e2e_run(self, steps):
        """The step through the public API from pinned host buffers, `steps` steps: per
        step the H2D copy of its inputs, the three calls of the step and the D2H copy of
        out and lse.  Uploads and downloads run on their own streams (one per direction,
        so a slow download never holds up an upload), uploads two steps ahead of the
        compute with three input and output buffer sets, as a serving loop would run it;
        every copy is inside the timed region."""
        torch = self.torch
        nb = self.E2E_BUFS
        comp = torch.cuda.current_stream()
        up, down = self.h2d_stream, self.d2h_stream
        ev_in = [torch.cuda.Event() for _ in range(nb)]      # inputs of a buffer landed
        ev_used = [torch.cuda.Event() for _ in range(nb)]    # compute done reading an input buffer
        ev_out = [torch.cuda.Event() for _ in range(nb)]     # outputs of a buffer ready
        ev_read = [torch.cuda.Event() for _ in range(nb)]    # outputs of a buffer copied out

        def h2d(step):
            buf = self.e2e_in[step % nb]
            with torch.cuda.stream(up):
                up.wait_event(ev_used[step % nb])
                for k in buf:
                    buf[k].copy_(self.host[k], non_blocking=True)
                ev_in[step % nb].record(up)

        for e in ev_used + ev_read:
            e.record(comp)
        for step in range(min(nb - 1, steps)):
            h2d(step)
        for step in range(steps):
            if step + nb - 1 < steps:
                h2d(step + nb - 1)
            b = step % nb
            buf, ob = self.e2e_in[b], self.e2e_out[b]
            comp.wait_event(ev_in[b])
            comp.wait_event(ev_read[b])  # this output buffer's previous contents have left the device
            # the prologue is the only reader of the inputs: release them after it
            self.run(buf, ob["out"], ob["lse"], ev=[None, ev_used[b], None, ev_out[b]])
            with torch.cuda.stream(down):
                down.wait_event(ev_out[b])
                self.out_host.copy_(ob["out"], non_blocking=True)
                self.lse_host.copy_(ob["lse"], non_blocking=True)
                ev_read[b].record(down)
        comp.wait_stream(up)
        comp.wait_stream(down)

    def h2d_bytes(self):
        return sum(t.numel() * t.element_size() for t in self.host.values())

    def d2h_bytes(self):
        return self.out_host.numel() * 2 + self.lse_host.numel() * 4


def gpu_index() -> str:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if vis:
        ids = [v.strip() for v in vis.split(",") if v.strip()]
        if local < len(ids):
            return ids[local]
    return str(local)


def barrier(dist_on):
    """Barrier across ranks (when distributed) and a device synchronize (when CUDA is up)."""
    import torch
    if dist_on:
        import torch.distributed as dist
        dist.barrier()
    if torch.cuda.is_available() and torch.cuda.is_initialized():
        torch.cuda.synchronize()


def max_over_ranks(x: float, dist_on) -> float:
    """The slowest rank's time: all-reduce MAX over the process group (NCCL on GPUs, gloo on CPU)."""
    if not dist_on:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank: float, world: int, seconds_max: float) -> float:
    """Units all ranks processed over the slowest rank's time (replicas: every rank does the same work)."""
    return work_per_rank * world / seconds_max


def time_calls(fn, steps, warmup=2):
    """Mean device time (ms) of `fn` over `steps` back-to-back calls on the current stream."""
    import torch
    for _ in range(warmup):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps


def measure(w, n_chunks, P, steps, warmup, dist_on, with_e2e=True, clocks=True, step_only=False):
    import torch
    x = inputs.make_inputs(w)
    path = Path(w, n_chunks, P, x)
    for _ in range(warmup):
        path.step()
    torch.cuda.synchronize()
    nev = len(path.intervals) + 1
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nev)] for _ in range(steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(dist_on)
    clk = Clocks(gpu_index())
    with (clk if clocks else _Null()):
        t0.record()
        for s in range(steps):
            path.step(evs[s])
        t1.record()
        barrier(dist_on)
    total_ms = max_over_ranks(t0.elapsed_time(t1), dist_on)
    path.sync()
    per = np.array([[evs[s][i].elapsed_time(evs[s][i + 1]) for i in range(nev - 1)] for s in range(steps)])
    res = {"total_ms": total_ms, "per_kernel_ms": dict(zip(path.intervals, per.mean(axis=0).tolist())),
           "clocks": clk.summary() if clocks else None, "launches": path.launches_per_step * steps,
           "group": path.group, "parts": path.parts}
    # the LSE merge of one partial per chunk (the workload's n), into the sequence layout
    if not step_only:
        res["merge_per_chunk_ms"] = time_calls(path.merge_per_chunk, steps)
        res["standalone_ms"] = path.standalone_rows(steps)
        path.sync()
    if with_e2e and not step_only:
        # the constant-max variant of attention + merge on the same buffers
        res["const_max_ms"] = time_calls(path.const_max_step, steps)
        res["const_max_attn_ms"] = time_calls(path.bounded_attention, steps)
        path.sync()
        path.e2e_run(max(1, warmup))
        torch.cuda.synchronize()
        barrier(dist_on)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        path.e2e_run(steps)
        e1.record()
        barrier(dist_on)
        res["e2e_ms"] = max_over_ranks(e0.elapsed_time(e1), dist_on)
        res["h2d"] = path.h2d_bytes()
        res["d2h"] = path.d2h_bytes()
        path.sync()
    del path
    torch.cuda.empty_cache()
    return res, x


class _Null:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        pass


def measure_fp8(w, n_chunks, P, x, steps, warmup):
    """The step in the FP8 mode (rotated q/k stored as e4m3, Q.K^T on 8-bit operands, P.V bf16)."""
    import torch
    st = UlyssesStep(w, n_chunks, P, x, qk="e4m3")
    for _ in range(warmup):
        st.step()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(steps)]
    for s in range(steps):
        st.step(evs[s])
    torch.cuda.synchronize()
    st.sync()
    per = np.array([[evs[s][i].elapsed_time(evs[s][i + 1]) for i in range(3)] for s in range(steps)]).mean(axis=0)
    total = float(per.sum())
    flops = w.flops()
    del st
    torch.cuda.empty_cache()
    return {"what": f"{w.name}: the step with rotated q/k in e4m3 (Q.K^T on kind::f8f6f4, P.V bf16)",
            "value": round(flops / (total * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_step": round(total, 4),
            "attention_ms": round(float(per[1]), 4),
            "attention_TFLOP/s": round(flops / (float(per[1]) * 1e-3) / 1e12, 2), "kernel": STEP_KERNEL,
            "parity": "tests/test_gpu_fp8.py (bf16 bounds on exact e4m3 inputs; relative L2 4e-2 at this workload)"}


def measure_cross(w, steps, warmup, n_chunks=8, Sq=None):
    """Audio queries (the workload's joint tokens, or the first Sq of them) over the
    full visual sequence, K/V in n chunks (k6attn_cross_forward: attention with the
    library's chunk groups, then the merge of the group partials)."""
    import torch
    B, H, d, Sk = w.B, w.H, w.d, w.Nv
    Sq = w.Nj if Sq is None else Sq

    def dev(tid, rows, std):
        return torch.from_numpy(inputs.tensor(42, tid, (B, rows, H, d), "bf16", std).view(np.int16)).view(
            torch.bfloat16).cuda()

    q, k, v = dev(30, Sq, w.qk_std), dev(31, Sk, w.qk_std), dev(32, Sk, w.v_std)
    h = K.Handle(B, H, d, "bf16", (1, 1, 1), 0, (d, 0, 0))
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    ws = torch.empty(h.cross_workspace_bytes(Sq, n_chunks), dtype=torch.uint8, device="cuda")
    for _ in range(warmup):
        h.cross_forward(q, k, v, out, lse, n_chunks=n_chunks, workspace=ws)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        h.cross_forward(q, k, v, out, lse, n_chunks=n_chunks, workspace=ws)
    e1.record()
    torch.cuda.synchronize()
    h.sync()
    ms = e0.elapsed_time(e1) / steps
    flops = 4.0 * B * H * Sq * Sk * d
    kernel = STEP_KERNEL
    return {"workload": f"{Sq} audio queries over {Sk} video keys (B={B}, H={H}, d={d}), {n_chunks} K/V chunks",
            "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms_per_call": round(ms, 4),
            "kernel": kernel, "flops_counted": "4*B*H*Sq*Sk*d on the real query rows"}


def measure_backward(w, x, steps, warmup):
    """Attention backward on the workload: rotary into fp16 copies and the one-chunk
    forward (out, lse), then `steps` timed k6attn_backward calls (D pre-pass,
    dq kernel, dk/dv kernel).  FLOPs are the 5-GEMM count 10*B*H*S^2*d.  The
    one-chunk forward (bf16 out and lse written directly, no merge) is timed
    too, over the same number of calls: returns (backward, forward_n1)."""
    import torch
    B, S, Nv, Nj, H, d = w.B, w.S, w.Nv, w.Nj, w.H, w.d
    h = K.Handle.for_workload(w)

    def dev(a):
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()

    q, k, v, jk, jv = (dev(x[n]) for n in ("q", "k", "v", "jk", "jv"))
    qh, kh, jh = (torch.empty(t.shape, dtype=torch.float16, device="cuda") for t in (q, k, jk))
    h.rope_qk(q, k, jk, q_out=qh, k_out=kh, joint_k_out=jh, out_dtype=K.F16)
    out = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")

    def forward():
        h.attention_chunks(qh, kh, v, jh, jv, 1, out, lse, qk_dtype=K.F16)

    for _ in range(warmup):
        forward()
    torch.cuda.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record()
    for _ in range(steps):
        forward()
    f1.record()
    torch.cuda.synchronize()
    h.sync()
    fwd_ms = f0.elapsed_time(f1) / steps
    fwd = {"what": f"{w.name}: attention with one K/V chunk (bf16 out and lse written directly, no merge), "
                   "rotated fp16 q/k", "value": round(4.0 * B * H * S * S * d / (fwd_ms * 1e-3) / 1e12, 2),
           "unit": "TFLOP/s", "ms_per_call": round(fwd_ms, 3), "launches_per_call": 1}
    do = dev(inputs.tensor(42, 20, (B, S, H, d), "bf16"))
    f32 = dict(dtype=torch.float32, device="cuda")
    dq = torch.empty((B, S, H, d), **f32)
    dk, dv = torch.empty((B, Nv, H, d), **f32), torch.empty((B, Nv, H, d), **f32)
    djk, djv = torch.empty((B, Nj, H, d), **f32), torch.empty((B, Nj, H, d), **f32)
    ws = torch.empty(h.backward_workspace_bytes(), dtype=torch.uint8, device="cuda")

    def call():
        h.backward(qh, kh, v, jh, jv, out, do, lse, dq, dk, dv, djk, djv, workspace=ws, qk_dtype=K.F16)

    for _ in range(warmup):
        call()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        call()
    e1.record()
    torch.cuda.synchronize()
    h.sync()
    ms = e0.elapsed_time(e1) / steps
    flops = 10.0 * B * H * S * S * d
    return ({"workload": f"{w.name}: gradients of q, k, v, joint_k, joint_v over {S} tokens (B={B}, H={H}, d={d})",
             "value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s (5-GEMM count)",
             "ms_per_call": round(ms, 3), "launches_per_call": 3}, fwd)


def merge_bytes(w, n):
    """Algorithmic bytes of the LSE merge of n partials: n fp32 partial outputs and
    LSEs read, the bf16 output and fp32 LSE written."""
    rows = w.B * w.S * w.H
    return n * (rows * w.d * 4 + rows * 4) + rows * w.d * 2 + rows * 4


def prologue_bytes(w):
    """Algorithmic bytes of the fused rotary + head split: q, k, joint_k, v, joint_v
    read (bf16) and written (fp16 / bf16) once each."""
    return 2 * (w.S + 2 * w.Nv + 2 * w.Nj) * w.H * w.d * 2


def cpu_sample(w, x, rows_count, seed=7):
    """Oracle on `rows_count` query rows (all heads, all keys); returns (seconds, flops, threads)."""
    from oracle import oracle as O
    rng = np.random.default_rng(seed)
    rows = np.sort(rng.choice(w.S, size=rows_count, replace=False))
    g = O.Geom(w.B, w.H, w.d, w.grid, w.Nj, w.axis_dim, w.theta, w.joint_rope)
    t = time.perf_counter()
    O.attention(g, x["q"], x["k"], x["v"], x["jk"], x["jv"], rows=rows)
    dt = time.perf_counter() - t
    return dt, 4.0 * w.B * w.H * rows_count * w.S * w.d, O.num_threads()


def bench_config(w, n, P):
    """The workload keys both arms report (the reference arm times the oracle on the same workload)."""
    q_mb = w.B * w.S * w.H * w.d * 2 // 2**20
    return {"workload": f"{w.name}: {w.note}", "B": w.B, "H": w.H, "d": w.d, "S": w.S, "Nv": w.Nv, "Nj": w.Nj,
            "grid": list(w.grid), "n_chunks": n, "relayout_P": P, "parallelism": "replicas",
            "l2": f"inputs larger than L2 (q, k, v are {q_mb} MB each)"}


def workload_args(args):
    w = configs.WORKLOADS[args.config]
    return w, (args.chunks or w.chunks[0]), w.relayout_P[-1]


def run_ours(args, rank, world, dist_on):
    w, n, P = workload_args(args)
    pk = peaks()
    res, x = measure(w, n, P, args.steps, args.warmup, dist_on, step_only=args.step_only)
    flops = w.flops()
    ms = res["total_ms"] / args.steps
    value = whole_job_rate(flops, world, res["total_ms"] / args.steps * 1e-3) / 1e12
    k_ms = res["per_kernel_ms"]
    attn_tflops = flops / (k_ms["attention_chunk_groups"] * 1e-3) / 1e12
    # The attention kernel is timed with CUDA events inside a step of a few tens of
    # ms and a timed region of about a second: a burst, so the burst peak is its
    # denominator; the sustained (seconds-long, power-capped) figure is kept beside it.
    peak_b, peak_s = pk["bf16_tflops"], pk["bf16_tflops_sustained"]
    tag = "of measured" if pk["source"] == "measured" else "of fallback"
    hbm = pk["hbm_gbs"]

    def gbs(b, t_ms):
        return b / (t_ms * 1e-3) / 1e9

    def hbm_rec(nbytes, t_ms):
        return {"ms": round(t_ms, 4), "bytes": nbytes, "GB/s": round(gbs(nbytes, t_ms), 1),
                "frac": round(gbs(nbytes, t_ms) / hbm, 4)}

    kernels = {
        "rope_split_heads": hbm_rec(prologue_bytes(w), k_ms["rope_split_heads"]),
        "attention_chunk_groups": {"ms": round(k_ms["attention_chunk_groups"], 4), "TFLOP/s": round(attn_tflops, 2),
                                   "frac": round(attn_tflops / peak_b, 4),
                                   "frac_sustained": round(attn_tflops / peak_s, 4),
                                   "chunks": n, "chunks_per_cta": res["group"], "partials": res["parts"]},
        "lse_merge_heads": hbm_rec(merge_bytes(w, res["parts"]), k_ms["lse_merge_heads"]),
    }
    if "merge_per_chunk_ms" in res:  # secondary: the merge of one partial per chunk (not part of the step)
        kernels["lse_merge_per_chunk"] = hbm_rec(merge_bytes(w, n), res["merge_per_chunk_ms"])
    if "standalone_ms" in res:  # secondary: the unfused a1 and a4 rows, each alone
        sa = res["standalone_ms"]
        qkj = (w.S + w.Nv + w.Nj) * w.H * w.d * 2
        kernels["standalone_rope_qk"] = hbm_rec(2 * qkj, sa["rope_qk"])
        kernels["standalone_relayout_seq2head_qkv"] = hbm_rec(prologue_bytes(w), sa["relayout_seq2head_qkv"])
        kernels["standalone_relayout_head2seq_out"] = hbm_rec(2 * w.S * w.H * w.d * 2, sa["relayout_head2seq_out"])
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "pct_of_peak": round(100 * value / world / peak_b, 2),
        "peak_basis": f"bf16 burst {peak_b} {tag} (the step is a burst of a few tens of ms)",
        "config": bench_config(w, n, P),
        "roofline": {"bound": "tensor", "achieved": round(attn_tflops, 2), "peak": peak_b, "unit": "TFLOP/s",
                     "frac": round(attn_tflops / peak_b, 4), "frac_sustained": round(attn_tflops / peak_s, 4),
                     "traffic": traffic_record(STEP_KERNEL, f"{w.name}_n{n}"), "kernel": STEP_KERNEL,
                     "peak_kind": f"bf16 burst, {tag}; frac_sustained against {peak_s}",
                     "algorithmic_flops_per_launch": flops},
        "kernels": kernels,
        "gpu_launches": res["launches"],
        "clocks": res["clocks"],
        "peaks": pk,
    }
    if "e2e_ms" in res:
        line["e2e"] = {"value": round(flops * world / (res["e2e_ms"] / args.steps * 1e-3) / 1e12, 2),
                       "unit": "TFLOP/s", "h2d_bytes_per_step": res["h2d"], "d2h_bytes_per_step": res["d2h"],
                       "ms_per_step": round(res["e2e_ms"] / args.steps, 4)}
    if args.secondary and not args.step_only:
        w2 = configs.WORKLOADS["long"]
        n2, P2 = w2.chunks[-1], w2.relayout_P[-1]
        steps2 = max(3, args.steps // 5)
        r2, _ = measure(w2, n2, P2, steps2, max(3, args.warmup), dist_on, with_e2e=False, clocks=True)
        f2 = w2.flops()
        t2 = r2["total_ms"] / steps2
        k2 = r2["per_kernel_ms"]
        a2 = f2 / (k2["attention_chunk_groups"] * 1e-3) / 1e12
        line["long_video"] = {"workload": f"{w2.name}: {w2.note}", "n_chunks": n2, "relayout_P": P2,
                              "steps": steps2, "value": round(f2 * world / (t2 * 1e-3) / 1e12, 2),
                              "unit": "TFLOP/s", "ms_per_step": round(t2, 3),
                              "pct_of_peak": round(100 * f2 / (t2 * 1e-3) / 1e12 / peak_b, 2),
                              "roofline": {"bound": "tensor", "achieved": round(a2, 2), "peak": peak_b,
                                           "unit": "TFLOP/s", "frac": round(a2 / peak_b, 4),
                                           "frac_sustained": round(a2 / peak_s, 4),
                                           "traffic": traffic_record(STEP_KERNEL, f"{w2.name}_n{n2}"),
                                           "kernel": STEP_KERNEL, "algorithmic_flops_per_launch": f2},
                              "kernels": {
                                  "rope_split_heads": hbm_rec(prologue_bytes(w2), k2["rope_split_heads"]),
                                  "attention_chunk_groups": {"ms": round(k2["attention_chunk_groups"], 3),
                                                             "chunks_per_cta": r2["group"],
                                                             "partials": r2["parts"]},
                                  "lse_merge_heads": hbm_rec(merge_bytes(w2, r2["parts"]), k2["lse_merge_heads"]),
                                  "lse_merge_per_chunk": hbm_rec(merge_bytes(w2, n2), r2["merge_per_chunk_ms"])},
                              "clocks": r2["clocks"]}
    if "const_max_ms" in res:
        line["const_max"] = {"what": "row bounds + bounded attention (no running max, no rescale) in the step's "
                                      "chunk groups + merge of the group partials",
                              "ms": round(res["const_max_ms"], 3),
                              "TFLOP/s": round(flops / (res["const_max_ms"] * 1e-3) / 1e12, 2),
                              "attention_ms": round(res["const_max_attn_ms"], 3),
                              "attention_TFLOP/s": round(flops / (res["const_max_attn_ms"] * 1e-3) / 1e12, 2),
                              "step_attention_plus_merge_ms": round(k_ms["attention_chunk_groups"] +
                                                                    k_ms["lse_merge_heads"], 3)}
    if args.secondary and not args.step_only:
        line["cross_attention"] = measure_cross(w, max(5, args.steps // 2), args.warmup)
        line["cross_attention"]["frac"] = round(line["cross_attention"]["value"] / peak_b, 4)
        # a short query range (one 128-row tile: the single-tile kernel)
        line["cross_attention_short"] = measure_cross(w, max(10, args.steps), args.warmup, Sq=100)
        line["cross_attention_short"]["frac"] = round(line["cross_attention_short"]["value"] / peak_b, 4)
        bwd, fwd1 = measure_backward(w, x, max(3, args.steps // 10), max(3, args.warmup // 2))
        for rec in (bwd, fwd1):
            rec["frac"] = round(rec["value"] / peak_b, 4)
            rec["frac_sustained"] = round(rec["value"] / peak_s, 4)
        line["attention_n1"] = fwd1
        line["backward"] = bwd
        line["fp8_logits"] = measure_fp8(w, n, P, x, max(5, args.steps // 2), args.warmup)
        line["fp8_logits"]["frac_of_bf16_peak"] = round(line["fp8_logits"]["attention_TFLOP/s"] / peak_b, 4)
    if rank == 0 and world == 1 and not args.no_cpu and not args.step_only:
        dt, fl, thr = cpu_sample(w, x, args.cpu_rows)
        line["cpu_baseline"] = {"value": round(fl / dt / 1e12, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                                "sample": f"{args.cpu_rows} query rows x {w.H} heads x all {w.S} keys of "
                                          f"{w.name}, fp64, {dt:.1f} s"}
    return line


def run_reference(args, rank, world):
    """The reference arm of this benchmark is the fp64 oracle as it stands, on the
    host cores: each step a bounded sample of query rows (all heads, all keys) of
    the same workload, enough rows per step to keep every core busy."""
    if rank != 0:
        return None
    w, n, P = workload_args(args)
    x = inputs.make_inputs(w)
    for s in range(args.warmup):
        cpu_sample(w, x, args.ref_rows, seed=50 + s)
    times, flops, thr = [], 0.0, 1
    for s in range(args.steps):
        dt, fl, thr = cpu_sample(w, x, args.ref_rows, seed=100 + s)
        times.append(dt)
        flops = fl
    total = sum(times)
    value = flops * args.steps / total / 1e12
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": bench_config(w, n, P),
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": thr, "kind": "oracle",
                             "sample": f"per step {args.ref_rows} seeded query rows x {w.H} heads x all {w.S} "
                                       f"keys of {w.name}, fp64 (rotary, scores, softmax, output)"},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_only(args):
    """One measurement alone, for profiling (the capture's kernel is the only heavy one)."""
    w, n, P = workload_args(args)
    if args.only == "step":
        res, _ = measure(w, n, P, args.steps, args.warmup, False, step_only=True)
        return {"only": "step", "workload": w.name, "n_chunks": n, "ms_per_step": res["total_ms"] / args.steps,
                "per_kernel_ms": res["per_kernel_ms"], "chunks_per_cta": res["group"], "partials": res["parts"],
                "clocks": res["clocks"]}
    if args.only == "merge_per_chunk":
        res, _ = measure(w, n, P, args.steps, args.warmup, False, clocks=False)
        return {"only": "merge_per_chunk", "workload": w.name, "n_chunks": n, "ms": res["merge_per_chunk_ms"]}
    if args.only == "fp8":
        return dict(measure_fp8(w, n, P, inputs.make_inputs(w), args.steps, args.warmup), only="fp8")
    if args.only in ("cross", "cross_short"):
        r = measure_cross(w, args.steps, args.warmup, Sq=None if args.only == "cross" else 100)
        return dict(r, only=args.only)
    if args.only == "backward":
        bwd, fwd = measure_backward(w, inputs.make_inputs(w), args.steps, args.warmup)
        return {"only": "backward", "backward": bwd, "attention_n1": fwd}
    raise ValueError(args.only)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="pro", choices=["pro", "long", "lite", "image", "mid"])
    ap.add_argument("--chunks", type=int, default=0)
    ap.add_argument("--no-secondary", dest="secondary", action="store_false")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--step-only", action="store_true",
                    help="time the step alone (no secondary rows, end-to-end loop or CPU baseline)")
    ap.add_argument("--only", choices=["step", "merge_per_chunk", "cross", "cross_short", "backward", "fp8"],
                    help="run one measurement alone and print it (for profiling captures)")
    ap.add_argument("--cpu-rows", type=int, default=1536)
    ap.add_argument("--ref-rows", type=int, default=256)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    import torch
    dist_on = world > 1
    if dist_on:
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
    line = run_only(args) if args.only else run_ours(args, rank, world, dist_on)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist_on:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
