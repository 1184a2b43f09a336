"""GPU parity of the fused entry points of the Ulysses step.

- k6attn_rope_split_heads (rotary + seq->head relayout in one pass): bit for
  bit the unfused chain (k6attn_rope_qk into copies, then
  k6attn_seq2head_relayout of each tensor) for B = 1, and within one fp16
  rounding of the oracle's rotation, with v/joint_v bit-exact, for B = 2.
- k6attn_lse_merge_heads (merge written to the sequence layout): bit for bit
  k6attn_lse_merge on the head layout followed by the head->seq relayout
  (B = 1), and within the merge tolerance of the oracle's merge (B = 2).
- k6attn_attention_chunk_groups (each CTA's chunk group merged in the
  kernel): every group partial against the oracle's attention over the
  group's key range, and the merged result against the oracle, for group
  sizes 2, 3 and 4, with ragged tails, joint tokens shared with video keys,
  and query ranges of one tile (the single-tile kernel).
"""
import numpy as np
import pytest

from oracle import oracle as O
from video_dit_long_gb300 import configs, inputs
from video_dit_long_gb300.configs import Workload

from .helpers import compare, geom, to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def K():
    from video_dit_long_gb300 import k6attn
    return k6attn


SMALL = {
    # S = 600 + 40 = 640: chunks of 160 / 80 / 128 keys, ragged tiles, joint keys in the last chunk
    "ragged": Workload("ragged", 1, 8, 128, "bf16", (3, 10, 20), 40, (32, 48, 48), 0, 1.0, 1.0, (4,)),
    # B = 2, 1-D audio rotary, S = 256 + 32 = 288
    "audio1d": Workload("audio1d", 2, 4, 128, "bf16", (2, 8, 16), 32, (32, 48, 48), 1, 1.0, 1.0, (3,)),
    # one query tile: S = 63 + 9 = 72 (single-tile kernel)
    "short": Workload("short", 1, 4, 128, "bf16", (1, 7, 9), 9, (32, 48, 48), 0, 1.0, 1.0, (4,)),
}

NAMES = ("q", "k", "v", "jk", "jv")


def dev_inputs(w, x):
    return {n: to_dev(x[n], w.dtype) for n in NAMES}


def split_buffers(w, P, qk_dtype):
    rows = {"q": w.S, "k": w.Nv, "v": w.Nv, "jk": w.Nj, "jv": w.Nj}
    return {n: torch.empty((P * w.B, r, w.H // P, w.d), dtype=qk_dtype if n in ("q", "k", "jk") else torch.bfloat16,
                           device="cuda") for n, r in rows.items()}


@pytest.mark.parametrize("name,P", [("lite", 8), ("ragged", 4), ("ragged", 1)])
@pytest.mark.parametrize("fp16", [True, False])
def test_rope_split_heads_equals_rope_then_relayout(name, P, fp16):
    w = configs.WORKLOADS.get(name) or SMALL[name]
    k6 = K()
    x = inputs.make_inputs(w)
    d = dev_inputs(w, x)
    h = k6.Handle.for_workload(w)
    qk_t, qk_code = (torch.float16, k6.F16) if fp16 else (torch.bfloat16, k6.BF16)
    fused = split_buffers(w, P, qk_t)
    h.rope_split_heads(d["q"], d["k"], d["v"], d["jk"], d["jv"], P, fused["q"], fused["k"], fused["v"], fused["jk"],
                       fused["jv"], qk_out_dtype=qk_code)
    rot = {n: torch.empty(d[n].shape, dtype=qk_t, device="cuda") for n in ("q", "k", "jk")}
    h.rope_qk(d["q"], d["k"], d["jk"], q_out=rot["q"], k_out=rot["k"], joint_k_out=rot["jk"], out_dtype=qk_code)
    rows = {"q": w.S, "k": w.Nv, "v": w.Nv, "jk": w.Nj, "jv": w.Nj}
    src = {"q": rot["q"], "k": rot["k"], "jk": rot["jk"], "v": d["v"], "jv": d["jv"]}
    for n in NAMES:
        ref = torch.empty_like(fused[n])
        k6.seq2head_relayout(src[n], ref, w.B, rows[n], w.H, w.d, P, 0)
        torch.cuda.synchronize()
        assert torch.equal(fused[n].view(torch.int16), ref.view(torch.int16)), (name, P, n)
    h.sync()


def test_rope_split_heads_matches_oracle_with_batches():
    w = SMALL["audio1d"]
    P = 2
    k6 = K()
    x = inputs.make_inputs(w)
    d = dev_inputs(w, x)
    h = k6.Handle.for_workload(w)
    out = split_buffers(w, P, torch.float16)
    h.rope_split_heads(d["q"], d["k"], d["v"], d["jk"], d["jv"], P, out["q"], out["k"], out["v"], out["jk"],
                       out["jv"])
    h.sync()
    g = geom(w)
    Hl = w.H // P
    ref_q = O.rope(g, x["q"])
    ref_kall = O.rope(g, np.concatenate([x["k"], x["jk"]], axis=1))
    refs = {"q": ref_q, "k": ref_kall[:, :w.Nv], "jk": ref_kall[:, w.Nv:],
            "v": inputs.bf16_to_f32(x["v"]).astype(np.float64), "jv": inputs.bf16_to_f32(x["jv"]).astype(np.float64)}
    for n in NAMES:
        ref = refs[n]  # [B][R][H][d] -> head split [P][B][R][Hl][d]
        R = ref.shape[1]
        ref = ref.reshape(w.B, R, P, Hl, w.d).transpose(2, 0, 1, 3, 4).reshape(P * w.B, R, Hl, w.d)
        got = to_host(out[n])
        if n in ("v", "jv"):
            assert np.array_equal(got, ref), n
        else:
            bound = np.abs(ref) * 2.0**-10 + 2.0**-24 + 1e-6  # one fp16 rounding plus fp32 table error
            assert (np.abs(got - ref) <= bound).all(), (n, float(np.abs(got - ref).max()))


@pytest.mark.parametrize("B,S,H,P,n", [(1, 1000, 24, 8, 2), (1, 132, 8, 4, 3), (1, 64, 4, 1, 2)])
def test_lse_merge_heads_equals_merge_then_relayout(B, S, H, P, n):
    k6 = K()
    Hl, d = H // P, 128
    full = Workload("m", B, H, d, "bf16", (1, 1, S), 0, (d, 0, 0), 0, 1.0, 1.0, (n,))
    head = Workload("mh", P * B, Hl, d, "bf16", (1, 1, S), 0, (d, 0, 0), 0, 1.0, 1.0, (n,))
    hf, hh = k6.Handle.for_workload(full), k6.Handle.for_workload(head)
    po = torch.from_numpy(inputs.normal_f32(9, 20, n * P * B * S * Hl * d).reshape(n, P * B, S, Hl, d)).cuda()
    pl = torch.from_numpy(inputs.normal_f32(9, 21, n * P * B * Hl * S, std=3.0).reshape(n, P * B, Hl, S)).cuda()
    out = torch.empty((B, S, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    hf.lse_merge_heads(po, pl, n, P, out, lse)
    out_h = torch.empty((P * B, S, Hl, d), dtype=torch.bfloat16, device="cuda")
    lse_h = torch.empty((P * B, Hl, S), dtype=torch.float32, device="cuda")
    hh.lse_merge(po, pl, n, out_h, lse_h)
    ref = torch.empty_like(out)
    k6.seq2head_relayout(out_h, ref, B, S, H, d, P, 1)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_h.reshape(B, H, S).view(torch.int32))


def test_lse_merge_heads_matches_oracle_with_batches():
    k6 = K()
    B, S, H, P, n, d = 2, 96, 6, 3, 4, 128
    Hl = H // P
    full = Workload("m", B, H, d, "bf16", (1, 1, S), 0, (d, 0, 0), 0, 1.0, 1.0, (n,))
    hf = k6.Handle.for_workload(full)
    po = inputs.normal_f32(5, 20, n * P * B * S * Hl * d).reshape(n, P * B, S, Hl, d)
    pl = inputs.normal_f32(5, 21, n * P * B * Hl * S, std=3.0).reshape(n, P * B, Hl, S)
    out = torch.empty((B, S, H, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
    hf.lse_merge_heads(torch.from_numpy(po).cuda(), torch.from_numpy(pl).cuda(), n, P, out, lse)
    torch.cuda.synchronize()
    ref_h, ref_lse_h = O.lse_merge(po, pl)  # [P*B][S][Hl][d], [P*B][Hl][S]
    ref = ref_h.reshape(P, B, S, Hl, d).transpose(1, 2, 0, 3, 4).reshape(B, S, H, d)
    ref_lse = ref_lse_h.reshape(P, B, Hl, S).transpose(1, 0, 2, 3).reshape(B, H, S)
    got = to_host(out)
    assert (np.abs(got - ref) <= np.abs(ref) * 2.0**-8 + 1e-5).all(), float(np.abs(got - ref).max())
    assert np.abs(lse.cpu().numpy() - ref_lse).max() < 1e-5


def run_groups(w, x, n, group):
    """Rotary into fp16, then attention_chunk_groups: returns the rotated
    inputs' handle, the group partials (or the output) and their LSE."""
    k6 = K()
    d = dev_inputs(w, x)
    h = k6.Handle.for_workload(w)
    rot = {nm: torch.empty(d[nm].shape, dtype=torch.float16, device="cuda") for nm in ("q", "k", "jk")}
    jk = d["jk"] if w.Nj else None
    h.rope_qk(d["q"], d["k"], jk, q_out=rot["q"], k_out=rot["k"], joint_k_out=rot["jk"] if w.Nj else None,
              out_dtype=k6.F16)
    parts = n // group
    if parts > 1:
        out = torch.empty((parts, w.B, w.S, w.H, w.d), dtype=torch.float32, device="cuda")
        lse = torch.empty((parts, w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    else:
        out = torch.empty((w.B, w.S, w.H, w.d), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    h.attention_chunk_groups(rot["q"], rot["k"], d["v"], rot["jk"] if w.Nj else None, d["jv"] if w.Nj else None,
                             n, group, out, lse, qk_dtype=k6.F16)
    h.sync()
    return h, out, lse


@pytest.mark.parametrize("name,n,group", [("ragged", 4, 2), ("ragged", 4, 4), ("ragged", 8, 4), ("ragged", 5, 5),
                                          ("audio1d", 9, 3), ("audio1d", 4, 2), ("short", 4, 2), ("short", 8, 4),
                                          ("short", 3, 3)])
def test_chunk_groups_match_oracle(name, n, group):
    w = SMALL[name]
    x = inputs.make_inputs(w)
    h, out, lse = run_groups(w, x, n, group)
    g = geom(w)
    parts = n // group
    L = w.S // n
    jk, jv = (x["jk"], x["jv"]) if w.Nj else (None, None)
    if parts == 1:
        ref, ref_lse = O.attention(g, x["q"], x["k"], x["v"], jk, jv)
        compare(to_host(out), ref, lse.cpu().numpy().astype(np.float64), ref_lse, "bf16")
        return
    # each group partial is the attention over the group's key range
    for gi in range(parts):
        ref, ref_lse = O.attention(g, x["q"], x["k"], x["v"], jk, jv, kv_range=(gi * group * L, (gi + 1) * group * L))
        compare(to_host(out[gi]), ref, lse[gi].cpu().numpy().astype(np.float64), ref_lse, "bf16")
    # and the merge of the group partials is the attention over all keys
    merged = torch.empty((w.B, w.S, w.H, w.d), dtype=torch.bfloat16, device="cuda")
    mlse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    h.lse_merge(out, lse, parts, merged, mlse)
    h.sync()
    ref, ref_lse = O.attention(g, x["q"], x["k"], x["v"], jk, jv)
    compare(to_host(merged), ref, mlse.cpu().numpy().astype(np.float64), ref_lse, "bf16")


def test_per_chunk_partials_of_multi_chunk_ctas_match_oracle():
    """k6attn_attention_chunks at a size where the library gives each CTA
    several chunks (here 2) but still writes one partial per chunk: every
    CTA runs an epilogue per chunk and starts the next chunk afresh.  Sampled
    rows of three chunks' partials against the oracle's attention over that
    chunk's keys, and the merge of all eight against all keys."""
    k6 = K()
    w = Workload("groups", 1, 8, 128, "bf16", (4, 32, 32), 96, (32, 48, 48), 0, 1.0, 1.0, (8,))  # S = 4,192
    n = 8
    x = inputs.make_inputs(w)
    d = dev_inputs(w, x)
    h = k6.Handle.for_workload(w)
    assert h.chunk_group(n) >= 2  # the path under test: several chunks per CTA
    rot = {nm: torch.empty(d[nm].shape, dtype=torch.float16, device="cuda") for nm in ("q", "k", "jk")}
    h.rope_qk(d["q"], d["k"], d["jk"], q_out=rot["q"], k_out=rot["k"], joint_k_out=rot["jk"], out_dtype=k6.F16)
    po = torch.empty((n, w.B, w.S, w.H, w.d), dtype=torch.float32, device="cuda")
    pl = torch.empty((n, w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    h.attention_chunks(rot["q"], rot["k"], d["v"], rot["jk"], d["jv"], n, po, pl, qk_dtype=k6.F16)
    merged = torch.empty((w.B, w.S, w.H, w.d), dtype=torch.bfloat16, device="cuda")
    mlse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    h.lse_merge(po, pl, n, merged, mlse)
    h.sync()
    g = geom(w)
    L = w.S // n
    rows = inputs.sample_rows(w.S, w.Nv, L, count=256)
    for c in (0, 3, 7):  # chunk 7 holds the joint keys
        ref, ref_lse = O.attention(g, x["q"], x["k"], x["v"], x["jk"], x["jv"], kv_range=(c * L, (c + 1) * L),
                                   rows=rows)
        got, got_lse = to_host(po[c])[:, rows], pl[c].cpu().numpy().astype(np.float64)[:, :, rows]
        compare(got, ref, got_lse, ref_lse, "bf16")
    ref, ref_lse = O.attention(g, x["q"], x["k"], x["v"], x["jk"], x["jv"], rows=rows)
    compare(to_host(merged)[:, rows], ref, mlse.cpu().numpy().astype(np.float64)[:, :, rows], ref_lse, "bf16")


def test_chunk_groups_peaked_rescale_across_chunks():
    """Q, K x 4 with pre-rotated inputs: the running max moves (and O is rescaled)
    at chunk boundaries inside a group, not only between tiles of one chunk."""
    w = SMALL["ragged"]
    k6 = K()
    x = inputs.make_inputs(w, qk_scale=4.0)
    d = dev_inputs(w, x)
    h = k6.Handle.for_workload(w)
    out = torch.empty((2, w.B, w.S, w.H, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((2, w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    h.attention_chunk_groups(d["q"], d["k"], d["v"], d["jk"], d["jv"], 8, 4, out, lse)
    merged = torch.empty((w.B, w.S, w.H, w.d), dtype=torch.bfloat16, device="cuda")
    mlse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    h.lse_merge(out, lse, 2, merged, mlse)
    h.sync()
    ref, ref_lse = O.attention(geom(w), x["q"], x["k"], x["v"], x["jk"], x["jv"], rope=False)
    compare(to_host(merged), ref, mlse.cpu().numpy().astype(np.float64), ref_lse, "bf16")


def test_forward_uses_chunk_groups_and_matches_the_explicit_calls():
    """k6attn_forward = rotary into fp16 + attention_chunk_groups with the
    library's group + merge of the group partials (same bits)."""
    w = Workload("grp", 1, 24, 128, "bf16", (8, 16, 32), 64, (32, 48, 48), 0, 1.0, 1.0, (8,))  # 4160 tokens
    k6 = K()
    x = inputs.make_inputs(w)
    d = dev_inputs(w, x)
    h = k6.Handle.for_workload(w)
    n = 8
    grp = h.chunk_group(n)
    assert grp >= 1 and n % grp == 0
    out_f = torch.empty_like(d["q"])
    lse_f = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    ws = torch.empty(h.workspace_bytes(n, True), dtype=torch.uint8, device="cuda")
    h.forward(d["q"], d["k"], d["v"], d["jk"], d["jv"], out_f, lse_f, rope=True, n_chunks=n, workspace=ws)
    _, part, plse = run_groups(w, x, n, grp)
    out = torch.empty_like(d["q"])
    lse = torch.empty_like(lse_f)
    if n // grp > 1:
        h.lse_merge(part, plse, n // grp, out, lse)
    else:
        out, lse = part, plse
    h.sync()
    assert torch.equal(out.view(torch.int16), out_f.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), lse_f.view(torch.int32))


def test_chunk_group_argument_errors():
    w = SMALL["ragged"]
    k6 = K()
    x = inputs.make_inputs(w)
    d = dev_inputs(w, x)
    h = k6.Handle.for_workload(w)
    out = torch.empty((2, w.B, w.S, w.H, w.d), dtype=torch.float32, device="cuda")
    lse = torch.empty((2, w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    for n, grp in ((4, 3), (4, 0), (3, 1)):  # group must divide n; n must divide S = 640
        with pytest.raises(k6.K6Error) as e:
            h.attention_chunk_groups(d["q"], d["k"], d["v"], d["jk"], d["jv"], n, grp, out, lse)
        assert e.value.status == k6.ERR_INVALID_ARG
    with pytest.raises(k6.K6Error) as e:  # partial lse required
        h.attention_chunk_groups(d["q"], d["k"], d["v"], d["jk"], d["jv"], 4, 2, out, None)
    assert e.value.status == k6.ERR_INVALID_ARG


def test_fused_calls_without_joint_tokens():
    """No joint segment (Nj = 0): the prologue moves only q, k, v (null joint pointers), the chunk
    groups run on video keys alone, and the merged step result equals the oracle."""
    w = Workload("nojoint", 1, 4, 128, "bf16", (2, 10, 24), 0, (32, 48, 48), 0, 1.0, 1.0, (4,))  # S = 480
    k6 = K()
    x = inputs.make_inputs(w)
    d = dev_inputs(w, x)
    P = 2
    hf = k6.Handle.for_workload(w)
    hh = k6.Handle(P * w.B, w.H // P, w.d, "bf16", w.grid, 0, w.axis_dim)
    sp = split_buffers(w, P, torch.float16)
    hf.rope_split_heads(d["q"], d["k"], d["v"], None, None, P, sp["q"], sp["k"], sp["v"])
    po = torch.empty((2, P * w.B, w.S, w.H // P, w.d), dtype=torch.float32, device="cuda")
    pl = torch.empty((2, P * w.B, w.H // P, w.S), dtype=torch.float32, device="cuda")
    hh.attention_chunk_groups(sp["q"], sp["k"], sp["v"], None, None, 4, 2, po, pl, qk_dtype=k6.F16)
    out = torch.empty_like(d["q"])
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    hf.lse_merge_heads(po, pl, 2, P, out, lse)
    hf.sync()
    hh.sync()
    ref, ref_lse = O.attention(geom(w), x["q"], x["k"], x["v"])
    compare(to_host(out), ref, lse.cpu().numpy().astype(np.float64), ref_lse, "bf16")
