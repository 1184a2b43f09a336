"""GPU parity of the constant-max softmax (row bounds in place of the running
max) against the oracle: the bounds themselves, the attention result, and the
underflow guard when the Cauchy-Schwarz bound is far above every logit."""
import numpy as np
import pytest

from oracle import oracle as O
from video_dit_long_gb300 import configs, inputs
from video_dit_long_gb300.configs import Workload

from .helpers import compare, geom, to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CASES = {
    "ragged": Workload("ragged", 1, 2, 128, "bf16", (3, 10, 20), 40, (32, 48, 48), 0, 1.0, 1.0, (1, 4)),
    "audio1d": Workload("audio1d", 2, 2, 128, "bf16", (2, 8, 16), 62, (32, 48, 48), 1, 1.0, 1.0, (1, 3)),
    "lite": configs.WORKLOADS["lite"],
    # 63 tokens: a query range of one tile (the single-tile kernel), chunks of 21 keys
    "one_tile": Workload("one_tile", 1, 3, 128, "bf16", (1, 7, 9), 0, (32, 48, 48), 0, 1.0, 1.0, (1, 3)),
}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_bounded(w, x, n, rope=True, group=0):
    from video_dit_long_gb300 import k6attn as K
    h = K.Handle.for_workload(w)
    q, k, v, jk, jv = (to_dev(x[nm], w.dtype) for nm in ("q", "k", "v", "jk", "jv"))
    if w.Nj == 0:
        jk = jv = None
    if rope:
        qo, ko = (torch.empty(t.shape, dtype=torch.float16, device="cuda") for t in (q, k))
        jo = torch.empty(jk.shape, dtype=torch.float16, device="cuda") if jk is not None else None
        h.rope_qk(q, k, jk, q_out=qo, k_out=ko, joint_k_out=jo, out_dtype=K.F16)
        qd = K.F16
    else:
        qo, ko, jo, qd = q, k, jk, K.BF16
    bounds = torch.empty(h.row_bounds_bytes() // 4, dtype=torch.float32, device="cuda")
    h.row_bounds(qo, ko, jo, bounds, qk_dtype=qd)
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    if group:  # each CTA's group of chunks merged in the kernel
        parts = n // group
        if parts == 1:
            h.attention_chunk_groups_bounded(qo, ko, v, jo, jv, bounds, n, group, out, lse, qk_dtype=qd)
        else:
            po = torch.empty((parts, w.B, w.S, w.H, w.d), dtype=torch.float32, device="cuda")
            pl = torch.empty((parts, w.B, w.H, w.S), dtype=torch.float32, device="cuda")
            h.attention_chunk_groups_bounded(qo, ko, v, jo, jv, bounds, n, group, po, pl, qk_dtype=qd)
            h.lse_merge(po, pl, parts, out, lse)
    elif n == 1:
        h.attention_chunks_bounded(qo, ko, v, jo, jv, bounds, 1, out, lse, qk_dtype=qd)
    else:
        po = torch.empty((n, w.B, w.S, w.H, w.d), dtype=torch.float32, device="cuda")
        pl = torch.empty((n, w.B, w.H, w.S), dtype=torch.float32, device="cuda")
        h.attention_chunks_bounded(qo, ko, v, jo, jv, bounds, n, po, pl, qk_dtype=qd)
        h.lse_merge(po, pl, n, out, lse)
    return h, out, lse, bounds


@pytest.mark.parametrize("name", ["ragged", "audio1d", "lite", "one_tile"])
def test_bounded_attention_matches_oracle(name):
    w = CASES[name]
    x = inputs.make_inputs(w)
    for n in (1, w.chunks[-1]):
        h, out, lse, bounds = run_bounded(w, x, n)
        h.sync()
        ref, ref_lse = O.attention(geom(w), x["q"], x["k"], x["v"], x["jk"] if w.Nj else None,
                                   x["jv"] if w.Nj else None)
        compare(to_host(out), ref, lse.cpu().numpy().astype(np.float64), ref_lse, "bf16")
        # the bounds: within fp16 rounding of the oracle's, and above every logit
        rb = O.row_bounds(geom(w), x["q"], x["k"], x["jk"] if w.Nj else None)
        got = bounds[: w.B * w.H * w.S].cpu().numpy().reshape(w.B, w.H, w.S)
        np.testing.assert_allclose(got, rb, rtol=2e-3, atol=0)


def test_bounded_attention_mildly_peaked():
    w = CASES["ragged"]
    x = inputs.make_inputs(w, qk_scale=2.0)
    h, out, lse, _ = run_bounded(w, x, 4, rope=False)
    h.sync()
    ref, ref_lse = O.attention(geom(w), x["q"], x["k"], x["v"], x["jk"], x["jv"], rope=False)
    compare(to_host(out), ref, lse.cpu().numpy().astype(np.float64), ref_lse, "bf16")


def test_loose_bound_underflow_is_reported():
    from video_dit_long_gb300 import k6attn as K
    w = CASES["ragged"]
    x = inputs.make_inputs(w, qk_scale=5.0)  # |q||k|/sqrt(d) ~ 330 against logits ~ 110: exp underflows
    g = geom(w)
    rb = O.row_bounds(g, x["q"], x["k"], x["jk"], rope=False)
    _, ref_lse = O.attention(g, x["q"], x["k"], x["v"], x["jk"], x["jv"], rope=False)
    assert (rb - ref_lse).max() > 90  # the oracle agrees the bound is that loose somewhere
    h, out, lse, _ = run_bounded(w, x, 1, rope=False)
    with pytest.raises(K.K6Error) as e:
        h.sync()
    assert e.value.status == K.ERR_RANGE
    assert torch.isfinite(out.float()).all()


@pytest.mark.parametrize("name,n,group", [("ragged", 4, 2), ("ragged", 4, 4), ("audio1d", 3, 3), ("one_tile", 3, 3)])
def test_bounded_chunk_groups_match_oracle(name, n, group):
    """Constant max with each CTA's chunk group merged in the kernel (the chunks' terms share one bound)."""
    w = CASES[name]
    x = inputs.make_inputs(w)
    h, out, lse, _ = run_bounded(w, x, n, group=group)
    h.sync()
    ref, ref_lse = O.attention(geom(w), x["q"], x["k"], x["v"], x["jk"] if w.Nj else None,
                               x["jv"] if w.Nj else None)
    compare(to_host(out), ref, lse.cpu().numpy().astype(np.float64), ref_lse, "bf16")


@pytest.mark.slow
def test_bounded_step_on_the_pro_workload_matches_oracle():
    """The constant-max variant as the benchmark times it: row bounds, bounded attention over the 8 chunks in
    the step's chunk groups on the head layout, merge into the sequence layout; 1024 sampled query rows x all
    heads x all keys of the Pro workload against the oracle."""
    from video_dit_long_gb300 import k6attn as K
    from video_dit_long_gb300.step import UlyssesStep
    from .helpers import oracle_sampled
    w = configs.WORKLOADS["pro"]
    x = inputs.make_inputs(w)
    st = UlyssesStep(w, 8, 8, x)
    st.step()
    hd = st.head
    bounds = torch.empty(st.h.row_bounds_bytes() // 4, dtype=torch.float32, device="cuda")
    st.h.row_bounds(hd["q"], hd["k"], hd["jk"], bounds, qk_dtype=K.F16)
    st.h.attention_chunk_groups_bounded(hd["q"], hd["k"], hd["v"], hd["jk"], hd["jv"], bounds, 8, st.group,
                                        st.part_o, st.part_lse, qk_dtype=K.F16)
    out = torch.empty_like(st.out)
    lse = torch.empty_like(st.lse)
    st.hs.lse_merge_heads(st.part_o, st.part_lse, st.parts, 8, out, lse)
    st.sync()
    rows = inputs.sample_rows(w.S, w.Nv, w.S // 8, count=1024)
    idx = torch.from_numpy(rows).cuda()
    got = to_host(out.index_select(1, idx))
    got_lse = lse.index_select(2, idx).cpu().numpy().astype(np.float64)
    del st
    torch.cuda.empty_cache()
    ref, ref_lse = oracle_sampled(w, x, rows)
    print(compare(got, ref, got_lse, ref_lse, "bf16"))
