"""GPU parity of the attention backward pass against the fp64 oracle.

Gradients of sum(out * dout) with respect to the rotated q, k and to v,
joint_k, joint_v.  The GPU side runs the product path: rotary embeddings into
fp16 copies, the one-chunk forward for out and lse, then the backward kernels;
the oracle rotates in fp64 itself from the same seeded bf16 inputs.

Tolerance per gradient tensor, from the arithmetic of the kernels: P is
rounded to bf16 (relative 2^-9) before dv += P^T dout; dS is rounded to the
q/k type (fp16 2^-11, bf16 2^-9) before dq and dk; the rotated q/k are fp16
(logit error about 7e-4 for unit inputs); and D_i comes from the bf16 forward
output (2^-9 per element).  Rounding errors of random sign add in
quadrature, about 1.5e-3 of the gradient's own RMS.  The D_i term is not
damped where attention is peaked: for the dominant key dP_ij - D_i is small
while D_i carries its full 2^-9 error, which lifts dq/dk to about 3.5e-3 for
q/k of std 2 with bf16 dS.  The bounds sit above that:
  rms(g - ref) <= 5e-3 rms(ref),  max|g - ref| <= 2e-2 max|ref|.
A plausible kernel mistake (a transposed operand, a missing scale, a dropped
D_i term, a wrong key tile) moves the error to order one.
"""
import numpy as np
import pytest

from oracle import oracle as O
from video_dit_long_gb300 import configs, inputs
from video_dit_long_gb300.configs import Workload

from .helpers import geom, to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

GRAD_RMS_REL = 5e-3
GRAD_MAX_REL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def K():
    from video_dit_long_gb300 import k6attn
    return k6attn


CASES = {
    # several key tiles, ragged video and joint tails, rotary on (fp16 q/k)
    "ragged": (Workload("ragged", 1, 2, 128, "bf16", (3, 10, 20), 40, (32, 48, 48), 0, 1.0, 1.0, (1,)), "f16"),
    # B = 2, joint tokens with 1-D rotary, joint tail of 62 rows
    "audio1d": (Workload("audio1d", 2, 2, 128, "bf16", (2, 8, 16), 62, (32, 48, 48), 1, 1.0, 1.0, (1,)), "f16"),
    # one partial tile, no joint tokens, bf16 q/k without rotary
    "one_tile": (Workload("one_tile", 1, 3, 128, "bf16", (1, 7, 9), 0, (32, 48, 48), 0, 1.0, 1.0, (1,)), "bf16"),
    # tile-aligned sequence, no joint tokens, bf16 q/k
    "aligned": (Workload("aligned", 1, 2, 128, "bf16", (1, 16, 16), 0, (32, 48, 48), 0, 1.0, 1.0, (1,)), "bf16"),
    # peaked attention (q/k std 2), joint tail of 5 rows, bf16 q/k
    "peaked": (Workload("peaked", 1, 2, 128, "bf16", (1, 10, 30), 5, (32, 48, 48), 0, 2.0, 1.0, (1,)), "bf16"),
    # a longer sequence: 9 key tiles plus a joint tile
    "long9": (Workload("long9", 1, 2, 128, "bf16", (4, 12, 24), 100, (32, 48, 48), 0, 1.0, 1.0, (1,)), "f16"),
}


def gpu_backward(w, x, dout_bits, qk):
    k6 = K()
    h = k6.Handle.for_workload(w)
    q, k, v, jk, jv = (to_dev(x[n], "bf16") for n in ("q", "k", "v", "jk", "jv"))
    has_j = w.Nj > 0
    if not has_j:
        jk = jv = None
    if qk == "f16":
        qh = torch.empty(q.shape, dtype=torch.float16, device="cuda")
        kh = torch.empty(k.shape, dtype=torch.float16, device="cuda")
        jh = torch.empty(jk.shape, dtype=torch.float16, device="cuda") if has_j else None
        h.rope_qk(q, k, jk, q_out=qh, k_out=kh, joint_k_out=jh, out_dtype=k6.F16)
        qd = k6.F16
    else:
        qh, kh, jh, qd = q, k, jk, k6.BF16
    out = torch.empty_like(q)
    lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    h.attention_chunks(qh, kh, v, jh, jv, 1, out, lse, qk_dtype=qd)
    do = to_dev(dout_bits, "bf16")
    f32 = dict(dtype=torch.float32, device="cuda")
    dq = torch.full((w.B, w.S, w.H, w.d), float("nan"), **f32)
    dk = torch.full((w.B, w.Nv, w.H, w.d), float("nan"), **f32)
    dv = torch.full((w.B, w.Nv, w.H, w.d), float("nan"), **f32)
    djk = torch.full((w.B, w.Nj, w.H, w.d), float("nan"), **f32) if has_j else None
    djv = torch.full((w.B, w.Nj, w.H, w.d), float("nan"), **f32) if has_j else None
    ws = torch.empty(h.backward_workspace_bytes(), dtype=torch.uint8, device="cuda")
    h.backward(qh, kh, v, jh, jv, out, do, lse, dq, dk, dv, djk, djv, workspace=ws, qk_dtype=qd)
    h.sync()
    res = [dq, dk, dv] + ([djk, djv] if has_j else [])
    return [t.cpu().numpy().astype(np.float64) for t in res]


def check_grad(name, g, ref):
    assert np.isfinite(g).all(), f"{name}: non-finite gradient"
    err = g - ref
    rms_ref = float(np.sqrt(np.mean(ref * ref)))
    m = {"name": name, "rms_rel": float(np.sqrt(np.mean(err * err))) / max(rms_ref, 1e-300),
         "max_rel": float(np.abs(err).max()) / max(float(np.abs(ref).max()), 1e-300)}
    assert m["rms_rel"] <= GRAD_RMS_REL, m
    assert m["max_rel"] <= GRAD_MAX_REL, m
    return m


@pytest.mark.parametrize("case", list(CASES))
def test_backward_matches_oracle(case):
    w, qk = CASES[case]
    x = inputs.make_inputs(w, seed=42)
    dout = inputs.tensor(42, 20, (w.B, w.S, w.H, w.d), "bf16")
    got = gpu_backward(w, x, dout, qk)
    ref = O.attention_backward(geom(w), x["q"], x["k"], x["v"], x["jk"] if w.Nj else None,
                               x["jv"] if w.Nj else None, inputs.bf16_to_f32(dout).astype(np.float64),
                               rope=(qk == "f16"))
    names = ["dq", "dk", "dv", "djk", "djv"]
    for n, g, r in zip(names, got, ref):
        print(check_grad(n, g, r))


def test_backward_full_size_invariants():
    """At the Kandinsky 6 Pro geometry (52,360 tokens, 24 heads), two identities
    that hold at any size: every row of P sums to one, so the sum over all keys
    of dv equals the sum over all queries of dout; and every row of dS sums to
    zero (sum_j P_ij (dP_ij - D_i) = O_i.dout_i - D_i), so the sum over all keys
    of dk vanishes.  Bounds: bf16 rounding of P (2^-9, random sign) gives a
    standard deviation below 1.2e-3 of the root sum of squares of dout; the
    dk sum is compared with the root sum of squares of dk itself."""
    k6 = K()
    w = configs.WORKLOADS["pro"]
    x = inputs.make_inputs(w, seed=7)
    dout = inputs.tensor(7, 20, (w.B, w.S, w.H, w.d), "bf16")
    got = gpu_backward(w, x, dout, "f16")
    dq, dk, dv, djk, djv = got
    do = inputs.bf16_to_f32(dout).astype(np.float64)
    sum_dv = dv.sum(axis=1) + djv.sum(axis=1)           # [B][H][d]
    sum_do = do.sum(axis=1)
    rss_do = np.sqrt((do * do).sum(axis=1))
    assert np.all(np.abs(sum_dv - sum_do) <= 6e-3 * rss_do + 1e-3), float(np.abs(sum_dv - sum_do).max())
    sum_dk = dk.sum(axis=1) + djk.sum(axis=1)
    rss_dk = np.sqrt((dk * dk).sum(axis=1) + (djk * djk).sum(axis=1))
    assert np.all(np.abs(sum_dk) <= 1e-2 * rss_dk), float((np.abs(sum_dk) / rss_dk).max())
    assert np.isfinite(dq).all() and np.abs(dq).max() > 0
    del k6


def test_backward_rejects_bad_arguments():
    k6 = K()
    w = CASES["one_tile"][0]
    h = k6.Handle.for_workload(w)
    t = torch.zeros((w.B, w.S, w.H, w.d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((w.B, w.H, w.S), dtype=torch.float32, device="cuda")
    g = [torch.zeros((w.B, w.S, w.H, w.d), dtype=torch.float32, device="cuda") for _ in range(3)]
    ws = torch.empty(h.backward_workspace_bytes(), dtype=torch.uint8, device="cuda")
    with pytest.raises(k6.K6Error) as e:
        h.backward(t, t, t, None, None, t, t, lse, g[0], g[1], g[2], workspace=ws[:16])
    assert e.value.status == k6.ERR_WORKSPACE
    with pytest.raises(k6.K6Error) as e:
        h.backward(t, t, t, None, None, t, t, lse, g[0], g[0], g[2], workspace=ws)
    assert e.value.status == k6.ERR_INVALID_ARG
    with pytest.raises(k6.K6Error) as e:
        h.backward(t, t, t, None, None, t, t, lse, g[0], g[1], g[2], workspace=ws, qk_dtype=k6.F32)
    assert e.value.status == k6.ERR_INVALID_ARG
    f = k6.Handle(1, 2, 64, "f32", (1, 1, 8), 0, (64, 0, 0))
    with pytest.raises(k6.K6Error) as e:
        f.backward(t, t, t, None, None, t, t, lse, g[0], g[1], g[2], workspace=ws)
    assert e.value.status == k6.ERR_UNSUPPORTED
