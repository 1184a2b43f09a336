"""GPU parity of the fused QK-norm + rotary prologue against the oracle
(RMSNorm over each token's H*d row, then the rotation)."""
import numpy as np
import pytest

from oracle import oracle as O
from video_dit_long_gb300 import configs, inputs
from video_dit_long_gb300.configs import Workload

from .helpers import geom, to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

CASES = {
    "lite": configs.WORKLOADS["lite"],
    "ragged": Workload("ragged", 2, 2, 128, "bf16", (3, 10, 20), 40, (32, 48, 48), 0, 1.0, 1.0, (1,)),
    "tiny": configs.WORKLOADS["tiny"],
}


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def weights(n, tid):
    return inputs.normal_f32(42, tid, n, std=0.2, mean=1.0)


def oracle_norm_rope(w, x, wq, wk, wjq, wjk, eps):
    g = geom(w)
    HD = w.H * w.d
    qn = np.empty((w.B, w.S, HD))
    qr = x["q"].reshape(w.B, w.S, HD)
    qn[:, :w.Nv] = O.rms_norm(qr[:, :w.Nv], wq, eps)
    if w.Nj:
        qn[:, w.Nv:] = O.rms_norm(qr[:, w.Nv:], wjq, eps)
    kn = O.rms_norm(x["k"].reshape(w.B, w.Nv, HD), wk, eps)
    parts = [kn]
    if w.Nj:
        parts.append(O.rms_norm(x["jk"].reshape(w.B, w.Nj, HD), wjk, eps))
    kall = np.concatenate(parts, axis=1).reshape(w.B, w.S, w.H, w.d)
    return O.rope(g, qn.reshape(w.B, w.S, w.H, w.d)), O.rope(g, kall)


@pytest.mark.parametrize("name,to_f16", [("lite", True), ("ragged", True), ("ragged", False), ("tiny", False)])
def test_norm_rope_matches_oracle(name, to_f16):
    from video_dit_long_gb300 import k6attn as K
    w = CASES[name]
    x = inputs.make_inputs(w)
    HD = w.H * w.d
    wq, wk, wjq, wjk = (weights(HD, t) for t in (40, 41, 42, 43))
    eps = 1e-6
    h = K.Handle.for_workload(w)
    q, k, jk = (to_dev(x[n], w.dtype) for n in ("q", "k", "jk"))
    tw = [torch.from_numpy(a).cuda() for a in (wq, wk, wjq, wjk)]
    if to_f16:
        outs = [torch.empty(t.shape, dtype=torch.float16, device="cuda") for t in (q, k, jk)]
        h.norm_rope_qk(q, k, jk, tw[0], tw[1], eps, joint_q_weight=tw[2], joint_k_weight=tw[3], q_out=outs[0],
                       k_out=outs[1], joint_k_out=outs[2], out_dtype=K.F16)
        rel = 2.0 ** -10
    else:
        h.norm_rope_qk(q, k, jk, tw[0], tw[1], eps, joint_q_weight=tw[2], joint_k_weight=tw[3])
        outs = [q, k, jk]
        rel = 2.0 ** -8 if w.dtype == "bf16" else 1e-5
    h.sync()
    ref_q, ref_k = oracle_norm_rope(w, x, wq, wk, wjq, wjk, eps)
    got_k = np.concatenate([to_host(outs[1]), to_host(outs[2])], axis=1)
    for got, ref in ((to_host(outs[0]), ref_q), (got_k, ref_k)):
        bound = np.abs(ref) * rel + 1e-5
        assert (np.abs(got - ref) <= bound).all(), float((np.abs(got - ref) - bound).max())


def test_norm_rope_rejects_missing_weights():
    from video_dit_long_gb300 import k6attn as K
    w = CASES["ragged"]
    h = K.Handle.for_workload(w)
    x = inputs.make_inputs(w)
    q, k, jk = (to_dev(x[n], w.dtype) for n in ("q", "k", "jk"))
    wq = torch.ones(w.H * w.d, device="cuda")
    with pytest.raises(K.K6Error) as e:
        h.norm_rope_qk(q, k, jk, wq, None, 1e-6)
    assert e.value.status == K.ERR_INVALID_ARG
