"""GPU parity at the degenerate sizes of the method, against the fp64 oracle:
a single token (one query, one key), one-key chunks, a sequence one row past a
full 128-row tile, a joint segment of one token, and the backward pass on a
single token and on a ragged two-tile sequence.  Bounds as in the other bf16
parity tests (forward: max-abs 2e-2, mean-abs 2e-3, relative L2 1e-2, LSE
1e-3; backward: RMS 5e-3 and max 2e-2 of the reference's RMS / max).
"""
import numpy as np
import pytest

from oracle import oracle as O
from video_dit_long_gb300 import inputs
from video_dit_long_gb300.configs import Workload

from .helpers import compare, geom
from .test_gpu_backward import check_grad, gpu_backward
from .test_gpu_parity import run_forward

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def wl(name, grid, Nj, H=2, joint_rope=0):
    return Workload(name, 1, H, 128, "bf16", grid, Nj, (32, 48, 48), joint_rope, 1.0, 1.0, (1,))


EDGES = [
    (wl("one_token", (1, 1, 1), 0), 1),          # S = 1: one query, one key
    (wl("two_tokens", (1, 1, 2), 0), 2),         # chunks of one key
    (wl("tile_plus_one", (1, 1, 129), 0), 3),    # 129 rows: a full tile and one more; chunks of 43 keys
    (wl("one_joint", (1, 4, 8), 1), 1),          # a joint segment of one token
    (wl("one_joint_chunked", (1, 4, 8), 1), 3),  # ... and the last chunk holds video keys and the joint key
]


@pytest.mark.parametrize("w,n", EDGES, ids=[e[0].name + f"_n{e[1]}" for e in EDGES])
def test_forward_at_degenerate_sizes(w, n):
    # unit-variance q/k, the distribution the LSE bound is derived for with rotary on
    # (fp16 rotated copies); peaked inputs are covered with rotary off elsewhere
    x = inputs.make_inputs(w)
    out, lse, _ = run_forward(w, x, n)
    ref, ref_lse = O.attention(geom(w), x["q"], x["k"], x["v"], x["jk"] if w.Nj else None,
                               x["jv"] if w.Nj else None, rope=True)
    print(w.name, n, compare(out, ref, lse, ref_lse, "bf16"))


def test_single_token_output_is_its_value():
    """With one key the softmax weight is exactly 1: out = v (bf16 exact) and LSE = the logit."""
    w = wl("one_token", (1, 1, 1), 0)
    x = inputs.make_inputs(w)
    out, lse, _ = run_forward(w, x, 1)
    assert np.array_equal(out, inputs.bf16_to_f32(x["v"]).astype(np.float64))


@pytest.mark.parametrize("grid,Nj", [((1, 1, 1), 0), ((1, 10, 13), 0), ((1, 2, 64), 2)],
                         ids=["one_token", "ragged_130", "two_tiles_joint_2"])
def test_backward_at_degenerate_sizes(grid, Nj):
    w = wl("bwd_edge", grid, Nj)
    x = inputs.make_inputs(w, seed=11)
    dout = inputs.tensor(11, 20, (w.B, w.S, w.H, w.d), "bf16")
    got = gpu_backward(w, x, dout, "f16")
    ref = O.attention_backward(geom(w), x["q"], x["k"], x["v"], x["jk"] if w.Nj else None,
                               x["jv"] if w.Nj else None, inputs.bf16_to_f32(dout).astype(np.float64), rope=True)
    for name, g, r in zip(["dq", "dk", "dv", "djk", "djv"], got, ref):
        if w.S == 1 and name in ("dq", "dk"):
            # one key: P = 1 and dS = P (dP - D) = 0, so dq = dk = 0 (on the GPU up to the
            # rounding of LSE and of the two fp32 sums dP and D, about 1e-6 of |dout||v|)
            assert np.abs(g).max() < 1e-3 and np.abs(r).max() < 1e-12, (name, np.abs(g).max())
            continue
        print(check_grad(name, g, r))
