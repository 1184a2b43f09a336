"""The static-scratch forward (k6attn_forward_static_scratch) gives the same
results as k6attn_forward with a caller workspace.

It serves callers that cannot allocate device memory (a plugin whose host
framework owns all allocations, a fixed memory budget, a binding that only
receives tensors): the scratch comes from one device array inside the
library.  Both entry points run the same kernels on the same inputs, so their
outputs must agree bit for bit.  Two calls in a row, with different inputs,
the larger chunk count first, check that the second call is not disturbed by
the partials the first left in the array.  This file is collected last so
that a stop at its first failure has already run every other test.
"""
import pytest

from video_dit_long_gb300 import inputs
from video_dit_long_gb300.configs import Workload

from .helpers import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

W = Workload("noalloc", 1, 2, 128, "bf16", (3, 10, 20), 40, (32, 48, 48), 0, 1.0, 1.0, (2, 4))


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def test_static_scratch_forward_matches_workspace_forward_twice():
    from video_dit_long_gb300 import k6attn as K
    h = K.Handle.for_workload(W)
    for seed, n in ((42, 4), (7, 2)):
        x = inputs.make_inputs(W, seed=seed)
        q, k, v, jk, jv = (to_dev(x[name], W.dtype) for name in ("q", "k", "v", "jk", "jv"))
        ws = torch.empty(h.workspace_bytes(n, True), dtype=torch.uint8, device="cuda")
        ref = torch.empty_like(q)
        ref_lse = torch.empty((W.B, W.H, W.S), dtype=torch.float32, device="cuda")
        h.forward(q, k, v, jk, jv, ref, ref_lse, rope=True, n_chunks=n, workspace=ws)
        out = torch.full_like(q, float("nan"))
        lse = torch.full_like(ref_lse, float("nan"))
        h.forward_static_scratch(q, k, v, jk, jv, out, lse, rope=True, n_chunks=n)
        h.sync()
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16)), (seed, n)
        assert torch.equal(lse.view(torch.int32), ref_lse.view(torch.int32)), (seed, n)


def test_static_scratch_rejects_problems_beyond_its_size():
    from video_dit_long_gb300 import k6attn as K
    big = Workload("big", 1, 24, 128, "bf16", (7, 16, 27), 128, (32, 48, 48), 1, 1.0, 1.0, (2,))
    h = K.Handle.for_workload(big)
    assert h.workspace_bytes(2, True) > 32 << 20
    q = torch.zeros((1, big.S, 24, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, big.Nv, 24, 128), dtype=torch.bfloat16, device="cuda")
    j = torch.zeros((1, big.Nj, 24, 128), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(K.K6Error) as e:
        h.forward_static_scratch(q, kv, kv, j, j, out, None, rope=True, n_chunks=2)
    assert e.value.status == K.ERR_WORKSPACE
