"""A handle is bound to the device it was created on: a call made while
another device is current is refused on the host (INVALID_ARG) before any
launch, instead of running on the wrong device with the handle's tables and
error word from the other one.  Needs two GPUs; skipped otherwise."""
import pytest

from video_dit_long_gb300 import inputs
from video_dit_long_gb300.configs import Workload

from .helpers import to_dev

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

W = Workload("devices", 1, 2, 128, "bf16", (1, 8, 16), 0, (32, 48, 48), 0, 1.0, 1.0, (1,))


@pytest.fixture(scope="module", autouse=True)
def _need_two_gpus():
    if not torch.cuda.is_available() or torch.cuda.device_count() < 2:
        pytest.skip("needs two CUDA devices")


def test_calls_on_another_device_are_refused():
    from video_dit_long_gb300 import k6attn as K
    with torch.cuda.device(0):
        h = K.Handle.for_workload(W)
    x = inputs.make_inputs(W)
    with torch.cuda.device(1):
        q, k, v = (to_dev(x[n], W.dtype).to("cuda:1") for n in ("q", "k", "v"))
        out = torch.empty_like(q)
        for call in (lambda: h.forward(q, k, v, None, None, out, rope=False, n_chunks=1),
                     lambda: h.forward_static_scratch(q, k, v, None, None, out, rope=False, n_chunks=1),
                     lambda: h.rope_qk(q, k, None),
                     lambda: h.sync()):
            with pytest.raises(K.K6Error) as e:
                call()
            assert e.value.status == K.ERR_INVALID_ARG
            assert b"device" in K.load().k6attn_last_error()
        h.close()  # destroy frees on the handle's own device from any current device
