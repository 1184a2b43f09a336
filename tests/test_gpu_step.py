"""Parity of the benchmarked step as composed (`UlyssesStep.step`, the exact
sequence of C-ABI calls `bench.py` times) against the fp64 oracle.

The step runs the Ulysses layout on one GPU ("Context Parallelism in vLLM
Omni Neuron", "Comparison with Other CP Strategies"; xDiT PR #586, USP
dispatch listing): rotary into fp16 fused with the seq->head relayout,
attention over the K/V chunks on the head-partitioned layout with each CTA's
chunk group merged in the kernel, and the LSE merge of the group partials
written back to the sequence layout.  Each piece has its own
parity test; this one checks the chain the headline number is measured on, at
the full workload sizes, on 1024 sampled query rows x all heads x all keys.
"""
import numpy as np
import pytest

from video_dit_long_gb300 import configs, inputs

from .helpers import compare, oracle_sampled, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_step(w, n, P, x):
    from video_dit_long_gb300.step import UlyssesStep
    st = UlyssesStep(w, n, P, x)
    st.step()
    st.sync()
    return st


@pytest.mark.slow
@pytest.mark.parametrize("name,n", [("pro", 8), ("long", 16)])
def test_benchmarked_step_matches_oracle(name, n):
    w = configs.WORKLOADS[name]
    x = inputs.make_inputs(w)
    st = run_step(w, n, w.relayout_P[-1], x)
    rows = inputs.sample_rows(w.S, w.Nv, w.S // n, count=1024)
    idx = torch.from_numpy(rows).cuda()
    out = to_host(st.out.index_select(1, idx))
    lse = st.lse.index_select(2, idx).cpu().numpy().astype(np.float64)
    del st
    torch.cuda.empty_cache()
    ref, ref_lse = oracle_sampled(w, x, rows)
    m = compare(out, ref, lse, ref_lse, "bf16")
    print(name, n, m)


def test_step_on_a_small_workload_matches_oracle():
    """The same chain on the Lite geometry (1-D audio rotary, 8-way relayout), every row."""
    w = configs.WORKLOADS["lite"]
    x = inputs.make_inputs(w)
    st = run_step(w, 2, 8, x)
    out = to_host(st.out)
    lse = st.lse.cpu().numpy().astype(np.float64)
    rows = np.arange(w.S)
    ref, ref_lse = oracle_sampled(w, x, rows)
    compare(out, ref, lse, ref_lse, "bf16")


def test_step_with_two_batches_matches_oracle():
    """The chain with B = 2 (image workload: 2-D rotary, 256 text tokens; 8-way head split of 24
    heads, 4 chunks in the library's groups), every row of both batches."""
    w = configs.WORKLOADS["image"].with_batch(2)
    x = inputs.make_inputs(w)
    st = run_step(w, 4, 8, x)
    out = to_host(st.out)
    lse = st.lse.cpu().numpy().astype(np.float64)
    ref, ref_lse = oracle_sampled(w, x, np.arange(w.S))
    compare(out, ref, lse, ref_lse, "bf16")
