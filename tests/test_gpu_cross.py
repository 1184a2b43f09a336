"""GPU parity of cross-attention (Sq != Sk, no rotary) against the fp64 oracle.

Workloads: audio queries over the full visual sequence at the Kandinsky 6 Pro
geometry (520 audio tokens over 51,840 video tokens), visual queries over
text (the image workload's 4,096 tokens over 256 text tokens, B = 2), and
small ragged cases in bf16 and fp32; with one and several K/V chunks.
"""
import numpy as np
import pytest

from oracle import oracle as O
from video_dit_long_gb300 import inputs

from .helpers import compare, to_dev, to_host

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _need_gpu():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")


def run_cross(B, H, d, dtype, Sq, Sk, n, seed=42, std=1.0, strict=False, raw=False):
    from video_dit_long_gb300 import k6attn as K
    q = inputs.tensor(seed, 30, (B, Sq, H, d), dtype, std)
    k = inputs.tensor(seed, 31, (B, Sk, H, d), dtype, std)
    v = inputs.tensor(seed, 32, (B, Sk, H, d), dtype)
    h = K.Handle(B, H, d, dtype, (1, 1, 1), 0, (d, 0, 0))
    if strict:
        h.set_option(K.OPT_STRICT_MMA_ORDER, 1)
    tq, tk, tv = (to_dev(a, dtype) for a in (q, k, v))
    out = torch.empty_like(tq)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    nb = h.cross_workspace_bytes(Sq, n)
    ws = torch.empty(nb, dtype=torch.uint8, device="cuda") if nb else None
    h.cross_forward(tq, tk, tv, out, lse, n_chunks=n, workspace=ws)
    h.sync()
    if raw:
        return to_host(out), lse.cpu().numpy()
    ref, ref_lse = O.cross_attention(q, k, v)
    return compare(to_host(out), ref, lse.cpu().numpy().astype(np.float64), ref_lse, dtype)


@pytest.mark.parametrize("n", [1, 8])
def test_audio_queries_over_full_visual_sequence(n):
    print(run_cross(1, 24, 128, "bf16", 520, 51840, n))


@pytest.mark.parametrize("n", [1, 2])
def test_visual_queries_over_text(n):
    run_cross(2, 24, 128, "bf16", 4096, 256, n)


@pytest.mark.parametrize("Sq,Sk,n", [(333, 700, 7), (1, 128, 1), (129, 1, 1), (257, 255, 5),
                                     (77, 1000, 1), (128, 2000, 1)])
def test_ragged_cross_bf16(Sq, Sk, n):
    run_cross(1, 2, 128, "bf16", Sq, Sk, n, std=2.0)


@pytest.mark.parametrize("Sq,Sk,n", [(100, 96, 4), (130, 64, 1)])
def test_cross_fp32(Sq, Sk, n):
    run_cross(1, 3, 64, "f32", Sq, Sk, n)


def test_cross_rejects_indivisible_chunks():
    from video_dit_long_gb300 import k6attn as K
    h = K.Handle(1, 2, 128, "bf16", (1, 1, 1), 0, (128, 0, 0))
    q = torch.zeros((1, 10, 2, 128), dtype=torch.bfloat16, device="cuda")
    kv = torch.zeros((1, 15, 2, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(K.K6Error) as e:
        h.cross_forward(q, kv, kv, torch.empty_like(q), n_chunks=4)
    assert e.value.status == K.ERR_INVALID_ARG


def test_short_queries_several_chunks_per_cta():
    # 100 query rows: every CTA runs a single Q tile; 32 heads x 80 chunks make
    # enough work units that each CTA takes four chunks in turn, carrying its
    # S buffers and barrier phases from one chunk to the next
    print(run_cross(1, 32, 128, "bf16", 100, 80 * 130, 80))


@pytest.mark.parametrize("n", [1, 2])
def test_single_tile_strict_mma_order_gives_identical_bits(n):
    # 77 queries (the single-tile kernel) over 16 K/V tiles per chunk, logits peaked
    # enough to rescale O: waiting for every P.V before S(j+2) reuses its tensor memory
    # must change nothing
    a = run_cross(1, 2, 128, "bf16", 77, 2048, n, std=2.0, raw=True)
    b = run_cross(1, 2, 128, "bf16", 77, 2048, n, std=2.0, raw=True, strict=True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_short_queries_split_into_sub_chunks_match_oracle():
    # 100 audio queries over the Pro visual sequence in 8 chunks: with the full
    # workspace the call runs each chunk as sub-chunks (the HBM-bound single-tile
    # CTAs fill the last wave); with room for 8 partials only, unsplit.  Both
    # equal the oracle, and each other within the bf16 bounds.
    from video_dit_long_gb300 import k6attn as K
    B, H, d, Sq, Sk, n = 1, 24, 128, 100, 51840, 8
    q = inputs.tensor(42, 30, (B, Sq, H, d), "bf16", 0.5)
    k = inputs.tensor(42, 31, (B, Sk, H, d), "bf16", 0.5)
    v = inputs.tensor(42, 32, (B, Sk, H, d), "bf16")
    h = K.Handle(B, H, d, "bf16", (1, 1, 1), 0, (d, 0, 0))
    tq, tk, tv = (to_dev(a, "bf16") for a in (q, k, v))
    ref, ref_lse = O.cross_attention(q, k, v)
    full = h.cross_workspace_bytes(Sq, n)
    unsplit = (n * B * Sq * H * d * 4 + 255) // 256 * 256 + (n * B * H * Sq * 4 + 255) // 256 * 256
    assert full > unsplit
    got = []
    for nb in (full, unsplit):
        out = torch.empty_like(tq)
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
        ws = torch.empty(nb, dtype=torch.uint8, device="cuda")
        h.cross_forward(tq, tk, tv, out, lse, n_chunks=n, workspace=ws)
        h.sync()
        got.append((to_host(out), lse.cpu().numpy().astype(np.float64)))
        compare(got[-1][0], ref, got[-1][1], ref_lse, "bf16")
    assert np.abs(got[0][0] - got[1][0]).max() <= 2e-2 and np.abs(got[0][1] - got[1][1]).max() <= 1e-3
