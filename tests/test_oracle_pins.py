"""Pins of the fp64 oracle against what mathematics and the pages fix.

None of these recomputes the oracle's own formula the oracle's way: attention
is checked against a high-precision brute force without max subtraction,
against torch's scaled_dot_product_attention, against closed forms and
invariants; the rotary embedding against its defining properties; the merge
against the unchunked result; the relayout against a reshape/transpose
formulation; the geometry against the worked examples the pages print.
"""
import math
import os
from decimal import Decimal, getcontext

import numpy as np
import pytest

from oracle import oracle as O
from video_dit_long_gb300 import configs, inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(shape, seed, std=1.0):
    return np.random.default_rng(seed).normal(0.0, std, size=shape)


def tiny_geom(B=1, H=2, d=8, grid=(1, 2, 3), Nj=2, axis=None, joint_rope=0):
    axis = axis or (d, 0, 0)
    return O.Geom(B, H, d, grid, Nj, axis, 10000.0, joint_rope)


def tiny_inputs(g, seed=0, std=1.0):
    return (rnd((g.B, g.S, g.H, g.d), seed, std), rnd((g.B, g.Nv, g.H, g.d), seed + 1, std),
            rnd((g.B, g.Nv, g.H, g.d), seed + 2), rnd((g.B, g.Nj, g.H, g.d), seed + 3, std),
            rnd((g.B, g.Nj, g.H, g.d), seed + 4))


# ---------------------------------------------------------------- attention


def brute_attention_decimal(q, K, V, prec=40):
    """softmax(q K^T / sqrt(d)) V by direct definition in 40-digit decimal,
    no max subtraction: E_j = exp(s_j), Z = sum E_j, out = sum E_j v_j / Z."""
    getcontext().prec = prec
    d = len(q)
    inv = Decimal(1) / Decimal(d).sqrt()
    E = []
    for kj in K:
        s = sum(Decimal(float(a)) * Decimal(float(b)) for a, b in zip(q, kj)) * inv
        E.append(s.exp())
    Z = sum(E)
    out = [sum(E[j] * Decimal(float(V[j][e])) for j in range(len(K))) / Z for e in range(d)]
    return [float(x) for x in out], float(Z.ln())


@pytest.mark.parametrize("d,Nj,std", [(4, 2, 1.0), (8, 3, 2.0), (8, 0, 3.0)])
def test_attention_matches_decimal_brute_force(d, Nj, std):
    g = tiny_geom(B=2, H=2, d=d, grid=(1, 3, 4), Nj=Nj)
    q, k, v, jk, jv = tiny_inputs(g, seed=d + Nj, std=std)
    out, lse = O.attention(g, q, k, v, jk if Nj else None, jv if Nj else None, rope=False)
    for b in range(g.B):
        for h in range(g.H):
            K = [k[b, j, h] for j in range(g.Nv)] + [jk[b, j, h] for j in range(Nj)]
            V = [v[b, j, h] for j in range(g.Nv)] + [jv[b, j, h] for j in range(Nj)]
            for i in range(g.S):
                ref_o, ref_l = brute_attention_decimal(q[b, i, h], K, V)
                np.testing.assert_allclose(out[b, i, h], ref_o, rtol=0, atol=1e-13)
                assert abs(lse[b, h, i] - ref_l) < 1e-13


def test_attention_matches_torch_sdpa_fp64():
    torch = pytest.importorskip("torch")
    g = O.Geom(2, 3, 16, (2, 3, 5), 7, (4, 6, 6), 10000.0, 0)
    q, k, v, jk, jv = tiny_inputs(g, seed=11, std=1.5)
    out, lse = O.attention(g, q, k, v, jk, jv, rope=True)
    qr = O.rope(g, q)
    # keys: rotate the concatenated sequence as a whole (joint keys at the rear)
    K = np.concatenate([k, jk], axis=1)
    V = np.concatenate([v, jv], axis=1)
    kr = O.rope(g, K)
    tq = torch.from_numpy(qr).permute(0, 2, 1, 3)
    tk = torch.from_numpy(kr).permute(0, 2, 1, 3)
    tv = torch.from_numpy(V).permute(0, 2, 1, 3)
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).permute(0, 2, 1, 3).numpy()
    ref_lse = torch.logsumexp(tq @ tk.transpose(-1, -2) / math.sqrt(g.d), dim=-1).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_constant_values_give_that_value():
    g = O.Geom(1, 2, 16, (2, 2, 3), 5, (4, 6, 6), 10000.0, 0)
    q, k, v, jk, jv = tiny_inputs(g, seed=3, std=2.0)
    c = rnd((g.H, g.d), 99)
    v[:] = c[None, None]
    jv[:] = c[None, None]
    out, _ = O.attention(g, q, k, v, jk, jv, rope=True)
    np.testing.assert_allclose(out, np.broadcast_to(c[None, None], out.shape), rtol=0, atol=1e-13)


def test_identical_keys_give_mean_of_values():
    g = tiny_geom(B=1, H=2, d=8, grid=(1, 4, 5), Nj=3)
    q, k, v, jk, jv = tiny_inputs(g, seed=5)
    key = rnd((g.H, g.d), 77)
    k[:] = key[None, None]
    jk[:] = key[None, None]
    out, lse = O.attention(g, q, k, v, jk, jv, rope=False)
    Vall = np.concatenate([v, jv], axis=1)
    mean_v = Vall.mean(axis=1)  # [B][H][d]
    np.testing.assert_allclose(out, np.broadcast_to(mean_v[:, None], out.shape), rtol=0, atol=1e-13)
    s = np.einsum("bihd,hd->bhi", q, key) / math.sqrt(g.d)
    np.testing.assert_allclose(lse, s + math.log(g.S), rtol=0, atol=1e-12)


def test_dominant_key_selects_its_value():
    g = tiny_geom(B=1, H=1, d=8, grid=(1, 3, 3), Nj=2)
    q, k, v, jk, jv = tiny_inputs(g, seed=8, std=0.1)
    # row 4 aligned with key 6 (video) at a large scale: that key dominates
    k[0, 6, 0] = q[0, 4, 0] * 4000.0
    out, _ = O.attention(g, q, k, v, jk, jv, rope=False, rows=[4])
    np.testing.assert_allclose(out[0, 0, 0], v[0, 6, 0], rtol=0, atol=1e-9)


def test_key_value_permutation_invariance():
    g = tiny_geom(B=2, H=3, d=8, grid=(2, 3, 4), Nj=5)
    q, k, v, jk, jv = tiny_inputs(g, seed=21)
    out, lse = O.attention(g, q, k, v, jk, jv, rope=False)
    K = np.concatenate([k, jk], axis=1)
    V = np.concatenate([v, jv], axis=1)
    perm = np.random.default_rng(4).permutation(g.S)
    Kp, Vp = K[:, perm], V[:, perm]
    out2, lse2 = O.attention(g, q, Kp[:, :g.Nv], Vp[:, :g.Nv], Kp[:, g.Nv:], Vp[:, g.Nv:], rope=False)
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


def test_rows_subset_equals_full():
    g = O.Geom(1, 2, 16, (2, 3, 4), 4, (4, 6, 6), 10000.0, 1)
    q, k, v, jk, jv = tiny_inputs(g, seed=2)
    out, lse = O.attention(g, q, k, v, jk, jv)
    rows = np.array([0, 5, 23, 24, 27])
    o2, l2 = O.attention(g, q, k, v, jk, jv, rows=rows)
    np.testing.assert_array_equal(o2, out[:, rows])
    np.testing.assert_array_equal(l2, lse[:, :, rows])


def test_bf16_and_f32_inputs_are_widened_exactly():
    g = tiny_geom(B=1, H=2, d=8, grid=(1, 2, 4), Nj=2)
    raw = inputs.make_inputs(configs.Workload("t", 1, 2, 8, "bf16", (1, 2, 4), 2, (8, 0, 0), 0, 1.0, 1.0, (1,)))
    wide = {k: inputs.bf16_to_f32(x).astype(np.float64) for k, x in raw.items()}
    a = O.attention(g, raw["q"], raw["k"], raw["v"], raw["jk"], raw["jv"])
    b = O.attention(g, wide["q"], wide["k"], wide["v"], wide["jk"], wide["jv"])
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------- chunked + merge


def chunked(g, q, k, v, jk, jv, bounds, rope=True):
    parts = [O.attention(g, q, k, v, jk, jv, rope=rope, kv_range=b) for b in bounds]
    po = np.stack([p[0] for p in parts])
    pl = np.stack([p[1] for p in parts])
    return O.lse_merge(po, pl)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16])
def test_chunked_merge_equals_unchunked(n):
    g = O.Geom(1, 2, 16, (2, 4, 5), 8, (4, 6, 6), 10000.0, 1)  # S = 48
    q, k, v, jk, jv = tiny_inputs(g, seed=n, std=2.0)
    out, lse = O.attention(g, q, k, v, jk, jv)
    mo, ml = chunked(g, q, k, v, jk, jv, O.chunk_bounds(g.S, n))
    np.testing.assert_allclose(mo, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=0, atol=1e-12)


def test_unequal_chunks_merge_equals_unchunked():
    g = O.Geom(2, 2, 16, (2, 4, 5), 8, (4, 6, 6), 10000.0, 0)
    q, k, v, jk, jv = tiny_inputs(g, seed=31, std=3.0)
    out, lse = O.attention(g, q, k, v, jk, jv)
    mo, ml = chunked(g, q, k, v, jk, jv, [(0, 1), (1, 17), (17, 40), (40, 41), (41, 48)])
    np.testing.assert_allclose(mo, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=0, atol=1e-12)


def test_chunk_bounds_reject_indivisible():
    assert O.chunk_bounds(52360, 8)[-1] == (45815, 52360)
    with pytest.raises(ValueError):
        O.chunk_bounds(3645, 8)


def test_merge_matches_decimal_definition():
    getcontext().prec = 40
    n, B, S, H, d = 3, 1, 4, 2, 3
    po = rnd((n, B, S, H, d), 1)
    pl = rnd((n, B, H, S), 2, 5.0)
    out, lse = O.lse_merge(po, pl)
    for s in range(S):
        for h in range(H):
            E = [Decimal(float(pl[c, 0, h, s])).exp() for c in range(n)]
            Z = sum(E)
            assert abs(float(Z.ln()) - lse[0, h, s]) < 1e-13
            for e in range(d):
                ref = sum(E[c] * Decimal(float(po[c, 0, s, h, e])) for c in range(n)) / Z
                assert abs(float(ref) - out[0, s, h, e]) < 1e-13


def test_merge_single_chunk_is_identity_and_equal_lse_is_mean():
    po = rnd((1, 2, 5, 3, 4), 3)
    pl = rnd((1, 2, 3, 5), 4)
    out, lse = O.lse_merge(po, pl)
    np.testing.assert_allclose(out, po[0], rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse, pl[0], rtol=0, atol=1e-15)
    po = rnd((4, 1, 5, 3, 4), 5)
    pl = np.full((4, 1, 3, 5), 1.25)
    out, lse = O.lse_merge(po, pl)
    np.testing.assert_allclose(out, po.mean(axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, 1.25 + math.log(4), rtol=0, atol=1e-14)


def test_merge_accepts_f32_partials_exactly():
    po = rnd((3, 1, 6, 2, 8), 6).astype(np.float32)
    pl = rnd((3, 1, 2, 6), 7).astype(np.float32)
    a = O.lse_merge(po, pl)
    b = O.lse_merge(po.astype(np.float64), pl.astype(np.float64))
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ---------------------------------------------------------------- backward


def test_backward_matches_central_differences_of_the_forward():
    """d/dx sum(out * G) by central differences through the forward oracle (rope off)."""
    g = tiny_geom(B=1, H=2, d=8, grid=(1, 2, 3), Nj=2)
    q, k, v, jk, jv = tiny_inputs(g, seed=71, std=1.5)
    G = rnd((g.B, g.S, g.H, g.d), 72)
    grads = dict(zip(("q", "k", "v", "jk", "jv"), O.attention_backward(g, q, k, v, jk, jv, G, rope=False)))
    x = {"q": q, "k": k, "v": v, "jk": jk, "jv": jv}

    def loss():
        out, _ = O.attention(g, x["q"], x["k"], x["v"], x["jk"], x["jv"], rope=False)
        return float((out * G).sum())

    eps = 1e-5
    rng = np.random.default_rng(73)
    for name in x:
        for _ in range(6):
            idx = tuple(int(rng.integers(0, n)) for n in x[name].shape)
            keep = x[name][idx]
            x[name][idx] = keep + eps
            up = loss()
            x[name][idx] = keep - eps
            dn = loss()
            x[name][idx] = keep
            fd = (up - dn) / (2 * eps)
            assert abs(fd - grads[name][idx]) < 1e-7 * max(1.0, abs(fd)), (name, idx, fd, grads[name][idx])


def test_backward_with_rope_is_the_rotated_gradient():
    """With rotary on, dq/dk are gradients w.r.t. the rotated q~, k~: identical to
    running the rope-off backward on the oracle-rotated inputs."""
    g = O.Geom(1, 2, 16, (2, 2, 3), 3, (4, 6, 6), 10000.0, 1)
    q, k, v, jk, jv = tiny_inputs(g, seed=74)
    G = rnd((g.B, g.S, g.H, g.d), 75)
    a = O.attention_backward(g, q, k, v, jk, jv, G, rope=True)
    K = O.rope(g, np.concatenate([k, jk], axis=1))
    b = O.attention_backward(g, O.rope(g, q), K[:, :g.Nv], v, K[:, g.Nv:], jv, G, rope=False)
    for x, y in zip(a, b):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-13)


def test_backward_closed_forms():
    """sum_j dV_j = sum_i dO_i (each row of P sums to 1); with every value
    equal, the output does not depend on q or k: their gradients vanish."""
    g = tiny_geom(B=1, H=1, d=8, grid=(1, 3, 3), Nj=1)
    q, k, v, jk, jv = tiny_inputs(g, seed=76)
    G = rnd((g.B, g.S, g.H, g.d), 77)
    dq, dk, dv, djk, djv = O.attention_backward(g, q, k, v, jk, jv, G, rope=False)
    np.testing.assert_allclose(dv.sum(axis=1) + djv.sum(axis=1), G.sum(axis=1), rtol=0, atol=1e-12)
    vc = np.broadcast_to(v[:, :1], v.shape).copy()
    jvc = np.broadcast_to(v[:, :1], jv.shape).copy()
    dq, dk, _, djk, _ = O.attention_backward(g, q, k, vc, jk, jvc, G, rope=False)
    assert np.abs(dq).max() < 1e-13 and np.abs(dk).max() < 1e-13 and np.abs(djk).max() < 1e-13


# ------------------------------------------------------------ cross-attention


@pytest.mark.parametrize("Sq,Sk,d", [(3, 11, 4), (13, 5, 8), (1, 1, 4)])
def test_cross_attention_matches_decimal_brute_force(Sq, Sk, d):
    B, H = 2, 2
    q, k, v = rnd((B, Sq, H, d), Sq, 2.0), rnd((B, Sk, H, d), Sk + 1, 2.0), rnd((B, Sk, H, d), Sk + 2)
    out, lse = O.cross_attention(q, k, v)
    for b in range(B):
        for h in range(H):
            K = [k[b, j, h] for j in range(Sk)]
            V = [v[b, j, h] for j in range(Sk)]
            for i in range(Sq):
                ref_o, ref_l = brute_attention_decimal(q[b, i, h], K, V)
                np.testing.assert_allclose(out[b, i, h], ref_o, rtol=0, atol=1e-13)
                assert abs(lse[b, h, i] - ref_l) < 1e-13


def test_cross_attention_matches_torch_sdpa_and_merges():
    torch = pytest.importorskip("torch")
    B, Sq, Sk, H, d = 2, 9, 40, 3, 16
    q, k, v = rnd((B, Sq, H, d), 1, 1.5), rnd((B, Sk, H, d), 2, 1.5), rnd((B, Sk, H, d), 3)
    out, lse = O.cross_attention(q, k, v)
    tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv).permute(0, 2, 1, 3).numpy()
    ref_lse = torch.logsumexp(tq @ tk.transpose(-1, -2) / math.sqrt(d), dim=-1).numpy()
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    parts = [O.cross_attention(q, k, v, kv_range=r) for r in O.chunk_bounds(Sk, 4)]
    mo, ml = O.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    np.testing.assert_allclose(mo, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=0, atol=1e-12)


def test_cross_attention_equals_self_attention_without_rotary():
    g = tiny_geom(B=1, H=2, d=8, grid=(1, 3, 4), Nj=0)
    q, k, v, _, _ = tiny_inputs(g, seed=12)
    a = O.attention(g, q, k, v, rope=False)
    b = O.cross_attention(q, k, v)
    np.testing.assert_array_equal(a[0], b[0])
    np.testing.assert_array_equal(a[1], b[1])


# ------------------------------------------------------- constant-max bound


def test_row_bounds_dominate_every_logit_and_are_tight_for_aligned_keys():
    g = O.Geom(2, 3, 16, (2, 3, 4), 5, (4, 6, 6), 10000.0, 1)
    q, k, v, jk, jv = tiny_inputs(g, seed=61, std=2.0)
    bound = O.row_bounds(g, q, k, jk)
    qr = O.rope(g, q)
    kr = O.rope(g, np.concatenate([k, jk], axis=1))
    s = np.einsum("bihe,bjhe->bhij", qr, kr) / math.sqrt(g.d)
    assert (s.max(axis=-1) <= bound + 1e-12).all()          # Cauchy-Schwarz
    # a key equal to the longest key direction aligned with q reaches the bound
    g0 = tiny_geom(B=1, H=1, d=8, grid=(1, 1, 3), Nj=0)
    q0 = rnd((1, 3, 1, 8), 62)
    k0 = np.stack([q0[0, 0, 0] * 2.0, q0[0, 1, 0] * 0.1, q0[0, 2, 0] * 0.3])[None, :, None, :]
    b0 = O.row_bounds(g0, q0, k0, rope=False)
    s00 = q0[0, 0, 0] @ k0[0, 0, 0] / math.sqrt(8)
    assert abs(b0[0, 0, 0] - s00) < 1e-12


# ----------------------------------------------------------------- QK-norm


def test_rms_norm_unit_rms_scale_invariance_and_weights():
    x = rnd((5, 3, 48), 40, 3.0)
    flat = x.reshape(5, 3 * 48)
    ones = np.ones(3 * 48)
    y = O.rms_norm(flat, ones, 0.0)
    np.testing.assert_allclose(np.sqrt((y ** 2).mean(axis=1)), 1.0, rtol=1e-14)   # unit RMS per row
    np.testing.assert_allclose(O.rms_norm(7.5 * flat, ones, 0.0), y, rtol=1e-13)   # scale invariance
    w = rnd(3 * 48, 41)
    np.testing.assert_allclose(O.rms_norm(flat, w, 0.0), y * w, rtol=1e-14)        # weights scale per dim
    # eps: a row of zeros stays zero; a constant row c gives c / sqrt(c^2 + eps)
    z = O.rms_norm(np.zeros((1, 8)), np.ones(8), 1e-6)
    assert not z.any()
    c = O.rms_norm(np.full((1, 8), 2.0), np.ones(8), 0.25)
    np.testing.assert_allclose(c, 2.0 / np.sqrt(4.25), rtol=1e-15)


def test_rms_norm_accepts_bf16_rows_exactly():
    raw = inputs.tensor(42, 50, (4, 256), "bf16")
    w = rnd(256, 51)
    np.testing.assert_array_equal(O.rms_norm(raw, w, 1e-6),
                                  O.rms_norm(inputs.bf16_to_f32(raw).astype(np.float64), w, 1e-6))


# ------------------------------------------------------------------- rotary


def video_token(g, t, h, w):
    return (t * g.grid[1] + h) * g.grid[2] + w


def test_rope_identity_at_position_zero_and_on_unrotated_joint_tokens():
    g = O.Geom(1, 1, 16, (3, 4, 5), 3, (4, 6, 6), 10000.0, 0)
    x = rnd(16, 1)
    np.testing.assert_array_equal(O.rope_vec(g, 0, x), x)
    for j in range(3):
        np.testing.assert_array_equal(O.rope_vec(g, g.Nv + j, x), x)
    g1 = O.Geom(1, 1, 16, (3, 4, 5), 3, (4, 6, 6), 10000.0, 1)
    np.testing.assert_array_equal(O.rope_vec(g1, g1.Nv, x), x)  # joint index 0
    assert np.abs(O.rope_vec(g1, g1.Nv + 1, x) - x).max() > 1e-3


def test_rope_preserves_each_pair_norm():
    g = O.Geom(1, 1, 16, (3, 4, 5), 3, (4, 6, 6), 10000.0, 1)
    x = rnd(16, 2)
    for n in range(g.S):
        y = O.rope_vec(g, n, x)
        np.testing.assert_allclose(np.hypot(y[0::2], y[1::2]), np.hypot(x[0::2], x[1::2]), rtol=1e-14)


@pytest.mark.parametrize("axis", [0, 1, 2])
def test_rope_relative_position_property(axis):
    """Shifting both tokens by the same amount along one axis keeps q~ . k~."""
    g = O.Geom(1, 1, 32, (6, 7, 8), 0, (8, 12, 12), 10000.0, 0)
    qv, kv = rnd(32, 10 + axis), rnd(32, 20 + axis)
    base_q, base_k = [1, 2, 3], [0, 1, 5]
    dot0 = None
    for shift in range(0, 3):
        pq, pk = list(base_q), list(base_k)
        pq[axis] += shift
        pk[axis] += shift
        dot = O.rope_vec(g, video_token(g, *pq), qv) @ O.rope_vec(g, video_token(g, *pk), kv)
        if dot0 is None:
            dot0 = dot
        assert abs(dot - dot0) < 1e-12
    # but a relative shift changes it
    pq = list(base_q)
    pq[axis] += 1
    assert abs(O.rope_vec(g, video_token(g, *pq), qv) @ O.rope_vec(g, video_token(g, *base_k), kv) - dot0) > 1e-6


def test_rope_frequency_ladder_and_axis_segments():
    """At position 1 on one axis, unit vectors reveal each pair's angle:
    pair 0 of every axis turns by 1 rad, successive pairs by a factor theta^(-2/d_a),
    and only the dims owned by that axis move."""
    axis_dim = (8, 12, 12)
    g = O.Geom(1, 1, 32, (3, 3, 3), 0, axis_dim, 10000.0, 0)
    offs = [0, 8, 20]
    for a in range(3):
        pos = [0, 0, 0]
        pos[a] = 1
        n = video_token(g, *pos)
        angles = []
        for p in range(16):
            e = np.zeros(32)
            e[2 * p] = 1.0
            y = O.rope_vec(g, n, e)
            ang = math.atan2(y[2 * p + 1], y[2 * p])
            owned = offs[a] <= 2 * p < offs[a] + axis_dim[a]
            if owned:
                angles.append(ang)
            else:
                assert ang == 0.0 and y[2 * p] == 1.0
            others = np.delete(y, [2 * p, 2 * p + 1])
            assert not others.any()
        assert abs(angles[0] - 1.0) < 1e-15
        ratio = 10000.0 ** (-2.0 / axis_dim[a])
        for i in range(1, len(angles)):
            assert abs(angles[i] / angles[i - 1] - ratio) < 1e-12


def test_rope_2d_geometry_has_empty_time_part():
    g = O.Geom(1, 1, 16, (3, 4, 5), 0, (0, 8, 8), 10000.0, 0)
    x = rnd(16, 3)
    for t in range(3):
        np.testing.assert_array_equal(O.rope_vec(g, video_token(g, t, 2, 3), x),
                                      O.rope_vec(g, video_token(g, 0, 2, 3), x))


def test_rope_1d_joint_equals_complex_product():
    """joint_rope=1: full-dim 1-D rotary at the joint index, as complex products."""
    g = O.Geom(1, 1, 16, (1, 2, 2), 6, (4, 6, 6), 10000.0, 1)
    x = rnd(16, 4)
    z = x[0::2] + 1j * x[1::2]
    for j in range(6):
        y = O.rope_vec(g, g.Nv + j, x)
        ref = z * np.exp(1j * j * 10000.0 ** (-np.arange(8) * 2.0 / 16))
        np.testing.assert_allclose(y[0::2] + 1j * y[1::2], ref, rtol=0, atol=1e-14)


def test_rope_tensor_matches_per_token():
    g = O.Geom(2, 3, 16, (2, 3, 4), 5, (4, 6, 6), 10000.0, 1)
    x = rnd((2, g.S, 3, 16), 9)
    y = O.rope(g, x)
    for b in range(2):
        for n in range(g.S):
            for h in range(3):
                np.testing.assert_array_equal(y[b, n, h], O.rope_vec(g, n, x[b, n, h]))


# ----------------------------------------------------------------- relayout


def relayout_by_transpose(src, B, S, H, d, P, direction):
    Sl, Hl = S // P, H // P
    if direction == 0:  # seq [r][b][s][p][hh][e] -> head [p][b][r][s][hh][e]
        return src.reshape(P, B, Sl, P, Hl, d).transpose(3, 1, 0, 2, 4, 5).reshape(P, B, S, Hl, d)
    return src.reshape(P, B, P, Sl, Hl, d).transpose(2, 1, 3, 0, 4, 5).reshape(P, B, Sl, H, d)


@pytest.mark.parametrize("B,S,H,d,P,dt", [(1, 16, 4, 8, 2, np.uint16), (2, 24, 6, 4, 3, np.float32),
                                          (1, 40, 24, 8, 8, np.uint16), (3, 10, 2, 2, 1, np.float32)])
def test_relayout_matches_transpose_and_round_trips(B, S, H, d, P, dt):
    rng = np.random.default_rng(S * H)
    src = rng.integers(0, 2**15, size=(P, B, S // P, H, d)).astype(dt)
    head = O.relayout(src, B, S, H, d, P, 0)
    np.testing.assert_array_equal(head, relayout_by_transpose(src, B, S, H, d, P, 0).reshape(head.shape))
    back = O.relayout(head, B, S, H, d, P, 1)
    np.testing.assert_array_equal(back, src)
    np.testing.assert_array_equal(relayout_by_transpose(head.reshape(P, B, S, H // P, d), B, S, H, d, P, 1)
                                  .reshape(src.shape), src)
    if P == 1:
        np.testing.assert_array_equal(head, src)


def test_relayout_rejects_indivisible():
    src = np.zeros(3645 * 8 * 4, np.uint16)
    with pytest.raises(ValueError):
        O.relayout(src, 1, 3645, 8, 4, 8, 0)
    with pytest.raises(ValueError):
        O.relayout(np.zeros(16 * 24 * 8, np.uint16), 1, 16, 24, 8, 16, 0)  # H % P != 0


# ----------------------------------------------------------------- geometry


def read_golden_geometry():
    rows, div = [], []
    with open(os.path.join(GOLDEN, "latent_geometry.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            lhs, rhs = line.split("->")
            if lhs.startswith("divisible"):
                _, s, p = lhs.split()
                div.append((int(s), int(p), int(rhs)))
            else:
                rows.append((tuple(map(int, lhs.split())), tuple(map(int, rhs.split()))))
    return rows, div


def test_latent_geometry_worked_examples():
    rows, div = read_golden_geometry()
    assert len(rows) == 5
    for (hgt, wid, fr), (t, h, w, n) in rows:
        assert O.latent_grid(hgt, wid, fr) == (t, h, w)
        assert t * h * w == n
    for s, p, rem in div:
        assert s % p == rem
    grids = {w.grid for w in configs.WORKLOADS.values()}
    for _, (t, h, w, _) in rows[1:]:
        assert (t, h, w) in grids


def test_workload_token_counts():
    W = configs.WORKLOADS
    assert [W[k].S for k in ("tiny", "lite", "image", "pro", "long")] == [1088, 3152, 4352, 52360, 119056]
    for w in W.values():
        for n in w.chunks:
            assert w.S % n == 0
        for P in w.relayout_P:
            assert w.S % P == 0 and w.H % P == 0
    assert abs(W["pro"].flops() / 1e12 - 33.69) < 0.01
    assert abs(W["long"].flops() / 1e12 - 174.17) < 0.01


# ------------------------------------------------------- full tiny workload


def test_tiny_workload_chunked_equals_unchunked():
    w = configs.WORKLOADS["tiny"]
    g = O.Geom(w.B, w.H, w.d, w.grid, w.Nj, w.axis_dim, w.theta, w.joint_rope)
    x = inputs.make_inputs(w)
    out, lse = O.attention(g, x["q"], x["k"], x["v"], x["jk"], x["jv"])
    mo, ml = chunked(g, x["q"], x["k"], x["v"], x["jk"], x["jv"], O.chunk_bounds(g.S, 4))
    np.testing.assert_allclose(mo, out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(ml, lse, rtol=0, atol=1e-12)
    # statistical sanity (not a tolerance): LSE ~ ln S + |q|^2 sigma_k^2 / (2 d)
    assert abs(lse.mean() - (math.log(g.S) + 0.5)) < 0.1
