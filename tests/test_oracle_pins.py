"""CPU pins for the float64 oracle.

Each test ties an oracle function to something other than itself: a closed
form, a worked number printed on the pages, a library routine, an identity the
pages derive, or a pure-Python brute force on tiny inputs.
"""
import cmath
import math
import os

import numpy as np
import pytest
import scipy.linalg
import scipy.special

from oracle import palu_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def test_rope_two_dims_is_plane_rotation_by_position_radians():
    # d_h = 2: one pair with omega_0 = theta^0 = 1, so position p rotates by p radians.
    for p in (0.0, 1.0, 2.5, 100.0):
        out = O.rope_rotate(np.array([1.0, 0.0]), p, 10000.0)
        np.testing.assert_allclose(out, [math.cos(p), math.sin(p)], atol=1e-15)
        out = O.rope_rotate(np.array([0.0, 1.0]), p, 10000.0)
        np.testing.assert_allclose(out, [-math.sin(p), math.cos(p)], atol=1e-15)


def test_rope_frequencies_closed_form():
    # d_h = 4, theta = 10000: omega = [1, 10000^(-1/2)] = [1, 0.01].
    np.testing.assert_allclose(O.rope_inv_freq(4, 10000.0), [1.0, 0.01], rtol=1e-15)
    # last pair of d_h = 128 at theta = 10000: 10000^(-126/128)
    w = O.rope_inv_freq(128, 10000.0)
    assert w[0] == 1.0 and abs(w[-1] - 10000.0 ** (-126 / 128)) < 1e-18
    assert np.all(np.diff(w) < 0)


def test_rope_undone_by_shard_inverse_formula():
    # Shard section 5 step 1: k_no_rope = k*cos(theta p) - rotate_half(k)*sin(theta p),
    # rotate_half([a, b]) = [-b, a]. It must undo the oracle's forward rotation.
    rng = np.random.default_rng(0)
    d = 16
    x = rng.standard_normal((5, d))
    pos = np.array([0, 1, 7, 300, 65535], dtype=np.float64)
    y = O.rope_rotate(x, pos, 10000.0)
    k = np.arange(d // 2)
    ang = pos[:, None] * (10000.0 ** (-2.0 * k / d))[None, :]
    cos = np.concatenate([np.cos(ang)] * 2, axis=1)
    sin = np.concatenate([np.sin(ang)] * 2, axis=1)
    rot_half = np.concatenate([-y[:, d // 2:], y[:, :d // 2]], axis=1)
    x_back = y * cos - rot_half * sin
    np.testing.assert_allclose(x_back, x, atol=1e-12)


def test_rope_identity_at_zero_norm_preserving_and_relative():
    rng = np.random.default_rng(1)
    d = 32
    x = rng.standard_normal(d)
    np.testing.assert_array_equal(O.rope_rotate(x, 0.0, 10000.0), x)
    for p in (1, 17, 4095, 65535):
        np.testing.assert_allclose(np.linalg.norm(O.rope_rotate(x, p, 1e4)), np.linalg.norm(x), rtol=1e-13)
    # scores depend only on the relative position (RoFormer property)
    q = rng.standard_normal(d)
    k = rng.standard_normal(d)
    base = O.rope_rotate(q, 100, 1e4) @ O.rope_rotate(k, 37, 1e4)
    for c in (1, 5, 1000):
        sh = O.rope_rotate(q, 100 + c, 1e4) @ O.rope_rotate(k, 37 + c, 1e4)
        assert abs(sh - base) < 1e-10


# ---------------------------------------------------------------------------
# Softmax / attention
# ---------------------------------------------------------------------------

def test_softmax_attend_matches_scipy():
    rng = np.random.default_rng(2)
    s = rng.standard_normal(50) * 3
    v = rng.standard_normal((50, 7))
    o, lse = O.softmax_attend(s, v)
    np.testing.assert_allclose(o, scipy.special.softmax(s) @ v, rtol=1e-13)
    assert abs(lse - scipy.special.logsumexp(s)) < 1e-12


def _tiny(seed=3, B=2, T=6, n=4, s=2, d_h=4, r=4, r_v=3):
    rng = np.random.default_rng(seed)
    n_g = n // s
    q = rng.standard_normal((B, n, d_h))
    hk = rng.standard_normal((B, T, n_g, r))
    hv = rng.standard_normal((B, T, n_g, r_v))
    bk = rng.standard_normal((n_g, r, s * d_h))
    return q, hk, hv, bk


def test_single_token_returns_its_value_latent():
    q, hk, hv, bk = _tiny(T=1)
    for mode in ("rope", "absorbed"):
        o, lse = O.decode(q, hk, hv, bk, [1, 1], 2, mode=mode)
        for b in range(2):
            for i in range(4):
                np.testing.assert_allclose(o[b, i], hv[b, 0, i // 2], rtol=1e-14)


def test_zero_query_is_mean_of_values_and_lse_log_T():
    q, hk, hv, bk = _tiny(T=6)
    q[:] = 0
    for mode in ("rope", "absorbed"):
        o, lse = O.decode(q, hk, hv, bk, [6, 4], 2, mode=mode)
        np.testing.assert_allclose(o[0, 1], hv[0, :6, 0].mean(axis=0), rtol=1e-13)
        np.testing.assert_allclose(o[1, 3], hv[1, :4, 1].mean(axis=0), rtol=1e-13)
        np.testing.assert_allclose(lse[0], math.log(6), rtol=1e-14)
        np.testing.assert_allclose(lse[1], math.log(4), rtol=1e-14)


def test_equal_key_latents_give_uniform_weights_absorbed():
    q, hk, hv, bk = _tiny(T=5)
    hk[:] = hk[:, :1]
    o, _ = O.decode(q, hk, hv, bk, [5, 5], 2, mode="absorbed")
    np.testing.assert_allclose(o[1, 2], hv[1, :, 1].mean(axis=0), rtol=1e-13)


def test_empty_sequence():
    q, hk, hv, bk = _tiny(T=3)
    o, lse = O.decode(q, hk, hv, bk, [0, 3], 2)
    assert np.all(o[0] == 0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


# ---------------------------------------------------------------------------
# Brute force on tiny inputs: scalar loops, math.fsum, complex-number rotation
# ---------------------------------------------------------------------------

def _brute_rope_decode(q, hk, hv, bk, T, s, theta, pos, qp):
    n, d_h = len(q), len(q[0])
    half = d_h // 2

    def rot(vec, p):
        out = [0.0] * d_h
        for c in range(half):
            z = complex(vec[c], vec[c + half]) * cmath.exp(1j * p * theta ** (-(2 * c) / d_h))
            out[c], out[c + half] = z.real, z.imag
        return out

    res = []
    for i in range(n):
        g, j = i // s, i % s
        qr = rot(list(q[i]), qp)
        scores = []
        for t in range(T):
            k = [math.fsum(hk[t][g][m] * bk[g][m][j * d_h + c] for m in range(len(bk[g])))
                 for c in range(d_h)]
            kr = rot(k, pos[t])
            scores.append(math.fsum(a * b for a, b in zip(qr, kr)) / math.sqrt(d_h))
        mx = max(scores)
        e = [math.exp(x - mx) for x in scores]
        l = math.fsum(e)
        o = [math.fsum(e[t] * hv[t][g][m] for t in range(T)) / l for m in range(len(hv[0][g]))]
        res.append((o, mx + math.log(l)))
    return res


def test_brute_force_rope_tiny():
    q, hk, hv, bk = _tiny(seed=4, B=2, T=7, n=4, s=2, d_h=4, r=4, r_v=3)
    pos = np.array([[3, 9, 1, 0, 22, 5, 6], [0, 1, 2, 3, 4, 5, 6]])
    qp = np.array([30, 6])
    theta = 100.0
    o, lse = O.decode(q, hk, hv, bk, [7, 5], 2, mode="rope", theta=theta, positions=pos, q_pos=qp)
    for b, T in ((0, 7), (1, 5)):
        ref = _brute_rope_decode(q[b].tolist(), hk[b].tolist(), hv[b].tolist(), bk.tolist(), T, 2,
                                 theta, pos[b].tolist(), float(qp[b]))
        for i, (ro, rl) in enumerate(ref):
            np.testing.assert_allclose(o[b, i], ro, rtol=1e-12, atol=1e-13)
            assert abs(lse[b, i] - rl) < 1e-12


def test_default_query_position_is_last_cached_token():
    q, hk, hv, bk = _tiny(seed=5, T=6)
    pos = np.array([[4, 8, 15, 16, 23, 42], [1, 2, 3, 5, 8, 13]])
    a = O.decode(q, hk, hv, bk, [6, 4], 2, positions=pos)
    b = O.decode(q, hk, hv, bk, [6, 4], 2, positions=pos, q_pos=[42, 5])
    np.testing.assert_array_equal(a[0], b[0])
    c = O.decode(q, hk, hv, bk, [6, 4], 2)
    d = O.decode(q, hk, hv, bk, [6, 4], 2, q_pos=[5, 3])
    np.testing.assert_array_equal(c[0], d[0])


# ---------------------------------------------------------------------------
# Identities the Palu notes derive
# ---------------------------------------------------------------------------

def _mha_setup(seed, B=2, T=9, d=64, n=4, s=2, d_h=8):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((B, T, d))
    wk = rng.standard_normal((d, n * d_h)) / math.sqrt(d)
    wv = rng.standard_normal((d, n * d_h)) / math.sqrt(d)
    q = rng.standard_normal((B, n, d_h))
    return x, wk, wv, q


def _group_factors(w, n_g, s, d_h, r):
    A, B = [], []
    for g in range(n_g):
        a, b = O.svd_factor(w[:, g * s * d_h:(g + 1) * s * d_h], r)
        A.append(a)
        B.append(b)
    return np.stack(A), np.stack(B)


@pytest.mark.parametrize("mode", ["rope", "absorbed"])
def test_full_rank_latent_decode_equals_uncompressed_mha(mode):
    # With r = s*d_h the group factors are exact, so decode over latents must be MHA.
    B, T, d, n, s, d_h = 2, 9, 64, 4, 2, 8
    x, wk, wv, q = _mha_setup(6, B, T, d, n, s, d_h)
    n_g, r = n // s, s * d_h
    Ak, Bk = _group_factors(wk, n_g, s, d_h, r)
    Av, Bv = _group_factors(wv, n_g, s, d_h, r)
    hk = np.einsum("btd,gdr->btgr", x, Ak)
    hv = np.einsum("btd,gdr->btgr", x, Av)
    seq = [9, 6]
    pos = np.array([[5, 1, 2, 9, 4, 7, 3, 0, 8], list(range(9))])
    o, lse = O.decode(q, hk, hv, Bk, seq, s, mode=mode, positions=pos, q_pos=[11, 5])
    a, lse_ref = O.mha_decode(q, x, wk, wv, seq, rope=(mode == "rope"), positions=pos, q_pos=[11, 5])
    for b in range(B):
        for i in range(n):
            g, j = i // s, i % s
            np.testing.assert_allclose(o[b, i] @ Bv[g][:, j * d_h:(j + 1) * d_h], a[b, i], atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-11)


def test_value_fusion_into_output_projection():
    # p H_v (B_v W_o) == (p V) W_o with V = H_v B_v, at truncated rank.
    B, T, d, n, s, d_h, r = 1, 12, 64, 4, 2, 8, 5
    x, wk, wv, q = _mha_setup(7, B, T, d, n, s, d_h)
    rng = np.random.default_rng(8)
    wo = rng.standard_normal((n * d_h, d)) / math.sqrt(d)
    n_g = n // s
    Ak, Bk = _group_factors(wk, n_g, s, d_h, r)
    Av, Bv = _group_factors(wv, n_g, s, d_h, r)
    hk = np.einsum("btd,gdr->btgr", x, Ak)
    hv = np.einsum("btd,gdr->btgr", x, Av)
    o, _ = O.decode(q, hk, hv, Bk, [T], s)
    # uncompressed MHA with the low-rank weights W' = A B (block columns per group)
    wk_lr = np.concatenate([Ak[g] @ Bk[g] for g in range(n_g)], axis=1)
    wv_lr = np.concatenate([Av[g] @ Bv[g] for g in range(n_g)], axis=1)
    a, _ = O.mha_decode(q, x, wk_lr, wv_lr, [T])
    y_ref = sum(a[0, i] @ wo[i * d_h:(i + 1) * d_h] for i in range(n))
    y = sum(o[0, i] @ (Bv[i // s][:, (i % s) * d_h:(i % s + 1) * d_h] @ wo[i * d_h:(i + 1) * d_h])
            for i in range(n))
    np.testing.assert_allclose(y, y_ref, atol=1e-11)


def test_fused_output_projection_equals_uncompressed_mha_output_at_full_rank():
    # At full rank r = s*d_h with exact SVD factors the latent path is the MHA layer itself, so
    # sum_i o_i (B_v^(i) W_o^(i)) must equal concat_i(a_i) W_o of plain multi-head attention.
    B, T, d, n, s, d_h = 2, 9, 32, 4, 2, 4
    x, wk, wv, q = _mha_setup(21, B, T, d, n, s, d_h)
    rng = np.random.default_rng(22)
    wo = rng.standard_normal((n * d_h, d)) / math.sqrt(d)
    n_g, r = n // s, s * d_h
    Ak, Bk = _group_factors(wk, n_g, s, d_h, r)
    Av, Bv = _group_factors(wv, n_g, s, d_h, r)
    hk = np.einsum("btd,gdr->btgr", x, Ak)
    hv = np.einsum("btd,gdr->btgr", x, Av)
    o, _ = O.decode(q, hk, hv, Bk, [T, T - 3], s)
    y = O.project_fused(o, O.fuse_value_output(Bv, wo, s))
    a, _ = O.mha_decode(q, x, wk, wv, [T, T - 3])
    y_ref = a.reshape(B, n * d_h) @ wo
    np.testing.assert_allclose(y, y_ref, rtol=1e-10, atol=1e-11)


def test_fused_output_projection_brute_force_tiny():
    # scalar loops with exact summation, written from the definition y_c = sum_i sum_m o_im W_f,(i m) c
    rng = np.random.default_rng(23)
    n_g, s, d_h, r, d, B = 2, 2, 3, 2, 5, 2
    bv = rng.standard_normal((n_g, r, s * d_h))
    wo = rng.standard_normal((n_g * s * d_h, d))
    o = rng.standard_normal((B, n_g * s, r))
    wf = O.fuse_value_output(bv, wo, s)
    for i in range(n_g * s):
        g, j = i // s, i % s
        for m in range(r):
            for c in range(d):
                want = math.fsum(bv[g, m, j * d_h + e] * wo[i * d_h + e, c] for e in range(d_h))
                assert abs(wf[i * r + m, c] - want) < 1e-12
    y = O.project_fused(o, wf)
    for b in range(B):
        for c in range(d):
            want = math.fsum(o[b, i, m] * wf[i * r + m, c] for i in range(n_g * s) for m in range(r))
            assert abs(y[b, c] - want) < 1e-12


def test_absorbed_equals_rebuild_when_rotation_is_identity():
    # Key fusion: q K^T = (q B^T) H^T. With every position 0, RoPE is the identity.
    q, hk, hv, bk = _tiny(seed=9, B=2, T=8, n=4, s=2, d_h=4, r=4, r_v=3)
    zeros = np.zeros((2, 8), dtype=np.int64)
    a = O.decode(q, hk, hv, bk, [8, 3], 2, mode="rope", positions=zeros, q_pos=[0, 0])
    b = O.decode(q, hk, hv, bk, [8, 3], 2, mode="absorbed")
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


# ---------------------------------------------------------------------------
# SVD factors and the Hadamard fold
# ---------------------------------------------------------------------------

def test_svd_factor_eckart_young_and_balanced_split():
    rng = np.random.default_rng(10)
    w = rng.standard_normal((40, 24))
    sv = np.linalg.svd(w, compute_uv=False)
    for r in (1, 5, 24):
        A, B = O.svd_factor(w, r)
        assert A.shape == (40, r) and B.shape == (r, 24)
        err = np.linalg.norm(w - A @ B) ** 2
        assert abs(err - np.sum(sv[r:] ** 2)) < 1e-9
        # A = U_r sqrt(S_r), B = sqrt(S_r) V_r^T  =>  A^T A = B B^T = diag(S_r)
        np.testing.assert_allclose(A.T @ A, np.diag(sv[:r]), atol=1e-10)
        np.testing.assert_allclose(B @ B.T, np.diag(sv[:r]), atol=1e-10)


def test_hadamard_matches_scipy_and_is_orthogonal():
    for r in (1, 2, 8, 16, 128, 256):
        R = O.hadamard(r)
        np.testing.assert_array_equal(R, scipy.linalg.hadamard(r) / math.sqrt(r))
        if r in (1, 16, 256):  # 1/sqrt(r) is a power of two: R R^T = I exactly
            np.testing.assert_array_equal(R @ R.T, np.eye(r))
        else:
            np.testing.assert_allclose(R @ R.T, np.eye(r), atol=1e-15)
    R = O.hadamard(256)
    assert set(np.unique(R)) == {-1 / 16, 1 / 16}


def test_hadamard_fold_preserves_product():
    rng = np.random.default_rng(11)
    A = rng.standard_normal((64, 16))
    B = rng.standard_normal((16, 32))
    R = O.hadamard(16)
    np.testing.assert_allclose((A @ R) @ (R.T @ B), A @ B, atol=1e-12)


# ---------------------------------------------------------------------------
# int4 quantisation
# ---------------------------------------------------------------------------

def _read_int4_golden():
    cases, cur = [], {}
    with open(os.path.join(GOLDEN, "int4_pack.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            cur[key] = vals
            if key == "bytes":
                cases.append(cur)
                cur = {}
    return cases


def test_int4_golden_codes_and_bytes():
    cases = _read_int4_golden()
    assert len(cases) == 5
    for c in cases:
        h = np.array([float(v) for v in c["h"]], dtype=np.float32)[None]
        codes, scale = O.quantize_int4(h)
        assert scale.view(np.uint16)[0] == int(c["scale"][0], 16)
        np.testing.assert_array_equal(codes[0], [int(v) for v in c["codes"]])
        packed = O.pack_int4(codes)
        np.testing.assert_array_equal(packed[0], [int(v, 16) for v in c["bytes"]])
        np.testing.assert_array_equal(O.unpack_int4(packed), codes)


def test_int4_properties():
    rng = np.random.default_rng(12)
    h = (rng.standard_normal((64, 256)) * rng.uniform(0.01, 30, (64, 1))).astype(np.float32)
    codes, scale = O.quantize_int4(h)
    assert codes.min() >= -7 and codes.max() <= 7
    sf = scale.astype(np.float64)
    deq = O.dequant_int4(O.pack_int4(codes), scale)
    # dequantised value is the exact product (<= 4 + 11 significant bits)
    np.testing.assert_array_equal(deq, codes.astype(np.float64) * sf[:, None])
    np.testing.assert_array_equal(deq.astype(np.float32).astype(np.float64), deq)
    # rounding error bounded by half a step where nothing is clamped
    inside = np.abs(h / sf[:, None]) <= 7
    assert np.all(np.abs(h - deq)[inside] <= sf[:, None].repeat(256, 1)[inside] / 2 * (1 + 1e-6))
    # the largest-magnitude element maps to +-7 (scale rounding never pushes it below 6.5)
    idx = np.argmax(np.abs(h), axis=1)
    assert np.all(np.abs(codes[np.arange(64), idx]) == 7)


def test_int4_integer_inputs_round_trip():
    rng = np.random.default_rng(13)
    codes_in = rng.integers(-7, 8, (32, 64)).astype(np.float32)
    codes_in[:, 0] = 7  # amax 7 -> scale exactly 1
    codes, scale = O.quantize_int4(codes_in)
    assert np.all(scale == 1.0)
    np.testing.assert_array_equal(codes, codes_in.astype(np.int8))
    np.testing.assert_array_equal(O.dequant_int4(O.pack_int4(codes), scale), codes_in)


def test_int4_huge_and_zero_rows():
    h = np.zeros((2, 8), np.float32)
    h[1] = 1e6
    codes, scale = O.quantize_int4(h)
    assert scale[0] == 0 and np.all(codes[0] == 0)
    assert scale[1] == np.float16(65504.0) and np.all(codes[1] == 7)


def test_projected_latents_brute_force_tiny():
    # scalar loops with exact summation: h[b, t, g, m] = sum_e x[b, t, e] A_g[e, m]
    rng = np.random.default_rng(31)
    B, T, d, n_g, r = 2, 3, 5, 2, 4
    x = rng.standard_normal((B, T, d))
    a = rng.standard_normal((n_g, d, r))
    h = O.project_latents(x, a)
    assert h.shape == (B, T, n_g, r)
    for b in range(B):
        for t in range(T):
            for g in range(n_g):
                for m in range(r):
                    want = math.fsum(x[b, t, e] * a[g, e, m] for e in range(d))
                    assert abs(h[b, t, g, m] - want) < 1e-12


def test_projected_latents_rebuild_the_keys_at_full_rank():
    # the SVD rewrite: (x A_g) B_g = x W_g when the factors are exact (full rank r = s*d_h), so
    # each group's latents rebuild exactly that group's block of keys x W
    B, T, d, n, s, d_h = 2, 6, 16, 4, 2, 4
    x, wk, _, _ = _mha_setup(32, B, T, d, n, s, d_h)
    n_g, r = n // s, s * d_h
    Ak, Bk = _group_factors(wk, n_g, s, d_h, r)
    h = O.project_latents(x, Ak)
    for g in range(n_g):
        np.testing.assert_allclose(h[:, :, g, :] @ Bk[g], x @ wk[:, g * s * d_h:(g + 1) * s * d_h], atol=1e-11)


# ---------------------------------------------------------------------------
# Hybrid cache: dense sink + window next to the latent middle
# ---------------------------------------------------------------------------

def _hybrid_split(x, wk, wv, Ak, Av, n, d_h, T, S, W, rope, theta=10000.0):
    """Tokens [0, S) and [T - W, T) as a dense cache (keys rotated at their positions when rope),
    tokens [S, T - W) as latents at positions S .. T - W - 1."""
    B = x.shape[0]
    dense_idx = list(range(S)) + list(range(T - W, T))
    D = len(dense_idx)
    dk = np.zeros((B, D, n, d_h))
    dv = np.zeros((B, D, n, d_h))
    for b in range(B):
        for i in range(n):
            K = x[b, dense_idx] @ wk[:, i * d_h:(i + 1) * d_h]
            if rope:
                K = O.rope_rotate(K, np.array(dense_idx, np.float64), theta)
            dk[b, :, i] = K
            dv[b, :, i] = x[b, dense_idx] @ wv[:, i * d_h:(i + 1) * d_h]
    mid = x[:, S:T - W]
    hk = np.einsum("btd,gdr->btgr", mid, Ak)
    hv = np.einsum("btd,gdr->btgr", mid, Av)
    pos = np.tile(np.arange(S, T - W), (B, 1))
    return dk, dv, hk, hv, pos


@pytest.mark.parametrize("mode", ["rope", "absorbed"])
def test_hybrid_at_full_rank_equals_uncompressed_mha_over_all_tokens(mode):
    # exact factors: sink + latent middle + window must be plain attention over every token
    B, T, d, n, s, d_h = 2, 14, 32, 4, 2, 4
    x, wk, wv, q = _mha_setup(41, B, T, d, n, s, d_h)
    n_g, r = n // s, s * d_h
    Ak, Bk = _group_factors(wk, n_g, s, d_h, r)
    Av, Bv = _group_factors(wv, n_g, s, d_h, r)
    S, W = 2, 3
    dk, dv, hk, hv, pos = _hybrid_split(x, wk, wv, Ak, Av, n, d_h, T, S, W, mode == "rope")
    qp = [T - 1] * B
    o_lat, o_den, lse = O.decode_hybrid(q, hk, hv, Bk, [T - S - W] * B, s, dk, dv, [S + W] * B, mode=mode,
                                        positions=pos, q_pos=qp)
    a, lse_ref = O.mha_decode(q, x, wk, wv, [T] * B, rope=(mode == "rope"), q_pos=qp)
    for b in range(B):
        for i in range(n):
            g, j = i // s, i % s
            np.testing.assert_allclose(o_lat[b, i] @ Bv[g][:, j * d_h:(j + 1) * d_h] + o_den[b, i], a[b, i],
                                       atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-11)


@pytest.mark.parametrize("mode", ["rope", "absorbed"])
def test_hybrid_without_dense_tokens_is_the_latent_decode(mode):
    q, hk, hv, bk = _tiny(seed=42, B=2, T=7, n=4, s=2, d_h=4, r=4, r_v=3)
    dk = np.zeros((2, 0, 4, 4))
    qp = [6, 6]
    o_lat, o_den, lse = O.decode_hybrid(q, hk, hv, bk, [7, 5], 2, dk, dk, [0, 0], mode=mode, q_pos=qp)
    o, lse_ref = O.decode(q, hk, hv, bk, [7, 5], 2, mode=mode, q_pos=qp)
    np.testing.assert_allclose(o_lat, o, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-13)
    assert np.all(o_den == 0)


def test_hybrid_with_an_empty_middle_is_dense_softmax_attention():
    import scipy.special
    rng = np.random.default_rng(43)
    B, n, d_h, D = 1, 2, 4, 5
    q = rng.standard_normal((B, n, d_h))
    dk = rng.standard_normal((B, D, n, d_h))
    dv = rng.standard_normal((B, D, n, d_h))
    hk = np.zeros((B, 1, 1, 3))
    bk = np.zeros((1, 3, 2 * d_h))
    o_lat, o_den, lse = O.decode_hybrid(q, hk, hk, bk, [0], 2, dk, dv, [D], mode="rope", q_pos=[0])
    for i in range(n):
        sc = dk[0, :, i] @ q[0, i] / math.sqrt(d_h)   # q_pos 0: the query is not rotated
        np.testing.assert_allclose(o_den[0, i], scipy.special.softmax(sc) @ dv[0, :, i], atol=1e-13)
        assert abs(lse[0, i] - scipy.special.logsumexp(sc)) < 1e-13
    assert np.all(o_lat == 0)


# ---------------------------------------------------------------------------
# Page-factorised cache ([Puzzle] section 3.3)
# ---------------------------------------------------------------------------

def test_page_factors_are_the_truncated_svd_and_match_the_gram_route():
    rng = np.random.default_rng(61)
    x = rng.standard_normal((8, 20)) * np.exp(-np.arange(20) / 6.0)[None, :]
    sv = np.linalg.svd(x, compute_uv=False)
    for r in (1, 3, 8):
        L, R = O.factor_page(x, r)
        Lg, Rg = O.factor_page_gram(x, r)
        # L has orthonormal columns, and the product is the same rank-r approximation both ways
        np.testing.assert_allclose(L.T @ L, np.eye(r), atol=1e-13)
        np.testing.assert_allclose(Lg.T @ Lg, np.eye(r), atol=1e-12)
        np.testing.assert_allclose(L @ R, Lg @ Rg, atol=1e-11)
        # Eckart-Young: the residual is the discarded singular values
        assert abs(np.sum((x - L @ R) ** 2) - np.sum(sv[r:] ** 2)) < 1e-10
    L, R = O.factor_page(x, 8)                      # full page rank: exact
    np.testing.assert_allclose(L @ R, x, atol=1e-12)


def _pages_of(keys, vals, P, r):
    """Factorise [T][n][d] keys and values page by page (T a multiple of P): [n_pages][n][...] factors."""
    T, n, _ = keys.shape
    lk, rk, lv, rv = [], [], [], []
    for p in range(T // P):
        f = [O.factor_page(keys[p * P:(p + 1) * P, i], r) for i in range(n)]
        g = [O.factor_page(vals[p * P:(p + 1) * P, i], r) for i in range(n)]
        lk.append([a for a, _ in f]); rk.append([b for _, b in f])
        lv.append([a for a, _ in g]); rv.append([b for _, b in g])
    return np.array(lk), np.array(rk), np.array(lv), np.array(rv)


@pytest.mark.parametrize("mode", ["rope", "absorbed"])
def test_paged_decode_at_full_page_rank_is_softmax_attention_over_every_token(mode):
    # exact page factors: factorised pages + dense tokens must be plain attention over all of them
    rng = np.random.default_rng(62)
    B, n, d_h, P, npg, D = 2, 3, 8, 4, 3, 5
    keys = rng.standard_normal((B, npg * P + D, n, d_h))
    vals = rng.standard_normal((B, npg * P + D, n, d_h))
    q = rng.standard_normal((B, n, d_h))
    f = [_pages_of(keys[b, :npg * P], vals[b, :npg * P], P, P) for b in range(B)]
    lk, rk, lv, rv = (np.array([fb[k] for fb in f]) for k in range(4))
    qp = [0, 0]        # q_pos 0: the rotation is the identity on the RoPE path
    o_pg, o_den, lse = O.decode_paged(q, lk, rk, lv, rv, [npg, 2], keys[:, npg * P:], vals[:, npg * P:], [D, 3],
                                      mode=mode, q_pos=qp)
    for b, (used_pages, used_dense) in enumerate([(npg, D), (2, 3)]):
        idx = list(range(used_pages * P)) + [npg * P + t for t in range(used_dense)]
        for i in range(n):
            sc = keys[b, idx, i] @ q[b, i] / math.sqrt(d_h)
            p = scipy.special.softmax(sc)
            np.testing.assert_allclose(o_pg[b, i] + o_den[b, i], p @ vals[b, idx, i], atol=1e-12)
            np.testing.assert_allclose(o_den[b, i], p[used_pages * P:] @ vals[b, idx[used_pages * P:], i],
                                       atol=1e-12)
            assert abs(lse[b, i] - scipy.special.logsumexp(sc)) < 1e-12


def test_paged_decode_rotates_the_query_like_the_dense_tokens():
    # RoPE path: scores use q rotated at q_pos against keys as stored (already rotated)
    rng = np.random.default_rng(63)
    B, n, d_h, P = 1, 2, 4, 2
    keys = rng.standard_normal((B, 2 * P, n, d_h))
    vals = rng.standard_normal((B, 2 * P, n, d_h))
    q = rng.standard_normal((B, n, d_h))
    lk, rk, lv, rv = (a[None] for a in _pages_of(keys[0], vals[0], P, P))
    o_pg, _, lse = O.decode_paged(q, lk, rk, lv, rv, [2], keys[:, :0], vals[:, :0], [0], mode="rope",
                                  q_pos=[5])
    for i in range(n):
        # the rotation by complex multiplication of the rotate-half pairs (k, k + d_h/2)
        w = O.rope_inv_freq(d_h, 10000.0)
        z = (q[0, i, :2] + 1j * q[0, i, 2:]) * np.exp(1j * 5 * w)
        qr = np.concatenate([z.real, z.imag])
        sc = keys[0, :, i] @ qr / math.sqrt(d_h)
        np.testing.assert_allclose(o_pg[0, i], scipy.special.softmax(sc) @ vals[0, :, i], atol=1e-12)
        assert abs(lse[0, i] - scipy.special.logsumexp(sc)) < 1e-12


def test_paged_decode_brute_force_low_rank():
    # rank below the page size: scalar loops over the printed formula, s_p = (q R^T) L^T / sqrt(d)
    rng = np.random.default_rng(64)
    B, n, d_h, P, r, npg, D = 1, 2, 4, 3, 2, 2, 2
    lk = rng.standard_normal((B, npg, n, P, r))
    rk = rng.standard_normal((B, npg, n, r, d_h))
    lv = rng.standard_normal((B, npg, n, P, r))
    rv = rng.standard_normal((B, npg, n, r, d_h))
    dk = rng.standard_normal((B, D, n, d_h))
    dv = rng.standard_normal((B, D, n, d_h))
    q = rng.standard_normal((B, n, d_h))
    o_pg, o_den, lse = O.decode_paged(q, lk, rk, lv, rv, [npg], dk, dv, [D], mode="absorbed")
    for i in range(n):
        scores, vecs = [], []
        for p in range(npg):
            u = [math.fsum(q[0, i, e] * rk[0, p, i, j, e] for e in range(d_h)) for j in range(r)]
            for t in range(P):
                scores.append(math.fsum(u[j] * lk[0, p, i, t, j] for j in range(r)) / math.sqrt(d_h))
                vecs.append([math.fsum(lv[0, p, i, t, j] * rv[0, p, i, j, e] for j in range(r)) for e in range(d_h)])
        for t in range(D):
            scores.append(math.fsum(q[0, i, e] * dk[0, t, i, e] for e in range(d_h)) / math.sqrt(d_h))
            vecs.append(list(dv[0, t, i]))
        m = max(scores)
        ex = [math.exp(x - m) for x in scores]
        l = math.fsum(ex)
        full = [math.fsum(ex[t] * vecs[t][e] for t in range(len(ex))) / l for e in range(d_h)]
        dense = [math.fsum(ex[t] * vecs[t][e] for t in range(npg * P, len(ex))) / l for e in range(d_h)]
        np.testing.assert_allclose(o_pg[0, i] + o_den[0, i], full, atol=1e-12)
        np.testing.assert_allclose(o_den[0, i], dense, atol=1e-12)
        assert abs(lse[0, i] - (m + math.log(l))) < 1e-12


def test_paged_decode_empty_row():
    z5 = np.zeros((1, 1, 1, 2, 1))
    zr = np.zeros((1, 1, 1, 1, 4))
    o_pg, o_den, lse = O.decode_paged(np.ones((1, 1, 4)), z5, zr, z5, zr, [0], np.zeros((1, 0, 1, 4)),
                                      np.zeros((1, 0, 1, 4)), [0], mode="absorbed")
    assert np.all(o_pg == 0) and np.all(o_den == 0) and lse[0, 0] == -math.inf


# ---------------------------------------------------------------------------
# ALiBi on the absorbed path
# ---------------------------------------------------------------------------

def test_alibi_slopes_closed_form():
    # the ALiBi paper's sequence for 8 heads is 1/2, 1/4, ..., 1/256; for 16 heads it starts at 2^-0.5
    np.testing.assert_array_equal(O.alibi_slopes(8), [2.0 ** -k for k in range(1, 9)])
    np.testing.assert_allclose(O.alibi_slopes(16)[:2], [2 ** -0.5, 0.5], rtol=1e-15)
    assert O.alibi_bias(0.25, [0, 3, 7], 7).tolist() == [-1.75, -1.0, 0.0]


def test_absorbed_alibi_at_full_rank_equals_mha_with_alibi():
    # key fusion stays exact under a bias that never touches the keys
    B, T, d, n, s, d_h = 2, 10, 32, 4, 2, 4
    x, wk, wv, q = _mha_setup(51, B, T, d, n, s, d_h)
    n_g, r = n // s, s * d_h
    Ak, Bk = _group_factors(wk, n_g, s, d_h, r)
    Av, Bv = _group_factors(wv, n_g, s, d_h, r)
    hk = np.einsum("btd,gdr->btgr", x, Ak)
    hv = np.einsum("btd,gdr->btgr", x, Av)
    pos = np.stack([np.arange(T) * 3 + 5, np.arange(T)[::-1] + 2])
    o, lse = O.decode(q, hk, hv, Bk, [T, T - 4], s, mode="absorbed", positions=pos, q_pos=[40, 30], alibi=True)
    a, lse_ref = O.mha_decode(q, x, wk, wv, [T, T - 4], rope=False, positions=pos, q_pos=[40, 30], alibi=True)
    for b in range(B):
        for i in range(n):
            g, j = i // s, i % s
            np.testing.assert_allclose(o[b, i] @ Bv[g][:, j * d_h:(j + 1) * d_h], a[b, i], atol=1e-11)
    np.testing.assert_allclose(lse, lse_ref, atol=1e-11)


def test_alibi_depends_only_on_distance_and_changes_the_result():
    q, hk, hv, bk = _tiny(seed=52, B=1, T=8, n=4, s=2, d_h=4, r=4, r_v=3)
    pos = np.arange(8)[None]
    o1, l1 = O.decode(q, hk, hv, bk, [8], 2, mode="absorbed", positions=pos, q_pos=[9], alibi=True)
    o2, l2 = O.decode(q, hk, hv, bk, [8], 2, mode="absorbed", positions=pos + 100, q_pos=[109], alibi=True)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)
    o0, _ = O.decode(q, hk, hv, bk, [8], 2, mode="absorbed")
    assert np.abs(o1 - o0).max() > 1e-3
