"""CPU checks of the two group reshapes the library runs (with the float64 oracle on both sides):

* packed groups: G-LRD groups of s = 1 or 2 heads with r = 64 s ranks decoded as groups of four heads at
  256 ranks, whose B_k is block-diagonal and whose latents are the neighbouring groups' rows side by side;
  each head's output is its own group's slice of the 256 latent columns;
* split groups (absorbed path): a group of 8 or 32 heads at rank 256 decoded as groups of four heads over
  the same latents, each with its column block of B_k.

Both are exact rewrites ("Palu" notes, method section: G-LRD rebuild per group; key-fusion paragraph for the
absorbed query): these tests check that, so that the GPU tests' comparison with the oracle's original shape
is a comparison with the same mathematics.
"""
import numpy as np
import pytest

from oracle import palu_oracle as O


def _draw(seed, B, T, n, s, d_h, r):
    rng = np.random.default_rng(seed)
    n_g = n // s
    return (rng.standard_normal((B, n, d_h)), rng.standard_normal((B, T, n_g, r)),
            rng.standard_normal((B, T, n_g, r)), rng.standard_normal((n_g, r, s * d_h)))


def _packed(hk, hv, bk, s, d_h):
    """Four-head groups: latents of 4 / s neighbouring groups side by side, block-diagonal B_k."""
    B, T, n_g, r = hk.shape
    pack = 4 // s
    hk4 = hk.reshape(B, T, n_g // pack, pack * r)
    hv4 = hv.reshape(B, T, n_g // pack, pack * r)
    bk4 = np.zeros((n_g // pack, pack * r, 4 * d_h))
    for g4 in range(n_g // pack):
        for jg in range(pack):
            bk4[g4, jg * r:(jg + 1) * r, jg * s * d_h:(jg + 1) * s * d_h] = bk[g4 * pack + jg]
    return hk4, hv4, bk4


@pytest.mark.parametrize("mode", ["rope", "absorbed"])
@pytest.mark.parametrize("s", [1, 2])
def test_packed_groups_reproduce_the_source_groups(mode, s):
    B, T, n, d_h = 2, 9, 8, 4
    r = 2 * s                                   # r = (64 / 32) s at the library's scale, kept small here
    q, hk, hv, bk = _draw(70 + s, B, T, n, s, d_h, r)
    pos = np.stack([np.random.default_rng(5).permutation(40)[:T] for _ in range(B)])
    kw = dict(mode=mode, positions=pos if mode == "rope" else None, q_pos=[33, 7] if mode == "rope" else None)
    o_src, lse_src = O.decode(q, hk, hv, bk, [T, 5], s, **kw)
    hk4, hv4, bk4 = _packed(hk, hv, bk, s, d_h)
    o_pk, lse_pk = O.decode(q, hk4, hv4, bk4, [T, 5], 4, **kw)
    np.testing.assert_allclose(lse_pk, lse_src, atol=1e-12)
    for i in range(n):
        jg = (i % 4) // s                       # the head's own group within its four-head group
        np.testing.assert_allclose(o_pk[:, i, jg * r:(jg + 1) * r], o_src[:, i], atol=1e-12)


@pytest.mark.parametrize("s", [8, 32])
def test_split_groups_reproduce_the_source_groups(s):
    B, T, d_h, r = 2, 7, 4, 5
    n = s                                       # one source group
    q, hk, hv, bk = _draw(80 + s, B, T, n, s, d_h, r)
    o_src, lse_src = O.decode(q, hk, hv, bk, [T, 3], s, mode="absorbed")
    split = s // 4
    hk_s = np.repeat(hk, split, axis=2)         # every kernel group reads its source group's latents
    hv_s = np.repeat(hv, split, axis=2)
    bk_s = np.stack([bk[g // split][:, (g % split) * 4 * d_h:(g % split + 1) * 4 * d_h]
                     for g in range(bk.shape[0] * split)])
    o_sp, lse_sp = O.decode(q, hk_s, hv_s, bk_s, [T, 3], 4, mode="absorbed")
    np.testing.assert_allclose(o_sp, o_src, atol=1e-12)
    np.testing.assert_allclose(lse_sp, lse_src, atol=1e-12)
