"""CPU checks of the seeded workload generator (shapes, spectrum, determinism)."""
import math

import numpy as np
import pytest

from oracle import palu_oracle as O
from synthetic import gen


def test_configs_follow_llama2_7b_group_shapes():
    for c in (gen.ROPE_FP16, gen.ROPE_BF16, gen.ABSORBED_FP16, gen.ROPE_INT4):
        assert (c.n_heads, c.head_dim, c.hidden, c.group_size, c.rank) == (32, 128, 4096, 4, 256)
        # G-LRD concatenation of s = 4 heads: a 4096 x 512 matrix (Palu notes, "补充细节")
        assert (c.hidden, c.head_dim * c.group_size) == (4096, 512)
    c1 = gen.TINY_FP32
    assert (c1.n_heads, c1.head_dim, c1.hidden, c1.n_groups, c1.rank, c1.T) == (8, 64, 512, 2, 128, 512)


def test_tiny_workload_deterministic_and_consistent():
    cfg = gen.TINY_FP32
    a = gen.make_inputs(cfg, with_x=True)
    b = gen.make_inputs(cfg, with_x=True)
    np.testing.assert_array_equal(a["hk"], b["hk"])
    np.testing.assert_array_equal(a["q"], b["q"])
    assert a["hk"].shape == (1, 512, 2, 128) and a["bk"].shape == (2, 128, 256)
    # latents are x A (exact draw)
    np.testing.assert_allclose(a["hk"][0, :, 1], a["x"][0] @ a["ak"][1], rtol=1e-4, atol=1e-4)
    # spectrum: W_k singular values are exp(-i/64)
    wk, _ = gen.weights(cfg)
    sv = np.linalg.svd(wk, compute_uv=False)
    np.testing.assert_allclose(sv, np.exp(-np.arange(512) / 64.0), rtol=1e-9, atol=1e-12)
    # factors reproduce each group's truncated SVD (Eckart-Young optimum)
    g = 1
    wg = wk[:, g * 256:(g + 1) * 256]
    ref = np.linalg.svd(wg, compute_uv=False)
    err = np.linalg.norm(wg - a["ak"][g] @ a["bk"][g]) ** 2
    assert abs(err - np.sum(ref[128:] ** 2)) < 1e-9


def test_hadamard_fold_in_generator_preserves_weights():
    cfg = gen.TINY_FP32.with_(hadamard=True)
    a = gen.make_inputs(cfg)
    plain = gen.make_inputs(gen.TINY_FP32)
    for g in range(cfg.n_groups):
        np.testing.assert_allclose(a["ak"][g] @ a["bk"][g], plain["ak"][g] @ plain["bk"][g], atol=1e-12)
    R = O.hadamard(cfg.rank)
    np.testing.assert_allclose(a["bk"][0], R.T @ plain["bk"][0], atol=1e-13)


def test_equivalent_latent_draw_matches_covariance():
    # The large-workload draw must have the covariance of x A: A^T A = diag(S_r).
    cfg = gen.TINY_FP32.with_(T=20000)
    a = gen.make_inputs(cfg, exact_x=False)
    h = a["hk"][0, :, 0, :].astype(np.float64)
    cov = h.T @ h / h.shape[0]
    np.testing.assert_allclose(np.diag(cov), a["sk"][0], rtol=0.05)
    off = cov - np.diag(np.diag(cov))
    assert np.max(np.abs(off)) < 0.05 * a["sk"][0][0]


def test_storage_round_bf16_is_round_to_nearest_even():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -2.5], np.float32)
    t = gen.storage_round(x, "bf16").float().numpy()
    np.testing.assert_array_equal(t, [1.0, 1.0, 1.0 + 2 ** -6, -2.5])
