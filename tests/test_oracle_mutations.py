"""Plant plausible mistakes in the oracle (CPU only) and check the pins catch each.

Every mutation below is a realistic slip: wrong rotation sign, wrong pairing,
wrong frequency schedule, wrong head-to-group map, wrong score scale, wrong
rounding mode, swapped nibbles, the wrong factor of a page. The pin tests must fail on each one.
"""
import math

import numpy as np
import pytest

from oracle import palu_oracle as O
from tests import test_oracle_pins as P


def _rope_wrong_sign(x, pos, theta):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, np.float64)[..., None] * O.rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :d // 2], x[..., d // 2:]
    return np.concatenate([a * c + b * s, b * c - a * s], axis=-1)


def _rope_interleaved(x, pos, theta):
    x = np.asarray(x, np.float64)
    d = x.shape[-1]
    ang = np.asarray(pos, np.float64)[..., None] * O.rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., 0::2], x[..., 1::2]
    out = np.empty(np.broadcast_shapes(x.shape, ang.shape[:-1] + (d,)))
    out[..., 0::2] = a * c - b * s
    out[..., 1::2] = b * c + a * s
    return out


def _inv_freq_half(head_dim, theta):
    k = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -k / head_dim)


def _group_of_modulo(head, group_size):
    # heads strided across groups instead of consecutive
    return head % group_size, head // group_size


def _rope_head_scale_r(q_i, hk_bg, hv_bg, bk_g, j, pos, qp, theta):
    d_h = q_i.shape[-1]
    r = hk_bg.shape[-1]
    K = hk_bg @ bk_g[:, j * d_h:(j + 1) * d_h]
    s = (O.rope_rotate(K, pos, theta) @ O.rope_rotate(q_i, qp, theta)) / math.sqrt(r)
    return O.softmax_attend(s, hv_bg)


def _absorbed_transposed(q_i, hk_bg, hv_bg, bk_g, j, bias=None):
    # uses the head's row block of B^T instead of its column block of B
    d_h = q_i.shape[-1]
    blk = bk_g[:, j * d_h:(j + 1) * d_h]
    q_lat = np.zeros(bk_g.shape[0])
    q_lat[:d_h] = blk[:d_h, :] @ q_i
    return O.softmax_attend(hk_bg @ q_lat / math.sqrt(d_h), hv_bg)


def _quantize_half_away(h):
    h = np.asarray(h, np.float32)
    amax = np.max(np.abs(h), axis=-1)
    scale = np.minimum(amax / np.float32(7), np.float32(O.FP16_MAX)).astype(np.float16)
    sf = scale.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = h / sf[..., None]
    codes = np.clip(np.sign(r) * np.floor(np.abs(r) + 0.5), -7, 7)
    return np.where((sf == 0)[..., None], 0, codes).astype(np.int8), scale


def _pack_swapped(codes):
    c = np.asarray(codes, np.int16) & 0xF
    return (c[..., 1::2] | (c[..., 0::2] << 4)).astype(np.uint8)


def _qpos_off_by_one(positions, q_pos, b, T):
    if q_pos is not None:
        return float(q_pos[b])
    return float(T) if positions is None else float(positions[b][T - 1]) + 1


def _softmax_no_norm(scores, values):
    scores = np.asarray(scores, np.float64)
    if scores.size == 0:
        return np.zeros(values.shape[-1]), -math.inf
    m = scores.max()
    e = np.exp(scores - m)
    return e @ values, m + math.log(e.sum())


def _fuse_wrong_head_block(bv, wo, group_size):
    # every head of a group takes the group's first column block of B_v
    bv, wo = np.asarray(bv, np.float64), np.asarray(wo, np.float64)
    n_g, r_v, cols = bv.shape
    d_h = cols // group_size
    return np.concatenate([bv[i // group_size][:, :d_h] @ wo[i * d_h:(i + 1) * d_h]
                           for i in range(n_g * group_size)], axis=0)


def _project_rows_of_next_head(o, w_fused):
    # off-by-one head: head i meets the rows of head (i + 1) % n
    o, w = np.asarray(o, np.float64), np.asarray(w_fused, np.float64)
    B, n, r_v = o.shape
    y = np.zeros((B, w.shape[1]))
    for b in range(B):
        for i in range(n):
            k = (i + 1) % n
            y[b] += o[b, i] @ w[k * r_v:(k + 1) * r_v]
    return y


def _project_latents_first_group(x, a):
    # every group's latents taken with group 0's down-projection
    x, a = np.asarray(x, np.float64), np.asarray(a, np.float64)
    h = np.einsum("btd,dr->btr", x, a[0])
    return np.repeat(h[:, :, None, :], a.shape[0], axis=2)


def _decode_hybrid_separate_softmax(q, hk, hv, bk, seq_lens, group_size, dense_k, dense_v, n_dense, **kw):
    # each segment normalised on its own: the merge of the two partial softmaxes is left out
    o_lat, lse_mid = O.decode(q, hk, hv, bk, seq_lens, group_size, mode=kw.get("mode", "rope"),
                              theta=kw.get("theta", 10000.0), positions=kw.get("positions"), q_pos=kw.get("q_pos"))
    B, n, d_h = q.shape
    o_den = np.zeros((B, n, d_h))
    lse = np.array(lse_mid)
    for b in range(B):
        D = int(n_dense[b])
        for i in range(n):
            qi = np.asarray(q[b, i], np.float64)
            if kw.get("mode", "rope") == "rope":
                qi = O.rope_rotate(qi, float(kw["q_pos"][b]), kw.get("theta", 10000.0))
            if D:
                sc = np.asarray(dense_k[b, :D, i], np.float64) @ qi / math.sqrt(d_h)
                o_den[b, i], _ = O.softmax_attend(sc, np.asarray(dense_v[b, :D, i], np.float64))
    return o_lat, o_den, lse


def _alibi_bias_wrong_sign(slope, pos, qp):
    # rewards distance instead of penalising it
    return slope * (float(qp) - np.asarray(pos, np.float64))


_decode_paged = O.decode_paged


def _decode_paged_values_from_key_factors(q, lk, rk, lv, rv, *a, **kw):
    # reads every page's values through its key factors
    return _decode_paged(q, lk, rk, lk, rk, *a, **kw)


def _factor_page_without_singular_values(x, r):
    # R = W_r^T: the singular values dropped from the right factor
    u, s, wt = np.linalg.svd(np.asarray(x, np.float64), full_matrices=False)
    return u[:, :r], wt[:r]


ALL_PINS = [getattr(P, n) for n in dir(P) if n.startswith("test_")]

MUTATIONS = {
    "rope_wrong_sign": ("rope_rotate", _rope_wrong_sign),
    "rope_interleaved_pairs": ("rope_rotate", _rope_interleaved),
    "rope_frequency_schedule": ("rope_inv_freq", _inv_freq_half),
    "head_group_map": ("_group_of", _group_of_modulo),
    "score_scale_sqrt_r": ("decode_rope_head", _rope_head_scale_r),
    "absorbed_transposed_block": ("decode_absorbed_head", _absorbed_transposed),
    "int4_round_half_away": ("quantize_int4", _quantize_half_away),
    "int4_nibble_order": ("pack_int4", _pack_swapped),
    "query_position_default": ("_query_position", _qpos_off_by_one),
    "softmax_unnormalised": ("softmax_attend", _softmax_no_norm),
    "fuse_wrong_head_block": ("fuse_value_output", _fuse_wrong_head_block),
    "project_rows_of_next_head": ("project_fused", _project_rows_of_next_head),
    "latents_first_group_only": ("project_latents", _project_latents_first_group),
    "hybrid_segments_normalised_apart": ("decode_hybrid", _decode_hybrid_separate_softmax),
    "alibi_bias_wrong_sign": ("alibi_bias", _alibi_bias_wrong_sign),
    "paged_values_from_key_factors": ("decode_paged", _decode_paged_values_from_key_factors),
    "page_factor_without_singular_values": ("factor_page", _factor_page_without_singular_values),
}


def _run_pins(pins):
    failed = []
    for fn in pins:
        params = getattr(fn, "pytestmark", [])
        arglists = [{}]
        for m in params:
            if m.name == "parametrize":
                name, vals = m.args[0], m.args[1]
                arglists = [{name: v} for v in vals]
        for kw in arglists:
            try:
                fn(**kw)
            except (AssertionError, ValueError, IndexError):
                failed.append(fn.__name__)
                break
    return failed


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, monkeypatch):
    attr, mutant = MUTATIONS[name]
    monkeypatch.setattr(O, attr, mutant)
    failed = _run_pins(ALL_PINS)
    assert failed, f"no pin caught the planted mistake {name}"


def test_unmutated_oracle_passes_every_pin():
    assert _run_pins(ALL_PINS) == []
