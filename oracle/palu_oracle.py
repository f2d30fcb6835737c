"""Float64 CPU oracle for Palu-style G-LRD decode attention over cached latents.

TEST INFRASTRUCTURE ONLY. This module exists to check the CUDA path. Only the
test suite, the smoke check in ``__graft_entry__`` and the benchmark's CPU
baseline / reference arm may import it. The library never imports it and has
no CPU fallback.

It is deliberately plain: NumPy float64, one (batch, head) at a time, every step
in the order the pages state it, no blocking, fusion or reordering. Library
primitives used as steps: ``numpy`` matmul, ``exp``/``log``, ``rint``, and the
LAPACK SVD.

Sources (page title, section):
  [Palu]    "Palu: KV-Cache Compression With Low-Rank Projection" (paper notes)
  [Puzzle]  "PuzzleKV: 基于页面的低秩分解用于KV缓存压缩" (translation)
  [Shard]   "Shard - 实现10倍KV缓存压缩" (blog translation)

Readings taken where the pages are silent (each is listed with its reason in the
design notes):
  * row-vector convention h = x A (the method section writes both h = Ax and
    h = xA; A in R^{d x r} fixes h = xA);
  * head i belongs to group i // s and is column block i % s of B_g;
  * score scale 1/sqrt(d_h) on both paths;
  * RoPE: rotate-half pairing (k, k + d_h/2) as [Shard] section 5 states for
    Llama, inverse frequencies theta^(-2k/d_h) (the RoFormer schedule; the
    [Palu] notes only cite RoFormer);
  * the query arrives unrotated and is rotated at q_pos, which defaults to the
    position of the last cached token; no mask (all cached tokens attend);
  * the output stays in latent space, o_i = p_i H_v (B_v is fused into W_o);
  * int4: per-token, per-group symmetric codes in [-7, 7], scale
    fp16_rn(min(amax/7, 65504)) with amax and the division in IEEE fp32, codes
    rint-half-even(h / scale) clamped to [-7, 7], zero codes when the scale is 0;
    element 2j in the low nibble, 2j+1 in the high nibble (two's complement);
  * an empty sequence yields o = 0 and lse = -inf.

The per-page factorised decode follows [Puzzle] section 3.3 (decode_paged, factor_page and
factor_page_gram); its readings are given in its docstring.

Every function below is pinned by a CPU test against something other than
itself (closed forms, the pages' worked numbers, library routines, brute force,
the identities the pages derive); none is "parity unpinned".
"""
from __future__ import annotations

import math

import numpy as np


# ---------------------------------------------------------------------------
# RoPE
# ---------------------------------------------------------------------------

def rope_inv_freq(head_dim: int, theta: float) -> np.ndarray:
    """omega_k = theta^(-2k/d_h), k = 0 .. d_h/2-1 (RoFormer schedule cited by
    [Palu] "方法细节", RoPE paragraph)."""
    k = np.arange(head_dim // 2, dtype=np.float64)
    return np.power(float(theta), -2.0 * k / head_dim)


def rope_rotate(x: np.ndarray, pos, theta: float) -> np.ndarray:
    """Rotate-half RoPE of the last axis of ``x`` at positions ``pos``.

    [Shard] section 5, step 1 states Llama's inverse as
    k_no_rope = k*cos(theta p) - rotate_half(k)*sin(theta p) with
    rotate_half([a, b]) = [-b, a]; the forward map is therefore
    out = x*cos + rotate_half(x)*sin, i.e. for each pair (a, b) = (x_k, x_{k+d/2}):
    out_k = a cos - b sin, out_{k+d/2} = b cos + a sin.
    ``pos`` broadcasts against x's leading axes.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    half = d // 2
    ang = np.asarray(pos, dtype=np.float64)[..., None] * rope_inv_freq(d, theta)
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# ---------------------------------------------------------------------------
# Softmax attention for one query head
# ---------------------------------------------------------------------------

def softmax_attend(scores: np.ndarray, values: np.ndarray):
    """p = softmax(scores); returns (p @ values, lse) with lse = log sum exp(scores).

    [Palu] "背景知识": p = Softmax(q K^T / sqrt(d_h)), a = p V. The max is
    subtracted before exponentiating, which leaves p unchanged.
    """
    scores = np.asarray(scores, dtype=np.float64)
    if scores.size == 0:
        return np.zeros(values.shape[-1]), -math.inf
    m = scores.max()
    e = np.exp(scores - m)
    l = e.sum()
    p = e / l
    return p @ values, m + math.log(l)


# ---------------------------------------------------------------------------
# Decode attention over G-LRD latents
# ---------------------------------------------------------------------------

def _group_of(head: int, group_size: int):
    return head // group_size, head % group_size


def _positions(positions, b: int, T: int):
    if positions is None:
        return np.arange(T, dtype=np.float64)
    return np.asarray(positions[b][:T], dtype=np.float64)


def _query_position(positions, q_pos, b: int, T: int):
    if q_pos is not None:
        return float(q_pos[b])
    if positions is None:
        return float(T - 1)
    return float(positions[b][T - 1])


def decode_rope_head(q_i, hk_bg, hv_bg, bk_g, j: int, pos, qp: float, theta: float):
    """One head of the RoPE path.

    Rebuild K_i = H_k,g B_g[:, j-block] ([Palu] "方法细节", G-LRD: the s heads of a
    group are the column blocks of h_g B_g), rotate every key at its own position
    and the query at qp, score q_rot K_rot^T / sqrt(d_h), softmax, and apply p to
    the value latents (V rebuild skipped because B_v is fused into W_o, [Palu]
    "方法细节", value fusion paragraph).
    """
    d_h = q_i.shape[-1]
    T = hk_bg.shape[0]
    if T == 0:
        return np.zeros(hv_bg.shape[-1]), -math.inf
    K = np.asarray(hk_bg, np.float64) @ np.asarray(bk_g, np.float64)[:, j * d_h:(j + 1) * d_h]
    K_rot = rope_rotate(K, pos, theta)
    q_rot = rope_rotate(np.asarray(q_i, np.float64), qp, theta)
    scores = (K_rot @ q_rot) / math.sqrt(d_h)
    return softmax_attend(scores, np.asarray(hv_bg, np.float64))


def decode_absorbed_head(q_i, hk_bg, hv_bg, bk_g, j: int, bias=None):
    """One head of the non-RoPE path: the query is absorbed into the latent space,
    q'_i = q_i (B_i^k)^T, and scored straight against H_k
    ([Palu] "方法细节", key fusion: q_i K_i^T = q_i (H_i^k B_i^k)^T = (q_i B_i^k^T) H_i^k^T).
    `bias` (one value per token) is added to the scores: a position bias that never touches
    the keys, such as ALiBi's, leaves the key fusion valid (same paragraph)."""
    d_h = q_i.shape[-1]
    if hk_bg.shape[0] == 0:
        return np.zeros(hv_bg.shape[-1]), -math.inf
    q_lat = np.asarray(bk_g, np.float64)[:, j * d_h:(j + 1) * d_h] @ np.asarray(q_i, np.float64)
    scores = (np.asarray(hk_bg, np.float64) @ q_lat) / math.sqrt(d_h)
    if bias is not None:
        scores = scores + np.asarray(bias, np.float64)
    return softmax_attend(scores, np.asarray(hv_bg, np.float64))


def alibi_slopes(n_heads: int) -> np.ndarray:
    """ALiBi's per-head slopes m_i = 2^(-8 (i + 1) / n), the geometric sequence of the paper the
    Palu notes cite for non-RoPE position encodings ("Train short, test long: attention with
    linear biases"): 1/2, 1/4, ..., 1/256 for 8 heads."""
    return np.power(2.0, -8.0 * (np.arange(n_heads, dtype=np.float64) + 1.0) / n_heads)


def alibi_bias(slope: float, pos, qp: float) -> np.ndarray:
    """The score bias of each key: -m (q_pos - pos_t), a penalty linear in the query's distance."""
    return -slope * (float(qp) - np.asarray(pos, np.float64))


def decode(q, hk, hv, bk, seq_lens, group_size: int, *, mode: str = "rope", theta: float = 10000.0,
           positions=None, q_pos=None, heads=None, alibi: bool = False):
    """Decode attention for every (batch, head), or only for ``heads`` = [(b, i), ...].

    q  [B][n][d_h], hk [B][T][n_g][r_k], hv [B][T][n_g][r_v] (already dequantised),
    bk [n_g][r_k][s*d_h], seq_lens [B]. Returns (o [B][n][r_v], lse [B][n]) float64;
    entries not requested through ``heads`` are NaN.
    """
    B, n, _ = q.shape
    r_v = hv.shape[-1]
    o = np.full((B, n, r_v), np.nan)
    lse = np.full((B, n), np.nan)
    todo = heads if heads is not None else [(b, i) for b in range(B) for i in range(n)]
    for b, i in todo:
        T = int(seq_lens[b])
        g, j = _group_of(i, group_size)
        hk_bg = np.asarray(hk[b, :T, g, :], np.float64)
        hv_bg = np.asarray(hv[b, :T, g, :], np.float64)
        if mode == "rope":
            pos = _positions(positions, b, T)
            qp = _query_position(positions, q_pos, b, T) if T > 0 else 0.0
            o[b, i], lse[b, i] = decode_rope_head(q[b, i], hk_bg, hv_bg, bk[g], j, pos, qp, theta)
        elif mode == "absorbed":
            bias = None
            if alibi and T > 0:
                bias = alibi_bias(alibi_slopes(n)[i], _positions(positions, b, T),
                                  _query_position(positions, q_pos, b, T))
            o[b, i], lse[b, i] = decode_absorbed_head(q[b, i], hk_bg, hv_bg, bk[g], j, bias)
        else:
            raise ValueError(mode)
    return o, lse


def decode_hybrid(q, hk, hv, bk, seq_lens, group_size: int, dense_k, dense_v, n_dense, *, mode: str = "rope",
                  theta: float = 10000.0, positions=None, q_pos=None, heads=None):
    """Decode over a hybrid cache: a dense segment (the attention-sink tokens and the recent window)
    next to the G-LRD latent middle ([Puzzle] section 3: the sink page and the local window stay
    dense, the other completed pages are factorised, and each query attends over dense and
    factorised pages at once, their partial results merged by online softmax; [Shard] section 7:
    four fp16 sink tokens and a 64-token fp16 window around the compressed middle).

    Readings: the dense keys are a standard KV cache, i.e. already rotated at their own positions
    on the RoPE path (unrotated on the absorbed path), so they are scored against q rotated at
    q_pos; the latent middle is scored as in decode(), at `positions`; one softmax spans both
    segments. The middle's output stays in latent space (B_v is fused into W_o) while the dense
    tokens' output is in value space, so head i's attention output is o_lat B_v^(i) + o_dense.

    dense_k, dense_v [B][D][n][d_h]; n_dense [B] (dense tokens used per row). Returns
    (o_lat [B][n][r_v], o_dense [B][n][d_h], lse [B][n]); rows not in ``heads`` are NaN.
    """
    B, n, d_h = q.shape
    r_v = hv.shape[-1]
    o_lat = np.full((B, n, r_v), np.nan)
    o_den = np.full((B, n, d_h), np.nan)
    lse = np.full((B, n), np.nan)
    todo = heads if heads is not None else [(b, i) for b in range(B) for i in range(n)]
    for b, i in todo:
        T = int(seq_lens[b])
        D = int(n_dense[b])
        g, j = _group_of(i, group_size)
        hk_bg = np.asarray(hk[b, :T, g, :], np.float64)
        hv_bg = np.asarray(hv[b, :T, g, :], np.float64)
        kd = np.asarray(dense_k[b, :D, i, :], np.float64)
        vd = np.asarray(dense_v[b, :D, i, :], np.float64)
        qi = np.asarray(q[b, i], np.float64)
        if mode == "rope":
            if q_pos is None:
                raise ValueError("the hybrid RoPE path needs q_pos")
            K = hk_bg @ np.asarray(bk[g], np.float64)[:, j * d_h:(j + 1) * d_h]
            K_rot = rope_rotate(K, _positions(positions, b, T), theta)
            q_use = rope_rotate(qi, float(q_pos[b]), theta)
            s_mid = (K_rot @ q_use) / math.sqrt(d_h) if T else np.zeros(0)
        elif mode == "absorbed":
            q_use = qi
            q_lat = np.asarray(bk[g], np.float64)[:, j * d_h:(j + 1) * d_h] @ qi
            s_mid = (hk_bg @ q_lat) / math.sqrt(d_h) if T else np.zeros(0)
        else:
            raise ValueError(mode)
        s_den = (kd @ q_use) / math.sqrt(d_h) if D else np.zeros(0)
        s_all = np.concatenate([s_mid, s_den])
        if s_all.size == 0:
            o_lat[b, i], o_den[b, i], lse[b, i] = 0.0, 0.0, -math.inf
            continue
        m = s_all.max()
        e = np.exp(s_all - m)
        l = e.sum()
        p = e / l
        o_lat[b, i] = p[:T] @ hv_bg if T else 0.0
        o_den[b, i] = p[T:] @ vd if D else 0.0
        lse[b, i] = m + math.log(l)
    return o_lat, o_den, lse


# ---------------------------------------------------------------------------
# Uncompressed multi-head attention (the definition the latent path must equal)
# ---------------------------------------------------------------------------

def mha_decode(q, x, wk, wv, seq_lens, *, theta: float = 10000.0, rope: bool = True,
               positions=None, q_pos=None, alibi: bool = False):
    """Plain MHA decode over cached activations x [B][T][d] ([Palu] "背景知识"):
    k_i = x W_i^k, v_i = x W_i^v, p = softmax(q_i K_i^T / sqrt(d_h)), a_i = p V_i.
    Returns a [B][n][d_h] and lse [B][n]."""
    B, n, d_h = q.shape
    a = np.zeros((B, n, d_h))
    lse = np.zeros((B, n))
    for b in range(B):
        T = int(seq_lens[b])
        xb = np.asarray(x[b, :T], np.float64)
        pos = _positions(positions, b, T)
        qp = _query_position(positions, q_pos, b, T)
        for i in range(n):
            K = xb @ wk[:, i * d_h:(i + 1) * d_h]
            V = xb @ wv[:, i * d_h:(i + 1) * d_h]
            qi = np.asarray(q[b, i], np.float64)
            if rope:
                K = rope_rotate(K, pos, theta)
                qi = rope_rotate(qi, qp, theta)
            sc = K @ qi / math.sqrt(d_h)
            if alibi:
                sc = sc + alibi_bias(alibi_slopes(n)[i], pos, qp)
            a[b, i], lse[b, i] = softmax_attend(sc, V)
    return a, lse


def factor_page(x: np.ndarray, r: int):
    """One page's rank-r factors ([Puzzle] section 3.3, eq. 2): the truncated SVD X ~= L R of a
    P x d page with L = U_r (P x r) and R = S_r W_r^T (r x d)."""
    u, s, wt = np.linalg.svd(np.asarray(x, np.float64), full_matrices=False)
    return u[:, :r], s[:r, None] * wt[:r]


def factor_page_gram(x: np.ndarray, r: int):
    """The same factors the way [Puzzle] section 3.3 obtains them for short, wide pages: the top-r
    eigenvectors Q_r of the P x P Gram matrix G = X X^T give L = Q_r and R = Q_r^T X."""
    x = np.asarray(x, np.float64)
    w, q = np.linalg.eigh(x @ x.T)
    qr = q[:, np.argsort(w)[::-1][:r]]
    return qr, qr.T @ x


def decode_paged(q, lk, rk, lv, rv, n_pages, dense_k, dense_v, n_dense, *, mode: str = "rope",
                 theta: float = 10000.0, q_pos=None, heads=None):
    """Decode over a page-factorised cache next to dense sink and window tokens ([Puzzle] section
    3.3, step 4: every completed page p of a head holds K_p ~= L_p^K R_p^K and V_p ~= L_p^V R_p^V;
    the page's scores are s_p = (q R_p^K^T) L_p^K^T / sqrt(d) and its values are read as
    L_p^V R_p^V without rebuilding the page; dense and factorised pages share one softmax).

    Readings: the factorised pages hold the keys as the cache holds them, i.e. already rotated on
    the RoPE path, so they are scored like the dense tokens against q rotated at q_pos (no
    rotation on the absorbed path); the value read is the plain product p (L^V R^V). The output is
    split like decode_hybrid's: the factorised pages' part and the dense tokens' part, both
    normalised by the shared denominator (their sum is the attention output).

    lk [B][Pmax][n][P][r_k], rk [B][Pmax][n][r_k][d_h], lv [B][Pmax][n][P][r_v],
    rv [B][Pmax][n][r_v][d_h]; n_pages [B]; dense_k, dense_v [B][D][n][d_h]; n_dense [B].
    Returns (o_pages [B][n][d_h], o_dense [B][n][d_h], lse [B][n]); rows not in ``heads`` are NaN.
    """
    B, n, d_h = q.shape
    o_pg = np.full((B, n, d_h), np.nan)
    o_den = np.full((B, n, d_h), np.nan)
    lse = np.full((B, n), np.nan)
    todo = heads if heads is not None else [(b, i) for b in range(B) for i in range(n)]
    for b, i in todo:
        npg = int(n_pages[b])
        D = int(n_dense[b])
        qi = np.asarray(q[b, i], np.float64)
        if mode == "rope":
            if q_pos is None:
                raise ValueError("the RoPE path needs q_pos")
            q_use = rope_rotate(qi, float(q_pos[b]), theta)
        elif mode == "absorbed":
            q_use = qi
        else:
            raise ValueError(mode)
        s_pages = []
        for p in range(npg):
            u = np.asarray(rk[b, p, i], np.float64) @ q_use              # q R^T: one value per rank
            s_pages.append((np.asarray(lk[b, p, i], np.float64) @ u) / math.sqrt(d_h))
        s_pg = np.concatenate(s_pages) if s_pages else np.zeros(0)
        kd = np.asarray(dense_k[b, :D, i, :], np.float64)
        s_den = (kd @ q_use) / math.sqrt(d_h) if D else np.zeros(0)
        s_all = np.concatenate([s_pg, s_den])
        if s_all.size == 0:
            o_pg[b, i], o_den[b, i], lse[b, i] = 0.0, 0.0, -math.inf
            continue
        m = s_all.max()
        e = np.exp(s_all - m)
        l = e.sum()
        prob = e / l
        acc = np.zeros(d_h)
        off = 0
        for p in range(npg):
            P = lk.shape[3]
            w = prob[off:off + P] @ np.asarray(lv[b, p, i], np.float64)   # p L^V: one value per rank
            acc += w @ np.asarray(rv[b, p, i], np.float64)
            off += P
        o_pg[b, i] = acc
        o_den[b, i] = prob[off:] @ np.asarray(dense_v[b, :D, i, :], np.float64) if D else 0.0
        lse[b, i] = m + math.log(l)
    return o_pg, o_den, lse


# ---------------------------------------------------------------------------
# Offline transforms the pins use
# ---------------------------------------------------------------------------

def svd_factor(w: np.ndarray, r: int):
    """W ~= A B with A = U_r sqrt(S_r), B = sqrt(S_r) V_r^T ([Palu] "背景知识", SVD)."""
    u, s, vt = np.linalg.svd(np.asarray(w, np.float64), full_matrices=False)
    rs = np.sqrt(s[:r])
    return u[:, :r] * rs[None, :], rs[:, None] * vt[:r]


def hadamard(r: int) -> np.ndarray:
    """Normalised Walsh-Hadamard matrix by Sylvester doubling, H_2m = [[H, H], [H, -H]],
    scaled by 1/sqrt(r) so that R R^T = I ([Palu] "方法细节", Hadamard fold)."""
    if r < 1 or r & (r - 1):
        raise ValueError("r must be a power of two")
    h = np.ones((1, 1))
    while h.shape[0] < r:
        h = np.block([[h, h], [h, -h]])
    return h / math.sqrt(r)


# ---------------------------------------------------------------------------
# Latent production (the step before decode)
# ---------------------------------------------------------------------------

def project_latents(x, a) -> np.ndarray:
    """H[b, t, g, :] = x[b, t, :] A_g, the latents a new token leaves in the cache ([Palu]
    "方法细节", SVD rewrite: the layer caches h = x A instead of the key or value itself, and
    the G-LRD paragraph gives one A_g per group). x [B][T][d], a [n_g][d][r] -> [B][T][n_g][r]."""
    x = np.asarray(x, np.float64)
    a = np.asarray(a, np.float64)
    B, T, _ = x.shape
    n_g, _, r = a.shape
    h = np.empty((B, T, n_g, r))
    for b in range(B):
        for g in range(n_g):
            h[b, :, g, :] = x[b] @ a[g]
    return h


# ---------------------------------------------------------------------------
# int4 per-token latent quantisation
# ---------------------------------------------------------------------------

FP16_MAX = 65504.0


def quantize_int4(h):
    """Per-token, per-group symmetric int4 codes ([Palu] "补充细节": simple per-token
    quantisation of the latents; code range [-7, 7] as in [Shard] section 5, step 4).

    h: float32 array [..., r]. Returns (codes int8 [..., r], scale float16 [...]).
    Arithmetic in IEEE float32 / float16 round-to-nearest-even.
    """
    h = np.asarray(h, dtype=np.float32)
    amax = np.max(np.abs(h), axis=-1)
    q = np.minimum(amax / np.float32(7.0), np.float32(FP16_MAX)).astype(np.float32)
    scale = q.astype(np.float16)
    sf = scale.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = h / sf[..., None]
    codes = np.clip(np.rint(ratio), -7, 7)
    codes = np.where((sf == 0)[..., None], 0.0, codes).astype(np.int8)
    return codes, scale


def pack_int4(codes) -> np.ndarray:
    """Two codes per byte: element 2j in bits 0-3, element 2j+1 in bits 4-7, each as
    a 4-bit two's-complement number."""
    c = np.asarray(codes, dtype=np.int16) & 0xF
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_int4(packed) -> np.ndarray:
    p = np.asarray(packed, dtype=np.uint8).astype(np.int16)
    lo = p & 0xF
    hi = (p >> 4) & 0xF
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.int8)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def dequant_int4(packed, scale) -> np.ndarray:
    """Latent value = code * scale, returned in float64 (exact)."""
    codes = unpack_int4(packed).astype(np.float64)
    return codes * np.asarray(scale, dtype=np.float16).astype(np.float64)[..., None]


# ---------------------------------------------------------------------------
# Value fusion into the output projection (the step after decode)
# ---------------------------------------------------------------------------

def fuse_value_output(bv, wo, group_size: int) -> np.ndarray:
    """The fused matrices W_f^(i) = B_v^(i) W_o^(i) of every head i, stacked as
    [n * r_v][d] ([Palu] "方法细节", value-fusion paragraph: head i's attention output
    p_i V_i = p_i H_v,g B_v^(i) meets its rows of W_o, so B_v^(i) W_o^(i) can be
    formed offline). B_v^(i) is column block j = i % s of group g = i // s of
    bv [n_g][r_v][s*d_h]; W_o^(i) is rows i*d_h .. (i+1)*d_h - 1 of wo [n*d_h][d]."""
    bv = np.asarray(bv, np.float64)
    wo = np.asarray(wo, np.float64)
    n_g, r_v, cols = bv.shape
    d_h = cols // group_size
    blocks = []
    for i in range(n_g * group_size):
        g, j = _group_of(i, group_size)
        blocks.append(bv[g][:, j * d_h:(j + 1) * d_h] @ wo[i * d_h:(i + 1) * d_h])
    return np.concatenate(blocks, axis=0)


def project_fused(o, w_fused) -> np.ndarray:
    """y[b] = sum_i o[b, i] W_f^(i): the layer output from the latent decode outputs
    o [B][n][r_v], with W_f^(i) = rows i*r_v .. (i+1)*r_v - 1 of w_fused [n*r_v][d]."""
    o = np.asarray(o, np.float64)
    w = np.asarray(w_fused, np.float64)
    B, n, r_v = o.shape
    y = np.zeros((B, w.shape[1]))
    for b in range(B):
        for i in range(n):
            y[b] += o[b, i] @ w[i * r_v:(i + 1) * r_v]
    return y
