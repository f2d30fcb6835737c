"""Seeded synthetic workloads for Palu-style G-LRD decode attention.

Every array here is a *draw*: random weights with a prescribed singular-value
decay, their per-group truncated SVD factors (the offline weight transform that
precedes decoding), Gaussian activations and queries. Nothing in this module
computes attention, RoPE, softmax or quantisation; the oracle and the CUDA path
both start from what it returns.

Workload recipe (all five shapes follow the Llama-2-7B attention layer that the
Palu notes evaluate, "实验环境"/"实验结果"):
  * W_k, W_v = U diag(sigma) V^T with Haar-orthogonal U, V (QR of a Gaussian
    matrix with the sign of R's diagonal folded into Q) and sigma_i = exp(-i/tau).
  * Group g holds consecutive heads g*s .. g*s+s-1, W_g = W[:, g*s*d_h:(g+1)*s*d_h]
    (the d x (d_h*s) concatenation of the G-LRD section of the Palu notes; 4096x512
    for Llama-2-7B with s=4).
  * Truncated SVD per group: A_g = U_r sqrt(S_r), B_g = sqrt(S_r) V_r^T
    (Palu notes, "背景知识", SVD paragraph).
  * Optional normalised Walsh-Hadamard fold: A_g <- A_g R, B_g <- R^T B_g
    (Palu notes, "方法细节", Hadamard paragraph).
  * Latents H = x A with x ~ N(0, I_d). For large workloads the equivalent draw
    H = z sqrt(S_r) [R] with z ~ N(0, I_r) is used: x U_r is exactly N(0, I_r)
    because U_r has orthonormal columns, so the latents have the same
    distribution (K and V latents are then drawn independently).
  * q ~ N(0, I) per head; positions 0..T-1.
Seeds: numpy PCG64 streams spawned from SeedSequence(20261202 + stream id), one
each for W_k, W_v, x, q and W_o; the four Llama-2-7B workloads are one layer and
draw W_k and W_v from the fp16 RoPE workload's streams.
"""
from __future__ import annotations

import dataclasses
import functools
import math

import numpy as np
import scipy.linalg

SEED_BASE = 20261202
# Above this many activation elements (B*T*d) the equivalent latent draw is used.
EXACT_X_LIMIT = 1 << 26


@dataclasses.dataclass(frozen=True)
class Config:
    stream: int          # seed-stream id (SEED_BASE + stream); the Llama-2-7B layers share weights
    name: str
    batch: int
    n_heads: int
    head_dim: int
    hidden: int
    group_size: int
    rank: int            # r_k = r_v = r_g
    T: int
    latent_dtype: str    # "f32" | "f16" | "bf16" | "int4"
    mode: str            # "rope" | "absorbed"
    sigma_tau: float     # sigma_i = exp(-i / tau)
    hadamard: bool = False
    theta: float = 10000.0
    v_dtype: str = ""    # value latents' dtype when it differs from the keys' ("int4": int4 values only)

    @property
    def n_groups(self) -> int:
        return self.n_heads // self.group_size

    @property
    def value_dtype(self) -> str:
        return self.v_dtype or self.latent_dtype

    @property
    def bk_dtype(self) -> str:
        # int4 latents are dequantised to fp16 before the rebuild contraction
        return "f16" if self.latent_dtype == "int4" else self.latent_dtype

    @property
    def q_dtype(self) -> str:
        return self.bk_dtype

    def with_(self, **kw) -> "Config":
        return dataclasses.replace(self, **kw)


# The workloads: a tiny fp32 layer (8 heads, d_h 64, hidden 512, rank 128, T 512) and one
# Llama-2-7B attention layer (32 heads, d_h 128, hidden 4096, group 4, rank 256) in four forms.
TINY_FP32 = Config(1, "tiny-fp32-b1-t512", 1, 8, 64, 512, 4, 128, 512, "f32", "rope", 64.0)
ROPE_FP16 = Config(2, "llama2-7b-rope-fp16-b1-t4k", 1, 32, 128, 4096, 4, 256, 4096, "f16", "rope", 512.0)
ROPE_BF16 = Config(3, "llama2-7b-rope-bf16-b8-t32k", 8, 32, 128, 4096, 4, 256, 32768, "bf16", "rope", 512.0)
ABSORBED_FP16 = Config(4, "llama2-7b-absorbed-fp16-b4-t64k", 4, 32, 128, 4096, 4, 256, 65536, "f16", "absorbed",
                       512.0)
ROPE_INT4 = Config(5, "llama2-7b-rope-int4-hadamard-b4-t64k", 4, 32, 128, 4096, 4, 256, 65536, "int4", "rope",
                   512.0, hadamard=True)
ALL = (TINY_FP32, ROPE_FP16, ROPE_BF16, ABSORBED_FP16, ROPE_INT4)
LLAMA_STREAM = ROPE_FP16.stream


def _streams(stream: int):
    ss = np.random.SeedSequence(SEED_BASE + stream)
    return [np.random.Generator(np.random.PCG64(s)) for s in ss.spawn(5)]


def _weight_stream(stream: int) -> int:
    # the four Llama-2-7B workloads describe the same layer, so they share its weights;
    # activations and queries keep their own streams
    return LLAMA_STREAM if stream in (s.stream for s in ALL[1:]) else stream


def _haar(rng: np.random.Generator, n: int) -> np.ndarray:
    z = rng.standard_normal((n, n))
    q, r = np.linalg.qr(z)
    return q * np.sign(np.diag(r))[None, :]


@functools.lru_cache(maxsize=8)
def _weights(stream: int, hidden: int, tau: float):
    """Spectrum-decay W_k, W_v (hidden x hidden), float64."""
    rk, rv, _, _, _ = _streams(stream)
    sig = np.exp(-np.arange(hidden) / tau)
    out = []
    for rng in (rk, rv):
        u = _haar(rng, hidden)
        v = _haar(rng, hidden)
        out.append((u * sig[None, :]) @ v.T)
    return out[0], out[1]


@functools.lru_cache(maxsize=8)
def _factors(cfg_key):
    stream, hidden, tau, n_g, s, d_h, r, had = cfg_key
    wk, wv = _weights(stream, hidden, tau)
    R = scipy.linalg.hadamard(r).astype(np.float64) / math.sqrt(r) if had else None
    res = {}
    for name, w in (("k", wk), ("v", wv)):
        A = np.empty((n_g, hidden, r))
        B = np.empty((n_g, r, s * d_h))
        S_all = np.empty((n_g, r))
        for g in range(n_g):
            wg = w[:, g * s * d_h:(g + 1) * s * d_h]
            u, sv, vt = np.linalg.svd(wg, full_matrices=False)
            rs = np.sqrt(sv[:r])
            A[g] = u[:, :r] * rs[None, :]
            B[g] = rs[:, None] * vt[:r]
            S_all[g] = sv[:r]
            if R is not None:
                A[g] = A[g] @ R
                B[g] = R.T @ B[g]
        res[name] = (A, B, S_all)
    return res, R


def weights(cfg: Config):
    """(W_k, W_v) float64 full projection matrices of the configuration."""
    return _weights(_weight_stream(cfg.stream), cfg.hidden, cfg.sigma_tau)


def factors(cfg: Config):
    key = (_weight_stream(cfg.stream), cfg.hidden, cfg.sigma_tau, cfg.n_groups, cfg.group_size, cfg.head_dim,
           cfg.rank, cfg.hadamard)
    return _factors(key)


def make_inputs(cfg: Config, *, exact_x: bool | None = None, q_scale: float = 1.0,
                with_x: bool = False, with_wo: bool = False) -> dict:
    """Draw one workload. Returns float32/float64 numpy arrays (unrounded):

    hk, hv : [B][T][n_g][r] float32 latents (cache layout)
    bk, bv : [n_g][r][s*d_h] float64 reconstruction factors (Hadamard-folded if set)
    ak, av : [n_g][d][r] float64 down-projections
    q      : [B][n][d_h] float32 query (not rotated)
    x      : [B][T][d] float32 activations (only when drawn exactly and with_x)
    wo     : [d][d] float64 output projection ~ N(0, 1/d) (only with with_wo)
    """
    B, T, d = cfg.batch, cfg.T, cfg.hidden
    n_g, r, s, d_h = cfg.n_groups, cfg.rank, cfg.group_size, cfg.head_dim
    fac, R = factors(cfg)
    _, _, rx, rq, ro = _streams(cfg.stream)
    if exact_x is None:
        exact_x = B * T * d <= EXACT_X_LIMIT
    out = {"cfg": cfg}
    if exact_x:
        x = rx.standard_normal((B, T, d), dtype=np.float32)
        ak = fac["k"][0].astype(np.float32)
        av = fac["v"][0].astype(np.float32)
        hk = np.ascontiguousarray(np.einsum("btd,gdr->btgr", x, ak, optimize=True), dtype=np.float32)
        hv = np.ascontiguousarray(np.einsum("btd,gdr->btgr", x, av, optimize=True), dtype=np.float32)
        if with_x:
            out["x"] = x
    else:
        hk = np.empty((B, T, n_g, r), np.float32)
        hv = np.empty((B, T, n_g, r), np.float32)
        for h, name in ((hk, "k"), (hv, "v")):
            sq = np.sqrt(fac[name][2]).astype(np.float32)       # [n_g][r]
            Rf = None if R is None else R.astype(np.float32)
            for b in range(B):
                z = rx.standard_normal((T, n_g, r), dtype=np.float32)
                z *= sq[None, :, :]
                if Rf is not None:
                    z = z @ Rf
                h[b] = z
    out["hk"], out["hv"] = hk, hv
    out["bk"], out["bv"] = fac["k"][1], fac["v"][1]
    out["ak"], out["av"] = fac["k"][0], fac["v"][0]
    out["sk"], out["sv"] = fac["k"][2], fac["v"][2]
    q = rq.standard_normal((B, cfg.n_heads, d_h), dtype=np.float32)
    out["q"] = q * np.float32(q_scale)
    if with_wo:
        out["wo"] = ro.standard_normal((d, d)) / math.sqrt(d)
    out["R"] = R
    return out


def draw_query(cfg: Config, q_scale: float = 1.0) -> np.ndarray:
    """The workload's query alone, [B][n][d_h] float32: the same draw make_inputs returns."""
    _, _, _, rq, _ = _streams(cfg.stream)
    q = rq.standard_normal((cfg.batch, cfg.n_heads, cfg.head_dim), dtype=np.float32)
    return q * np.float32(q_scale)


def sample_group_latents(cfg: Config, which: str = "k", b: int = 0, g: int = 0) -> np.ndarray:
    """[T][r] float32 latents of one (batch row, group), in the equivalent form
    H = z sqrt(S_r) [R], from a seed stream of their own (keyed by side, b and g).
    For CPU-side samples of a workload (timing the oracle) without drawing the
    whole cache."""
    fac, R = factors(cfg)
    key = (1000, 0 if which == "k" else 1, b, g)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(SEED_BASE + cfg.stream, spawn_key=key)))
    z = rng.standard_normal((cfg.T, cfg.rank), dtype=np.float32)
    z *= np.sqrt(fac[which][2][g]).astype(np.float32)[None, :]
    if R is not None:
        z = z @ R.astype(np.float32)
    return np.ascontiguousarray(z, dtype=np.float32)


def latent_rows_torch(cfg: Config, device, which: str = "k"):
    """Seeded latents drawn on a CUDA device, one batch row at a time (a generator of
    [T][n_g][r] float32 tensors, batch row b = 0 .. B-1).

    The draw is the equivalent form of H = x A used for large workloads,
    H = z sqrt(S_r) [R] with z ~ N(0, I_r) (x U_r is exactly N(0, I_r)), taken with
    torch's device generator seeded from SeedSequence(20261202 + stream) so that
    multi-gigabyte caches are drawn in well under a second. The benchmark uses it;
    the parity tests use make_inputs.
    """
    import torch
    fac, R = factors(cfg)
    seed = int(np.random.SeedSequence(SEED_BASE + cfg.stream).generate_state(1, np.uint64)[0] >> 1)
    seed += 0 if which == "k" else 1
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    sq = torch.from_numpy(np.sqrt(fac[which][2]).astype(np.float32)).to(device)       # [n_g][r]
    Rt = None if R is None else torch.from_numpy(R.astype(np.float32)).to(device)
    for _ in range(cfg.batch):
        z = torch.randn((cfg.T, cfg.n_groups, cfg.rank), generator=g, device=device, dtype=torch.float32)
        z.mul_(sq[None])
        if Rt is not None:
            z = z @ Rt
        yield z


_TORCH_DT = {"f32": "float32", "f16": "float16", "bf16": "bfloat16"}


def storage_round(a, dtype: str):
    """Round an array to a storage dtype ("f32"/"f16"/"bf16"); returns a CPU torch tensor.

    The rounded tensor is what both the CUDA path and the oracle consume (the
    oracle upcasts it to float64), so rounding never separates the two sides.
    """
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(getattr(torch, _TORCH_DT[dtype]))


def hadamard_sylvester(r: int) -> np.ndarray:
    """Normalised Sylvester Walsh-Hadamard matrix (input preparation only)."""
    return scipy.linalg.hadamard(r).astype(np.float64) / math.sqrt(r)


def page_factor_draw(seed: int, batch: int, n_pages: int, n_heads: int, page: int = 32, rank: int = 16,
                     head_dim: int = 128, tau: float = 4.0, key_scale: float = 1.0):
    """Seeded stand-ins for page-factorised keys and values (the PuzzleKV page cache, section 3.3):
    L [B][pages][n][P][r] with orthonormal columns (QR of a Gaussian matrix, sign-fixed) and
    R = diag(sigma) G [B][pages][n][r][d] with G's rows orthonormal and sigma_j = sqrt(P) exp(-j/tau),
    the shape a page's truncated SVD has. Returns (lk, rk, lv, rv) as float32 arrays; nothing here
    factorises or attends."""
    rng = np.random.default_rng(np.random.SeedSequence([SEED_BASE, 7, seed]))
    sig = math.sqrt(page) * np.exp(-np.arange(rank) / tau)

    def draw(scale):
        z = rng.standard_normal((batch, n_pages, n_heads, page, rank))
        q, r = np.linalg.qr(z)
        L = q * np.sign(np.diagonal(r, axis1=-2, axis2=-1))[..., None, :]
        g = rng.standard_normal((batch, n_pages, n_heads, head_dim, rank))
        qg, rg = np.linalg.qr(g)
        G = np.swapaxes(qg * np.sign(np.diagonal(rg, axis1=-2, axis2=-1))[..., None, :], -1, -2)
        return L.astype(np.float32), (scale * sig[:, None] * G).astype(np.float32)

    lk, rk = draw(key_scale)
    lv, rv = draw(1.0)
    return lk, rk, lv, rv


def page_records(lk, rk, lv, rv):
    """Pack page factors into the library's record layout [B][pages][n][L_K | R_K | L_V | R_V]
    (row-major, contiguous); pure reshaping."""
    B, npg, n = lk.shape[:3]
    parts = [np.reshape(a, (B, npg, n, -1)) for a in (lk, rk, lv, rv)]
    return np.ascontiguousarray(np.concatenate(parts, axis=-1))
