"""Bit-exact checks of the int4 unpack that the tensor-core RoPE kernel runs.

The stored format is fixed by the method (per-token int4 latents, Palu notes
"补充细节", KV-quantisation paragraph; codes in [-7, 7], Shard §5 step 4). The
decode kernel expands key codes to exact fp16 tensor-core operands with its own
converter, and multiplies value codes by integer weights with dp2a on biased codes.
Both routines are exported by test hooks that run the kernel's own device
functions; here their outputs are compared with the oracle's unpacking, bit for bit.

The cache bytes are written from the host: the oracle's quantised and packed
latents of the int4 workload, plus crafted rows in which every byte position of a
row takes every one of the 256 byte values (so every nibble value, -8 included,
reaches every position of the converter and of the dp2a routine).
"""
import numpy as np
import pytest

from oracle import palu_oracle as O
from synthetic import gen

pytestmark = pytest.mark.gpu

# operand position p within each run of eight ranks holds rank PERM8[p] (the order B_k^T uses too)
PERM8 = np.array([0, 2, 4, 6, 1, 3, 5, 7])
RANK_OF_POS = (np.arange(256) & ~7) | PERM8[np.arange(256) & 7]


def _cache_bytes(B, T, seed):
    """Packed int4 K and V rows [B][T][n_g][128] and their fp16 scales, from the oracle's quantiser,
    with crafted rows in batch row 0: byte j of token t is (t + 7 j) mod 256 for t < 256."""
    cfg = gen.ROPE_INT4.with_(T=T, batch=B)
    inp = gen.make_inputs(cfg)
    out = []
    rng = np.random.default_rng(seed)
    for h in (inp["hk"], inp["hv"]):
        codes, scale = O.quantize_int4(h)
        packed = O.pack_int4(codes)
        n = min(T, 256)
        t = np.arange(n)[:, None, None]
        j = np.arange(packed.shape[-1])[None, None, :]
        packed[0, :n] = np.broadcast_to(((t + 7 * j) % 256).astype(np.uint8), packed[0, :n].shape)
        scale[0, :n] = rng.uniform(1e-3, 3.0, size=(n, cfg.n_groups)).astype(np.float16)
        out.append((np.ascontiguousarray(packed), np.ascontiguousarray(scale)))
    return cfg, out


@pytest.fixture(scope="module")
def int4_cache(cuda_device):
    import torch
    from rank_kv_cache_gb300 import palu as P
    B, T = 2, 300
    cfg, ((pk, sk), (pv, sv)) = _cache_bytes(B, T, seed=7)
    bk = torch.zeros((cfg.n_groups, cfg.rank, cfg.group_size * cfg.head_dim), dtype=torch.float16, device="cuda")
    attn = P.PaluAttention(bk, n_heads=cfg.n_heads, head_dim=cfg.head_dim, group_size=cfg.group_size,
                           rank_k=cfg.rank, rank_v=cfg.rank, latent_dtype="int4", q_dtype="f16", mode="rope",
                           max_batch=B, max_tokens=T)
    cache = P.LatentCache(B, T, cfg.n_groups, cfg.rank, cfg.rank, "int4", device="cuda")
    cache.hk.copy_(torch.from_numpy(pk))
    cache.hv.copy_(torch.from_numpy(pv))
    cache.k_scale.copy_(torch.from_numpy(sk))
    cache.v_scale.copy_(torch.from_numpy(sv))
    torch.cuda.synchronize()
    return cfg, attn, cache, (pk, sk, pv, sv)


def test_crafted_rows_cover_every_byte_value_at_every_position(int4_cache):
    _, _, _, (pk, _, pv, _) = int4_cache
    for p in (pk, pv):
        for j in range(p.shape[-1]):
            assert len(np.unique(p[0, :256, 0, j])) == 256


def test_tensor_core_key_operand_bit_exact(int4_cache):
    import torch
    from rank_kv_cache_gb300 import palu as P
    cfg, attn, cache, (pk, sk, _, _) = int4_cache
    B, T = pk.shape[0], pk.shape[1]
    codes = torch.full((B, T, cfg.n_groups, cfg.rank), -1, dtype=torch.int16, device="cuda")
    deq = torch.full((B, T, cfg.n_groups, cfg.rank), float("nan"), dtype=torch.float32, device="cuda")
    st = P.palu_debug_int4_operand(attn.handle, cache.c_struct(), B, T, codes.data_ptr(), deq.data_ptr(),
                                   int(torch.cuda.current_stream().cuda_stream))
    assert st == P.PALU_OK
    torch.cuda.synchronize()
    attn.check_device()
    got_bits = codes.cpu().numpy().view(np.uint16)
    want_codes = O.unpack_int4(pk)[..., RANK_OF_POS]                 # oracle codes in operand order
    want_bits = want_codes.astype(np.float16).view(np.uint16)
    np.testing.assert_array_equal(got_bits, want_bits)
    # every code value the 4-bit field can hold reached the converter
    assert set(np.unique(want_codes)) == set(range(-8, 8))
    want_deq = O.dequant_int4(pk, sk)[..., RANK_OF_POS]              # exact in float64 and in float32
    np.testing.assert_array_equal(deq.cpu().numpy().astype(np.float64), want_deq)


@pytest.mark.parametrize("which", [1, 0], ids=["values", "keys"])
def test_dp2a_integer_sums_bit_exact(int4_cache, which):
    import torch
    from rank_kv_cache_gb300 import palu as P
    cfg, attn, cache, (pk, _, pv, _) = int4_cache
    packed = pv if which == 1 else pk
    B, T = packed.shape[0], packed.shape[1]
    rng = np.random.default_rng(100 + which)
    w = rng.integers(0, 32768, size=(B, T, 2), dtype=np.int32)
    w[0, :16] = 32767                                                 # the largest weights the kernel feeds
    w[1, 16:32] = 0
    w[1, 32:48, 0] = 32767
    nblk = (T + 15) // 16
    sums = torch.zeros((B, nblk, cfg.n_groups, 2, cfg.rank), dtype=torch.int32, device="cuda")
    w_dev = torch.from_numpy(w).to("cuda")
    st = P.palu_debug_int4_dp2a(attn.handle, cache.c_struct(), which, B, T, w_dev.data_ptr(), sums.data_ptr(),
                                int(torch.cuda.current_stream().cuda_stream))
    assert st == P.PALU_OK
    torch.cuda.synchronize()
    codes = O.unpack_int4(packed).astype(np.int64)                   # [B][T][n_g][r]
    cpad = np.zeros((B, nblk * 16) + codes.shape[2:], np.int64)
    cpad[:, :T] = codes
    wpad = np.zeros((B, nblk * 16, 2), np.int64)
    wpad[:, :T] = w
    want = np.einsum("bkth,bktgc->bkghc", wpad.reshape(B, nblk, 16, 2), cpad.reshape((B, nblk, 16) + codes.shape[2:]))
    np.testing.assert_array_equal(sums.cpu().numpy().astype(np.int64), want)


def test_int4_debug_hooks_reject_bad_arguments(int4_cache):
    import torch
    from rank_kv_cache_gb300 import palu as P
    cfg, attn, cache, _ = int4_cache
    s = int(torch.cuda.current_stream().cuda_stream)
    buf = torch.empty(16, dtype=torch.int32, device="cuda")
    assert P.palu_debug_int4_operand(attn.handle, cache.c_struct(), 2, 301, buf.data_ptr(), None, s) \
        == P.PALU_ERR_INVALID_ARG                                     # beyond the capacity
    assert P.palu_debug_int4_dp2a(attn.handle, cache.c_struct(), 2, 2, 16, buf.data_ptr(), buf.data_ptr(), s) \
        == P.PALU_ERR_INVALID_ARG                                     # which must be 0 or 1
    assert P.palu_debug_int4_operand(attn.handle, cache.c_struct(), 2, 0, buf.data_ptr(), None, s) == P.PALU_OK
