"""GPU parity of latent production H = x A_g (Palu notes, method section: the SVD rewrite
caches h = x A; supplementary section: per-token int4 quantisation of the cached latents),
through the C ABI, against the float64 oracle."""
import numpy as np
import pytest

from oracle import palu_oracle as O
from synthetic import gen

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    return cuda_device


def _torch():
    import torch
    return torch


class Producer:
    """A handle, a cache and the prepared down-projection of one configuration."""

    def __init__(self, cfg, latent_dtype, *, batch, capacity, x_dtype="f16", seed=0):
        torch = _torch()
        from rank_kv_cache_gb300 import palu as P
        self.P, self.cfg = P, cfg
        dev = torch.device("cuda:0")
        inp = gen.make_inputs(cfg.with_(T=1, batch=1))
        self.ak = gen.storage_round(inp["ak"], x_dtype)          # [n_g][d][r]
        self.av = gen.storage_round(inp["av"], x_dtype)
        # the handle reads B_k in the descriptor's dtype: the latent dtype, fp16 for int4 caches
        bk_dtype = "f16" if latent_dtype == "int4" else latent_dtype
        bk = gen.storage_round(inp["bk"], bk_dtype)
        self.attn = P.PaluAttention(bk.to(dev), n_heads=cfg.n_heads, head_dim=cfg.head_dim,
                                    group_size=cfg.group_size, rank_k=cfg.rank, rank_v=cfg.rank,
                                    latent_dtype=latent_dtype, q_dtype=bk_dtype, mode="rope", max_batch=batch,
                                    max_tokens=capacity)
        self.cache = P.LatentCache(batch, capacity, cfg.n_groups, cfg.rank, cfg.rank, latent_dtype, device=dev)
        self.w = self.attn.prepare_down_proj(self.ak.to(dev), self.av.to(dev), dtype=x_dtype)
        self.x_dtype = x_dtype
        torch.cuda.synchronize()

    def project(self, x, dst_slot):
        torch = _torch()
        self.attn.project(self.w, x.cuda(), self.cache, torch.tensor(dst_slot, dtype=torch.int32, device="cuda"))
        torch.cuda.synchronize()
        self.attn.check_device()


def _x(cfg, batch, n_new, dtype, seed):
    rng = np.random.default_rng(seed)
    return gen.storage_round(rng.standard_normal((batch, n_new, cfg.hidden)).astype(np.float32), dtype)


def _check_close(h32, x, a, slots, n_new):
    """fp32-accumulated H against the float64 oracle: each element within 3e-5 of the sum of the
    magnitudes of its d_model products (one missing or wrong product is ~1/d_model of that)."""
    ref = O.project_latents(x.double().numpy(), a.double().numpy())
    mag = O.project_latents(np.abs(x.double().numpy()), np.abs(a.double().numpy()))
    for b, s0 in enumerate(slots):
        got = h32[b, s0:s0 + n_new]
        err = np.abs(got - ref[b])
        assert np.all(err <= 3e-5 * mag[b] + 1e-7), float((err / (3e-5 * mag[b] + 1e-7)).max())


@pytest.mark.parametrize("x_dtype", ["f16", "bf16"])
def test_fp32_latents_match_oracle_ragged(x_dtype):
    # 3 batch rows x 200 tokens = 600 rows of x: five 128-token tiles, the last one partial;
    # different first slots per row
    cfg = gen.ROPE_FP16
    p = Producer(cfg, "f32", batch=3, capacity=300, x_dtype=x_dtype)
    x = _x(cfg, 3, 200, x_dtype, seed=1)
    slots = [0, 17, 100]
    p.project(x, slots)
    hk = p.cache.hk.cpu().double().numpy()
    hv = p.cache.hv.cpu().double().numpy()
    _check_close(hk, x, p.ak, slots, 200)
    _check_close(hv, x, p.av, slots, 200)
    # rows outside the written slots are untouched (the cache starts zeroed)
    assert np.all(hk[0, 200:] == 0) and np.all(hk[1, :17] == 0) and np.all(hk[2, :100] == 0)


def test_rank_128_small_model():
    cfg = gen.TINY_FP32
    p = Producer(cfg, "f32", batch=2, capacity=160, x_dtype="f16")
    x = _x(cfg, 2, 130, "f16", seed=2)
    p.project(x, [0, 30])
    _check_close(p.cache.hk.cpu().double().numpy(), x, p.ak, [0, 30], 130)
    _check_close(p.cache.hv.cpu().double().numpy(), x, p.av, [0, 30], 130)


def _fp32_reference_run(cfg, x, slots, batch, capacity, x_dtype="f16"):
    p = Producer(cfg, "f32", batch=batch, capacity=capacity, x_dtype=x_dtype)
    p.project(x, slots)
    return p.cache.hk.cpu().numpy(), p.cache.hv.cpu().numpy()


@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_float16_caches_are_the_fp32_values_rounded(dt):
    torch = _torch()
    cfg = gen.ROPE_FP16
    x = _x(cfg, 2, 257, "f16", seed=3)
    h32k, h32v = _fp32_reference_run(cfg, x, [0, 40], 2, 300)
    p = Producer(cfg, dt, batch=2, capacity=300)
    p.project(x, [0, 40])
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dt]
    for got, h32 in ((p.cache.hk, h32k), (p.cache.hv, h32v)):
        want = torch.from_numpy(h32).to(tdt)
        assert torch.equal(got.cpu().view(torch.int16), want.view(torch.int16))


def test_int4_codes_and_scales_are_the_oracle_quantiser_of_the_fp32_values():
    # the kernel is deterministic, so an fp32 run gives the exact values the int4 run quantised
    cfg = gen.ROPE_INT4
    x = _x(cfg, 2, 300, "f16", seed=4)
    slots = [0, 11]
    h32k, h32v = _fp32_reference_run(cfg, x, slots, 2, 320)
    p = Producer(cfg, "int4", batch=2, capacity=320)
    p.project(x, slots)
    for got, scale, h32 in ((p.cache.hk, p.cache.k_scale, h32k), (p.cache.hv, p.cache.v_scale, h32v)):
        got = got.cpu().numpy()
        scale = scale.cpu().numpy()
        for b, s0 in enumerate(slots):
            codes, sc = O.quantize_int4(h32[b, s0:s0 + 300])
            assert np.array_equal(scale[b, s0:s0 + 300].view(np.uint16), sc.view(np.uint16))
            assert np.array_equal(got[b, s0:s0 + 300], O.pack_int4(codes))


def test_projected_int4_cache_decodes_like_an_appended_one():
    # the producer's int4 cache and the append path's int4 cache of the same fp32 latents are
    # byte-identical, so the decode reads the same cache either way; checked on the bytes and
    # on the decode output against the oracle
    torch = _torch()
    from tests.gpu_cases import assert_close
    cfg = gen.ROPE_INT4.with_(T=260, batch=2)
    x = _x(cfg, 2, 260, "f16", seed=5)
    h32k, h32v = _fp32_reference_run(cfg, x, [0, 0], 2, 260)
    p = Producer(cfg, "int4", batch=2, capacity=260)
    p.project(x, [0, 0])
    q = gen.storage_round(gen.make_inputs(cfg)["q"], "f16").cuda()
    seq = torch.tensor([260, 199], dtype=torch.int32, device="cuda")
    lse = torch.empty((2, cfg.n_heads), dtype=torch.float32, device="cuda")
    out = p.attn.decode(q, p.cache, seq, max_seq_len=260, lse=lse)
    torch.cuda.synchronize()
    # the oracle on the dequantised fp32 values
    ck, sk = O.quantize_int4(h32k)
    cv, sv = O.quantize_int4(h32v)
    hk = O.dequant_int4(O.pack_int4(ck), sk)
    hv = O.dequant_int4(O.pack_int4(cv), sv)
    bk = p.attn._bk.cpu().double().numpy()
    ref, lse_ref = O.decode(q.cpu().double().numpy(), hk, hv, bk, [260, 199], cfg.group_size, theta=cfg.theta)
    assert_close(out.cpu().double().numpy(), ref, lse.cpu().double().numpy(), lse_ref)


def test_slot_past_capacity_is_recorded_and_skipped():
    torch = _torch()
    cfg = gen.ROPE_FP16
    p = Producer(cfg, "f16", batch=1, capacity=64)
    x = _x(cfg, 1, 40, "f16", seed=6)
    p.attn.project(p.w, x.cuda(), p.cache, torch.tensor([30], dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    with pytest.raises(p.P.PaluError) as e:
        p.attn.check_device()
    assert e.value.status == p.P.PALU_ERR_DEVICE
    # tokens 30..63 were written, 64..69 skipped
    assert torch.count_nonzero(p.cache.hk[0, 30:64]).item() > 0


def test_project_rejects_bad_arguments():
    torch = _torch()
    cfg = gen.ROPE_FP16
    p = Producer(cfg, "f16", batch=1, capacity=64)
    P_ = p.P
    x = _x(cfg, 1, 8, "f16", seed=7).cuda()
    slot = torch.zeros(1, dtype=torch.int32, device="cuda")
    s0 = torch.cuda.current_stream().cuda_stream
    c = p.cache.c_struct()
    st = P_.palu_project_latents(p.attn.handle, p.w.data_ptr(), P_.PALU_F16, cfg.hidden, x.data_ptr() + 2, c,
                                 slot.data_ptr(), 1, 8, s0)
    assert st == P_.PALU_ERR_INVALID_ARG                       # x not 16-byte aligned
    st = P_.palu_project_latents(p.attn.handle, p.w.data_ptr(), P_.PALU_F16, cfg.hidden - 32, x.data_ptr(), c,
                                 slot.data_ptr(), 1, 8, s0)
    assert st == P_.PALU_ERR_UNSUPPORTED                       # d_model not a multiple of 64
    st = P_.palu_project_latents(p.attn.handle, p.w.data_ptr(), P_.PALU_F16, cfg.hidden, x.data_ptr(), c,
                                 slot.data_ptr(), 2, 8, s0)
    assert st == P_.PALU_ERR_INVALID_ARG                       # batch above the handle's max_batch
    st = P_.palu_project_latents(p.attn.handle, p.w.data_ptr(), P_.PALU_F16, cfg.hidden, x.data_ptr(), c,
                                 slot.data_ptr(), 1, 0, s0)
    assert st == P_.PALU_OK                                    # nothing to do
    torch.cuda.synchronize()
