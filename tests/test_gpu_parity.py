"""GPU parity: the CUDA path through the C ABI against the float64 oracle on the
same seeded, storage-rounded inputs."""
import numpy as np
import pytest

from synthetic import gen
from tests.gpu_cases import Case, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    return cuda_device


def test_tiny_fp32_full():
    c = Case(gen.TINY_FP32)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref, f32=True)


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 1000])
def test_rope_fp16_tile_edges(T):
    cfg = gen.ROPE_FP16.with_(T=T, batch=2)
    c = Case(cfg, seq_lens=[T, max(1, (T * 2) // 3)])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_rope_bf16_explicit_positions_query_position_and_empty_row():
    cfg = gen.ROPE_BF16.with_(T=300, batch=3)
    rng = np.random.default_rng(5)
    pos = np.stack([rng.permutation(5000)[:300] for _ in range(3)]).astype(np.int32)
    c = Case(cfg, seq_lens=[300, 17, 0], positions=pos, q_pos=[4999, 123, 0], max_position=5000)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert np.all(out[2] == 0)
    assert_close(out, ref, lse, lse_ref)


def test_rope_default_query_position_with_positions():
    cfg = gen.ROPE_FP16.with_(T=200, batch=2)
    pos = (np.arange(200)[None, :] * 3 + np.array([[7], [1000]])).astype(np.int32)
    c = Case(cfg, seq_lens=[200, 150], positions=pos, max_position=2000)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


@pytest.mark.parametrize("T", [1, 63, 64, 65, 127, 128, 129])
@pytest.mark.parametrize("lat", ["f16", "bf16"])
def test_absorbed_stage_edges(lat, T):
    # the absorbed kernel streams 64-token stages, 8 tokens per warp: lengths at and around the
    # stage edges, with a shorter second row
    cfg = gen.ABSORBED_FP16.with_(T=T, batch=2, latent_dtype=lat)
    c = Case(cfg, seq_lens=[T, max(1, T - 37)])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


@pytest.mark.parametrize("lat", ["f16", "bf16"])
def test_absorbed_peaked_softmax_stress(lat):
    cfg = gen.ABSORBED_FP16.with_(T=777, batch=2, latent_dtype=lat)
    c = Case(cfg, seq_lens=[777, 300], q_scale=8.0)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


@pytest.mark.parametrize("T", [1, 2, 127, 128, 129, 1000])
def test_rope_bf16_tile_edges(T):
    cfg = gen.ROPE_BF16.with_(T=T, batch=2)
    c = Case(cfg, seq_lens=[T, max(1, (T * 2) // 3)])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_rope_bf16_peaked_softmax_stress():
    cfg = gen.ROPE_BF16.with_(T=600, batch=2)
    c = Case(cfg, seq_lens=[600, 257], q_scale=8.0)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_absorbed_fp16_ragged():
    cfg = gen.ABSORBED_FP16.with_(T=1000, batch=2)
    c = Case(cfg, seq_lens=[1000, 333])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_absorbed_bf16_ragged():
    cfg = gen.ABSORBED_FP16.with_(T=1000, batch=3, latent_dtype="bf16")
    c = Case(cfg, seq_lens=[1000, 1, 517])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_absorbed_int4_on_cuda_cores():
    cfg = gen.ABSORBED_FP16.with_(T=300, batch=2, latent_dtype="int4")
    c = Case(cfg, seq_lens=[300, 77])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


@pytest.mark.parametrize("base", [gen.ROPE_FP16, gen.ABSORBED_FP16], ids=lambda c: c.name)
def test_float32_query(base):
    cfg = base.with_(T=500, batch=2)
    c = Case(cfg, seq_lens=[500, 250], q_dtype="f32")
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_peaked_softmax_stress():
    cfg = gen.ROPE_FP16.with_(T=512, batch=1)
    c = Case(cfg, q_scale=8.0)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_split_plan_does_not_change_result():
    cfg = gen.ROPE_FP16.with_(T=700, batch=1)
    c = Case(cfg, capacity=4096)
    a, _ = c.run_gpu()
    b, _ = c.run_gpu(max_seq_len=4096)
    ref, _ = c.run_oracle()
    assert_close(a, ref)
    assert_close(b, ref)


def test_float_append_matches_round_to_nearest():
    import torch
    for lat in ("f16", "bf16"):
        cfg = gen.ROPE_FP16.with_(T=64, batch=2, latent_dtype=lat)
        c = Case(cfg)
        want = gen.storage_round(c.inp["hk"], lat)
        got = c.cache.hk[:, :64].cpu()
        assert torch.equal(got.view(torch.int16), want.view(torch.int16))


def test_int4_append_bit_exact_and_dequant():
    import torch
    cfg = gen.ROPE_INT4.with_(T=300, batch=2)
    c = Case(cfg)
    pk, sk, pv, sv = c.ref_packed
    np.testing.assert_array_equal(c.cache.hk[:, :300].cpu().numpy(), pk)
    np.testing.assert_array_equal(c.cache.hv[:, :300].cpu().numpy(), pv)
    np.testing.assert_array_equal(c.cache.k_scale[:, :300].cpu().numpy().view(np.uint16), sk.view(np.uint16))
    np.testing.assert_array_equal(c.cache.v_scale[:, :300].cpu().numpy().view(np.uint16), sv.view(np.uint16))
    from rank_kv_cache_gb300 import palu as P
    for which, ref in ((0, c.hk64), (1, c.hv64)):
        out = torch.empty((2, 300, cfg.n_groups, cfg.rank), dtype=torch.float32, device=c.dev)
        st = P.palu_debug_dequant(c.attn.handle, c.cache.c_struct(), which, 2, 300, out.data_ptr(),
                                  int(torch.cuda.current_stream().cuda_stream))
        assert st == 0
        np.testing.assert_array_equal(out.cpu().numpy(), ref)


def test_int4_rope_hadamard_ragged():
    cfg = gen.ROPE_INT4.with_(T=700, batch=2)
    c = Case(cfg, seq_lens=[700, 259])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


@pytest.mark.parametrize("T", [64, 127, 128, 129, 1000])
def test_int4_rope_tile_edges(T):
    # batch * capacity >= 128: the tensor-core kernel with the int4 converter
    cfg = gen.ROPE_INT4.with_(T=T, batch=2)
    c = Case(cfg, seq_lens=[T, max(1, (T * 2) // 3)])
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_int4_peaked_softmax_stress():
    # a few tokens dominate: the int4 p H_v path quantises each warp's 16 weights to 15 bits
    # against their largest, so the error stays a small fraction of the dominant term
    cfg = gen.ROPE_INT4.with_(T=900, batch=2)
    c = Case(cfg, seq_lens=[900, 611], q_scale=8.0)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_int4_rope_positions_and_split_plan():
    cfg = gen.ROPE_INT4.with_(T=700, batch=2)
    rng = np.random.default_rng(11)
    pos = np.stack([rng.permutation(3000)[:700] for _ in range(2)]).astype(np.int32)
    c = Case(cfg, seq_lens=[700, 450], positions=pos, q_pos=[2999, 5], capacity=4096, max_position=3000)
    a, la = c.run_gpu()
    b, lb = c.run_gpu(max_seq_len=4096)
    ref, lse_ref = c.run_oracle()
    assert_close(a, ref, la, lse_ref)
    assert_close(b, ref, lb, lse_ref)


def test_device_error_word_on_bad_position():
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_FP16.with_(T=64, batch=1)
    pos = np.arange(64, dtype=np.int32)[None, :].copy()
    pos[0, 10] = 100000  # outside the 64-entry table
    c = Case(cfg, positions=pos)
    with pytest.raises(P.PaluError) as ei:
        c.run_gpu()
    assert ei.value.status == P.PALU_ERR_DEVICE
    c.attn.check_device()  # cleared


# --- full workload sizes: every head where the oracle is quick, else sampled heads ---

def _sample_heads(B, n, k=6, seed=0):
    rng = np.random.default_rng(seed)
    hs = {(0, 0), (B - 1, n - 1)}
    while len(hs) < k:
        hs.add((int(rng.integers(B)), int(rng.integers(n))))
    return sorted(hs)


def test_full_rope_fp16_b1_t4k_all_heads():
    c = Case(gen.ROPE_FP16)
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


@pytest.mark.parametrize("base,T", [(gen.ROPE_BF16, 16384), (gen.ROPE_BF16, 32768), (gen.ABSORBED_FP16, 65536),
                                    (gen.ROPE_INT4, 65536)], ids=["rope-bf16-b8-t16k", "rope-bf16-b8-t32k",
                                                                  "absorbed-fp16-b4-t64k", "rope-int4-b4-t64k"])
def test_full_size_sampled_heads(base, T):
    cfg = base.with_(T=T)
    c = Case(cfg)
    out, lse = c.run_gpu()
    heads = _sample_heads(cfg.batch, cfg.n_heads)
    ref, lse_ref = c.run_oracle(heads=heads)
    assert_close(out, ref, lse, lse_ref, heads=heads)


@pytest.mark.parametrize("cfg,kernel", [(gen.TINY_FP32, "SIMT"), (gen.ROPE_FP16, "TC_ROPE"), (gen.ROPE_BF16, "TC_ROPE"),
                                        (gen.ABSORBED_FP16, "TMA_ABSORBED"), (gen.ROPE_INT4, "TC_ROPE")],
                         ids=lambda x: x.name if hasattr(x, "name") else x)
def test_kernel_choice_per_workload(cfg, kernel):
    # the fast kernels must be the ones the full-size workloads run on
    import torch
    from rank_kv_cache_gb300 import palu as P
    bk = torch.zeros((cfg.n_groups, cfg.rank, cfg.group_size * cfg.head_dim),
                     dtype={"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[cfg.bk_dtype],
                     device="cuda")
    attn = P.PaluAttention(bk, n_heads=cfg.n_heads, head_dim=cfg.head_dim, group_size=cfg.group_size,
                           rank_k=cfg.rank, rank_v=cfg.rank, latent_dtype=cfg.latent_dtype, q_dtype=cfg.q_dtype,
                           mode=cfg.mode, max_batch=cfg.batch, max_tokens=cfg.T)
    got, n_splits, launches = attn.plan(cfg.T, cfg.batch, cfg.T)
    assert got == getattr(P, "PALU_KERNEL_" + kernel)
    assert n_splits >= 1 and launches == (1 if kernel == "TC_ROPE" else 2)


def test_bounded_wait_gives_up_and_reports_timeout():
    # failure detection without a fault: with the test-stall flag the H_v producer of the
    # tensor-core kernel issues nothing, every consumer wait gives up after its bound, the
    # CTAs unwind, and the error word reports PALU_ERR_TIMEOUT; the context stays usable
    import torch
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_FP16.with_(T=300, batch=2)
    c = Case(cfg)
    stall = P.PaluAttention(c.bk_t.to(c.dev), n_heads=cfg.n_heads, head_dim=cfg.head_dim,
                            group_size=cfg.group_size, rank_k=cfg.rank, rank_v=cfg.rank, latent_dtype="f16",
                            q_dtype=cfg.q_dtype, mode="rope", max_batch=cfg.batch, max_tokens=cfg.T,
                            flags=P.PALU_FLAG_TEST_STALL)
    assert stall.plan(cfg.T, cfg.batch, cfg.T)[0] == P.PALU_KERNEL_TC_ROPE
    seq = torch.full((cfg.batch,), cfg.T, dtype=torch.int32, device=c.dev)
    stall.decode(c.q_t.to(c.dev), c.cache, seq, max_seq_len=cfg.T)
    torch.cuda.synchronize()
    with pytest.raises(P.PaluError) as ei:
        stall.check_device()
    assert ei.value.status == P.PALU_ERR_TIMEOUT
    stall.check_device()        # reading the error word cleared it
    out, lse = c.run_gpu()      # the normal handle still decodes correctly afterwards
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref)


def test_cache_saved_and_reloaded_decodes_identically():
    # the library keeps no state between calls: a cache copied out to the host and back
    # into fresh device buffers gives the same bits
    import torch
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_INT4.with_(T=400, batch=2)
    c = Case(cfg, seq_lens=[400, 123])
    out1, lse1 = c.run_gpu()
    saved = {k: getattr(c.cache, k).cpu() for k in ("hk", "hv", "k_scale", "v_scale")}
    fresh = P.LatentCache(cfg.batch, c.capacity, cfg.n_groups, cfg.rank, cfg.rank, "int4", device=c.dev)
    for k, v in saved.items():
        getattr(fresh, k).copy_(v.to(c.dev))
    c.cache = fresh
    out2, lse2 = c.run_gpu()
    assert np.array_equal(out1, out2) and np.array_equal(lse1, lse2)
