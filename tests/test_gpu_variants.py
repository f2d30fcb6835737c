"""GPU parity of the granularity and storage variants (Palu notes, method section: M-LRD, G-LRD
and J-LRD decompositions and the key-fusion paragraph's ALiBi; results section: 4-bit values
only), through the C ABI, against the float64 oracle."""
import numpy as np
import pytest

from synthetic import gen
from tests.gpu_cases import Case, assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    return cuda_device


def _check(c, **kw):
    out, lse = c.run_gpu()
    ref, lse_ref = c.run_oracle()
    assert_close(out, ref, lse, lse_ref, **kw)


def _kernel(c):
    return c.attn.plan(c.capacity, c.cfg.batch, int(c.seq_lens.max()))[0]


# ---------------------------------------------------------------- int4 values only

@pytest.mark.parametrize("T", [1, 129, 1000])
def test_value_only_int4_under_fp16_keys(T):
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_FP16.with_(T=T, batch=2, v_dtype="int4")
    c = Case(cfg, seq_lens=[T, max(1, (2 * T) // 3)])
    # the tensor-core kernel takes caches of at least 128 rows; smaller ones run on CUDA cores
    assert _kernel(c) == (P.PALU_KERNEL_TC_ROPE if 2 * T >= 128 else P.PALU_KERNEL_SIMT)
    _check(c)


def test_value_only_int4_under_bf16_keys_peaked():
    cfg = gen.ROPE_BF16.with_(T=500, batch=2, v_dtype="int4")
    _check(Case(cfg, seq_lens=[500, 77], q_scale=8.0))


def test_value_only_int4_absorbed():
    cfg = gen.ABSORBED_FP16.with_(T=333, batch=2, v_dtype="int4")
    _check(Case(cfg, seq_lens=[333, 100]))


def test_value_only_int4_long_sampled_heads():
    cfg = gen.ROPE_FP16.with_(T=32768, batch=2, v_dtype="int4")
    c = Case(cfg)
    out, lse = c.run_gpu()
    heads = [(0, 0), (0, 13), (1, 31)]
    ref, lse_ref = c.run_oracle(heads=heads)
    assert_close(out, ref, lse, lse_ref, heads=heads)


# ---------------------------------------------------------------- group sizes

@pytest.mark.parametrize("s", [2, 8])
def test_group_sizes_on_the_tensor_core_kernel(s):
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_FP16.with_(T=600, batch=2, group_size=s)
    c = Case(cfg, seq_lens=[600, 257])
    assert _kernel(c) == P.PALU_KERNEL_TC_ROPE
    _check(c)


# M-LRD (s = 1, rank 64 per head: the same total rank as G-LRD with s = 4 and rank 256) and G-LRD
# with s = 2 and rank 128 run as packed groups of four heads with a block-diagonal B_k on the
# tensor-core and TMA-stream kernels; every head's output is its own group's latent slice
@pytest.mark.parametrize("mode,lat,s,T,batch,seqs,qs", [
    ("rope", "f16", 1, 300, 2, [300, 150], 1.0),
    ("rope", "bf16", 1, 129, 2, [129, 128], 8.0),
    ("rope", "f16", 2, 1000, 2, [1000, 257], 1.0),
    ("rope", "f16", 1, 100, 1, [100], 1.0),          # fewer than 128 cache rows: CUDA-core kernel
    ("absorbed", "f16", 1, 333, 2, [333, 65], 1.0),
    ("absorbed", "bf16", 2, 200, 2, [200, 129], 8.0),
])
def test_packed_groups_m_lrd_and_s2(mode, lat, s, T, batch, seqs, qs):
    from rank_kv_cache_gb300 import palu as P
    base = gen.ROPE_FP16 if mode == "rope" else gen.ABSORBED_FP16
    cfg = base.with_(T=T, batch=batch, group_size=s, rank=64 * s, latent_dtype=lat)
    c = Case(cfg, seq_lens=seqs, q_scale=qs)
    fast = P.PALU_KERNEL_TC_ROPE if mode == "rope" else P.PALU_KERNEL_TMA_ABSORBED
    assert _kernel(c) == (fast if batch * T >= 128 else P.PALU_KERNEL_SIMT)
    _check(c)


def test_packed_m_lrd_long_sampled_heads():
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_FP16.with_(T=4096, batch=1, group_size=1, rank=64)
    c = Case(cfg)
    assert _kernel(c) == P.PALU_KERNEL_TC_ROPE
    out, lse = c.run_gpu()
    heads = [(0, 0), (0, 1), (0, 2), (0, 3), (0, 30)]
    ref, lse_ref = c.run_oracle(heads=heads)
    assert_close(out, ref, lse, lse_ref, heads=heads)


def test_joint_decomposition_j_lrd():
    # s = n = 32: one group for all heads, rank 256, on the tensor-core kernel
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_FP16.with_(T=300, batch=1, group_size=32)
    c = Case(cfg)
    assert _kernel(c) == P.PALU_KERNEL_TC_ROPE
    _check(c)


# G-LRD with s = 8, 16 and J-LRD (s = 32) at rank 256 on the absorbed path run as split groups: four
# heads per kernel group over their group's shared latents, on the TMA-streamed kernel
@pytest.mark.parametrize("lat,s,T,batch,seqs,qs,alibi", [
    ("f16", 8, 300, 2, [300, 150], 1.0, False),
    ("bf16", 16, 129, 2, [129, 64], 8.0, False),
    ("f16", 32, 1000, 1, [1000], 1.0, True),
    ("f16", 8, 40, 1, [40], 1.0, False),             # fewer than 64 cache rows: CUDA-core kernel
])
def test_split_groups_on_the_absorbed_path(lat, s, T, batch, seqs, qs, alibi):
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ABSORBED_FP16.with_(T=T, batch=batch, group_size=s, latent_dtype=lat)
    c = Case(cfg, seq_lens=seqs, q_scale=qs, alibi=alibi)
    assert _kernel(c) == (P.PALU_KERNEL_TMA_ABSORBED if batch * T >= 64 else P.PALU_KERNEL_SIMT)
    _check(c)


# ---------------------------------------------------------------- ALiBi on the absorbed path

@pytest.mark.parametrize("dt", ["f16", "bf16"])
def test_alibi_absorbed_stream_kernel(dt):
    from rank_kv_cache_gb300 import palu as P
    base = gen.ABSORBED_FP16 if dt == "f16" else gen.ABSORBED_FP16.with_(latent_dtype="bf16")
    cfg = base.with_(T=1000, batch=3)
    rng = np.random.default_rng(9)
    pos = np.stack([np.sort(rng.choice(5000, 1000, replace=False)) for _ in range(3)]).astype(np.int32)
    c = Case(cfg, seq_lens=[1000, 65, 0], positions=pos, q_pos=[5000, 700, 0], max_position=6000, alibi=True)
    assert _kernel(c) == P.PALU_KERNEL_TMA_ABSORBED
    _check(c)


def test_alibi_absorbed_default_positions_int4_and_s2_on_cuda_cores():
    _check(Case(gen.ABSORBED_FP16.with_(T=300, batch=2, latent_dtype="int4"), seq_lens=[300, 31], alibi=True))
    _check(Case(gen.ABSORBED_FP16.with_(T=300, batch=2, group_size=2), seq_lens=[300, 200], alibi=True))


def test_alibi_is_refused_where_it_cannot_apply():
    import torch
    from rank_kv_cache_gb300 import palu as P
    d = P.make_desc(n_heads=32, head_dim=128, group_size=4, rank_k=256, rank_v=256, latent_dtype="f16",
                    q_dtype="f16", mode="rope", flags=P.PALU_FLAG_ALIBI)
    assert P.palu_attn_workspace_size(d)[0] == P.PALU_ERR_INVALID_ARG
    cfg = gen.ABSORBED_FP16.with_(T=128, batch=1)
    c = Case(cfg, alibi=True)
    dev = c.dev
    seq = torch.full((1,), 128, dtype=torch.int32, device=dev)
    out = torch.empty((1, cfg.n_heads, cfg.rank), dtype=torch.float32, device=dev)
    s0 = torch.cuda.current_stream().cuda_stream
    st = P.palu_decode_attn_noalloc(c.attn.desc, c.attn._bk.data_ptr(), c.q_t.to(dev).data_ptr(), c.cache.c_struct(),
                                    seq.data_ptr(), 1, 128, out.data_ptr(), None, s0)
    assert st == P.PALU_ERR_UNSUPPORTED
    dk = torch.zeros((1, 4, cfg.n_heads, cfg.head_dim), dtype=torch.float16, device=dev)
    nd = torch.zeros(1, dtype=torch.int32, device=dev)
    with pytest.raises(P.PaluError) as e:
        c.attn.decode_hybrid(c.q_t.to(dev), c.cache, seq, dk, dk, nd, max_seq_len=128)
    assert e.value.status == P.PALU_ERR_UNSUPPORTED
    torch.cuda.synchronize()
