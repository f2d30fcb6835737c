"""GPU parity of decode over a hybrid cache (PuzzleKV section 3: dense sink page and local window
next to factorised pages, one softmax merged online; Shard section 7: fp16 sinks and window)
through the C ABI, against the float64 oracle."""
import numpy as np
import pytest

from oracle import palu_oracle as O
from synthetic import gen
from tests.gpu_cases import Case, assert_close

pytestmark = pytest.mark.gpu

SINKS, WINDOW = 4, 64


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    return cuda_device


def _dense_segment(cfg, c, n_dense, dtype, seed, sink_boost=3.0):
    """Seeded dense keys and values [B][D][n][d_h], scaled like the case's rebuilt keys and value
    latents; the first two tokens of each row are made large (attention sinks)."""
    rng = np.random.default_rng(seed)
    B, n, d_h = cfg.batch, cfg.n_heads, cfg.head_dim
    D = max(max(n_dense), 1)
    k_ref = c.hk64[0, :64, 0] @ c.bk64[0][:, :d_h]
    sk = float(np.std(k_ref)) if k_ref.size else 1.0
    dk = rng.standard_normal((B, D, n, d_h)).astype(np.float32) * sk
    dk[:, :2] *= sink_boost
    dv = rng.standard_normal((B, D, n, d_h)).astype(np.float32)
    return gen.storage_round(dk, dtype), gen.storage_round(dv, dtype)


def _run(cfg, seq_mid, n_dense, dense_dtype="f16", *, seed=0, q_scale=1.0):
    import torch
    B = cfg.batch
    T = cfg.T
    pos = np.stack([SINKS + np.arange(T) for _ in range(B)]).astype(np.int32)
    q_pos = [SINKS + int(s) + WINDOW - 1 for s in seq_mid]
    c = Case(cfg, seq_lens=seq_mid, positions=pos if cfg.mode == "rope" else None, q_pos=q_pos,
             max_position=SINKS + T + WINDOW, q_scale=q_scale)
    dk, dv = _dense_segment(cfg, c, n_dense, dense_dtype, seed)
    dev = c.dev
    seq = torch.tensor(seq_mid, dtype=torch.int32, device=dev)
    posd = torch.zeros((B, c.capacity), dtype=torch.int32, device=dev)
    posd[:, :T] = torch.from_numpy(pos).to(dev)
    qp = torch.tensor(q_pos, dtype=torch.int32, device=dev)
    nd = torch.tensor(n_dense, dtype=torch.int32, device=dev)
    out, out_d, lse = c.attn.decode_hybrid(c.q_t.to(dev), c.cache, seq, dk.to(dev), dv.to(dev), nd,
                                           max_seq_len=int(max(seq_mid)), positions=posd if cfg.mode == "rope" else None,
                                           q_pos=qp if cfg.mode == "rope" else None)
    torch.cuda.synchronize()
    c.attn.check_device()
    ref_l, ref_d, ref_lse = O.decode_hybrid(c.q64, c.hk64, c.hv64, c.bk64, seq_mid, cfg.group_size,
                                           dk.double().numpy(), dv.double().numpy(), n_dense, mode=cfg.mode,
                                           theta=cfg.theta, positions=pos if cfg.mode == "rope" else None,
                                           q_pos=q_pos)
    return (out.cpu().double().numpy(), out_d.cpu().double().numpy(), lse.cpu().double().numpy(),
            ref_l, ref_d, ref_lse)


def _check(res, f32=False):
    out, out_d, lse, ref_l, ref_d, ref_lse = res
    assert_close(out, ref_l, lse, ref_lse, f32=f32)
    assert_close(out_d, ref_d, f32=f32)


@pytest.mark.parametrize("T", [1, 129, 700])
def test_rope_fp16_middle_with_sinks_and_window(T):
    cfg = gen.ROPE_FP16.with_(T=T, batch=2)
    _check(_run(cfg, [T, max(1, T // 2)], [SINKS + WINDOW, SINKS + 10]))


def test_rope_m_lrd_middle_packed_groups():
    # s = 1 rank 64 runs as packed groups; the dense merge rescales each head's own latent slice
    cfg = gen.ROPE_FP16.with_(T=300, batch=2, group_size=1, rank=64)
    _check(_run(cfg, [300, 130], [SINKS + WINDOW, SINKS + 3], seed=3))


def test_rope_int4_middle_bf16_dense():
    cfg = gen.ROPE_INT4.with_(T=500, batch=2)
    _check(_run(cfg, [500, 300], [SINKS + WINDOW, SINKS + WINDOW], "bf16", seed=1))


def test_rope_bf16_middle_fp32_dense_peaked():
    cfg = gen.ROPE_BF16.with_(T=300, batch=2)
    _check(_run(cfg, [300, 1], [SINKS + WINDOW, 3], "f32", seed=2, q_scale=8.0))


def test_absorbed_middle_with_dense_segment():
    cfg = gen.ABSORBED_FP16.with_(T=333, batch=2)
    _check(_run(cfg, [333, 100], [SINKS + WINDOW, 20], seed=3))


@pytest.mark.parametrize("s,rank", [(1, 64), (8, 256)])
def test_absorbed_packed_and_split_groups_with_dense_segment(s, rank):
    # M-LRD packed four heads at a time, and s = 8 split into four-head groups, under the dense merge
    cfg = gen.ABSORBED_FP16.with_(T=400, batch=2, group_size=s, rank=rank)
    _check(_run(cfg, [400, 97], [SINKS + WINDOW, 2], seed=7))


def test_empty_middle_empty_dense_and_both_empty():
    cfg = gen.ROPE_FP16.with_(T=200, batch=3)
    out, out_d, lse, ref_l, ref_d, ref_lse = _run(cfg, [0, 200, 0], [SINKS + WINDOW, 0, 0], seed=4)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(out_d[1] == 0) and np.all(out_d[2] == 0)
    assert np.all(lse[2] == -np.inf)
    _check((out, out_d, lse, ref_l, ref_d, ref_lse))


def test_full_size_int4_middle_sampled_heads():
    # the 64K int4 layer with 4 sink and 64 window tokens around a 65468-token latent middle
    import torch
    cfg = gen.ROPE_INT4
    B, T = cfg.batch, cfg.T - SINKS - WINDOW
    cfg = cfg.with_(T=T)
    pos = np.stack([SINKS + np.arange(T) for _ in range(B)]).astype(np.int32)
    q_pos = [SINKS + T + WINDOW - 1] * B
    c = Case(cfg, positions=pos, q_pos=q_pos, max_position=SINKS + T + WINDOW)
    n_dense = [SINKS + WINDOW] * B
    dk, dv = _dense_segment(cfg, c, n_dense, "f16", 5)
    dev = c.dev
    posd = torch.from_numpy(pos).to(dev)
    out, out_d, lse = c.attn.decode_hybrid(c.q_t.to(dev), c.cache, torch.full((B,), T, dtype=torch.int32, device=dev),
                                           dk.to(dev), dv.to(dev), torch.tensor(n_dense, dtype=torch.int32, device=dev),
                                           max_seq_len=T, positions=posd,
                                           q_pos=torch.tensor(q_pos, dtype=torch.int32, device=dev))
    torch.cuda.synchronize()
    c.attn.check_device()
    heads = [(0, 0), (1, 17), (3, 31)]
    ref_l, ref_d, ref_lse = O.decode_hybrid(c.q64, c.hk64, c.hv64, c.bk64, [T] * B, cfg.group_size,
                                           dk.double().numpy(), dv.double().numpy(), n_dense, theta=cfg.theta,
                                           positions=pos, q_pos=q_pos, heads=heads)
    o, od, ls = out.cpu().double().numpy(), out_d.cpu().double().numpy(), lse.cpu().double().numpy()
    assert_close(o, ref_l, ls, ref_lse, heads=heads)
    assert_close(od, ref_d, heads=heads)


def test_hybrid_rejects_bad_arguments():
    import torch
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ROPE_FP16.with_(T=128, batch=1)
    c = Case(cfg)
    dev = c.dev
    dk = torch.zeros((1, 8, cfg.n_heads, cfg.head_dim), dtype=torch.float16, device=dev)
    nd = torch.zeros(1, dtype=torch.int32, device=dev)
    seq = torch.full((1,), 128, dtype=torch.int32, device=dev)
    out = torch.empty((1, cfg.n_heads, cfg.rank), dtype=torch.float32, device=dev)
    od = torch.empty((1, cfg.n_heads, cfg.head_dim), dtype=torch.float32, device=dev)
    lse = torch.empty((1, cfg.n_heads), dtype=torch.float32, device=dev)
    dense = P.palu_dense_cache(dk.data_ptr(), dk.data_ptr(), nd.data_ptr(), 8, P.PALU_F16)
    s0 = torch.cuda.current_stream().cuda_stream
    q = c.q_t.to(dev)
    st = P.palu_decode_hybrid(c.attn.handle, q.data_ptr(), c.cache.c_struct(), seq.data_ptr(), None, None, 1, 128,
                              dense, out.data_ptr(), od.data_ptr(), lse.data_ptr(), s0)
    assert st == P.PALU_ERR_INVALID_ARG                       # RoPE path without q_pos
    qp = torch.full((1,), 127, dtype=torch.int32, device=dev)
    st = P.palu_decode_hybrid(c.attn.handle, q.data_ptr(), c.cache.c_struct(), seq.data_ptr(), None, qp.data_ptr(),
                              1, 128, dense, out.data_ptr(), od.data_ptr(), None, s0)
    assert st == P.PALU_ERR_INVALID_ARG                       # lse is required
    bad = P.palu_dense_cache(dk.data_ptr(), dk.data_ptr(), nd.data_ptr(), 0, P.PALU_F16)
    st = P.palu_decode_hybrid(c.attn.handle, q.data_ptr(), c.cache.c_struct(), seq.data_ptr(), None, qp.data_ptr(),
                              1, 128, bad, out.data_ptr(), od.data_ptr(), lse.data_ptr(), s0)
    assert st == P.PALU_ERR_INVALID_ARG                       # zero dense capacity
    torch.cuda.synchronize()
