"""GPU parity of decode over a page-factorised cache (PuzzleKV section 3.3: every completed page
of a head stored as rank-r factors, scored as (q R_K^T) L_K^T / sqrt(d) and read as p L_V R_V,
one softmax with the dense sink and window tokens) through the C ABI, against the float64 oracle."""
import numpy as np
import pytest

from oracle import palu_oracle as O
from synthetic import gen
from tests.gpu_cases import assert_close

pytestmark = pytest.mark.gpu

N_HEADS, D_H = 32, 128


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    return cuda_device


def _handle(mode, q_dtype="f16", max_batch=4):
    """A handle for the heads, head_dim, mode and RoPE table (its latent shape is not used here)."""
    import torch
    from rank_kv_cache_gb300 import palu as P
    bk = torch.zeros((8, 256, 4 * D_H), dtype=torch.float16, device="cuda")
    return P.PaluAttention(bk, n_heads=N_HEADS, head_dim=D_H, group_size=4, rank_k=256, rank_v=256,
                           latent_dtype="f16", q_dtype=q_dtype, mode=mode, max_batch=max_batch,
                           max_tokens=4096, max_position=8192)


def _run(mode, dtype, rank, n_pages, n_dense, *, capacity=None, seed=0, q_scale=1.0, dense_dtype="f16"):
    import torch
    B = len(n_pages)
    cap = capacity or max(max(n_pages), 1)
    lk, rk, lv, rv = gen.page_factor_draw(seed, B, cap, N_HEADS, rank=rank)
    lk, rk, lv, rv = (gen.storage_round(a, dtype).float().numpy() for a in (lk, rk, lv, rv))
    rec = gen.storage_round(gen.page_records(lk, rk, lv, rv), dtype).to("cuda")
    rng = np.random.default_rng(1000 + seed)
    q = gen.storage_round(rng.standard_normal((B, N_HEADS, D_H)) * q_scale, "f16")
    D = max(max(n_dense), 1)
    dk = gen.storage_round(rng.standard_normal((B, D, N_HEADS, D_H)) * 1.5, dense_dtype)
    dk[:, :2] *= 3                                     # attention sinks
    dv = gen.storage_round(rng.standard_normal((B, D, N_HEADS, D_H)), dense_dtype)
    q_pos = [int(x) for x in rng.integers(0, 8000, B)]
    attn = _handle(mode)
    dev = "cuda"
    npg = torch.tensor(n_pages, dtype=torch.int32, device=dev)
    nd = torch.tensor(n_dense, dtype=torch.int32, device=dev)
    qp = torch.tensor(q_pos, dtype=torch.int32, device=dev)
    use_dense = any(n_dense)
    out, out_d, lse = attn.decode_paged(q.to(dev), rec, npg, max_pages=cap, q_pos=qp if mode == "rope" else None,
                                        dense_k=dk.to(dev) if use_dense else None,
                                        dense_v=dv.to(dev) if use_dense else None, dense_n=nd if use_dense else None)
    torch.cuda.synchronize()
    attn.check_device()
    ref_p, ref_d, ref_lse = O.decode_paged(q.double().numpy(), lk, rk, lv, rv, n_pages, dk.double().numpy(),
                                           dv.double().numpy(), n_dense if use_dense else [0] * B, mode=mode,
                                           q_pos=q_pos)
    attn.close()
    got_d = out_d.cpu().double().numpy() if use_dense else np.zeros_like(ref_d)
    return out.cpu().double().numpy(), got_d, lse.cpu().double().numpy(), ref_p, ref_d, ref_lse


def _check(res):
    out, out_d, lse, ref_p, ref_d, ref_lse = res
    assert_close(out, ref_p, lse, ref_lse)
    assert_close(out_d, ref_d)


@pytest.mark.parametrize("rank", [8, 16, 32])
def test_rope_fp16_pages_with_sinks_and_window(rank):
    _check(_run("rope", "f16", rank, [40, 17], [68, 5], seed=rank))


def test_absorbed_bf16_pages_without_dense_tokens():
    _check(_run("absorbed", "bf16", 8, [33, 1, 0], [0, 0, 0], seed=2))


def test_rope_bf16_pages_rank32_fp32_dense_peaked():
    _check(_run("rope", "bf16", 32, [70, 23], [68, 40], seed=6, q_scale=6.0, dense_dtype="f32"))


def test_peaked_softmax_fp16_rank16():
    _check(_run("rope", "f16", 16, [64, 9], [68, 68], seed=3, q_scale=8.0))


def test_many_pages_split_plan_and_ragged_rows():
    # enough pages that the plan splits each (row, head) over several CTAs; rows end mid-split
    _check(_run("rope", "f16", 16, [517, 300, 1], [4, 0, 68], capacity=600, seed=4))


def test_no_pages_is_dense_attention_and_empty_rows():
    res = _run("rope", "f16", 16, [0, 0], [68, 0], seed=5)
    out, out_d, lse, ref_p, ref_d, ref_lse = res
    assert np.all(out[0] == 0) and np.all(out[1] == 0)
    assert np.all(np.isneginf(lse[1]))
    _check(res)


def test_bad_arguments_are_refused():
    import torch
    from rank_kv_cache_gb300 import palu as P
    attn = _handle("rope")
    q = torch.zeros((1, N_HEADS, D_H), dtype=torch.float16, device="cuda")
    rec = torch.zeros((1, 2, N_HEADS, 320 * 16), dtype=torch.float16, device="cuda")
    npg = torch.ones(1, dtype=torch.int32, device="cuda")
    qp = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(P.PaluError) as e:                      # the RoPE path needs q_pos
        attn.decode_paged(q, rec, npg, max_pages=2)
    assert e.value.status == P.PALU_ERR_INVALID_ARG
    with pytest.raises(P.PaluError) as e:                      # max_pages above the capacity
        attn.decode_paged(q, rec, npg, max_pages=3, q_pos=qp)
    assert e.value.status == P.PALU_ERR_INVALID_ARG
    with pytest.raises(ValueError):                            # not a 640 r-byte record
        attn.decode_paged(q, rec[..., :100].contiguous(), npg, max_pages=2, q_pos=qp)
    torch.cuda.synchronize()
    attn.close()


def test_page_count_above_the_bound_is_clamped_and_recorded():
    import torch
    from rank_kv_cache_gb300 import palu as P
    B, cap, rank = 1, 6, 8
    lk, rk, lv, rv = gen.page_factor_draw(9, B, cap, N_HEADS, rank=rank)
    lk, rk, lv, rv = (gen.storage_round(a, "f16").float().numpy() for a in (lk, rk, lv, rv))
    rec = gen.storage_round(gen.page_records(lk, rk, lv, rv), "f16").to("cuda")
    q = gen.storage_round(np.random.default_rng(9).standard_normal((B, N_HEADS, D_H)), "f16")
    attn = _handle("absorbed")
    npg = torch.tensor([cap + 5], dtype=torch.int32, device="cuda")     # more pages than the call's bound
    out, _, lse = attn.decode_paged(q.to("cuda"), rec, npg, max_pages=cap)
    torch.cuda.synchronize()
    with pytest.raises(P.PaluError) as e:
        attn.check_device()
    assert e.value.status == P.PALU_ERR_DEVICE
    ref_p, _, ref_lse = O.decode_paged(q.double().numpy(), lk, rk, lv, rv, [cap], np.zeros((B, 0, N_HEADS, D_H)),
                                       np.zeros((B, 0, N_HEADS, D_H)), [0], mode="absorbed")
    assert_close(out.cpu().double().numpy(), ref_p, lse.cpu().double().numpy(), ref_lse)
    attn.close()
