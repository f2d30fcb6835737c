"""GPU parity of the layer's output projection with B_v fused into W_o (Palu notes,
method section, value-fusion paragraph): the fused weight W_f^(i) = B_v^(i) W_o^(i)
and the per-step GEMV y = o W_f, through the C ABI, against the float64 oracle."""
import numpy as np
import pytest

from oracle import palu_oracle as O
from synthetic import gen
from tests.gpu_cases import Case

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu(cuda_device):
    return cuda_device


def _torch():
    import torch
    return torch


def _draw(n_heads, head_dim, s, r_v, d, seed):
    rng = np.random.default_rng(seed)
    bv = rng.standard_normal((n_heads // s, r_v, s * head_dim)) / np.sqrt(r_v)
    wo = rng.standard_normal((n_heads * head_dim, d)) / np.sqrt(n_heads * head_dim)
    return bv, wo


def _fuse_gpu(bv_t, wo_t, n_heads, head_dim, s, r_v, out="f16"):
    from rank_kv_cache_gb300 import palu as P
    torch = _torch()
    dev = torch.device("cuda:0")
    proj = P.OutputProjection(bv_t.to(dev), wo_t.to(dev), n_heads=n_heads, head_dim=head_dim, group_size=s,
                              rank_v=r_v, max_batch=16, dtype=out)
    torch.cuda.synchronize()
    return proj


def _check_fused_weight(wf_gpu, bv64, wo64, s):
    """Each fused element within one unit in the last place of the float64 value rounded to the
    output dtype, plus fp32 accumulation error over head_dim terms."""
    ref = O.fuse_value_output(bv64, wo64, s)
    mag = O.fuse_value_output(np.abs(bv64), np.abs(wo64), s)   # sum of |terms| per element
    got = wf_gpu.double().numpy()
    if wf_gpu.dtype == _torch().float16:
        ulp = np.spacing(np.abs(ref).astype(np.float16)).astype(np.float64)     # subnormals included
    else:   # bf16: fp32's exponent range with 8 significant bits
        ulp = np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) * 2.0 ** 16
    bound = ulp + 1e-6 * mag
    err = np.abs(got - ref)
    assert np.all(err <= bound), f"fused weight off by {float((err / bound).max()):.2f} of its bound"
    return float(err.max())


@pytest.mark.parametrize("in_dt,out_dt", [("f32", "f16"), ("f16", "f16"), ("bf16", "bf16"), ("f16", "bf16")])
def test_fused_weight_matches_oracle_ragged(in_dt, out_dt):
    n, d_h, s, r_v, d = 6, 64, 3, 100, 4104
    bv, wo = _draw(n, d_h, s, r_v, d, seed=11)
    bv_t, wo_t = gen.storage_round(bv, in_dt), gen.storage_round(wo, in_dt)
    proj = _fuse_gpu(bv_t, wo_t, n, d_h, s, r_v, out=out_dt)
    _check_fused_weight(proj.w.cpu(), bv_t.double().numpy(), wo_t.double().numpy(), s)


@pytest.mark.parametrize("batch", [1, 2, 3, 5, 8, 13])
def test_projection_matches_oracle_on_ragged_shapes(batch):
    # k_dim = 600 (not a multiple of the 128-row quantum), d = 4104 (a 8-column tail block),
    # batch sizes over every batch-block width and a partial last block
    torch = _torch()
    n, d_h, s, r_v, d = 6, 64, 3, 100, 4104
    bv, wo = _draw(n, d_h, s, r_v, d, seed=12)
    proj = _fuse_gpu(gen.storage_round(bv, "f16"), gen.storage_round(wo, "f16"), n, d_h, s, r_v)
    o = np.random.default_rng(batch).standard_normal((batch, n, r_v)).astype(np.float32)
    y = proj(torch.from_numpy(o).cuda().reshape(batch, -1))
    torch.cuda.synchronize()
    w64 = proj.w.cpu().double().numpy()
    ref = O.project_fused(o.astype(np.float64), w64)
    mag = O.project_fused(np.abs(o.astype(np.float64)), np.abs(w64))
    err = np.abs(y.cpu().double().numpy() - ref)
    assert np.all(err <= 2e-6 * mag + 1e-6), float((err / (2e-6 * mag + 1e-6)).max())


def test_projection_is_deterministic_and_leaves_workspace_ready():
    torch = _torch()
    n, d_h, s, r_v, d = 32, 128, 4, 256, 4096
    bv, wo = _draw(n, d_h, s, r_v, d, seed=13)
    proj = _fuse_gpu(gen.storage_round(bv, "f16"), gen.storage_round(wo, "f16"), n, d_h, s, r_v)
    o1 = torch.randn((4, n * r_v), generator=torch.Generator().manual_seed(1)).cuda()
    o2 = torch.randn((3, n * r_v), generator=torch.Generator().manual_seed(2)).cuda()
    y1a = proj(o1).clone()
    y2 = proj(o2).clone()
    y1b = proj(o1).clone()
    torch.cuda.synchronize()
    assert torch.equal(y1a, y1b)
    w64 = proj.w.cpu().double().numpy()
    for o, y in ((o1, y1a), (o2, y2)):
        ref = O.project_fused(o.cpu().double().numpy().reshape(o.shape[0], n, r_v), w64)
        assert float(np.abs(y.cpu().double().numpy() - ref).max()) <= 1e-4 * float(np.abs(ref).max())


def test_layer_output_from_decode_matches_oracle():
    # the decode kernel's latent output o, projected with the fused weight, against the oracle's
    # o projected with the float64 fused weight of the same storage-rounded B_v and W_o
    torch = _torch()
    cfg = gen.ROPE_FP16.with_(T=700, batch=2)
    c = Case(cfg, seq_lens=[700, 333])
    out, _ = c.run_gpu(with_lse=False)
    ref_o, _ = c.run_oracle()
    inp = gen.make_inputs(cfg, with_wo=True)
    bv_t, wo_t = gen.storage_round(inp["bv"], "f16"), gen.storage_round(inp["wo"], "f16")
    n, d_h, s, r_v = cfg.n_heads, cfg.head_dim, cfg.group_size, cfg.rank
    proj = _fuse_gpu(bv_t, wo_t, n, d_h, s, r_v)
    o_dev = torch.from_numpy(out.astype(np.float32)).cuda().reshape(cfg.batch, -1)
    y = proj(o_dev).cpu().double().numpy()
    y_ref = O.project_fused(ref_o, O.fuse_value_output(bv_t.double().numpy(), wo_t.double().numpy(), s))
    rel = float(np.abs(y - y_ref).max() / np.abs(y_ref).max())
    assert rel <= 1e-2, rel


def test_full_size_fused_weight_and_projection():
    # Llama-2-7B layer: 32 heads, d_h 128, s 4, r_v 256, d 4096 (a 64 MB fp16 fused weight)
    torch = _torch()
    cfg = gen.ROPE_FP16
    inp = gen.make_inputs(cfg.with_(T=1, batch=1), with_wo=True)
    bv_t, wo_t = gen.storage_round(inp["bv"], "f16"), gen.storage_round(inp["wo"], "f16")
    n, d_h, s, r_v = cfg.n_heads, cfg.head_dim, cfg.group_size, cfg.rank
    proj = _fuse_gpu(bv_t, wo_t, n, d_h, s, r_v)
    _check_fused_weight(proj.w.cpu(), bv_t.double().numpy(), wo_t.double().numpy(), s)
    o = torch.randn((4, n * r_v), generator=torch.Generator().manual_seed(3)).cuda()
    y = proj(o).cpu().double().numpy()
    w64 = proj.w.cpu().double().numpy()
    on = o.cpu().double().numpy().reshape(4, n, r_v)
    ref = O.project_fused(on, w64)
    mag = O.project_fused(np.abs(on), np.abs(w64))
    assert np.all(np.abs(y - ref) <= 2e-6 * mag + 1e-6)


def test_projection_rejects_bad_arguments():
    torch = _torch()
    from rank_kv_cache_gb300 import palu as P
    dev = torch.device("cuda:0")
    w = torch.zeros((256, 4096), dtype=torch.float16, device=dev)
    o = torch.zeros((2, 256), dtype=torch.float32, device=dev)
    y = torch.zeros((2, 4096), dtype=torch.float32, device=dev)
    st, nbytes = P.palu_output_proj_workspace_size(256, 4096, 2)
    assert st == P.PALU_OK
    ws = torch.zeros(nbytes + 256, dtype=torch.uint8, device=dev)
    base = int(ws.data_ptr())
    wsp = base + (-base) % 256
    s0 = torch.cuda.current_stream().cuda_stream
    ok = P.palu_output_proj(w.data_ptr(), P.PALU_F16, 256, 4096, o.data_ptr(), 2, y.data_ptr(), wsp, nbytes, s0)
    assert ok == P.PALU_OK
    assert P.palu_output_proj(w.data_ptr(), P.PALU_F16, 256, 4100, o.data_ptr(), 2, y.data_ptr(), wsp, nbytes,
                              s0) == P.PALU_ERR_INVALID_ARG          # d_model not a multiple of 8
    assert P.palu_output_proj(w.data_ptr(), P.PALU_F16, 1 << 17, 4096, o.data_ptr(), 2, y.data_ptr(), wsp, nbytes,
                              s0) == P.PALU_ERR_UNSUPPORTED          # k_dim above 65536
    assert P.palu_output_proj(w.data_ptr(), P.PALU_F16, 256, 4096, o.data_ptr(), 2, y.data_ptr(), wsp, 16,
                              s0) == P.PALU_ERR_WORKSPACE            # workspace too small
    assert P.palu_output_proj(w.data_ptr() + 2, P.PALU_F16, 256, 4096, o.data_ptr(), 2, y.data_ptr(), wsp,
                              nbytes, s0) == P.PALU_ERR_INVALID_ARG  # weight not 16-byte aligned
    assert P.palu_output_proj(w.data_ptr(), P.PALU_F16, 256, 4096, o.data_ptr(), 0, y.data_ptr(), wsp, nbytes,
                              s0) == P.PALU_OK                       # empty batch: nothing to do
    torch.cuda.synchronize()
