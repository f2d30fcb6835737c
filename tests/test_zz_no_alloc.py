"""The no-allocation decode entry point against the oracle and the regular one.

Callers that cannot call cudaMalloc (a plugin whose host process owns all device
memory, an engine with a fixed memory plan) use palu_decode_attn_noalloc, which
keeps its scratch in a fixed device array inside the library. Each case runs two
calls in a row with different sequence lengths, so that scratch left over from the
first call would show up in the second. This file is collected last so that a
stop-at-first-failure run has already run every other test; it also passes on its
own in a fresh process.
"""
import numpy as np
import pytest
import torch

from synthetic import gen
from tests.gpu_cases import Case, assert_close

pytestmark = pytest.mark.gpu


def _noalloc(c, seq, max_seq_len, out, lse):
    from rank_kv_cache_gb300 import palu as P
    bk_dev = c.attn._bk
    return P.palu_decode_attn_noalloc(c.attn.desc, bk_dev.data_ptr(), c.q_dev.data_ptr(), c.cache.c_struct(),
                                      seq.data_ptr(), c.cfg.batch, max_seq_len, out.data_ptr(),
                                      lse.data_ptr(), int(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("lat,T,batch", [("f16", 1000, 2), ("f16", 4096, 4), ("bf16", 777, 3), ("int4", 600, 2)])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(cuda_device, lat, T, batch):
    cfg = gen.ABSORBED_FP16.with_(T=T, batch=batch, latent_dtype=lat)
    seq_a = [T] + [max(1, T // (k + 2)) for k in range(batch - 1)]
    seq_b = [max(1, T // 3)] + [T - 5 * k for k in range(1, batch)]
    c = Case(cfg, seq_lens=seq_a)
    c.q_dev = c.q_t.to(c.dev)
    for seq_lens in (seq_a, seq_b):                     # two calls in a row share the fixed scratch
        c.seq_lens = np.array(seq_lens, dtype=np.int32)
        ref, lse_ref = c.run_oracle()
        ws_out, ws_lse = c.run_gpu(max_seq_len=T)       # regular entry point (workspace)
        seq = torch.tensor(seq_lens, dtype=torch.int32, device=c.dev)
        out = torch.full((batch, cfg.n_heads, cfg.rank), float("nan"), dtype=torch.float32, device=c.dev)
        lse = torch.full((batch, cfg.n_heads), float("nan"), dtype=torch.float32, device=c.dev)
        assert _noalloc(c, seq, T, out, lse) == 0
        torch.cuda.synchronize()
        got, got_lse = out.cpu().double().numpy(), lse.cpu().double().numpy()
        assert_close(got, ref, got_lse, lse_ref)
        assert_close(got, ws_out, got_lse, ws_lse)


def test_noalloc_rejects_bad_requests(cuda_device):
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ABSORBED_FP16.with_(T=64, batch=1)
    c = Case(cfg)
    c.q_dev = c.q_t.to(c.dev)
    stream = int(torch.cuda.current_stream().cuda_stream)
    big = P.make_desc(n_heads=1024, head_dim=128, group_size=4, rank_k=256, rank_v=256, latent_dtype="f16",
                      q_dtype="f16", mode="absorbed", max_batch=8, max_tokens=64)
    seq = torch.full((8,), 64, dtype=torch.int32, device=c.dev)
    out = torch.empty((8, 1024, 256), dtype=torch.float32, device=c.dev)
    st = P.palu_decode_attn_noalloc(big, c.attn._bk.data_ptr(), c.q_dev.data_ptr(), c.cache.c_struct(),
                                    seq.data_ptr(), 8, 64, out.data_ptr(), None, stream)
    assert st == P.PALU_ERR_WORKSPACE                   # beyond the fixed scratch
    rope = P.make_desc(n_heads=32, head_dim=128, group_size=4, rank_k=256, rank_v=256, latent_dtype="f16",
                       q_dtype="f16", mode="rope", max_batch=1, max_tokens=64)
    st = P.palu_decode_attn_noalloc(rope, c.attn._bk.data_ptr(), c.q_dev.data_ptr(), c.cache.c_struct(),
                                    seq.data_ptr(), 1, 64, out.data_ptr(), None, stream)
    assert st == P.PALU_ERR_UNSUPPORTED
    i4 = P.make_desc(n_heads=32, head_dim=128, group_size=4, rank_k=256, rank_v=256, latent_dtype="int4",
                     q_dtype="f16", mode="absorbed", max_batch=1, max_tokens=64)
    cache = c.cache.c_struct()                          # no scales: an int4 cache needs both
    st = P.palu_decode_attn_noalloc(i4, c.attn._bk.data_ptr(), c.q_dev.data_ptr(), cache, seq.data_ptr(), 1, 64,
                                    out.data_ptr(), None, stream)
    assert st == P.PALU_ERR_INVALID_ARG
    scale = torch.zeros(130, dtype=torch.float16, device=c.dev)
    cache.k_scale = cache.v_scale = scale.data_ptr() + 1  # misaligned scales
    st = P.palu_decode_attn_noalloc(i4, c.attn._bk.data_ptr(), c.q_dev.data_ptr(), cache, seq.data_ptr(), 1, 64,
                                    out.data_ptr(), None, stream)
    assert st == P.PALU_ERR_INVALID_ARG
