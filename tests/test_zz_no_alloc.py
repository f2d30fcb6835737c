"""The no-allocation decode entry point against the regular one.

Callers that cannot call cudaMalloc (a plugin whose host process owns all device
memory, an engine with a fixed memory plan) use palu_decode_attn_noalloc, which
keeps its scratch in a fixed device array inside the library. This file is
collected last so that a stop-at-first-failure run has already run every other
test; it also passes on its own in a fresh process.
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


@pytest.mark.parametrize("T,batch", [(1000, 2), (4096, 4)])
def test_noalloc_matches_workspace_entry_point_twice(cuda_device, T, batch):
    cfg = gen.ABSORBED_FP16.with_(T=T, batch=batch)
    seq_lens = [T] + [max(1, T // (k + 2)) for k in range(batch - 1)]
    c = Case(cfg, seq_lens=seq_lens)
    ref_out, ref_lse = c.run_gpu()                      # regular entry point (workspace)
    c.q_dev = c.q_t.to(c.dev)
    seq = torch.tensor(seq_lens, dtype=torch.int32, device=c.dev)
    for _ in range(2):                                  # two calls in a row share the fixed scratch
        out = torch.full((batch, cfg.n_heads, cfg.rank), float("nan"), dtype=torch.float32, device=c.dev)
        lse = torch.full((batch, cfg.n_heads), float("nan"), dtype=torch.float32, device=c.dev)
        assert _noalloc(c, seq, T, out, lse) == 0
        torch.cuda.synchronize()
        assert_close(out.cpu().double().numpy(), ref_out, lse.cpu().double().numpy(), ref_lse)


def test_noalloc_rejects_requests_beyond_its_scratch(cuda_device):
    from rank_kv_cache_gb300 import palu as P
    cfg = gen.ABSORBED_FP16.with_(T=64, batch=1)
    c = Case(cfg)
    c.q_dev = c.q_t.to(c.dev)
    big = P.make_desc(n_heads=1024, head_dim=128, group_size=4, rank_k=256, rank_v=256, latent_dtype="f16",
                      q_dtype="f16", mode="absorbed", max_batch=8, max_tokens=64)
    seq = torch.full((8,), 64, dtype=torch.int32, device=c.dev)
    out = torch.empty((8, 1024, 256), dtype=torch.float32, device=c.dev)
    st = P.palu_decode_attn_noalloc(big, c.attn._bk.data_ptr(), c.q_dev.data_ptr(), c.cache.c_struct(),
                                    seq.data_ptr(), 8, 64, out.data_ptr(), None,
                                    int(torch.cuda.current_stream().cuda_stream))
    assert st == P.PALU_ERR_WORKSPACE
    rope = P.make_desc(n_heads=32, head_dim=128, group_size=4, rank_k=256, rank_v=256, latent_dtype="f16",
                       q_dtype="f16", mode="rope", max_batch=1, max_tokens=64)
    st = P.palu_decode_attn_noalloc(rope, c.attn._bk.data_ptr(), c.q_dev.data_ptr(), c.cache.c_struct(),
                                    seq.data_ptr(), 1, 64, out.data_ptr(), None,
                                    int(torch.cuda.current_stream().cuda_stream))
    assert st == P.PALU_ERR_UNSUPPORTED
