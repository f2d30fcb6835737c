"""Shared helpers for the GPU parity tests: run one seeded case through the C ABI
and through the oracle, on identical storage-rounded inputs."""
from __future__ import annotations

import math

import numpy as np

from oracle import palu_oracle as O
from synthetic import gen

# Tolerances for fp16/bf16 latents with fp32 accumulation (stated for the method's
# decode attention): max |delta| <= 2e-3 and max |delta| / max |ref| <= 1e-2, lse |delta| <= 1e-3.
ABS_TOL = 2e-3
REL_TOL = 1e-2
LSE_TOL = 1e-3
# fp32 latents: the only error is fp32 rounding of the rebuild, RoPE and softmax sums
# (relative ~1e-6 per score); 1e-4 absolute leaves two orders of magnitude of headroom.
ABS_TOL_F32 = 1e-4


def torch_dtype(name):
    import torch
    return {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[name]


class Case:
    """One workload on the GPU plus everything the oracle needs to check it."""

    def __init__(self, cfg: gen.Config, *, seq_lens=None, positions=None, q_pos=None, q_scale=1.0,
                 capacity=None, max_position=0, fill="append", q_dtype=None, alibi=False):
        import torch
        from rank_kv_cache_gb300 import palu as P
        self.cfg = cfg
        self.alibi = alibi
        dev = torch.device("cuda:0")
        inp = gen.make_inputs(cfg, q_scale=q_scale)
        self.inp = inp
        B, T = cfg.batch, cfg.T
        self.seq_lens = np.array(seq_lens if seq_lens is not None else [T] * B, dtype=np.int32)
        self.positions = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32)
        self.q_pos = None if q_pos is None else np.ascontiguousarray(q_pos, dtype=np.int32)
        self.capacity = capacity or T
        lat = cfg.latent_dtype
        self.q_dtype = q_dtype or cfg.q_dtype
        self.q_t = gen.storage_round(inp["q"], self.q_dtype)
        self.bk_t = gen.storage_round(inp["bk"], cfg.bk_dtype)
        vlat = cfg.value_dtype
        self.attn = P.PaluAttention(self.bk_t.to(dev), n_heads=cfg.n_heads, head_dim=cfg.head_dim,
                                    group_size=cfg.group_size, rank_k=cfg.rank, rank_v=cfg.rank, latent_dtype=lat,
                                    q_dtype=self.q_dtype, mode=cfg.mode, rope_theta=cfg.theta, max_batch=B,
                                    max_tokens=self.capacity, max_position=max_position, v_dtype=vlat,
                                    flags=P.PALU_FLAG_ALIBI if alibi else 0)
        self.cache = P.LatentCache(B, self.capacity, cfg.n_groups, cfg.rank, cfg.rank, lat, device=dev, v_dtype=vlat)
        if "int4" in (lat, vlat):
            # one source dtype for both sides: float32, rounded or quantised by the append kernel
            src_k = torch.from_numpy(np.ascontiguousarray(inp["hk"]))
            src_v = torch.from_numpy(np.ascontiguousarray(inp["hv"]))
        else:
            src_k = gen.storage_round(inp["hk"], lat)
            src_v = gen.storage_round(inp["hv"], lat)
        if fill == "append" or "int4" in (lat, vlat):
            slot = torch.zeros(B, dtype=torch.int32, device=dev)
            self.attn.append(self.cache, src_k.to(dev), src_v.to(dev), slot)
        else:
            self.cache.hk[:, :T].copy_(src_k.to(dev))
            self.cache.hv[:, :T].copy_(src_v.to(dev))
        torch.cuda.synchronize()
        self.dev = dev
        self._oracle_latents()

    def _oracle_latents(self):
        cfg, inp = self.cfg, self.inp

        def side(h, dtype):
            if dtype == "int4":
                codes, sc = O.quantize_int4(h)
                # dequantised values are exact in float32 (pinned on the CPU); the oracle upcasts
                # each slice it reads to float64
                return O.pack_int4(codes), sc, O.dequant_int4(O.pack_int4(codes), sc).astype(np.float32)
            # fp16/bf16 values are exact in float32; the oracle upcasts to float64 per slice
            return None, None, gen.storage_round(h, dtype).float().numpy()

        pk, sk, self.hk64 = side(inp["hk"], cfg.latent_dtype)
        pv, sv, self.hv64 = side(inp["hv"], cfg.value_dtype)
        if cfg.latent_dtype == "int4":
            self.ref_packed = (pk, sk, pv, sv)
        self.q64 = self.q_t.double().numpy()
        self.bk64 = self.bk_t.double().numpy()

    def run_gpu(self, max_seq_len=None, with_lse=True):
        import torch
        B = self.cfg.batch
        dev = self.dev
        seq = torch.from_numpy(self.seq_lens).to(dev)
        pos = None
        if self.positions is not None:
            pos = torch.zeros((B, self.capacity), dtype=torch.int32, device=dev)
            pos[:, :self.positions.shape[1]] = torch.from_numpy(self.positions).to(dev)
        qp = None if self.q_pos is None else torch.from_numpy(self.q_pos).to(dev)
        lse = torch.empty((B, self.cfg.n_heads), dtype=torch.float32, device=dev) if with_lse else None
        msl = int(self.seq_lens.max()) if max_seq_len is None else max_seq_len
        out = self.attn.decode(self.q_t.to(dev), self.cache, seq, max_seq_len=msl, positions=pos, q_pos=qp,
                               lse=lse)
        torch.cuda.synchronize()
        self.attn.check_device()
        return out.cpu().double().numpy(), (lse.cpu().double().numpy() if with_lse else None)

    def run_oracle(self, heads=None):
        cfg = self.cfg
        return O.decode(self.q64, self.hk64, self.hv64, self.bk64, self.seq_lens, cfg.group_size, mode=cfg.mode,
                        theta=cfg.theta, positions=self.positions, q_pos=self.q_pos, heads=heads, alibi=self.alibi)


def assert_close(out, ref, lse=None, lse_ref=None, *, f32=False, heads=None):
    if heads is not None:
        idx = tuple(np.array(heads).T)
        out, ref = out[idx], ref[idx]
        if lse is not None:
            lse, lse_ref = lse[idx], lse_ref[idx]
    d = np.abs(out - ref)
    max_abs = float(d.max()) if d.size else 0.0
    ref_inf = float(np.abs(ref).max()) if ref.size else 0.0
    rel = max_abs / ref_inf if ref_inf > 0 else max_abs
    tol = ABS_TOL_F32 if f32 else ABS_TOL
    assert np.all(np.isfinite(out)), "non-finite output"
    assert max_abs <= tol, f"max abs err {max_abs:.3e} > {tol}"
    assert rel <= REL_TOL, f"max err / max ref {rel:.3e} > {REL_TOL}"
    if lse is not None:
        fin = np.isfinite(lse_ref)
        assert np.array_equal(np.isfinite(lse), fin)
        if fin.any():
            dl = float(np.abs(lse[fin] - lse_ref[fin]).max())
            assert dl <= LSE_TOL, f"lse err {dl:.3e}"
        assert np.all(lse[~fin] == -math.inf)
    return max_abs, rel
