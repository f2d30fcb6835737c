"""Python binding of the G-LRD decode-attention C ABI (include/palu_attn.h).

Argument marshalling only: every step of the decode path runs in the CUDA
kernels of ``_lib/libpalu_attn.so``. Importing this package loads that library
and raises if it has not been built (``rank_kv_cache_gb300.build.build()``);
there is no CPU fallback.

Low-level functions carry the C names and take raw integers (device pointers,
stream handles); ``PaluAttention`` and ``LatentCache`` wrap them for torch
tensors.
"""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "libpalu_attn.so")

PALU_ABI_VERSION = 1
PALU_OK, PALU_ERR_INVALID_ARG, PALU_ERR_UNSUPPORTED, PALU_ERR_CUDA, PALU_ERR_DEVICE, PALU_ERR_TIMEOUT, \
    PALU_ERR_WORKSPACE = range(7)
PALU_F32, PALU_F16, PALU_BF16, PALU_INT4 = range(4)
PALU_MODE_ROPE, PALU_MODE_ABSORBED = 0, 1
PALU_KERNEL_TC_ROPE, PALU_KERNEL_TMA_ABSORBED, PALU_KERNEL_SIMT = 1, 2, 3
PALU_FLAG_TEST_STALL = 0x80000000
PALU_FLAG_ALIBI = 0x1

DTYPES = {"f32": PALU_F32, "f16": PALU_F16, "bf16": PALU_BF16, "int4": PALU_INT4}
MODES = {"rope": PALU_MODE_ROPE, "absorbed": PALU_MODE_ABSORBED}

# every symbol include/palu_attn.h declares
EXPORTS = ("palu_attn_workspace_size", "palu_attn_create", "palu_append_latents", "palu_decode_attn",
           "palu_destroy", "palu_attn_check", "palu_status_string", "palu_debug_dequant",
           "palu_attn_trace_enable", "palu_attn_trace_read", "palu_decode_attn_noalloc", "palu_decode_plan",
           "palu_debug_int4_operand", "palu_debug_int4_dp2a", "palu_attn_trace_times",
           "palu_fuse_value_output", "palu_output_proj_workspace_size", "palu_output_proj",
           "palu_down_proj_size", "palu_prepare_down_proj", "palu_project_latents", "palu_decode_hybrid",
           "palu_decode_paged")
PALU_TRACE_CAPACITY = 4096


class palu_attn_desc(ctypes.Structure):
    _fields_ = [("abi_version", ctypes.c_int), ("n_heads", ctypes.c_int), ("head_dim", ctypes.c_int),
                ("group_size", ctypes.c_int), ("rank_k", ctypes.c_int), ("rank_v", ctypes.c_int),
                ("k_dtype", ctypes.c_int), ("v_dtype", ctypes.c_int), ("bk_dtype", ctypes.c_int),
                ("q_dtype", ctypes.c_int), ("mode", ctypes.c_int), ("rope_theta", ctypes.c_double),
                ("max_batch", ctypes.c_int), ("max_tokens", ctypes.c_int64), ("max_position", ctypes.c_int64),
                ("flags", ctypes.c_uint32)]


class palu_cache(ctypes.Structure):
    _fields_ = [("hk", ctypes.c_void_p), ("hv", ctypes.c_void_p), ("k_scale", ctypes.c_void_p),
                ("v_scale", ctypes.c_void_p), ("capacity", ctypes.c_int64)]


class palu_dense_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("n_tokens", ctypes.c_void_p),
                ("capacity", ctypes.c_int64), ("dtype", ctypes.c_int)]


class palu_page_cache(ctypes.Structure):
    _fields_ = [("pages", ctypes.c_void_p), ("n_pages", ctypes.c_void_p), ("capacity", ctypes.c_int64),
                ("page_size", ctypes.c_int), ("rank", ctypes.c_int), ("dtype", ctypes.c_int)]


class PaluError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {palu_status_string(status)} (status {status})")


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with rank_kv_cache_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, I64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "palu_attn_workspace_size": (I, [ctypes.POINTER(palu_attn_desc), ctypes.POINTER(SZ)]),
        "palu_attn_create": (I, [ctypes.POINTER(palu_attn_desc), P, P, SZ, P, ctypes.POINTER(P)]),
        "palu_append_latents": (I, [P, ctypes.POINTER(palu_cache), P, P, I, P, I, I, P]),
        "palu_decode_attn": (I, [P, P, ctypes.POINTER(palu_cache), P, P, P, I, I64, P, P, P]),
        "palu_destroy": (I, [P]),
        "palu_attn_check": (I, [P, P]),
        "palu_status_string": (ctypes.c_char_p, [I]),
        "palu_debug_dequant": (I, [P, ctypes.POINTER(palu_cache), I, I, I64, P, P]),
        "palu_attn_trace_enable": (I, [P, I]),
        "palu_attn_trace_read": (I, [P, ctypes.POINTER(I), ctypes.POINTER(ctypes.c_double)]),
        "palu_decode_attn_noalloc": (I, [ctypes.POINTER(palu_attn_desc), P, P, ctypes.POINTER(palu_cache), P, I,
                                         I64, P, P, P]),
        "palu_decode_plan": (I, [P, I64, I, I64, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)]),
        "palu_attn_trace_times": (I, [P, ctypes.POINTER(ctypes.c_float), I, ctypes.POINTER(I)]),
        "palu_fuse_value_output": (I, [P, P, I, I, I, I, I, I64, P, I, P]),
        "palu_output_proj_workspace_size": (I, [I64, I64, I, ctypes.POINTER(SZ)]),
        "palu_output_proj": (I, [P, I, I64, I64, P, I, P, P, SZ, P]),
        "palu_debug_int4_operand": (I, [P, ctypes.POINTER(palu_cache), I, I64, P, P, P]),
        "palu_debug_int4_dp2a": (I, [P, ctypes.POINTER(palu_cache), I, I, I64, P, P, P]),
        "palu_down_proj_size": (I, [P, I64, ctypes.POINTER(SZ)]),
        "palu_prepare_down_proj": (I, [P, P, P, I, I64, I, P, SZ, P]),
        "palu_project_latents": (I, [P, P, I, I64, P, ctypes.POINTER(palu_cache), P, I, I, P]),
        "palu_decode_hybrid": (I, [P, P, ctypes.POINTER(palu_cache), P, P, P, I, I64,
                                   ctypes.POINTER(palu_dense_cache), P, P, P, P]),
        "palu_decode_paged": (I, [P, P, ctypes.POINTER(palu_page_cache), P, I, I64,
                                  ctypes.POINTER(palu_dense_cache), P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    return lib


_lib = _load()


# ---------------------------------------------------------------------------
# C-named entry points (raw integers for pointers and streams)
# ---------------------------------------------------------------------------

def palu_status_string(status: int) -> str:
    return _lib.palu_status_string(int(status)).decode()


def palu_attn_workspace_size(desc: palu_attn_desc):
    n = ctypes.c_size_t(0)
    st = _lib.palu_attn_workspace_size(ctypes.byref(desc), ctypes.byref(n))
    return st, n.value


def palu_attn_create(desc: palu_attn_desc, bk_ptr: int, ws_ptr: int, ws_bytes: int, stream: int):
    h = ctypes.c_void_p()
    st = _lib.palu_attn_create(ctypes.byref(desc), bk_ptr, ws_ptr, ws_bytes, stream, ctypes.byref(h))
    return st, h.value


def palu_append_latents(h, cache: palu_cache, hk_new: int, hv_new: int, src_dtype: int, dst_slot: int,
                        batch: int, n_new: int, stream: int) -> int:
    return _lib.palu_append_latents(h, ctypes.byref(cache), hk_new, hv_new, src_dtype, dst_slot, batch, n_new,
                                    stream)


def palu_decode_attn(h, q: int, cache: palu_cache, seq_lens: int, positions, q_pos, batch: int,
                     max_seq_len: int, out: int, lse, stream: int) -> int:
    return _lib.palu_decode_attn(h, q, ctypes.byref(cache), seq_lens, positions, q_pos, batch, max_seq_len, out,
                                 lse, stream)


def palu_destroy(h) -> int:
    return _lib.palu_destroy(h)


def palu_attn_check(h, stream: int) -> int:
    return _lib.palu_attn_check(h, stream)


def palu_debug_dequant(h, cache: palu_cache, which: int, batch: int, n_tokens: int, out: int, stream: int) -> int:
    return _lib.palu_debug_dequant(h, ctypes.byref(cache), which, batch, n_tokens, out, stream)


def palu_debug_int4_operand(h, cache: palu_cache, batch: int, n_tokens: int, codes: int, deq, stream: int) -> int:
    return _lib.palu_debug_int4_operand(h, ctypes.byref(cache), batch, n_tokens, codes, deq, stream)


def palu_debug_int4_dp2a(h, cache: palu_cache, which: int, batch: int, n_tokens: int, weights: int, sums: int,
                         stream: int) -> int:
    return _lib.palu_debug_int4_dp2a(h, ctypes.byref(cache), which, batch, n_tokens, weights, sums, stream)


def palu_attn_trace_enable(h, enable: int) -> int:
    return _lib.palu_attn_trace_enable(h, int(enable))


def palu_attn_trace_read(h):
    n = ctypes.c_int(0)
    ms = ctypes.c_double(0.0)
    st = _lib.palu_attn_trace_read(h, ctypes.byref(n), ctypes.byref(ms))
    return st, n.value, ms.value


def palu_attn_trace_times(h, capacity: int = PALU_TRACE_CAPACITY):
    """(status, [ms per recorded launch]) and empties the trace ring."""
    buf = (ctypes.c_float * max(capacity, 1))()
    n = ctypes.c_int(0)
    st = _lib.palu_attn_trace_times(h, buf, capacity, ctypes.byref(n))
    return st, [float(buf[i]) for i in range(n.value)]


def palu_decode_attn_noalloc(desc: palu_attn_desc, bk: int, q: int, cache: palu_cache, seq_lens: int, batch: int,
                             max_seq_len: int, out: int, lse, stream: int) -> int:
    """Absorbed-mode decode with the library's fixed device scratch (no allocation anywhere)."""
    return _lib.palu_decode_attn_noalloc(ctypes.byref(desc), bk, q, ctypes.byref(cache), seq_lens, batch,
                                         max_seq_len, out, lse, stream)


def palu_decode_plan(h, cache_capacity: int, batch: int, max_seq_len: int):
    """(status, kernel, n_splits, launches) of the decode call for this shape; host-only."""
    k, n, l = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = _lib.palu_decode_plan(h, cache_capacity, batch, max_seq_len, ctypes.byref(k), ctypes.byref(n),
                               ctypes.byref(l))
    return st, k.value, n.value, l.value


def palu_fuse_value_output(bv: int, wo: int, in_dtype: int, n_heads: int, head_dim: int, group_size: int,
                           rank_v: int, d_model: int, w_fused: int, out_dtype: int, stream: int) -> int:
    return _lib.palu_fuse_value_output(bv, wo, in_dtype, n_heads, head_dim, group_size, rank_v, d_model, w_fused,
                                       out_dtype, stream)


def palu_output_proj_workspace_size(k_dim: int, d_model: int, max_batch: int):
    n = ctypes.c_size_t(0)
    st = _lib.palu_output_proj_workspace_size(k_dim, d_model, max_batch, ctypes.byref(n))
    return st, n.value


def palu_output_proj(w_fused: int, w_dtype: int, k_dim: int, d_model: int, o: int, batch: int, y: int,
                     workspace: int, ws_bytes: int, stream: int) -> int:
    return _lib.palu_output_proj(w_fused, w_dtype, k_dim, d_model, o, batch, y, workspace, ws_bytes, stream)


def palu_down_proj_size(h, d_model: int):
    n = ctypes.c_size_t(0)
    st = _lib.palu_down_proj_size(h, d_model, ctypes.byref(n))
    return st, n.value


def palu_prepare_down_proj(h, a_k: int, a_v: int, a_dtype: int, d_model: int, w_dtype: int, w: int, w_bytes: int,
                           stream: int) -> int:
    return _lib.palu_prepare_down_proj(h, a_k, a_v, a_dtype, d_model, w_dtype, w, w_bytes, stream)


def palu_project_latents(h, w: int, w_dtype: int, d_model: int, x: int, cache: palu_cache, dst_slot: int,
                         batch: int, n_new: int, stream: int) -> int:
    return _lib.palu_project_latents(h, w, w_dtype, d_model, x, ctypes.byref(cache), dst_slot, batch, n_new, stream)


def palu_decode_paged(h, q: int, pages: palu_page_cache, q_pos, batch: int, max_pages: int, dense, out: int,
                      out_dense, lse: int, stream: int) -> int:
    return _lib.palu_decode_paged(h, q, ctypes.byref(pages), q_pos, batch, max_pages,
                                  ctypes.byref(dense) if dense is not None else None, out, out_dense, lse, stream)


def palu_decode_hybrid(h, q: int, cache: palu_cache, seq_lens: int, positions, q_pos, batch: int,
                       max_seq_len: int, dense: palu_dense_cache, out: int, out_dense: int, lse: int,
                       stream: int) -> int:
    return _lib.palu_decode_hybrid(h, q, ctypes.byref(cache), seq_lens, positions, q_pos, batch, max_seq_len,
                                   ctypes.byref(dense), out, out_dense, lse, stream)


def check(status: int, what: str = "palu") -> None:
    if status != PALU_OK:
        raise PaluError(status, what)


# ---------------------------------------------------------------------------
# torch helpers
# ---------------------------------------------------------------------------

def _torch():
    import torch
    return torch


def _stream_handle(stream) -> int:
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _ptr(t) -> int | None:
    return None if t is None else int(t.data_ptr())


def _require_contiguous(**tensors):
    for name, t in tensors.items():
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")


def make_desc(*, n_heads, head_dim, group_size, rank_k, rank_v, latent_dtype, q_dtype, mode, rope_theta=10000.0,
              max_batch=1, max_tokens=1, max_position=0, flags=0, v_dtype=None) -> palu_attn_desc:
    """latent_dtype is the key latents' dtype and, unless v_dtype is given, the values' too
    (v_dtype="int4" under fp16 / bf16 keys: int4 values only)."""
    k = DTYPES[latent_dtype]
    v = DTYPES[v_dtype or latent_dtype]
    bk = PALU_F16 if k == PALU_INT4 else k
    return palu_attn_desc(PALU_ABI_VERSION, n_heads, head_dim, group_size, rank_k, rank_v, k, v, bk,
                          DTYPES[q_dtype], MODES[mode], float(rope_theta), max_batch, max_tokens, max_position, flags)


class LatentCache:
    """Device latent cache in the layout palu_cache describes ([rows][capacity][n_g][r])."""

    def __init__(self, rows, capacity, n_g, rank_k, rank_v, latent_dtype, device="cuda", v_dtype=None):
        torch = _torch()
        self.rows, self.capacity, self.n_g = rows, capacity, n_g
        self.rank_k, self.rank_v, self.latent_dtype = rank_k, rank_v, latent_dtype
        self.v_dtype = v_dtype or latent_dtype

        def side(dtype, rank):
            if dtype == "int4":
                return (torch.zeros((rows, capacity, n_g, rank // 2), dtype=torch.uint8, device=device),
                        torch.zeros((rows, capacity, n_g), dtype=torch.float16, device=device))
            dt = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16}[dtype]
            return torch.zeros((rows, capacity, n_g, rank), dtype=dt, device=device), None

        self.hk, self.k_scale = side(latent_dtype, rank_k)
        self.hv, self.v_scale = side(self.v_dtype, rank_v)

    def c_struct(self) -> palu_cache:
        return palu_cache(_ptr(self.hk), _ptr(self.hv), _ptr(self.k_scale), _ptr(self.v_scale), self.capacity)


class PaluAttention:
    """Owns one handle and its torch-allocated workspace."""

    def __init__(self, bk, *, n_heads, head_dim, group_size, rank_k, rank_v, latent_dtype, q_dtype, mode,
                 rope_theta=10000.0, max_batch=1, max_tokens=1, max_position=0, flags=0, v_dtype=None, stream=None):
        torch = _torch()
        self.desc = make_desc(n_heads=n_heads, head_dim=head_dim, group_size=group_size, rank_k=rank_k,
                              rank_v=rank_v, latent_dtype=latent_dtype, q_dtype=q_dtype, mode=mode,
                              rope_theta=rope_theta, max_batch=max_batch, max_tokens=max_tokens,
                              max_position=max_position, flags=flags, v_dtype=v_dtype)
        st, nbytes = palu_attn_workspace_size(self.desc)
        check(st, "palu_attn_workspace_size")
        self.workspace = torch.empty(nbytes + 256, dtype=torch.uint8, device=bk.device)
        base = int(self.workspace.data_ptr())
        off = (-base) % 256
        self.ws_ptr, self.ws_bytes = base + off, nbytes
        self.n_heads, self.head_dim, self.group_size = n_heads, head_dim, group_size
        self.rank_k, self.rank_v, self.mode = rank_k, rank_v, mode
        self._bk = bk.contiguous()
        st, self.handle = palu_attn_create(self.desc, _ptr(self._bk), self.ws_ptr, self.ws_bytes,
                                           _stream_handle(stream))
        check(st, "palu_attn_create")

    def close(self):
        if getattr(self, "handle", None):
            palu_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def append(self, cache: LatentCache, hk_new, hv_new, dst_slot, stream=None):
        torch = _torch()
        if hk_new.dtype != hv_new.dtype:
            raise ValueError("hk_new and hv_new must share a dtype")
        src = {torch.float32: PALU_F32, torch.float16: PALU_F16, torch.bfloat16: PALU_BF16}[hk_new.dtype]
        _require_contiguous(hk_new=hk_new, hv_new=hv_new, dst_slot=dst_slot)
        b, n_new = hk_new.shape[0], hk_new.shape[1]
        st = palu_append_latents(self.handle, cache.c_struct(), _ptr(hk_new), _ptr(hv_new), src, _ptr(dst_slot), b,
                                 n_new, _stream_handle(stream))
        check(st, "palu_append_latents")

    def decode(self, q, cache: LatentCache, seq_lens, *, max_seq_len, positions=None, q_pos=None, out=None,
               lse=None, stream=None):
        torch = _torch()
        _require_contiguous(q=q, seq_lens=seq_lens, positions=positions, q_pos=q_pos, out=out, lse=lse)
        B = q.shape[0]
        if out is None:
            out = torch.empty((B, self.n_heads, self.rank_v), dtype=torch.float32, device=q.device)
        st = palu_decode_attn(self.handle, _ptr(q), cache.c_struct(), _ptr(seq_lens), _ptr(positions),
                              _ptr(q_pos), B, int(max_seq_len), _ptr(out), _ptr(lse), _stream_handle(stream))
        check(st, "palu_decode_attn")
        return out

    def decode_hybrid(self, q, cache: LatentCache, seq_lens, dense_k, dense_v, dense_n, *, max_seq_len,
                      positions=None, q_pos=None, out=None, out_dense=None, lse=None, stream=None):
        """Decode over the latent middle (cache, seq_lens, positions) and a dense segment
        (dense_k / dense_v [rows][capacity][n_heads][head_dim], dense_n [batch] tokens per row),
        one softmax over both. Returns (out [B][n][rank_v], out_dense [B][n][head_dim], lse [B][n])."""
        torch = _torch()
        _require_contiguous(q=q, seq_lens=seq_lens, positions=positions, q_pos=q_pos, dense_k=dense_k,
                            dense_v=dense_v, dense_n=dense_n)
        B = q.shape[0]
        if out is None:
            out = torch.empty((B, self.n_heads, self.rank_v), dtype=torch.float32, device=q.device)
        if out_dense is None:
            out_dense = torch.empty((B, self.n_heads, self.head_dim), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((B, self.n_heads), dtype=torch.float32, device=q.device)
        ddt = {torch.float32: PALU_F32, torch.float16: PALU_F16, torch.bfloat16: PALU_BF16}[dense_k.dtype]
        dense = palu_dense_cache(_ptr(dense_k), _ptr(dense_v), _ptr(dense_n), int(dense_k.shape[1]), ddt)
        st = palu_decode_hybrid(self.handle, _ptr(q), cache.c_struct(), _ptr(seq_lens), _ptr(positions), _ptr(q_pos),
                                B, int(max_seq_len), dense, _ptr(out), _ptr(out_dense), _ptr(lse),
                                _stream_handle(stream))
        check(st, "palu_decode_hybrid")
        return out, out_dense, lse

    def decode_paged(self, q, pages, n_pages, *, max_pages, q_pos=None, dense_k=None, dense_v=None, dense_n=None,
                     out=None, out_dense=None, lse=None, stream=None):
        """Decode over a page-factorised cache (pages: a float16 / bfloat16 tensor [rows][capacity][n_heads]
        [320 r] of page records L_K [32][r], R_K [r][128], L_V [32][r], R_V [r][128]; n_pages [batch]) and,
        when dense_k is given, the dense sink / window tokens. Returns (out [B][n][d_h], out_dense or None,
        lse [B][n])."""
        torch = _torch()
        _require_contiguous(q=q, pages=pages, n_pages=n_pages, q_pos=q_pos, dense_k=dense_k, dense_v=dense_v,
                            dense_n=dense_n)
        B = q.shape[0]
        rec_bytes = pages[0, 0, 0].numel() * pages.element_size()
        rank = rec_bytes // 640
        if rec_bytes != 640 * rank:
            raise ValueError("a page record holds 640 r bytes (P = 32, head_dim 128)")
        pdt = {torch.float16: PALU_F16, torch.bfloat16: PALU_BF16}[pages.dtype]
        pc = palu_page_cache(_ptr(pages), _ptr(n_pages), int(pages.shape[1]), 32, int(rank), pdt)
        if out is None:
            out = torch.empty((B, self.n_heads, self.head_dim), dtype=torch.float32, device=q.device)
        if lse is None:
            lse = torch.empty((B, self.n_heads), dtype=torch.float32, device=q.device)
        dense = None
        if dense_k is not None:
            if out_dense is None:
                out_dense = torch.empty((B, self.n_heads, self.head_dim), dtype=torch.float32, device=q.device)
            ddt = {torch.float32: PALU_F32, torch.float16: PALU_F16, torch.bfloat16: PALU_BF16}[dense_k.dtype]
            dense = palu_dense_cache(_ptr(dense_k), _ptr(dense_v), _ptr(dense_n), int(dense_k.shape[1]), ddt)
        st = palu_decode_paged(self.handle, _ptr(q), pc, _ptr(q_pos), B, int(max_pages), dense, _ptr(out),
                               _ptr(out_dense), _ptr(lse), _stream_handle(stream))
        check(st, "palu_decode_paged")
        return out, out_dense, lse

    def prepare_down_proj(self, a_k, a_v, *, dtype="f16", stream=None):
        """The down-projections A_k, A_v ([n_g][d_model][rank] device tensors) as the tensor-core
        operand for project(): a [2][n_g][rank][d_model] tensor of `dtype` ("f16" or "bf16")."""
        torch = _torch()
        _require_contiguous(a_k=a_k, a_v=a_v)
        if a_k.dtype != a_v.dtype or a_k.shape != a_v.shape:
            raise ValueError("a_k and a_v must share dtype and shape")
        d_model = int(a_k.shape[1])
        st, nbytes = palu_down_proj_size(self.handle, d_model)
        check(st, "palu_down_proj_size")
        tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
        w = torch.empty((2, a_k.shape[0], self.rank_k, d_model), dtype=tdt, device=a_k.device)
        src = {torch.float32: PALU_F32, torch.float16: PALU_F16, torch.bfloat16: PALU_BF16}[a_k.dtype]
        check(palu_prepare_down_proj(self.handle, _ptr(a_k), _ptr(a_v), src, d_model, DTYPES[dtype], _ptr(w),
                                     nbytes, _stream_handle(stream)), "palu_prepare_down_proj")
        return w

    def project(self, w, x, cache: LatentCache, dst_slot, stream=None):
        """H = x A for x [batch][n_new][d_model] (the dtype of w), written into the cache at
        dst_slot[b] .. dst_slot[b] + n_new - 1."""
        torch = _torch()
        _require_contiguous(w=w, x=x, dst_slot=dst_slot)
        if x.dtype != w.dtype:
            raise ValueError("x and w must share a dtype")
        wdt = {torch.float16: PALU_F16, torch.bfloat16: PALU_BF16}[w.dtype]
        st = palu_project_latents(self.handle, _ptr(w), wdt, int(w.shape[-1]), _ptr(x), cache.c_struct(),
                                  _ptr(dst_slot), int(x.shape[0]), int(x.shape[1]), _stream_handle(stream))
        check(st, "palu_project_latents")

    def plan(self, cache_capacity, batch, max_seq_len):
        """(kernel, n_splits, launches) that decode() would use; host-only."""
        st, kernel, n_splits, launches = palu_decode_plan(self.handle, int(cache_capacity), int(batch),
                                                          int(max_seq_len))
        check(st, "palu_decode_plan")
        return kernel, n_splits, launches

    def check_device(self, stream=None):
        check(palu_attn_check(self.handle, _stream_handle(stream)), "palu_attn_check")


class OutputProjection:
    """The fused (B_v W_o) weight of one layer and the workspace of its GEMV."""

    def __init__(self, bv, wo, *, n_heads, head_dim, group_size, rank_v, max_batch=1, dtype="f16", stream=None):
        torch = _torch()
        _require_contiguous(bv=bv, wo=wo)
        tmap = {torch.float32: PALU_F32, torch.float16: PALU_F16, torch.bfloat16: PALU_BF16}
        if bv.dtype != wo.dtype:
            raise ValueError("bv and wo must share a dtype")
        self.d_model = int(wo.shape[1])
        self.k_dim = n_heads * rank_v
        self.w_dtype = DTYPES[dtype]
        self.w = torch.empty((self.k_dim, self.d_model), dtype={"f16": torch.float16, "bf16": torch.bfloat16}[dtype],
                             device=wo.device)
        check(palu_fuse_value_output(_ptr(bv), _ptr(wo), tmap[bv.dtype], n_heads, head_dim, group_size, rank_v,
                                     self.d_model, _ptr(self.w), self.w_dtype, _stream_handle(stream)),
              "palu_fuse_value_output")
        self._alloc_ws(max_batch, wo.device)

    def _alloc_ws(self, max_batch, device):
        torch = _torch()
        st, n = palu_output_proj_workspace_size(self.k_dim, self.d_model, max_batch)
        check(st, "palu_output_proj_workspace_size")
        self.max_batch = max_batch
        self.workspace = torch.zeros(n + 256, dtype=torch.uint8, device=device)
        base = int(self.workspace.data_ptr())
        self.ws_ptr, self.ws_bytes = base + (-base) % 256, n

    def __call__(self, o, y=None, stream=None):
        torch = _torch()
        _require_contiguous(o=o, y=y)
        B = o.shape[0]
        if B > self.max_batch:
            raise ValueError("batch larger than max_batch")
        if y is None:
            y = torch.empty((B, self.d_model), dtype=torch.float32, device=o.device)
        check(palu_output_proj(_ptr(self.w), self.w_dtype, self.k_dim, self.d_model, _ptr(o), B, _ptr(y),
                               self.ws_ptr, self.ws_bytes, _stream_handle(stream)), "palu_output_proj")
        return y
