"""CPU tests of the C ABI: the library loads, exports every declared symbol, and
rejects bad descriptors and arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

from rank_kv_cache_gb300 import palu as P

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "palu_attn.h")


def _declared_functions():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(palu_\w+)\s*\(", txt)))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert set(names) == set(P.EXPORTS)
    lib = ctypes.CDLL(P.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def _desc(**kw):
    base = dict(n_heads=32, head_dim=128, group_size=4, rank_k=256, rank_v=256, latent_dtype="f16",
                q_dtype="f16", mode="rope", max_batch=4, max_tokens=4096)
    base.update(kw)
    return P.make_desc(**base)


def test_workspace_size_accepts_every_config_shape():
    for lat, mode in (("f32", "rope"), ("f16", "rope"), ("bf16", "rope"), ("f16", "absorbed"), ("int4", "rope"),
                      ("int4", "absorbed")):
        st, n = P.palu_attn_workspace_size(_desc(latent_dtype=lat, mode=mode))
        assert st == P.PALU_OK and n > 0 and n % 256 == 0
    st, n = P.palu_attn_workspace_size(_desc(n_heads=8, head_dim=64, group_size=4, rank_k=128, rank_v=128,
                                             latent_dtype="f32", q_dtype="f32", max_batch=1, max_tokens=512))
    assert st == P.PALU_OK


def test_workspace_grows_with_positions_table():
    _, a = P.palu_attn_workspace_size(_desc(max_tokens=4096))
    _, b = P.palu_attn_workspace_size(_desc(max_tokens=4096, max_position=65536))
    assert b - a >= (65536 - 4096) * 64 * 8


@pytest.mark.parametrize("field,value,status", [
    ("abi_version", 2, P.PALU_ERR_INVALID_ARG),
    ("n_heads", 0, P.PALU_ERR_INVALID_ARG),
    ("group_size", 3, P.PALU_ERR_INVALID_ARG),
    ("head_dim", 96, P.PALU_ERR_UNSUPPORTED),
    ("rank_k", 192, P.PALU_ERR_UNSUPPORTED),
    ("rank_v", 512, P.PALU_ERR_UNSUPPORTED),
    ("v_dtype", P.PALU_F32, P.PALU_ERR_UNSUPPORTED),
    ("bk_dtype", P.PALU_BF16, P.PALU_ERR_UNSUPPORTED),
    ("q_dtype", P.PALU_INT4, P.PALU_ERR_INVALID_ARG),
    ("mode", 7, P.PALU_ERR_INVALID_ARG),
    ("rope_theta", 0.0, P.PALU_ERR_INVALID_ARG),
    ("max_batch", 0, P.PALU_ERR_INVALID_ARG),
    ("max_tokens", 0, P.PALU_ERR_INVALID_ARG),
    ("flags", 1, P.PALU_ERR_INVALID_ARG),
])
def test_bad_descriptor_rejected(field, value, status):
    d = _desc()
    setattr(d, field, value)
    st, _ = P.palu_attn_workspace_size(d)
    assert st == status


def test_flags_accepted_per_mode():
    st, _ = P.palu_attn_workspace_size(_desc(flags=P.PALU_FLAG_TEST_STALL))
    assert st == P.PALU_OK
    st, _ = P.palu_attn_workspace_size(_desc(flags=P.PALU_FLAG_TEST_STALL | 2))
    assert st == P.PALU_ERR_INVALID_ARG
    # ALiBi biases scores outside the keys: the absorbed path only
    st, _ = P.palu_attn_workspace_size(_desc(mode="absorbed", flags=P.PALU_FLAG_ALIBI))
    assert st == P.PALU_OK
    st, _ = P.palu_attn_workspace_size(_desc(mode="rope", flags=P.PALU_FLAG_ALIBI))
    assert st == P.PALU_ERR_INVALID_ARG


@pytest.mark.parametrize("kw,status", [
    (dict(latent_dtype="f16", v_dtype="int4"), P.PALU_OK),            # V-only int4
    (dict(latent_dtype="bf16", v_dtype="int4"), P.PALU_OK),
    (dict(latent_dtype="f16", v_dtype="int4", mode="absorbed"), P.PALU_OK),
    (dict(latent_dtype="int4", v_dtype="f16"), P.PALU_ERR_UNSUPPORTED),
    (dict(latent_dtype="f32", v_dtype="int4"), P.PALU_ERR_UNSUPPORTED),
    (dict(group_size=1, rank_k=64, rank_v=64), P.PALU_OK),            # M-LRD
    (dict(group_size=32), P.PALU_OK),                                 # J-LRD on the tensor-core path
    (dict(group_size=16, latent_dtype="int4"), P.PALU_OK),
    (dict(group_size=32, mode="absorbed"), P.PALU_OK),                # J-LRD absorbed as split groups
    (dict(group_size=16, mode="absorbed", latent_dtype="bf16"), P.PALU_OK),
    (dict(group_size=32, mode="absorbed", latent_dtype="int4"), P.PALU_ERR_UNSUPPORTED),
    (dict(group_size=16, mode="absorbed", rank_k=128, rank_v=128), P.PALU_ERR_UNSUPPORTED),
    (dict(group_size=32, rank_k=128, rank_v=128), P.PALU_ERR_UNSUPPORTED),
    (dict(group_size=32, latent_dtype="f32", q_dtype="f32"), P.PALU_ERR_UNSUPPORTED),
    (dict(group_size=64, n_heads=64), P.PALU_ERR_UNSUPPORTED),
])
def test_granularity_and_value_dtype_variants(kw, status):
    st, _ = P.palu_attn_workspace_size(_desc(**kw))
    assert st == status


def test_null_arguments_rejected_without_gpu():
    d = _desc()
    assert P._lib.palu_attn_workspace_size(ctypes.byref(d), None) == P.PALU_ERR_INVALID_ARG
    # no workspace -> PALU_ERR_WORKSPACE, before any CUDA call
    st, h = P.palu_attn_create(d, 0x1000, 0, 0, 0)
    assert st == P.PALU_ERR_INVALID_ARG or st == P.PALU_ERR_WORKSPACE
    st, h = P.palu_attn_create(d, 0x1000, 0x2000, 1, 0)
    assert st == P.PALU_ERR_WORKSPACE and h is None
    st, h = P.palu_attn_create(d, 0x1001, 0x2000, 1 << 30, 0)   # misaligned B_k
    assert st == P.PALU_ERR_INVALID_ARG
    cache = P.palu_cache(0, 0, 0, 0, 16)
    assert P.palu_decode_attn(None, 0, cache, 0, None, None, 1, 1, 0, None, 0) == P.PALU_ERR_INVALID_ARG
    assert P.palu_append_latents(None, cache, 0, 0, 0, 0, 1, 1, 0) == P.PALU_ERR_INVALID_ARG
    assert P.palu_attn_check(None, 0) == P.PALU_ERR_INVALID_ARG
    assert P.palu_destroy(None) == P.PALU_OK


def test_status_strings():
    for s in range(7):
        assert P.palu_status_string(s)
    assert "unknown" in P.palu_status_string(99)


def test_noalloc_refuses_groups_above_eight_heads_before_any_cuda_call():
    # split groups exist only on the workspace path; the fixed-scratch entry point runs the
    # CUDA-core kernel, which takes up to eight heads a group
    for s in (16, 32):
        d = _desc(mode="absorbed", group_size=s)
        assert P.palu_attn_workspace_size(d)[0] == P.PALU_OK
        st = P.palu_decode_attn_noalloc(d, 0x1000, 0x1000, P.palu_cache(), 0x1000, 1, 16, 0x1000, None, 0)
        assert st == P.PALU_ERR_UNSUPPORTED


def test_packed_and_split_group_workspaces():
    # packed M-LRD / s = 2 groups are laid out as G-LRD groups of four heads at rank 256 (block-diagonal
    # B_k, 256-wide partials); split absorbed groups keep the source B_k bytes in four-head blocks
    _, s4 = P.palu_attn_workspace_size(_desc())
    for s in (1, 2):
        _, packed = P.palu_attn_workspace_size(_desc(group_size=s, rank_k=64 * s, rank_v=64 * s))
        assert packed == s4
    _, unpacked = P.palu_attn_workspace_size(_desc(group_size=1, rank_k=64, rank_v=64, latent_dtype="f32",
                                                    q_dtype="f32"))
    assert unpacked < s4
    _, a4 = P.palu_attn_workspace_size(_desc(mode="absorbed"))
    for s in (8, 16, 32):
        assert P.palu_attn_workspace_size(_desc(mode="absorbed", group_size=s))[1] == a4
