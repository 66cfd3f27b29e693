"""CPU checks of the C ABI: the library loads, exports every symbol the header
declares, and its host-side validation rejects bad arguments without touching
a GPU (these calls fail before any launch)."""
import ctypes
import os
import re

import pytest

from gqa_decode_attention_02_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gqa_decode.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gqa_[a-z_]+)\s*\(", src)))


def test_header_declares_the_four_operations():
    names = declared_functions()
    for op in ("gqa_kv_append", "gqa_decode_attention", "gqa_verify_attention",
               "gqa_accept_prefix"):
        assert op in names


def test_library_exports_every_declared_symbol(cuda_lib):
    for name in declared_functions():
        assert hasattr(cuda_lib, name), name
    assert set(_lib.EXPORTS) <= set(declared_functions())


def test_version_and_status_strings(cuda_lib):
    assert cuda_lib.gqa_version() >= 100
    assert _lib.status_string(0) == "ok"
    assert "aligned" in _lib.status_string(4)
    assert _lib.status_string(12345) == "unknown status"


def _shape(**kw):
    d = dict(B=2, T=1, N=8, K=2, H=128, block_size=16, num_blocks=10, max_blocks_per_seq=4,
             dtype=1, scale=0.0)
    d.update(kw)
    return _lib.Shape(**d)


@pytest.mark.parametrize("kw,code", [
    (dict(N=7), 2),            # N % K != 0
    (dict(H=96), 2),           # unsupported head size
    (dict(block_size=32), 2),  # only 16-token blocks
    (dict(T=0), 2),
    (dict(dtype=5), 3),
    (dict(N=2 * 8193, K=2), 2),  # 8193 query rows per KV head > 8192
])
def test_validation_rejects_bad_shapes(cuda_lib, kw, code):
    s = _shape(**kw)
    fake = ctypes.c_void_p(16)
    rc = cuda_lib.gqa_verify_attention(ctypes.byref(s), fake, fake, fake, fake, fake, fake,
                                       fake, 1 << 30, None, None)
    assert rc == code


def test_validation_rejects_null_and_misaligned(cuda_lib):
    s = _shape()
    fake = ctypes.c_void_p(16)
    rc = cuda_lib.gqa_decode_attention(ctypes.byref(s), None, fake, fake, fake, fake, fake,
                                       fake, 1 << 30, None, None)
    assert rc == 1
    odd = ctypes.c_void_p(18)
    rc = cuda_lib.gqa_decode_attention(ctypes.byref(s), odd, fake, fake, fake, fake, fake,
                                       fake, 1 << 30, None, None)
    assert rc == 4
    rc = cuda_lib.gqa_decode_attention(ctypes.byref(_shape(T=2)), fake, fake, fake, fake, fake,
                                       fake, fake, 1 << 30, None, None)
    assert rc == 2  # decode is T == 1 only
    rc = cuda_lib.gqa_kv_append(ctypes.byref(s), None, fake, fake, fake, fake, fake, None, None)
    assert rc == 1
    rc = cuda_lib.gqa_accept_prefix(2, 0, 10, fake, fake, fake, fake, None, None, 0, None,
                                    None)
    assert rc == 2
    rc = cuda_lib.gqa_accept_prefix(2, 3, 10, odd, fake, fake, fake, None, None, 0, None, None)
    assert rc == 4
    # a workspace smaller than the size query, or misaligned
    need = cuda_lib.gqa_accept_workspace_size(2, 3)
    assert need >= 8 * 2 * 3 + 4 * 2 and need % 16 == 0
    rc = cuda_lib.gqa_accept_prefix(2, 3, 10, fake, fake, fake, fake, None, fake, need - 1,
                                    None, None)
    assert rc == 5
    rc = cuda_lib.gqa_accept_prefix(2, 3, 10, fake, fake, fake, fake, None, odd, need, None,
                                    None)
    assert rc == 4
    assert cuda_lib.gqa_accept_workspace_size(2, 65) == 0  # T > 64
    # more sequences than one cluster per sequence can take need the workspace
    rc = cuda_lib.gqa_accept_prefix(70000, 1, 10, fake, None, fake, fake, None, None, 0, None,
                                    None)
    assert rc == 2


def test_fused_quant_entry_points_check_their_arguments(cuda_lib):
    fake = ctypes.c_void_p(16)
    s = _shape(kv_dtype=1)
    for name in ("gqa_append_decode_attention_quant", "gqa_append_verify_attention_quant"):
        f = getattr(cuda_lib, name)
        # missing scale arrays
        assert f(ctypes.byref(s), fake, fake, fake, fake, fake, None, fake, fake, fake, fake,
                 fake, 1 << 20, None, None) == 1
        # a two-byte cache shape with scales: dtype mismatch
        plain = _shape()
        assert f(ctypes.byref(plain), fake, fake, fake, fake, fake, fake, fake, fake, fake,
                 fake, fake, 1 << 20, None, None) == 3


def test_tree_acceptance_and_compaction_check_their_arguments(cuda_lib):
    fake = ctypes.c_void_p(16)
    odd = ctypes.c_void_p(18)
    f = cuda_lib.gqa_accept_tree
    # (B, T, V, logits, draft, parents, accepted, next, path, ctx, ws, ws_bytes, status, stream)
    assert f(2, 65, 10, fake, fake, fake, fake, fake, fake, None, None, 0, None, None) == 2
    assert f(2, 3, 10, fake, fake, None, fake, fake, fake, None, None, 0, None, None) == 1
    assert f(2, 3, 10, fake, fake, fake, fake, fake, None, None, None, 0, None, None) == 1
    assert f(2, 3, 10, odd, fake, fake, fake, fake, fake, None, None, 0, None, None) == 4
    need = cuda_lib.gqa_accept_workspace_size(2, 3)
    assert f(2, 3, 10, fake, fake, fake, fake, fake, fake, None, fake, need - 1, None,
             None) == 5
    assert f(0, 3, 10, None, None, None, None, None, None, None, None, 0, None, None) == 0
    g = cuda_lib.gqa_kv_compact
    # (shape, k_cache, v_cache, k_scale, v_scale, tables, ctx, path, accepted, status, stream)
    assert g(ctypes.byref(_shape(T=65)), fake, fake, None, None, fake, fake, fake, fake, None,
             None) == 2
    assert g(ctypes.byref(_shape(T=4)), fake, fake, fake, fake, fake, fake, fake, fake, None,
             None) == 3  # scales with a two-byte cache
    assert g(ctypes.byref(_shape(T=4, kv_dtype=1)), fake, fake, None, None, fake, fake, fake,
             fake, None, None) == 1  # a one-byte cache without its scales
    assert g(ctypes.byref(_shape(T=4)), fake, fake, None, None, fake, fake, None, fake, None,
             None) == 1
    assert g(ctypes.byref(_shape(T=4)), odd, fake, None, None, fake, fake, fake, fake, None,
             None) == 4
    # nothing can move: an empty batch, or a tree of one node
    assert g(ctypes.byref(_shape(B=0, T=4)), None, None, None, None, None, None, None, None,
             None, None) == 0
    assert g(ctypes.byref(_shape(T=1)), None, None, None, None, None, None, None, None, None,
             None) == 0


def test_empty_batch_is_a_no_op(cuda_lib):
    s = _shape(B=0)
    rc = cuda_lib.gqa_kv_append(ctypes.byref(s), None, None, None, None, None, None, None,
                                None)
    assert rc == 0
    rc = cuda_lib.gqa_accept_prefix(0, 3, 10, None, None, None, None, None, None, 0, None,
                                    None)
    assert rc == 0


@pytest.mark.parametrize("kw,want", [
    (dict(T=1, N=32, K=8), 3),                 # 4 rows per KV head, a small call: direct
    (dict(T=2, N=32, K=8), 3),                 # 8 rows: direct
    (dict(T=3, N=32, K=8), 1),                 # 12 rows: persistent warp-level
    (dict(T=1, N=32, K=8, B=38), 3),           # 304 segments: direct
    (dict(T=1, N=32, K=8, B=39), 1),           # 312 segments: persistent
    (dict(T=1, N=32, K=8, max_blocks_per_seq=48), 3),  # H = 128 up to 48 blocks
    (dict(T=1, N=32, K=8, max_blocks_per_seq=49), 1),
    (dict(T=1, N=32, K=8, H=64, max_blocks_per_seq=64), 3),  # H = 64 up to 64 blocks
    (dict(T=1, N=32, K=8, H=64, max_blocks_per_seq=65), 1),
    (dict(T=1, N=32, K=8, window=8), 1),       # a window: persistent
    (dict(T=1, N=32, K=8, kv_dtype=1), 1),     # one-byte cache: persistent
    (dict(T=1, N=32, K=8, flags=4), 1),        # GQA_FLAG_WARP_MMA: persistent
    (dict(T=1, N=32, K=8, B=500, max_blocks_per_seq=1000, flags=16), 3),  # GQA_FLAG_DIRECT
    (dict(T=5, N=64, K=8, flags=16), 0),       # forced direct, 40 rows: not served
    (dict(T=1, N=32, K=8, flags=20), 0),       # two forced
    (dict(T=5, N=64, K=8), 2),                 # 40 rows: tensor memory
    (dict(T=4, N=64, K=8), 2),                 # 32 rows: tensor memory (threshold)
    (dict(T=3, N=64, K=8), 1),                 # 24 rows: warp-level
    (dict(T=5, N=64, K=8, H=64), 2),           # H = 64, 40 rows: tensor memory too
    (dict(T=5, N=64, K=8, window=128), 2),     # a window, 40 rows: tensor memory
    (dict(T=5, N=64, K=8, window=128, H=64), 2),  # ... also at H = 64
    (dict(T=3, N=64, K=8, H=64), 1),           # 24 rows: warp-level
    (dict(T=5, N=64, K=8, flags=4), 1),        # GQA_FLAG_WARP_MMA
    (dict(T=1, N=8, K=8, flags=8), 2),         # GQA_FLAG_TENSOR_MEMORY
    (dict(T=1, N=8, K=8, H=64, flags=8), 2),   # forced: served at H = 64 too
    (dict(T=1, N=8, K=8, kv_dtype=1, flags=8), 0),  # forced, one-byte cache: not served
    (dict(T=5, N=64, K=8, flags=12), 0),       # both forced
    (dict(N=7), 0),                            # invalid shape
])
def test_attention_engine_choice(cuda_lib, kw, want):
    """The kernel choice is host logic, checked without a GPU."""
    assert cuda_lib.gqa_attention_engine(ctypes.byref(_shape(**kw))) == want


def test_attention_engine_python_binding(cuda_lib):
    import torch

    import gqa_decode_attention_02_gb300 as gq

    bt = torch.zeros(2, 4, dtype=torch.int32)
    kc = torch.zeros(10, 16, 8, 128, dtype=torch.bfloat16)
    verify = torch.zeros(2, 5, 64, 128, dtype=torch.bfloat16)   # 40 rows per KV head
    decode = torch.zeros(2, 1, 32, 128, dtype=torch.bfloat16)   # 4 rows per KV head
    assert gq.attention_engine(verify, kc, bt) == "tmem"
    assert gq.attention_engine(decode, kc, bt) == "direct"
    assert gq.attention_engine(decode, kc, bt, engine="warp") == "warp"
    assert gq.attention_engine(verify, kc, bt, engine="warp") == "warp"
    assert gq.attention_engine(verify, kc, bt, window=64) == "tmem"
    assert gq.attention_engine(torch.zeros(2, 1, 32, 64, dtype=torch.bfloat16),  # H = 64, forced
                               torch.zeros(10, 16, 8, 64, dtype=torch.bfloat16), bt,
                               engine="tmem") == "tmem"
