"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every function include/kvq.h declares, sizes buffers as the
packed format says, and rejects bad arguments before launching anything."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvq():
    from bit_kv_cache_02_gb300 import build
    build.build()
    from bit_kv_cache_02_gb300 import kvq as mod
    return mod


def _declared():
    text = open(os.path.join(ROOT, "include", "kvq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kvq?_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol(kvq):
    names = _declared()
    assert {"kv_quant_append", "kv_decode_attn", "kv_dequant", "kv_decode_workspace_bytes"} <= set(names)
    lib = ctypes.CDLL(kvq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(kvq.EXPORTED) == set(names)


def _struct(kvq, **kw):
    d = dict(num_seqs=2, num_kv_heads=3, head_dim=128, bits=2, group=32, residual=128, num_sink=1,
             pre_rope=0, rope_theta=10000.0, capacity=1000)
    d.update(kw)
    st = kvq.CacheStruct()
    for k, v in d.items():
        setattr(st, k, v)
    return st


def test_sizes(kvq):
    bb = kvq.lib.kvq_block_bytes
    assert bb(2, 128, 0, 0) == 3328 and bb(4, 128, 0, 0) == 5376
    assert bb(2, 128, 1, 0) == 2560 and bb(4, 128, 1, 0) == 4608
    assert bb(2, 128, 0, 1) == 3968 and bb(4, 128, 0, 1) == 6016     # + one entry per key channel and value token
    assert bb(2, 128, 1, 1) == 2816 and bb(4, 128, 1, 1) == 4864
    assert bb(3, 128, 0, 0) == 0 and bb(2, 64, 0, 0) == 0 and bb(2, 128, 0, 2) == 0
    st = _struct(kvq)
    # (1000 - 1) // 128 * 128 = 896 quantized tokens -> 28 groups
    assert kvq.lib.kvq_max_groups(ctypes.byref(st)) == 28
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(st), kvq.BUF_BLOCKS) == 2 * 3 * 28 * 3328
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(st), kvq.BUF_K_RES) == 2 * 3 * 128 * 128 * 2
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(st), kvq.BUF_K_SINK) == 2 * 3 * 1 * 128 * 2
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(st), kvq.BUF_SEQ_LEN) == 8
    st0 = _struct(kvq, num_sink=0)
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(st0), kvq.BUF_K_SINK) == 0
    stk = _struct(kvq, key_per_token=1)   # per-token key metadata: 2560-byte blocks
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(stk), kvq.BUF_BLOCKS) == 2 * 3 * 28 * 2560
    stp = _struct(kvq, num_blocks=100)    # paged: a pool of 100 blocks plus the table
    stp.block_table = 1 << 20
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(stp), kvq.BUF_BLOCKS) == 100 * 3328
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(stp), kvq.BUF_BLOCK_TABLE) == 2 * 3 * 28 * 4
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(st), kvq.BUF_BLOCK_TABLE) == 0


@pytest.mark.parametrize("field,value,code", [
    ("head_dim", 64, -2), ("bits", 3, -2), ("group", 16, -2), ("residual", 100, -2),
    ("residual", 256, -2), ("num_sink", 2, -2), ("num_seqs", 0, -1), ("capacity", 0, -1),
    ("key_per_token", 2, -1), ("hadamard", 2, -1), ("outliers", 2, -1),
])
def test_bad_geometry_rejected(kvq, field, value, code):
    st = _struct(kvq, **{field: value})
    assert kvq.lib.kvq_max_groups(ctypes.byref(st)) == -1
    assert kvq.lib.kv_decode_workspace_bytes(ctypes.byref(st), 3, 10) == -1
    fake = ctypes.c_void_p(1 << 20)
    assert kvq.lib.kv_quant_append(ctypes.byref(st), fake, fake, fake, 1, None) == code


def test_paged_validation(kvq):
    """A paged cache needs a pool when it can hold groups and an aligned table."""
    st = _struct(kvq, num_blocks=0)
    base = 1 << 30
    st.blocks, st.k_res, st.v_res = base, base + 4096, base + 8192
    st.k_sink, st.v_sink, st.seq_len = base + 12288, base + 16384, base + 20480
    st.block_table = base + 24576
    fake = ctypes.c_void_p(base + (1 << 24))
    assert kvq.lib.kv_quant_append(ctypes.byref(st), fake, fake, fake, 1, None) == -1
    st.num_blocks = 10
    st.block_table = base + 24578
    assert kvq.lib.kv_quant_append(ctypes.byref(st), fake, fake, fake, 1, None) == -5


def test_key_per_token_with_pre_rope_unsupported(kvq):
    """Per-token key grouping is the ablation of the per-channel method and is
    not combined with pre-RoPE keys."""
    st = _struct(kvq, key_per_token=1, pre_rope=1)
    assert kvq.lib.kvq_max_groups(ctypes.byref(st)) == -1
    fake = ctypes.c_void_p(1 << 20)
    assert kvq.lib.kv_quant_append(ctypes.byref(st), fake, fake, fake, 1, None) == -2


def test_hadamard_with_pre_rope_unsupported(kvq):
    """The rotation is not combined with pre-RoPE keys (it does not commute
    with the per-position RoPE rotation); with per-token keys it is fine."""
    st = _struct(kvq, hadamard=1, pre_rope=1)
    assert kvq.lib.kvq_max_groups(ctypes.byref(st)) == -1
    fake = ctypes.c_void_p(1 << 20)
    assert kvq.lib.kv_quant_append(ctypes.byref(st), fake, fake, fake, 1, None) == -2
    assert kvq.lib.kvq_max_groups(ctypes.byref(_struct(kvq, hadamard=1, key_per_token=1))) == 28


def test_outliers_combinations(kvq):
    """Dense-and-sparse blocks work with both key groupings and with paging,
    not with pre-RoPE keys or the rotation; the pool grows by the entries."""
    fake = ctypes.c_void_p(1 << 20)
    for kw in (dict(pre_rope=1), dict(hadamard=1)):
        st = _struct(kvq, outliers=1, **kw)
        assert kvq.lib.kv_quant_append(ctypes.byref(st), fake, fake, fake, 1, None) == -2
    st = _struct(kvq, outliers=1, key_per_token=1)
    assert kvq.lib.kvq_buffer_bytes(ctypes.byref(st), kvq.BUF_BLOCKS) == 2 * 3 * 28 * 2816


def test_struct_layout_matches_header(kvq):
    """The ctypes mirror has the header's field order and offsets: 14 int32
    or float fields, then eight pointers from byte 56."""
    names = [f[0] for f in kvq.CacheStruct._fields_]
    assert names[:14] == ["num_seqs", "num_kv_heads", "head_dim", "bits", "group", "residual", "num_sink",
                          "pre_rope", "rope_theta", "capacity", "key_per_token", "num_blocks", "hadamard",
                          "outliers"]
    assert kvq.CacheStruct.blocks.offset == 56 and ctypes.sizeof(kvq.CacheStruct) == 56 + 8 * 8


def test_workspace_sizing(kvq):
    st = _struct(kvq)
    n = kvq.lib.kv_decode_workspace_bytes(ctypes.byref(st), 6, 1000)
    assert n > 0 and n % 256 == 0
    assert kvq.lib.kv_decode_workspace_bytes(ctypes.byref(st), 5, 1000) == -1   # not a multiple of Hkv
    assert kvq.lib.kv_decode_workspace_bytes(ctypes.byref(st), 24, 1000) == -1  # group of 8 unsupported
    assert kvq.lib.kv_decode_workspace_bytes(ctypes.byref(st), 6, 1001) == -1   # past capacity


def test_null_and_misaligned_buffers_rejected_before_launch(kvq):
    st = _struct(kvq)
    base = 1 << 30
    st.blocks, st.k_res, st.v_res = base, base + 4096, base + 8192
    st.k_sink, st.v_sink, st.seq_len = base + 12288, base + 16384, base + 20480
    p = ctypes.byref(st)
    kn = ctypes.c_void_p(base + (1 << 24))
    nl = ctypes.c_void_p(base + (1 << 25))
    assert kvq.lib.kv_quant_append(p, None, kn, nl, 4, None) == -1          # null k_new
    assert kvq.lib.kv_quant_append(p, kn, kn, None, 4, None) == -1          # null new_len
    assert kvq.lib.kv_quant_append(p, kn, kn, nl, 1001, None) == -3         # max_new > capacity
    assert kvq.lib.kv_quant_append(p, ctypes.c_void_p(base + 2), kn, nl, 4, None) == -5
    st.blocks = base + 64                                                     # blocks need 128 B
    assert kvq.lib.kv_quant_append(p, kn, kn, nl, 4, None) == -5
    st.blocks = base
    st.k_sink = None                                                          # sink needed when num_sink=1
    assert kvq.lib.kv_quant_append(p, kn, kn, nl, 4, None) == -1
    st.k_sink = base + 12288
    q = ctypes.c_void_p(base + (1 << 26))
    ws = ctypes.c_void_p(base + (1 << 27))
    need = kvq.lib.kv_decode_workspace_bytes(p, 6, 1000)
    assert kvq.lib.kv_decode_attn(p, 6, q, 0.0, q, ws, need - 1, 1000, None) == -4
    assert kvq.lib.kv_decode_attn(p, 6, q, 0.0, q, None, need, 1000, None) == -4
    assert kvq.lib.kv_decode_attn(p, 6, q, 0.0, q, ctypes.c_void_p(base + (1 << 27) + 16), need, 1000, None) == -5
    assert kvq.lib.kv_decode_attn(p, 6, q, 0.0, q, ws, need, 1001, None) == -3
    assert kvq.lib.kv_decode_attn(p, 24, q, 0.0, q, ws, need, 1000, None) == -2
    assert kvq.lib.kv_decode_attn(p, 6, None, 0.0, q, ws, need, 1000, None) == -1
    assert kvq.lib.kv_dequant(p, None, q, None) == -1
    assert kvq.lib.kvq_set_decode_warps(-1) == -1 and kvq.lib.kvq_set_decode_warps(2561) == -1
    assert kvq.lib.kvq_set_decode_warps(7) == 0 and kvq.lib.kvq_set_decode_warps(0) == 0
    assert kvq.lib.kvq_set_wait_test(-1, 0) == -1 and kvq.lib.kvq_set_wait_test(4000000001, 0) == -1
    assert kvq.lib.kvq_set_wait_test(0, 1) == -1 and kvq.lib.kvq_set_wait_test(100, 2) == -1
    assert kvq.lib.kvq_set_wait_test(100, 1) == 0 and kvq.lib.kvq_set_wait_test(0, 0) == 0
    assert kvq.lib.kvq_strerror(-4) == b"workspace missing or too small"
