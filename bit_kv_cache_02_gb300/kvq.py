"""Python binding of the C ABI in include/kvq.h (ctypes).

Argument marshalling only: every step of the hot path runs in the CUDA
kernels of libkvq.so.  torch tensors serve as device memory and torch streams
as CUDA streams.  If the shared object is missing the import of this module
fails; there is no fallback implementation.
"""

from __future__ import annotations

import ctypes
import os
from ctypes import c_float, c_int32, c_int64, c_size_t, c_uint64, c_void_p

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# KVQ_LIB_PATH selects another build of the same library (the bounds-checking
# debug build of build.build_debug); by default the in-tree release build.
LIB_PATH = os.environ.get("KVQ_LIB_PATH") or os.path.join(_HERE, "libkvq.so")

KVQ_OK = 0
KVQ_STATUS_CAPACITY = 1
KVQ_STATUS_BAD_LEN = 2
KVQ_STATUS_TIMEOUT = 4
KVQ_STATUS_MAX_LEN = 8
KVQ_STATUS_BAD_BLOCK = 16
KVQ_STATUS_BOUNDS = 32
BUF_BLOCKS, BUF_K_RES, BUF_V_RES, BUF_K_SINK, BUF_V_SINK, BUF_SEQ_LEN, BUF_BLOCK_TABLE = range(7)

EXPORTED = (
    "kvq_block_bytes", "kvq_max_groups", "kvq_buffer_bytes", "kv_quant_append",
    "kv_decode_workspace_bytes", "kv_decode_attn", "kv_dequant", "kvq_strerror",
    "kvq_launch_count", "kvq_set_decode_warps", "kv_decode_attn_noalloc", "kvq_set_wait_test",
)


class CacheStruct(ctypes.Structure):
    """Mirror of `kvq_cache` (include/kvq.h)."""
    _fields_ = [
        ("num_seqs", c_int32), ("num_kv_heads", c_int32), ("head_dim", c_int32),
        ("bits", c_int32), ("group", c_int32), ("residual", c_int32),
        ("num_sink", c_int32), ("pre_rope", c_int32), ("rope_theta", c_float),
        ("capacity", c_int32), ("key_per_token", c_int32), ("num_blocks", c_int32), ("hadamard", c_int32),
        ("outliers", c_int32),
        ("blocks", c_void_p), ("k_res", c_void_p), ("v_res", c_void_p),
        ("k_sink", c_void_p), ("v_sink", c_void_p), ("seq_len", c_void_p),
        ("status", c_void_p), ("block_table", c_void_p),
    ]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with bit_kv_cache_02_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.POINTER(CacheStruct)
    sig = {
        "kvq_block_bytes": (c_int32, [c_int32, c_int32, c_int32, c_int32]),
        "kvq_max_groups": (c_int32, [P]),
        "kvq_buffer_bytes": (c_int64, [P, c_int32]),
        "kv_quant_append": (ctypes.c_int, [P, c_void_p, c_void_p, c_void_p, c_int32, c_void_p]),
        "kv_decode_workspace_bytes": (c_int64, [P, c_int32, c_int32]),
        "kv_decode_attn": (ctypes.c_int, [P, c_int32, c_void_p, c_float, c_void_p, c_void_p, c_size_t,
                                          c_int32, c_void_p]),
        "kv_dequant": (ctypes.c_int, [P, c_void_p, c_void_p, c_void_p]),
        "kvq_strerror": (ctypes.c_char_p, [ctypes.c_int]),
        "kvq_launch_count": (c_uint64, []),
        "kvq_set_decode_warps": (ctypes.c_int, [c_int32]),
        "kvq_set_wait_test": (ctypes.c_int, [c_int64, c_int32]),
        "kv_decode_attn_noalloc": (ctypes.c_int, [P, c_int32, c_void_p, c_float, c_void_p, c_int32, c_void_p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


class KvqError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what}: {lib.kvq_strerror(code).decode()} ({code})")
        self.code = code


def _check(code: int, what: str):
    if code != KVQ_OK:
        raise KvqError(code, what)


def _ptr(t):
    return None if t is None else c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def block_bytes(bits: int, head_dim: int = 128, key_per_token: bool = False, outliers: bool = False) -> int:
    return lib.kvq_block_bytes(bits, head_dim, int(key_per_token), int(outliers))


class KVCache:
    """Device buffers of one quantized KV cache (one layer) and its descriptor.

    All tensors are allocated by torch on `device`; the library itself
    allocates nothing.  seq_len starts at zero (an empty cache).
    """

    def __init__(self, num_seqs, num_kv_heads, capacity, bits=2, residual=128, num_sink=0,
                 pre_rope=False, rope_theta=10000.0, head_dim=128, device="cuda", key_per_token=False,
                 num_blocks=None, paged=False, hadamard=False, outliers=False):
        """num_blocks (or paged=True, for a pool of one block per logical
        group): a paged layout with a pool of that many blocks and a block
        table [S][Hkv][max_groups] (int32, filled with -1: the caller assigns
        pool blocks before the appends that need them).  hadamard: tokens are
        Walsh-Hadamard rotated before quantization; outliers: dense-and-sparse
        blocks (include/kvq.h)."""
        st = CacheStruct(num_seqs, num_kv_heads, head_dim, bits, 32, residual, num_sink,
                         int(bool(pre_rope)), float(rope_theta), capacity, int(bool(key_per_token)),
                         int(num_blocks or 0), int(bool(hadamard)), int(bool(outliers)))
        self.num_seqs, self.num_kv_heads, self.capacity = num_seqs, num_kv_heads, capacity
        self.bits, self.residual, self.num_sink, self.head_dim = bits, residual, num_sink, head_dim
        self.pre_rope, self.rope_theta = bool(pre_rope), rope_theta
        self.key_per_token = bool(key_per_token)
        self.hadamard = bool(hadamard)
        self.outliers = bool(outliers)
        self.max_groups = lib.kvq_max_groups(ctypes.byref(st))
        if self.max_groups < 0:
            raise KvqError(-2, "kvq_max_groups")
        self.block_bytes = block_bytes(bits, head_dim, key_per_token, outliers)
        self.paged = paged or num_blocks is not None
        if self.paged and num_blocks is None:
            num_blocks = num_seqs * num_kv_heads * self.max_groups
        st.num_blocks = int(num_blocks or 0)

        def nbytes(which):
            n = lib.kvq_buffer_bytes(ctypes.byref(st), which)
            if n < 0:
                raise KvqError(-1, "kvq_buffer_bytes")
            return n

        S, H, D = num_seqs, num_kv_heads, head_dim
        self.num_blocks = int(num_blocks) if self.paged else S * H * self.max_groups
        self.block_table = None
        if self.paged:
            tbl = torch.full((S * H * self.max_groups + 1,), -1, dtype=torch.int32, device=device)
            self.block_table = tbl[:-1].view(S, H, self.max_groups)
            st.block_table = tbl.data_ptr()
        self.blocks = torch.zeros(max(nbytes(BUF_BLOCKS), 128), dtype=torch.uint8, device=device)
        assert nbytes(BUF_BLOCKS) == self.num_blocks * self.block_bytes
        self.k_res = torch.zeros((S, H, residual, D), dtype=torch.float16, device=device)
        self.v_res = torch.zeros_like(self.k_res)
        self.k_sink = torch.zeros((S, H, max(num_sink, 1), D), dtype=torch.float16, device=device)
        self.v_sink = torch.zeros_like(self.k_sink)
        self.seq_len = torch.zeros(S, dtype=torch.int32, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        st.blocks = self.blocks.data_ptr()
        st.k_res, st.v_res = self.k_res.data_ptr(), self.v_res.data_ptr()
        st.k_sink, st.v_sink = self.k_sink.data_ptr(), self.v_sink.data_ptr()
        st.seq_len, st.status = self.seq_len.data_ptr(), self.status.data_ptr()
        self.struct = st

    @property
    def ref(self):
        return ctypes.byref(self.struct)

    def blocks_view(self):
        """blocks as [S][H][max_groups][block_bytes] (a view; contiguous layout)."""
        assert not self.paged
        return self.blocks[:self.num_blocks * self.block_bytes].view(
            self.num_seqs, self.num_kv_heads, self.max_groups, self.block_bytes)

    def logical_blocks(self):
        """[S][H][max_groups][block_bytes] in logical order (a copy through the
        block table when paged; entries outside the pool give zeros)."""
        if not self.paged:
            return self.blocks_view().clone()
        pool = self.blocks[:self.num_blocks * self.block_bytes].view(self.num_blocks, self.block_bytes)
        idx = self.block_table.long()
        ok = (idx >= 0) & (idx < self.num_blocks)
        out = pool[idx.clamp(0, max(self.num_blocks - 1, 0))]
        return out * ok[..., None].to(out.dtype)


def kv_quant_append(cache: KVCache, k_new, v_new, new_len, max_new: int, stream=None):
    """k_new/v_new: fp16 [S][Hkv][max_new][D] contiguous device tensors;
    new_len: int32 [S] device tensor."""
    for t in (k_new, v_new):
        assert t.dtype == torch.float16 and t.is_contiguous() and t.is_cuda
    assert new_len.dtype == torch.int32 and new_len.is_cuda
    _check(lib.kv_quant_append(cache.ref, _ptr(k_new), _ptr(v_new), _ptr(new_len), int(max_new),
                               _stream(stream)), "kv_quant_append")


def kv_decode_workspace_bytes(cache: KVCache, num_q_heads: int, max_len: int) -> int:
    n = lib.kv_decode_workspace_bytes(cache.ref, num_q_heads, max_len)
    if n < 0:
        raise KvqError(-1, "kv_decode_workspace_bytes")
    return n


def alloc_workspace(cache: KVCache, num_q_heads: int, max_len: int):
    """A torch-allocated, zero-filled workspace for kv_decode_attn (256-byte
    aligned); it stays valid for calls on caches of this geometry."""
    n = kv_decode_workspace_bytes(cache, num_q_heads, max_len)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=cache.blocks.device)


def kv_decode_attn(cache: KVCache, q, out, workspace, max_len: int, softmax_scale: float = 0.0,
                   stream=None):
    """q, out: fp16 [S][Hq][D] contiguous device tensors."""
    assert q.dtype == torch.float16 and q.is_contiguous() and out.dtype == torch.float16
    assert out.is_contiguous() and q.shape == out.shape
    _check(lib.kv_decode_attn(cache.ref, q.shape[1], _ptr(q), float(softmax_scale), _ptr(out),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              int(max_len), _stream(stream)), "kv_decode_attn")


def kv_dequant(cache: KVCache, k_out, v_out, stream=None):
    """k_out, v_out: fp32 [S][Hkv][capacity][D] device tensors."""
    assert k_out.dtype == torch.float32 and v_out.dtype == torch.float32
    _check(lib.kv_dequant(cache.ref, _ptr(k_out), _ptr(v_out), _stream(stream)), "kv_dequant")


def launch_count() -> int:
    return lib.kvq_launch_count()


def set_decode_warps(warps: int):
    """Warps a decode launch cuts its work into (0: every resident warp)."""
    _check(lib.kvq_set_decode_warps(warps), "kvq_set_decode_warps")


def set_wait_test(limit_cycles: int, wait_before_fetch: bool = False):
    """Test aid for the decode kernel's bounded waits: their cycle limit (0:
    the default of about two seconds) and whether each warp's first wait
    comes before its first copy (so that it runs out)."""
    _check(lib.kvq_set_wait_test(int(limit_cycles), int(bool(wait_before_fetch))), "kvq_set_wait_test")
