"""kv_decode_attn_noalloc: the decode-attention entry point for callers that
cannot allocate device memory (their device memory is owned by another
runtime, or cudaMalloc is off limits on their path).  It must give the same
result as kv_decode_attn with a caller-provided workspace, call after call,
using only the scratch built into the library.  Collected last on purpose."""

import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ATOL, RTOL = 2e-3, 1e-2


@pytest.fixture(scope="module")
def kvq():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from bit_kv_cache_02_gb300 import build
    build.build()
    from bit_kv_cache_02_gb300 import kvq as mod
    return mod


def _cache(kvq, S, H, T, bits, ns, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((S, H, T, 128), dtype=np.float32)
    v = rng.standard_normal((S, H, T, 128), dtype=np.float32)
    k[..., [3, 17, 64, 101]] *= 15
    k, v = k.astype(np.float16), v.astype(np.float16)
    lens = np.array([T - 37 * s for s in range(S)], np.int32)
    cache = kvq.KVCache(S, H, T + 8, bits=bits, num_sink=ns)
    kvq.kv_quant_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                        torch.from_numpy(lens).cuda(), T)
    orc = oracle.OracleCache(S, H, T + 8, bits, num_sink=ns)
    orc.append(k, v, lens)
    return cache, orc, lens


@pytest.mark.parametrize("bits,gq,ns", [(2, 1, 0), (4, 4, 1)])
def test_noalloc_matches_workspace_entry_point(kvq, bits, gq, ns):
    S, H, T = 3, 2, 900
    cache, orc, lens = _cache(kvq, S, H, T, bits, ns, seed=bits + gq)
    max_len = int(lens.max())
    rng = np.random.default_rng(1)
    ws = kvq.alloc_workspace(cache, H * gq, max_len)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):                      # two calls in a row share the scratch
        q = torch.from_numpy(rng.standard_normal((S, H * gq, 128), dtype=np.float32).astype(np.float16)).cuda()
        ref = torch.empty_like(q)
        kvq.kv_decode_attn(cache, q, ref, ws, max_len)
        out = torch.full_like(q, float("nan"))
        rc = kvq.lib.kv_decode_attn_noalloc(cache.ref, H * gq, ctypes.c_void_p(q.data_ptr()), 0.0,
                                            ctypes.c_void_p(out.data_ptr()), max_len, stream)
        assert rc == 0, kvq.lib.kvq_strerror(rc)
        torch.cuda.synchronize()
        got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert (np.abs(got - want) <= ATOL + RTOL * np.abs(want)).all(), f"call {call}"
        o = orc.attention(q.cpu().numpy()).astype(np.float64)
        assert (np.abs(got - o) <= ATOL + RTOL * np.abs(o)).all(), f"call {call} vs oracle"
    assert int(cache.status.item()) == 0


def test_noalloc_rejects_requests_beyond_its_scratch(kvq):
    """16 MiB of built-in scratch: a request that needs more fails cleanly."""
    st = kvq.CacheStruct(4096, 8, 128, 2, 32, 128, 0, 0, 10000.0, 1 << 17)
    base = 1 << 30
    st.blocks, st.k_res, st.v_res, st.seq_len = base, base + 4096, base + 8192, base + 12288
    st.k_sink = st.v_sink = base + 16384
    need = kvq.lib.kv_decode_workspace_bytes(ctypes.byref(st), 32, 1 << 17)
    assert need > (16 << 20)
    q = ctypes.c_void_p(base + (1 << 26))
    rc = kvq.lib.kv_decode_attn_noalloc(ctypes.byref(st), 32, q, 0.0, q, 1 << 17, None)
    assert rc == -4
