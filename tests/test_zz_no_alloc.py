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


def _cache(kvq, S, H, T, bits, ns, pre_rope, seed):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((S, H, T, 128), dtype=np.float32)
    v = rng.standard_normal((S, H, T, 128), dtype=np.float32)
    k[..., [3, 17, 64, 101]] *= 15
    k, v = k.astype(np.float16), v.astype(np.float16)
    lens = np.array([T - (37 * s) % (T - 1) for s in range(S)], np.int32)
    cache = kvq.KVCache(S, H, T + 8, bits=bits, num_sink=ns, pre_rope=pre_rope)
    kvq.kv_quant_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                        torch.from_numpy(lens).cuda(), T)
    orc = oracle.OracleCache(S, H, T + 8, bits, num_sink=ns)
    orc.append(k, v, lens)
    return cache, orc, lens


@pytest.mark.parametrize("S,H,T,bits,gq,ns,pre_rope", [
    (3, 2, 900, 2, 1, 0, False),
    (3, 2, 900, 4, 4, 1, False),
    (3, 2, 700, 2, 2, 1, True),     # keys stored before RoPE: the RoPE tables live in the scratch too
    (257, 1, 200, 2, 1, 0, False),  # more than 256 sequences: the work prefix is planned in the scratch
])
def test_noalloc_matches_workspace_entry_point(kvq, S, H, T, bits, gq, ns, pre_rope):
    """Three calls in a row share the built-in scratch; each must give the
    workspace entry point's output (and the oracle's), and device memory
    must not change across them."""
    cache, orc, lens = _cache(kvq, S, H, T, bits, ns, pre_rope, seed=bits + gq + S)
    max_len = int(lens.max())
    rng = np.random.default_rng(1)
    ws = kvq.alloc_workspace(cache, H * gq, max_len)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    qs = [torch.from_numpy(rng.standard_normal((S, H * gq, 128), dtype=np.float32).astype(np.float16)).cuda()
          for _ in range(3)]
    refs = [torch.empty_like(q) for q in qs]
    outs = [torch.full_like(q, float("nan")) for q in qs]
    free = []
    for call, (q, ref, out) in enumerate(zip(qs, refs, outs)):
        kvq.kv_decode_attn(cache, q, ref, ws, max_len)
        rc = kvq.lib.kv_decode_attn_noalloc(cache.ref, H * gq, ctypes.c_void_p(q.data_ptr()), 0.0,
                                            ctypes.c_void_p(out.data_ptr()), max_len, stream)
        assert rc == 0, kvq.lib.kvq_strerror(rc)
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
        got, want = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert (np.abs(got - want) <= ATOL + RTOL * np.abs(want)).all(), f"call {call}"
        o = orc.attention(q.cpu().numpy(), pre_rope=pre_rope).astype(np.float64)
        assert (np.abs(got - o) <= ATOL + RTOL * np.abs(o)).all(), f"call {call} vs oracle"
    assert free[1] == free[2], "device memory changed across calls"
    assert int(cache.status.item()) == 0


def test_noalloc_rejects_requests_beyond_its_scratch(kvq):
    """16 MiB of built-in scratch: a valid request that needs more fails
    cleanly and enqueues nothing.  Every buffer is a real allocation of the
    size the geometry needs (an empty cache of 3000 KV heads, four query
    heads each), so a launch by mistake would stay in bounds."""
    S, H, gq, R = 1, 3000, 4, 32
    cache = kvq.KVCache(S, H, 1, bits=2, residual=R)
    need = kvq.kv_decode_workspace_bytes(cache, H * gq, 1)
    assert need > (16 << 20)
    q = torch.zeros((S, H * gq, 128), dtype=torch.float16, device="cuda")
    out = torch.full_like(q, 7.0)
    torch.cuda.synchronize()
    rc = kvq.lib.kv_decode_attn_noalloc(cache.ref, H * gq, ctypes.c_void_p(q.data_ptr()), 0.0,
                                        ctypes.c_void_p(out.data_ptr()), 1, None)
    assert rc == -4
    torch.cuda.synchronize()
    assert bool((out == 7.0).all()), "nothing may be written"
    # argument errors are reported as kv_decode_attn reports them, before the size
    assert kvq.lib.kv_decode_attn_noalloc(cache.ref, H * gq, None, 0.0, ctypes.c_void_p(out.data_ptr()), 1,
                                          None) == -1
    assert kvq.lib.kv_decode_attn_noalloc(cache.ref, H * gq, ctypes.c_void_p(q.data_ptr() + 2), 0.0,
                                          ctypes.c_void_p(out.data_ptr()), 1, None) == -5
