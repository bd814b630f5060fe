"""Parity at the benchmark workloads' full sizes, in the launch configuration
bench.py times (one layer: prefill of the whole context, one decode append,
decode attention with the grid sized for the cache capacity).

The oracle recomputes a few sampled (sequence, KV head) pairs from host
copies of the same seeded inputs: their packed blocks, window, sink and
length must match byte for byte, and the attention outputs of their query
heads within |gpu - oracle| <= 2e-3 + 1e-2 |oracle|."""

import numpy as np
import pytest
import torch

import oracle
from bit_kv_cache_02_gb300 import synth

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


def _run(kvq, name, pairs):
    w = synth.WORKLOADS[name]
    dev = "cuda"
    lens = synth.context_lengths(w)
    T = int(lens.max())
    cap = T + 8
    cache = kvq.KVCache(w.seqs, w.kv_heads, cap, bits=w.bits, residual=w.residual, num_sink=w.num_sink,
                        pre_rope=w.pre_rope, device=dev, key_per_token=w.key_per_token, paged=w.paged,
                        hadamard=w.hadamard, outliers=w.dense_sparse)
    if w.paged:
        tbl = synth.block_table(w, 0, w.seqs, w.kv_heads, cache.max_groups)
        cache.block_table.copy_(torch.from_numpy(tbl).to(dev))
    k, v = synth.kv_tokens(w, 0, T, device=dev)
    kvq.kv_quant_append(cache, k.contiguous(), v.contiguous(), torch.as_tensor(lens, device=dev), T)
    k1, v1 = synth.kv_tokens(w, 0, 1, device=dev, stream_id=1)
    ones = torch.ones(w.seqs, dtype=torch.int32, device=dev)
    kvq.kv_quant_append(cache, k1.contiguous(), v1.contiguous(), ones, 1)
    q = synth.queries(w, 0, 0, device=dev)
    out = torch.empty_like(q)
    ws = kvq.alloc_workspace(cache, w.q_heads, cap)
    kvq.kv_decode_attn(cache, q, out, ws, cap)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    gq = w.q_heads // w.kv_heads
    blocks = cache.logical_blocks()
    got = out.cpu().numpy().astype(np.float64)
    qh = q.cpu().numpy()
    worst = 0.0
    for s, h in pairs:
        L = int(lens[s])
        orc = oracle.OracleCache(1, 1, cap, w.bits, residual=w.residual, num_sink=w.num_sink,
                                 key_per_token=w.key_per_token, hadamard=w.hadamard,
                                 outliers=w.dense_sparse)
        ks = k[s:s + 1, h:h + 1, :L].cpu().numpy()
        vs = v[s:s + 1, h:h + 1, :L].cpu().numpy()
        orc.append(ks, vs, [L])
        orc.append(k1[s:s + 1, h:h + 1].cpu().numpy(), v1[s:s + 1, h:h + 1].cpu().numpy(), [1])
        assert int(cache.seq_len[s].item()) == L + 1 == int(orc.seq_len[0])
        ns, Lq, r = orc.split(0)
        ng = Lq // 32
        np.testing.assert_array_equal(blocks[s, h, :ng].cpu().numpy(), orc.blocks[0, 0, :ng],
                                      err_msg=f"{name}: blocks of ({s}, {h})")
        np.testing.assert_array_equal(cache.k_res[s, h, :r].cpu().numpy().view(np.uint16),
                                      orc.k_res[0, 0, :r].view(np.uint16))
        np.testing.assert_array_equal(cache.v_res[s, h, :r].cpu().numpy().view(np.uint16),
                                      orc.v_res[0, 0, :r].view(np.uint16))
        if ns:
            np.testing.assert_array_equal(cache.k_sink[s, h, :ns].cpu().numpy().view(np.uint16),
                                          orc.k_sink[0, 0, :ns].view(np.uint16))
        want = orc.attention(qh[s:s + 1, h * gq:(h + 1) * gq], pre_rope=w.pre_rope).astype(np.float64)[0]
        g = got[s, h * gq:(h + 1) * gq]
        err = np.abs(g - want)
        assert (err <= ATOL + RTOL * np.abs(want)).all(), f"{name} ({s}, {h}): max abs err {err.max():.3e}"
        worst = max(worst, float(err.max()))
    return worst


def test_llama2_7b_mha_2bit(kvq):
    """16 sequences x 32 heads, context 4096 (+1), 2-bit."""
    _run(kvq, "llama2_7b_mha", [(0, 0), (15, 31), (7, 3), (11, 19)])


@pytest.mark.parametrize("name", ["llama3_8b_gqa_2bit", "llama3_8b_gqa_4bit"])
def test_llama3_8b_gqa_ragged(kvq, name):
    """64 sequences of ragged length (U{1024..8192}), 8 KV heads x 4 query heads."""
    lens = synth.context_lengths(synth.WORKLOADS[name])
    pairs = [(0, 0), (63, 7), (int(np.argmin(lens)), 3), (int(np.argmax(lens)), 5)]
    _run(kvq, name, pairs)


def test_kvquant_prerope_sink(kvq):
    """8 sequences x 32 heads, context 16384 (+1), keys quantized before RoPE,
    token 0 kept in fp16."""
    _run(kvq, "kvquant_prerope", [(0, 0), (7, 31), (3, 17)])


def test_long_context_1m(kvq):
    """One sequence x 32 heads, 2^20 context tokens (+1), split-K decode: the
    first and last pairs on the work line (whose range and merge edges
    differ) and one between."""
    _run(kvq, "long_1m", [(0, 0), (0, 13), (0, 31)])


@pytest.mark.parametrize("name", ["llama2_7b_mha_key_per_token", "llama2_7b_mha_paged", "llama2_7b_mha_hadamard",
                                  "llama2_7b_mha_key_per_token_hadamard", "llama2_7b_mha_outliers"])
def test_llama2_7b_mha_variants(kvq, name):
    """The Llama-2 shape with keys grouped per token, with its group blocks
    paged through a shuffled block table, and with Walsh-Hadamard rotated
    tokens (per-channel and per-token keys), and with dense-and-sparse
    blocks."""
    _run(kvq, name, [(0, 0), (15, 31), (9, 12)])
