"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.

Packed codes, scales, mins, the fp16 window, the sink and seq_len must match
byte for byte; dequantized values within 1 fp32 ulp; attention outputs within
|gpu - oracle| <= 2e-3 + 1e-2 * |oracle| per element (fp16 outputs)."""

import math

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


def _rand_kv(S, H, T, seed, outliers=(3, 17, 64, 101), mult=15.0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((S, H, T, 128), dtype=np.float32)
    v = rng.standard_normal((S, H, T, 128), dtype=np.float32)
    k[..., list(outliers)] *= mult
    return k.astype(np.float16), v.astype(np.float16)


def _rand_q(S, Hq, seed):
    return np.random.default_rng(seed).standard_normal((S, Hq, 128), dtype=np.float32).astype(np.float16)


def _compare_state(cache, orc, heads=None):
    """Byte-compare the valid parts of the device state with the oracle's."""
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    sl = cache.seq_len.cpu().numpy()
    np.testing.assert_array_equal(sl, orc.seq_len)
    blocks = cache.logical_blocks().cpu().numpy()
    kres, vres = cache.k_res.cpu().numpy(), cache.v_res.cpu().numpy()
    ksink, vsink = cache.k_sink.cpu().numpy(), cache.v_sink.cpu().numpy()
    for s in range(orc.S):
        ns, Lq, r = orc.split(s)
        ng = Lq // 32
        np.testing.assert_array_equal(blocks[s, :, :ng], orc.blocks[s, :, :ng], err_msg=f"blocks seq {s}")
        np.testing.assert_array_equal(kres[s, :, :r].view(np.uint16), orc.k_res[s, :, :r].view(np.uint16))
        np.testing.assert_array_equal(vres[s, :, :r].view(np.uint16), orc.v_res[s, :, :r].view(np.uint16))
        if ns:
            np.testing.assert_array_equal(ksink[s, :, :ns].view(np.uint16), orc.k_sink[s, :, :ns].view(np.uint16))
            np.testing.assert_array_equal(vsink[s, :, :ns].view(np.uint16), orc.v_sink[s, :, :ns].view(np.uint16))


def _attn_close(got, want):
    got = got.astype(np.float64)
    want = want.astype(np.float64)
    err = np.abs(got - want)
    bad = err > ATOL + RTOL * np.abs(want)
    assert not bad.any(), f"{bad.sum()} elements out of tolerance, max abs err {err.max():.3e}"
    return float(err.max())


def _build(kvq, S, H, cap, bits, ns=0, pre_rope=False, R=128, kpt=False, num_blocks=None, rot=False, sp=False):
    cache = kvq.KVCache(S, H, cap, bits=bits, residual=R, num_sink=ns, pre_rope=pre_rope, key_per_token=kpt,
                        num_blocks=num_blocks, hadamard=rot, outliers=sp)
    orc = oracle.OracleCache(S, H, cap, bits, residual=R, num_sink=ns, key_per_token=kpt, hadamard=rot,
                             outliers=sp)
    return cache, orc


def _append(kvq, cache, orc, k, v, lens):
    dk = torch.from_numpy(np.ascontiguousarray(k)).cuda()
    dv = torch.from_numpy(np.ascontiguousarray(v)).cuda()
    nl = torch.as_tensor(np.asarray(lens, np.int32)).cuda()
    kvq.kv_quant_append(cache, dk, dv, nl, k.shape[2])
    orc.append(k, v, lens)


def _attend(kvq, cache, q, max_len):
    dq = torch.from_numpy(q).cuda()
    out = torch.empty_like(dq)
    ws = kvq.alloc_workspace(cache, q.shape[1], max_len)
    kvq.kv_decode_attn(cache, dq, out, ws, max_len)
    torch.cuda.synchronize()
    return out.cpu().numpy()


# ------------------------------------------------------------------- Tiny

def test_tiny_full(kvq):
    w = synth.WORKLOADS["tiny"]
    k, v = synth.kv_tokens(w, 0, w.ctx)
    k, v = k.numpy(), v.numpy()
    cache, orc = _build(kvq, 1, 1, 512, 2)
    _append(kvq, cache, orc, k, v, [256])
    _compare_state(cache, orc)
    q = synth.queries(w, 0).numpy()
    got = _attend(kvq, cache, q, 256)
    _attn_close(got, orc.attention(q))
    # dequant within one fp32 ulp
    K = torch.full((1, 1, 512, 128), float("nan"), device="cuda")
    V = torch.full_like(K, float("nan"))
    kvq.kv_dequant(cache, K, V)
    Ko, Vo = orc.dequant_all()
    np.testing.assert_array_max_ulp(K.cpu().numpy()[:, :, :256], Ko[:, :, :256].astype(np.float32), maxulp=1)
    np.testing.assert_array_max_ulp(V.cpu().numpy()[:, :, :256], Vo[:, :, :256].astype(np.float32), maxulp=1)
    assert torch.isnan(K[:, :, 256:]).all()


# ------------------------------------------------------------ boundary sweep

LENS = [1, 2, 31, 32, 33, 127, 128, 129, 255, 256, 257]


@pytest.mark.parametrize("spiky", [False, True])
@pytest.mark.parametrize("pre_rope", [False, True])
@pytest.mark.parametrize("ns", [0, 1])
@pytest.mark.parametrize("bits", [2, 4])
def test_boundary_sweep(kvq, bits, ns, pre_rope, spiky):
    """Lengths around every group and window boundary, plain caches (keys
    per channel, post- or pre-RoPE): blocks byte for byte, attention,
    dequantized rows within one fp32 ulp.  The spiky inputs add random x30
    entries, ties and constant rows to keys and values: a value token whose
    range a spike stretches has |min| >> |x|, where code * scale and the min
    nearly cancel, so its attention weight must keep its precision."""
    S, H, gq = len(LENS), 2, 2
    T = max(LENS)
    seed = 100 + bits + 10 * ns
    k, v = _spiky_kv(S, H, T, seed) if spiky else _rand_kv(S, H, T, seed)
    cache, orc = _build(kvq, S, H, 300, bits, ns=ns, pre_rope=pre_rope)
    _append(kvq, cache, orc, k, v, LENS)
    _compare_state(cache, orc)
    q = _rand_q(S, H * gq, seed=7)
    got = _attend(kvq, cache, q, T)
    _attn_close(got, orc.attention(q, pre_rope=pre_rope))
    K = torch.full((S, H, 300, 128), float("nan"), device="cuda")
    V = torch.full_like(K, float("nan"))
    kvq.kv_dequant(cache, K, V)
    Ko, Vo = orc.dequant_all()
    Kg, Vg = K.cpu().numpy(), V.cpu().numpy()
    for s, L in enumerate(LENS):
        np.testing.assert_array_max_ulp(Kg[s, :, :L], Ko[s, :, :L].astype(np.float32), maxulp=1)
        np.testing.assert_array_max_ulp(Vg[s, :, :L], Vo[s, :, :L].astype(np.float32), maxulp=1)
        assert np.isnan(Kg[s, :, L:]).all()


@pytest.mark.parametrize("option", ["key_per_token", "rotation", "outliers", "rotation_kpt", "outliers_kpt"])
@pytest.mark.parametrize("ns", [0, 1])
@pytest.mark.parametrize("bits", [2, 4])
def test_boundary_sweep_options(kvq, bits, ns, option):
    """The same lengths around every group and window boundary with each
    option of the descriptor: blocks byte for byte, attention, and the
    dequantized rows (within one fp32 ulp, outliers exact; with the rotation
    within the back-rotation's 2^-20 ||x_hat|| per row).  Keys and values
    carry random x30 spikes, ties and constant rows with every option."""
    S, H, gq = len(LENS), 2, 2
    T = max(LENS)
    kpt = option == "key_per_token" or option.endswith("kpt")
    rot, sp = option.startswith("rotation"), option.startswith("outliers")
    k, v = _spiky_kv(S, H, T, seed=170 + bits + 10 * ns)
    cache, orc = _build(kvq, S, H, 300, bits, ns=ns, kpt=kpt, rot=rot, sp=sp)
    _append(kvq, cache, orc, k, v, LENS)
    _compare_state(cache, orc)
    q = _rand_q(S, H * gq, seed=8)
    _attn_close(_attend(kvq, cache, q, T), orc.attention(q))
    K = torch.full((S, H, 300, 128), float("nan"), device="cuda")
    V = torch.full_like(K, float("nan"))
    kvq.kv_dequant(cache, K, V)
    Ko, Vo = orc.dequant_all()
    Kg, Vg = K.cpu().numpy().astype(np.float64), V.cpu().numpy().astype(np.float64)
    for s, L in enumerate(LENS):
        for got, want in ((Kg[s, :, :L], Ko[s, :, :L]), (Vg[s, :, :L], Vo[s, :, :L])):
            if rot:
                tol = 2.0 ** -20 * np.linalg.norm(want, axis=-1, keepdims=True)
                assert (np.abs(got - want) <= tol).all()
            else:
                np.testing.assert_array_max_ulp(got.astype(np.float32), want.astype(np.float32), maxulp=1)
        assert np.isnan(Kg[s, :, L:]).all()


@pytest.mark.parametrize("gq", [1, 2, 4])
@pytest.mark.parametrize("bits", [2, 4])
def test_gqa_group_sizes(kvq, gq, bits):
    S, H, T = 3, 2, 700
    k, v = _rand_kv(S, H, T, seed=31 + gq)
    cache, orc = _build(kvq, S, H, 800, bits)
    _append(kvq, cache, orc, k, v, [700, 333, 129])
    _compare_state(cache, orc)
    q = _rand_q(S, H * gq, seed=gq)
    _attn_close(_attend(kvq, cache, q, 700), orc.attention(q))


# ------------------------------------------------------------- streaming

@pytest.mark.parametrize("ns", [0, 1])
def test_streaming_appends_match_prefill(kvq, ns):
    """One-token appends, ragged chunks and one prefill all leave the oracle's
    bytes, across several window flushes."""
    S, H, T = 3, 2, 300
    k, v = _rand_kv(S, H, T, seed=5)
    lens = np.array([300, 257, 128 + ns])
    caches = []
    for mode in ("prefill", "tokens", "chunks"):
        cache, orc = _build(kvq, S, H, 320, 2, ns=ns)
        if mode == "prefill":
            _append(kvq, cache, orc, k, v, lens)
        elif mode == "tokens":
            for t in range(T):
                _append(kvq, cache, orc, k[:, :, t:t + 1], v[:, :, t:t + 1], (t < lens).astype(np.int32))
        else:
            pos = 0
            for step in (1, 126, 2, 64, 107):
                sl = np.clip(lens - pos, 0, step).astype(np.int32)
                _append(kvq, cache, orc, k[:, :, pos:pos + step], v[:, :, pos:pos + step], sl)
                pos += step
        _compare_state(cache, orc)
        caches.append(cache)
    b0 = caches[0].blocks.cpu()
    for c in caches[1:]:
        assert torch.equal(c.blocks.cpu(), b0)


@pytest.mark.parametrize("R,bits,ns,pre_rope", [(32, 2, 1, False), (64, 4, 0, False), (96, 2, 1, True),
                                                 (32, 4, 1, True)])
def test_residual_window_sizes(kvq, R, bits, ns, pre_rope):
    """Windows of R = 32, 64, 96 tokens: per-token appends (the one-kernel
    step path), then appends of up to R tokens, then a prefill-sized append
    (the two-kernel path) leave the oracle's bytes, and attention matches
    after each phase."""
    S, H, T = 2, 2, 4 * R + 40  # the last append (1.5 R + 32 tokens) exceeds R
    k, v = _rand_kv(S, H, T, seed=R + bits)
    cache, orc = _build(kvq, S, H, T + 8, bits, ns=ns, pre_rope=pre_rope, R=R)
    lens = np.array([T, T - 17])
    pos = 0
    steps = [1] * (R + 3) + [R, R // 2 + 5]
    steps.append(T - pos - sum(steps))
    for i, step in enumerate(steps):
        sl = np.clip(lens - pos, 0, step).astype(np.int32)
        _append(kvq, cache, orc, k[:, :, pos:pos + step], v[:, :, pos:pos + step], sl)
        pos += step
        if i in (R + 2, len(steps) - 2, len(steps) - 1):
            _compare_state(cache, orc)
            q = _rand_q(S, 2 * H, seed=i)
            _attn_close(_attend(kvq, cache, q, T), orc.attention(q, pre_rope=pre_rope))
    assert pos == T


@pytest.mark.parametrize("bits,gq,ns", [(2, 1, 0), (2, 4, 1), (4, 2, 0), (4, 1, 1)])
def test_key_per_token_ablation(kvq, bits, gq, ns):
    """Keys grouped per token (the ablation): a prefill (two-kernel path), then
    per-token and chunked appends (one-kernel path) leave the oracle's bytes
    (per-token key scales and mins in the blocks), and attention and
    dequantization match."""
    S, H, T = 3, 2, 420
    k, v = _rand_kv(S, H, T, seed=70 + bits + gq)
    cache, orc = _build(kvq, S, H, T + 8, bits, ns=ns, kpt=True)
    assert cache.block_bytes == (2560 if bits == 2 else 4608)
    lens = np.array([T, T - 29, 140])
    _append(kvq, cache, orc, k[:, :, :200], v[:, :, :200], np.minimum(lens, 200))
    pos = 200
    for step in [1] * 70 + [64, 86]:
        sl = np.clip(lens - pos, 0, step).astype(np.int32)
        _append(kvq, cache, orc, k[:, :, pos:pos + step], v[:, :, pos:pos + step], sl)
        pos += step
    assert pos == T
    _compare_state(cache, orc)
    q = _rand_q(S, H * gq, seed=gq)
    _attn_close(_attend(kvq, cache, q, T), orc.attention(q))
    K = torch.full((S, H, T + 8, 128), float("nan"), device="cuda")
    V = torch.full_like(K, float("nan"))
    kvq.kv_dequant(cache, K, V)
    Ko, Vo = orc.dequant_all()
    for s, L in enumerate(lens):
        np.testing.assert_array_max_ulp(K.cpu().numpy()[s, :, :L], Ko[s, :, :L].astype(np.float32), maxulp=1)
        np.testing.assert_array_max_ulp(V.cpu().numpy()[s, :, :L], Vo[s, :, :L].astype(np.float32), maxulp=1)


@pytest.mark.parametrize("bits,gq,ns,kpt,paged", [(2, 1, 0, False, False), (4, 4, 1, False, False),
                                                  (2, 2, 1, True, False), (4, 1, 0, True, True),
                                                  (2, 4, 1, True, False)])
def test_hadamard_rotation(kvq, bits, gq, ns, kpt, paged):
    """Walsh-Hadamard rotation before quantization: the fp32 fast transform
    and fp16 rounding of the quantize kernels leave the oracle's codes,
    scales and mins byte for byte (prefill, per-token and chunked appends);
    attention matches; dequantization rotates back within 2^-20 ||x_hat||
    per row (one fma and seven fp32 butterfly stages, each within 2^-24 sum
    |y_hat| <= 2^-24 ||x_hat||), and sink and window rows are exact."""
    S, H, T = 3, 2, 450
    k, v = _rand_kv(S, H, T, seed=110 + bits + gq + 2 * ns)
    nb = S * H * 16 + 5 if paged else None
    cache, orc = _build(kvq, S, H, T + 8, bits, ns=ns, kpt=kpt, num_blocks=nb, rot=True)
    if paged:
        rng = np.random.default_rng(bits)
        perm = rng.permutation(cache.num_blocks)[:S * H * cache.max_groups].astype(np.int32)
        cache.block_table.copy_(torch.from_numpy(perm.reshape(S, H, cache.max_groups)).cuda())
    lens = np.array([T, T - 41, 161])
    _append(kvq, cache, orc, k[:, :, :230], v[:, :, :230], np.minimum(lens, 230))
    pos = 230
    for step in [1] * 60 + [128, 32]:
        sl = np.clip(lens - pos, 0, step).astype(np.int32)
        _append(kvq, cache, orc, k[:, :, pos:pos + step], v[:, :, pos:pos + step], sl)
        pos += step
    assert pos == T
    _compare_state(cache, orc)
    q = _rand_q(S, H * gq, seed=gq + 7)
    _attn_close(_attend(kvq, cache, q, T), orc.attention(q))
    K = torch.full((S, H, T + 8, 128), float("nan"), device="cuda")
    V = torch.full_like(K, float("nan"))
    kvq.kv_dequant(cache, K, V)
    Ko, Vo = orc.dequant_all()
    for got, want in ((K.cpu().numpy().astype(np.float64), Ko), (V.cpu().numpy().astype(np.float64), Vo)):
        for s, L in enumerate(lens):
            g, w = got[s, :, :L], want[s, :, :L]
            tol = 2.0 ** -20 * np.linalg.norm(w, axis=-1, keepdims=True)
            assert (np.abs(g - w) <= tol).all(), f"dequant of sequence {s}: {np.abs(g - w).max():.3e}"
            ns_s, Lq, r = orc.split(s)
            np.testing.assert_array_equal(g[:, :ns_s], w[:, :ns_s])
            np.testing.assert_array_equal(g[:, ns_s + Lq:], w[:, ns_s + Lq:])


def _spiky_kv(S, H, T, seed):
    """Keys with fixed outlier channels plus, in keys and values, random x30
    spikes, planted equal-magnitude ties (a token row with +8 and -8, a key
    channel with +9 and -9 in one group) and constant rows."""
    k, v = _rand_kv(S, H, T, seed)
    rng = np.random.default_rng(seed + 1000)
    k, v = k.astype(np.float32), v.astype(np.float32)
    for a in (k, v):
        a[rng.random(a.shape) < 0.004] *= 30
        a[:, :, 5, :] = 0.5
        a[:, :, 5, 3] = 8.0       # ties inside token rows: the earlier channel wins
        a[:, :, 5, 70] = -8.0
        a[:, :, 40, :] = -1.25    # a constant row
    k[:, :, 64 + 3, 20] = -9.0    # a tie inside a key channel of one group: the earlier token wins
    k[:, :, 64 + 17, 20] = 9.0
    return k.astype(np.float16), v.astype(np.float16)


@pytest.mark.parametrize("bits,gq,ns,kpt,paged", [(2, 1, 0, False, False), (4, 4, 1, False, False),
                                                  (2, 2, 1, True, False), (4, 1, 0, True, True),
                                                  (2, 4, 0, False, True), (4, 2, 1, False, False)])
def test_dense_and_sparse(kvq, bits, gq, ns, kpt, paged):
    """Dense-and-sparse blocks: the quantize kernels leave the oracle's bytes
    (outlier entries, codes with the outlier at 0, statistics of the rest)
    after a prefill and per-token and chunked appends; attention matches;
    dequantization returns the outliers exactly and the rest within one fp32
    ulp."""
    S, H, T = 3, 2, 450
    k, v = _spiky_kv(S, H, T, seed=130 + bits + gq + 2 * ns)
    nb = S * H * 16 + 3 if paged else None
    cache, orc = _build(kvq, S, H, T + 8, bits, ns=ns, kpt=kpt, num_blocks=nb, sp=True)
    assert cache.block_bytes == oracle.block_bytes(bits, key_per_token=kpt, outliers=True)
    if paged:
        rng = np.random.default_rng(bits + 5)
        perm = rng.permutation(cache.num_blocks)[:S * H * cache.max_groups].astype(np.int32)
        cache.block_table.copy_(torch.from_numpy(perm.reshape(S, H, cache.max_groups)).cuda())
    lens = np.array([T, T - 53, 170])
    _append(kvq, cache, orc, k[:, :, :230], v[:, :, :230], np.minimum(lens, 230))
    pos = 230
    for step in [1] * 60 + [128, 32]:
        sl = np.clip(lens - pos, 0, step).astype(np.int32)
        _append(kvq, cache, orc, k[:, :, pos:pos + step], v[:, :, pos:pos + step], sl)
        pos += step
    assert pos == T
    _compare_state(cache, orc)
    q = _rand_q(S, H * gq, seed=gq + 11)
    _attn_close(_attend(kvq, cache, q, T), orc.attention(q))
    K = torch.full((S, H, T + 8, 128), float("nan"), device="cuda")
    V = torch.full_like(K, float("nan"))
    kvq.kv_dequant(cache, K, V)
    Ko, Vo = orc.dequant_all()
    for s, L in enumerate(lens):
        np.testing.assert_array_max_ulp(K.cpu().numpy()[s, :, :L], Ko[s, :, :L].astype(np.float32), maxulp=1)
        np.testing.assert_array_max_ulp(V.cpu().numpy()[s, :, :L], Vo[s, :, :L].astype(np.float32), maxulp=1)


@pytest.mark.parametrize("bits,gq,ns,kpt", [(2, 1, 0, False), (4, 4, 1, False), (2, 2, 1, True)])
def test_paged_layout(kvq, bits, gq, ns, kpt):
    """Block-paged layout: logical groups scattered over a larger pool by a
    random block table.  Prefill, per-token and chunked appends leave the
    oracle's bytes in logical order, attention and dequantization match, and
    pool blocks no group maps to stay untouched."""
    S, H, T = 3, 2, 600
    k, v = _rand_kv(S, H, T, seed=90 + bits + gq)
    cache, orc = _build(kvq, S, H, T + 8, bits, ns=ns, kpt=kpt, num_blocks=S * H * 20 + 37)
    rng = np.random.default_rng(bits + gq)
    perm = rng.permutation(cache.num_blocks)[:S * H * cache.max_groups].astype(np.int32)
    cache.block_table.copy_(torch.from_numpy(perm.reshape(S, H, cache.max_groups)).cuda())
    pool0 = cache.blocks.clone()
    lens = np.array([T, T - 77, 260])
    _append(kvq, cache, orc, k[:, :, :300], v[:, :, :300], np.minimum(lens, 300))
    pos = 300
    for step in [1] * 40 + [128, 95, 37]:
        sl = np.clip(lens - pos, 0, step).astype(np.int32)
        _append(kvq, cache, orc, k[:, :, pos:pos + step], v[:, :, pos:pos + step], sl)
        pos += step
    assert pos == T
    _compare_state(cache, orc)
    q = _rand_q(S, H * gq, seed=gq)
    _attn_close(_attend(kvq, cache, q, T), orc.attention(q))
    K = torch.full((S, H, T + 8, 128), float("nan"), device="cuda")
    V = torch.full_like(K, float("nan"))
    kvq.kv_dequant(cache, K, V)
    Ko, Vo = orc.dequant_all()
    for s, L in enumerate(lens):
        np.testing.assert_array_max_ulp(K.cpu().numpy()[s, :, :L], Ko[s, :, :L].astype(np.float32), maxulp=1)
    unused = np.setdiff1d(np.arange(cache.num_blocks), perm)
    bb = cache.block_bytes
    pool = cache.blocks[:cache.num_blocks * bb].view(cache.num_blocks, bb).cpu()
    assert torch.equal(pool[unused], pool0[:cache.num_blocks * bb].view(cache.num_blocks, bb).cpu()[unused])


def test_paged_bad_table_entry_sets_status(kvq):
    """A block-table entry outside the pool is never dereferenced: the group
    is not written, decode reads pool block 0 in its place, and
    KVQ_STATUS_BAD_BLOCK is set; groups with valid entries are intact."""
    S, H, T = 2, 1, 300
    k, v = _rand_kv(S, H, T, seed=5)
    cache, orc = _build(kvq, S, H, T + 8, 2, num_blocks=S * H * 8)
    tbl = np.arange(S * H * cache.max_groups, dtype=np.int32).reshape(S, H, cache.max_groups)
    tbl[1, 0, 3] = cache.num_blocks + 5     # group 3 of sequence 1: outside the pool
    tbl[1, 0, 5] = -2                       # and a negative entry
    cache.block_table.copy_(torch.from_numpy(tbl).cuda())
    _append(kvq, cache, orc, k, v, [T, T])
    torch.cuda.synchronize()
    assert int(cache.status.item()) & kvq.KVQ_STATUS_BAD_BLOCK
    got = cache.logical_blocks().cpu().numpy()
    np.testing.assert_array_equal(got[0, 0, :8], orc.blocks[0, 0, :8])
    np.testing.assert_array_equal(got[1, 0, :3], orc.blocks[1, 0, :3])
    np.testing.assert_array_equal(got[1, 0, 4], orc.blocks[1, 0, 4])
    cache.status.zero_()
    q = _rand_q(S, H, seed=1)
    out = _attend(kvq, cache, q, T)
    assert int(cache.status.item()) & kvq.KVQ_STATUS_BAD_BLOCK
    _attn_close(out[:1], orc.attention(q)[:1])          # sequence 0 is unaffected


@pytest.mark.parametrize("S,H,cap", [(1, 2, (1 << 22) + 64), (1, 512, 400)])
def test_appends_past_the_length_bits(kvq, S, H, cap):
    """The one-kernel step append and the split tail count arrivals in the
    bits of seq_len above 22 length bits, so caches of capacity >= 2^22 or
    with 512 KV heads append through the flush and the one-CTA-per-sequence
    tail instead: a prefill, one-token appends across a window flush and a
    chunk leave the oracle's bytes, and attention matches."""
    T = 300
    k, v = _rand_kv(S, H, T, seed=H + 7)
    cache = kvq.KVCache(S, H, cap, bits=2, num_sink=1)
    orc = oracle.OracleCache(S, H, 400, 2, num_sink=1)  # the oracle only needs room for T tokens
    pos = 0
    for step in [150] + [1] * 40 + [110]:
        sl = np.full(S, step, np.int32)
        _append(kvq, cache, orc, k[:, :, pos:pos + step], v[:, :, pos:pos + step], sl)
        pos += step
    _compare_state(cache, orc)
    q = _rand_q(S, H, seed=3)
    _attn_close(_attend(kvq, cache, q, 400), orc.attention(q))


@pytest.mark.parametrize("S", [2048, 2100])
def test_prefill_at_and_past_the_tile_kernel_batch_limit(kvq, S):
    """The tile kernel flushes batches of up to 2048 sequences (its largest
    line); a prefill of 2100 ragged sequences goes through the
    one-group-per-CTA flush kernel.  Both leave the oracle's bytes, and
    decode (planned by the plan kernel) matches."""
    H, T = 1, 70
    rng = np.random.default_rng(S)
    lens = rng.integers(0, T + 1, S).astype(np.int32)
    k, v = _rand_kv(S, H, T, seed=S + 1)
    cache, orc = _build(kvq, S, H, T + 8, 2, R=32)  # up to two groups flushed per sequence
    _append(kvq, cache, orc, k, v, lens)
    _compare_state(cache, orc)
    q = _rand_q(S, H, seed=4)
    got = _attend(kvq, cache, q, T)
    keep = lens > 0
    assert (got[~keep] == 0).all()
    _attn_close(got[keep], orc.attention(q)[keep])


def test_decode_step_flush_then_attend(kvq):
    """A window holding R-1 tokens plus one appended token flushes; attention
    then reads only quantized groups."""
    S, H, T = 2, 2, 256
    k, v = _rand_kv(S, H, T, seed=9)
    cache, orc = _build(kvq, S, H, 300, 2)
    _append(kvq, cache, orc, k[:, :, :255], v[:, :, :255], [255, 255])
    assert orc.split(0) == (0, 128, 127)
    _append(kvq, cache, orc, k[:, :, 255:], v[:, :, 255:], [1, 1])
    assert orc.split(0) == (0, 256, 0)
    _compare_state(cache, orc)
    q = _rand_q(S, 2 * H, seed=3)
    _attn_close(_attend(kvq, cache, q, 256), orc.attention(q))


# ------------------------------------------------------ edge and error cases

def test_empty_cache_outputs_zero(kvq):
    cache, orc = _build(kvq, 2, 1, 64, 2)
    q = _rand_q(2, 1, seed=1)
    got = _attend(kvq, cache, q, 64)
    assert (got == 0).all()


def test_capacity_overflow_sets_status_and_skips(kvq):
    cache, orc = _build(kvq, 2, 1, 160, 2)
    k, v = _rand_kv(2, 1, 150, seed=2)
    _append(kvq, cache, orc, k, v, [150, 20])
    k2, v2 = _rand_kv(2, 1, 20, seed=3)
    before = cache.blocks.clone()
    dk, dv = torch.from_numpy(k2).cuda(), torch.from_numpy(v2).cuda()
    kvq.kv_quant_append(cache, dk, dv, torch.tensor([20, 5], dtype=torch.int32, device="cuda"), 20)
    torch.cuda.synchronize()
    assert int(cache.status.item()) & kvq.KVQ_STATUS_CAPACITY
    assert cache.seq_len.cpu().tolist() == [150, 25]          # seq 0 skipped, seq 1 appended
    assert torch.equal(cache.blocks[: before.numel() // 2], before[: before.numel() // 2])


def test_bad_new_len_sets_status(kvq):
    cache, _ = _build(kvq, 1, 1, 64, 2)
    k, v = _rand_kv(1, 1, 4, seed=2)
    kvq.kv_quant_append(cache, torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(),
                        torch.tensor([9], dtype=torch.int32, device="cuda"), 4)
    torch.cuda.synchronize()
    assert int(cache.status.item()) & kvq.KVQ_STATUS_BAD_LEN
    assert cache.seq_len.item() == 0


def test_workspace_too_small_raises(kvq):
    cache, _ = _build(kvq, 1, 1, 64, 2)
    q = torch.zeros((1, 1, 128), dtype=torch.float16, device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(kvq.KvqError) as e:
        kvq.kv_decode_attn(cache, q, torch.empty_like(q), ws, 64)
    assert e.value.code == -4


@pytest.mark.parametrize("pre_rope", [False, True])
def test_wait_timeout_sets_status_and_recovers(kvq, pre_rope):
    """The decode kernel's ring waits are bounded.  In normal operation every
    copy lands before its first poll, so the test makes each warp's first
    wait come before its first copy is issued, on a barrier that nothing
    completes, with a limit of 20000 SM cycles: the wait runs out, the
    kernel records KVQ_STATUS_TIMEOUT and returns, and the device stays
    usable.  With the defaults restored and the workspace zeroed again, the
    same call matches the oracle.  Nothing faults and nothing hangs."""
    S, H, T = 8, 4, 3000
    k, v = _rand_kv(S, H, T, seed=41)
    cache, orc = _build(kvq, S, H, T + 8, 2, ns=int(pre_rope), pre_rope=pre_rope)
    _append(kvq, cache, orc, k, v, [T - 97 * s for s in range(S)])
    q = _rand_q(S, 2 * H, seed=42)
    dq = torch.from_numpy(q).cuda()
    out = torch.empty_like(dq)
    ws = kvq.alloc_workspace(cache, 2 * H, T)
    try:
        kvq.set_wait_test(20000, True)
        kvq.kv_decode_attn(cache, dq, out, ws, T)
        torch.cuda.synchronize()
    finally:
        kvq.set_wait_test(0, False)
    assert int(cache.status.item()) == kvq.KVQ_STATUS_TIMEOUT
    cache.status.zero_()
    ws.zero_()
    kvq.kv_decode_attn(cache, dq, out, ws, T)
    torch.cuda.synchronize()
    assert int(cache.status.item()) == 0
    _attn_close(out.cpu().numpy(), orc.attention(q, pre_rope=pre_rope))


@pytest.mark.parametrize("warps", [1, 3, 7, 50, 333, 2560])
def test_split_sizes_agree(kvq, warps):
    """The answer does not depend on how the work is cut into warp ranges:
    one warp for everything, ranges that end inside window passes and
    groups, and more warps than units (empty ranges)."""
    S, H, T = 2, 2, 1500
    k, v = _rand_kv(S, H, T, seed=12)
    cache, orc = _build(kvq, S, H, 1600, 2, ns=1)
    _append(kvq, cache, orc, k, v, [1500, 1100])
    q = _rand_q(S, 4 * H, seed=4)
    want = orc.attention(q)
    try:
        kvq.set_decode_warps(warps)
        _attn_close(_attend(kvq, cache, q, 1500), want)
    finally:
        kvq.set_decode_warps(0)


@pytest.mark.parametrize("variant", ["rotation", "outliers", "outliers_kpt", "paged_rotation", "paged_outliers"])
@pytest.mark.parametrize("warps", [1, 7, 64, 2560])
def test_split_sizes_agree_variants(kvq, variant, warps):
    """The kernels for rotated tokens, dense-and-sparse blocks and paged
    caches carry per-warp state across pairs (the query rotated in place,
    outlier corrections zeroed by their readers, the table check): their
    answers must not depend on the warp ranges either, with one warp
    crossing every pair, ranges ending inside passes and groups, and empty
    ranges."""
    S, H, T = 3, 2, 700
    k, v = _spiky_kv(S, H, T, seed=150)
    rot = "rotation" in variant
    sp = "outliers" in variant
    kpt = variant.endswith("kpt")
    nb = S * H * 24 + 7 if variant.startswith("paged") else None
    cache, orc = _build(kvq, S, H, T + 8, 2, ns=1, kpt=kpt, num_blocks=nb, rot=rot, sp=sp)
    if nb:
        perm = np.random.default_rng(3).permutation(nb)[:S * H * cache.max_groups].astype(np.int32)
        cache.block_table.copy_(torch.from_numpy(perm.reshape(S, H, cache.max_groups)).cuda())
    _append(kvq, cache, orc, k, v, [T, T - 211, 333])
    q = _rand_q(S, 4 * H, seed=9)
    want = orc.attention(q)
    dq = torch.from_numpy(q).cuda()
    ws = kvq.alloc_workspace(cache, q.shape[1], T)
    try:
        kvq.set_decode_warps(warps)
        for _ in range(2):  # the second call reuses the workspace's self-cleaning counters
            out = torch.empty_like(dq)
            kvq.kv_decode_attn(cache, dq, out, ws, T)
            torch.cuda.synchronize()
            _attn_close(out.cpu().numpy(), want)
    finally:
        kvq.set_decode_warps(0)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("S", [20, 32, 33, 200, 300])
def test_many_sequences_with_empty_and_overlong(kvq, S):
    """Batches planned inside the decode kernel from one read of seq_len
    (S <= 32) or by chunks of 32 sequences (S <= 256), and by the plan
    kernel (S > 256): ragged lengths with empty sequences and sequences
    longer than max_len, whose rows come back zero with
    KVQ_STATUS_MAX_LEN set."""
    H, T, max_len = 1, 200, 150
    rng = np.random.default_rng(S)
    lens = rng.integers(0, T + 1, S).astype(np.int32)
    lens[::17] = 0
    k, v = _rand_kv(S, H, T, seed=S + 1)
    cache, orc = _build(kvq, S, H, T + 8, 2, ns=1)
    _append(kvq, cache, orc, k, v, lens)
    q = _rand_q(S, 2 * H, seed=5)
    dq = torch.from_numpy(q).cuda()
    out = torch.full_like(dq, float("nan"))
    ws = kvq.alloc_workspace(cache, 2 * H, max_len)
    kvq.kv_decode_attn(cache, dq, out, ws, max_len)
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    over = lens > max_len
    assert over.any() and (lens == 0).any()
    assert bool(int(cache.status.item()) & kvq.KVQ_STATUS_MAX_LEN) == bool(over.any())
    assert (got[over | (lens == 0)] == 0).all()
    want = orc.attention(q)
    keep = ~over
    _attn_close(got[keep], want[keep])


def test_workspace_reused_across_calls(kvq):
    """The merge counters a call leaves behind are the zeros the next call
    starts from: several calls on one workspace, with the work cut into
    different numbers of warp ranges, all match the oracle."""
    S, H, T = 3, 2, 700
    k, v = _rand_kv(S, H, T, seed=21)
    cache, orc = _build(kvq, S, H, 720, 2)
    _append(kvq, cache, orc, k, v, [700, 333, 64])
    ws = kvq.alloc_workspace(cache, 2 * H, 720)
    try:
        for i, warps in enumerate([0, 5, 0, 77, 1, 0]):
            kvq.set_decode_warps(warps)
            q = _rand_q(S, 2 * H, seed=30 + i)
            dq = torch.from_numpy(q).cuda()
            out = torch.empty_like(dq)
            kvq.kv_decode_attn(cache, dq, out, ws, 720)
            torch.cuda.synchronize()
            _attn_close(out.cpu().numpy(), orc.attention(q))
    finally:
        kvq.set_decode_warps(0)
    assert int(cache.status.item()) == 0


@pytest.mark.parametrize("bits", [2, 4])
def test_ties_and_near_ties_bit_exact(kvq, bits):
    """Inputs on a half-step grid put many quotients exactly on rounding
    boundaries (and fp16 neighbours just beside them); codes must match the
    oracle's round-half-even of the IEEE quotient bit for bit."""
    S, H, T = 2, 3, 256
    rng = np.random.default_rng(40 + bits)
    top = 2 ** bits - 1
    k = (rng.integers(0, 2 * top + 1, (S, H, T, 128)) / 2.0).astype(np.float16)
    v = (rng.integers(0, 2 * top + 1, (S, H, T, 128)) / 2.0).astype(np.float16)
    # shift some slices by one fp16 ulp so quotients land just beside k + 1/2
    k[:, :, ::3, ::5] = np.nextafter(k[:, :, ::3, ::5], np.float16(100))
    v[:, 1] = (v[:, 1].astype(np.float32) * 0.3 - 7).astype(np.float16)
    cache, orc = _build(kvq, S, H, 300, bits)
    _append(kvq, cache, orc, k, v, [256, 256])
    _compare_state(cache, orc)
