"""Pins of the CPU oracle against what the pages and the mathematics fix
(closed forms, invariants, hand-derived fixtures, brute force).  No GPU."""

import cmath
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import kivi

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
rng0 = np.random.default_rng(12345)


def _normal(shape, rng=rng0, scale=1.0):
    return (rng.standard_normal(shape) * scale).astype(np.float16)


# ----------------------------------------------------------------- quantization

@pytest.mark.parametrize("bits", [2, 4])
def test_codes_in_range(bits):
    x = _normal((8, 32, 128), scale=3.0)
    for axis in (-1, -2):
        c, s, m = oracle.quantize_asymmetric(x, axis, bits)
        assert c.dtype == np.uint8 and c.min() >= 0 and c.max() <= 2 ** bits - 1
        assert (c.max(axis=axis) == 2 ** bits - 1).all()   # max element hits the top code
        assert (c.min(axis=axis) == 0).all()               # min element hits code 0


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("kind", ["keys", "values"])
def test_roundtrip_error_at_most_half_scale(bits, kind):
    x = _normal((4, 32, 128), scale=2.0)
    x[..., 5] *= 20  # an outlier channel
    if kind == "keys":
        c, s, m = oracle.quantize_key_group(x, bits)
        xh = oracle.dequantize(c, s[:, None, :], m[:, None, :])
        s_b = np.broadcast_to(s[:, None, :], x.shape)
        m_b = np.broadcast_to(m[:, None, :], x.shape)
    else:
        c, s, m = oracle.quantize_value_tokens(x, bits)
        xh = oracle.dequantize(c, s[..., None], m[..., None])
        s_b = np.broadcast_to(s[..., None], x.shape)
        m_b = np.broadcast_to(m[..., None], x.shape)
    x64 = x.astype(np.float64)
    # fp32 subtraction + division contribute a few ulps on top of scale/2
    bound = s_b * (0.5 + 2.0 ** -16) + 2.0 ** -22 * (np.abs(x64) + np.abs(m_b))
    assert (np.abs(x64 - xh) <= bound).all()


@pytest.mark.parametrize("bits", [2, 4])
def test_grid_values_roundtrip_exactly(bits):
    levels = 2 ** bits - 1
    mn, scale = -2.0, 0.25
    grid = mn + scale * np.arange(levels + 1)            # all exact in fp16
    rng = np.random.default_rng(1)
    x = rng.choice(grid, size=(32, 128)).astype(np.float16)
    x[0, :] = mn
    x[1, :] = grid[-1]                                   # every channel spans the grid
    c, s, m = oracle.quantize_key_group(x, bits)
    assert (s == np.float32(scale)).all() and (m == np.float32(mn)).all()
    assert (c == np.rint((x.astype(np.float64) - mn) / scale)).all()
    assert (oracle.dequantize(c, s, m) == x.astype(np.float64)).all()


def test_constant_slice_gives_scale_zero():
    x = np.full((32, 128), 1.5, np.float16)
    for fn in (oracle.quantize_key_group, oracle.quantize_value_tokens):
        c, s, m = fn(x, 2)
        assert (c == 0).all() and (s == 0).all() and (m == np.float32(1.5)).all()
        assert (oracle.dequantize(c, s[..., None] if fn is oracle.quantize_value_tokens else s,
                                  m[..., None] if fn is oracle.quantize_value_tokens else m) == 1.5).all()


def test_round_half_even_golden():
    with open(os.path.join(GOLDEN, "quant_ties.json")) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        vals = case["channel0"]
        x = np.zeros((32, 128), np.float16)
        x[:len(vals), 0] = vals
        c, s, m = oracle.quantize_key_group(x, case["bits"])
        assert s[0] == case["scale"] and m[0] == case["min"]
        assert list(c[:len(vals), 0]) == case["codes"]


@pytest.mark.parametrize("bits", [2, 4])
def test_nearest_code_brute_force(bits):
    """Each code is the nearest grid point (scale * c + min) to x."""
    x = _normal((32, 128), rng=np.random.default_rng(7))
    c, s, m = oracle.quantize_key_group(x, bits)
    x64 = x.astype(np.float64)
    for d in range(0, 128, 9):
        for t in range(32):
            if s[d] == 0:
                continue
            errs = [abs(x64[t, d] - (k * float(s[d]) + float(m[d]))) for k in range(2 ** bits)]
            assert c[t, d] == int(np.argmin(errs))


# ------------------------------------------------------- grouping confines errors

OUTLIERS = [3, 17, 64, 101]


@pytest.mark.parametrize("bits", [2, 4])
def test_outlier_channel_error_confined_per_channel(bits):
    """Per-channel key grouping keeps an outlier channel's effect inside that
    channel (KIVI page, second paragraph); per-token grouping does not."""
    x = _normal((32, 128), rng=np.random.default_rng(3))
    xo = x.copy()
    xo[:, OUTLIERS] = (xo[:, OUTLIERS].astype(np.float32) * 20).astype(np.float16)
    normal = [d for d in range(128) if d not in OUTLIERS]
    c0, s0, m0 = oracle.quantize_key_group(x, bits)
    c1, s1, m1 = oracle.quantize_key_group(xo, bits)
    assert (c0[:, normal] == c1[:, normal]).all()
    assert (s0[normal] == s1[normal]).all() and (m0[normal] == m1[normal]).all()
    # the per-token baseline: the outliers set every token's scale
    p0, ps0, _ = oracle.quantize_keys_per_token(x, bits)
    p1, ps1, _ = oracle.quantize_keys_per_token(xo, bits)
    assert (ps1 > 2 * ps0).all() and ps1.mean() > 5 * ps0.mean()
    assert (p0[:, normal] != p1[:, normal]).mean() > 0.3
    # and its error on normal channels is far larger
    e_chan = np.abs(oracle.dequantize(c1, s1, m1) - xo.astype(np.float64))[:, normal].max()
    e_tok = np.abs(oracle.dequantize(p1, ps1[:, None], _[:, None]) - xo.astype(np.float64))[:, normal].max()
    assert e_tok > 5 * e_chan


def test_value_token_error_confined_per_token():
    """Per-token value grouping keeps one token's range from touching others."""
    v = _normal((32, 128), rng=np.random.default_rng(4))
    vo = v.copy()
    vo[9] = (vo[9].astype(np.float32) * 20).astype(np.float16)
    c0, s0, m0 = oracle.quantize_value_tokens(v, 2)
    c1, s1, m1 = oracle.quantize_value_tokens(vo, 2)
    others = [t for t in range(32) if t != 9]
    assert (c0[others] == c1[others]).all() and (s0[others] == s1[others]).all()
    assert s1[9] > 10 * s0[9]


# ------------------------------------------------------------------- packing

def test_pack_locations_golden():
    with open(os.path.join(GOLDEN, "pack_locations.json")) as f:
        entries = json.load(f)["entries"]
    for tile, bits, row, col, byte, bit, _why in entries:
        rows, cols = (32, 128) if tile == "K" else (128, 32)
        assert oracle.code_location(row, col, bits, rows, cols) == (byte, bit), (tile, bits, row, col)
        # and the packer puts a lone code there
        c = np.zeros((rows, cols), np.uint8)
        c[row, col] = 1
        buf = oracle.pack_tile(c, bits)
        nz = np.nonzero(buf)[0]
        assert list(nz) == [byte] and buf[byte] == (1 << bit)


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("shape", [(32, 128), (128, 32)])
def test_pack_is_bijection_and_roundtrips(bits, shape):
    rows, cols = shape
    byte, bit = oracle.code_location_table(rows, cols, bits)
    flat = byte * 8 + bit
    assert len(np.unique(flat)) == rows * cols
    assert flat.min() == 0 and flat.max() == rows * cols * bits - bits
    assert (flat % bits == 0).all()
    c = np.random.default_rng(5).integers(0, 2 ** bits, (3, rows, cols)).astype(np.uint8)
    assert (oracle.unpack_tile(oracle.pack_tile(c, bits), bits, rows, cols) == c).all()


def test_block_sizes_and_footprint_ratio():
    """2 vs 16 bits per element is an 8x reduction in code bytes ("2-Bit KV
    Cache Quantization...", "The capacity math")."""
    assert oracle.block_bytes(2) == 3328 and oracle.block_bytes(4) == 5376
    code_bytes_2 = 2 * 32 * 128 * 2 // 8          # K + V codes of one group
    fp16_bytes = 2 * 32 * 128 * 2
    assert fp16_bytes / code_bytes_2 == 8
    # with fp32 (scale, min) metadata the per-token-head cost is 104 B
    assert oracle.block_bytes(2) / 32 == 104 and oracle.block_bytes(4) / 32 == 168


# --------------------------------------------------------------- cache stream

def _cache_inputs(S, H, T, seed=0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((S, H, T, 128)).astype(np.float16)
    v = rng.standard_normal((S, H, T, 128)).astype(np.float16)
    k[..., OUTLIERS] = (k[..., OUTLIERS].astype(np.float32) * 15).astype(np.float16)
    return k, v


@pytest.mark.parametrize("ns", [0, 1])
@pytest.mark.parametrize("bits", [2, 4])
def test_streaming_equivalence(ns, bits):
    """prefill(L) leaves the same bytes as L one-token appends, or any chunking."""
    S, H, T = 2, 2, 300
    k, v = _cache_inputs(S, H, T)
    lens = np.array([300, 257])
    a = oracle.OracleCache(S, H, 320, bits, num_sink=ns)
    a.append(k, v, lens)
    b = oracle.OracleCache(S, H, 320, bits, num_sink=ns)
    for t in range(T):
        b.append(k[:, :, t:t + 1], v[:, :, t:t + 1], (t < lens).astype(int))
    c = oracle.OracleCache(S, H, 320, bits, num_sink=ns)
    pos = 0
    for step in (1, 126, 2, 64, 107):
        step_lens = np.clip(lens - pos, 0, step)
        c.append(k[:, :, pos:pos + step], v[:, :, pos:pos + step], step_lens)
        pos += step
    for other in (b, c):
        assert (a.seq_len == other.seq_len).all()
        assert (a.blocks == other.blocks).all()
        for s in range(S):
            ns_, Lq, r = a.split(s)
            assert (a.k_res[s, :, :r] == other.k_res[s, :, :r]).all()
            assert (a.v_res[s, :, :r] == other.v_res[s, :, :r]).all()
            assert (a.k_sink[s, :, :ns_] == other.k_sink[s, :, :ns_]).all()


def test_split_counts_follow_the_window_rule():
    c = oracle.OracleCache(1, 1, 1000, 2, num_sink=1)
    k, v = _cache_inputs(1, 1, 600)
    expect = {1: (1, 0, 0), 2: (1, 0, 1), 128: (1, 0, 127), 129: (1, 128, 0),
              130: (1, 128, 1), 257: (1, 256, 0), 600: (1, 512, 87)}
    done = 0
    for L in sorted(expect):
        c.append(k[:, :, done:L], v[:, :, done:L], [L - done])
        done = L
        assert c.split(0) == expect[L]


@pytest.mark.parametrize("ns", [0, 1])
def test_sink_and_window_are_exact(ns):
    k, v = _cache_inputs(1, 2, 200)
    c = oracle.OracleCache(1, 2, 256, 2, num_sink=ns)
    c.append(k, v, [200])
    ns_, Lq, r = c.split(0)
    for h in range(2):
        K, V = c.keys_values(0, h)
        assert K.shape == (200, 128)
        assert (K[:ns_] == k[0, h, :ns_].astype(np.float64)).all()
        assert (K[ns_ + Lq:] == k[0, h, ns_ + Lq:200].astype(np.float64)).all()
        assert (V[ns_ + Lq:] == v[0, h, ns_ + Lq:200].astype(np.float64)).all()
        # the quantized part is not exact but within its error bound
        assert np.abs(K[ns_:ns_ + Lq] - k[0, h, ns_:ns_ + Lq]).max() > 0


# ------------------------------------------------------------------ attention

def _textbook_attention(q, K, V, scale):
    """Pure-Python softmax attention (fp64 loops)."""
    L = len(K)
    z = [scale * sum(float(q[d]) * float(K[t][d]) for d in range(len(q))) for t in range(L)]
    m = max(z)
    p = [math.exp(zi - m) for zi in z]
    tot = sum(p)
    return [sum(p[t] * float(V[t][d]) for t in range(L)) / tot for d in range(len(q))]


@pytest.mark.parametrize("ns", [0, 1])
def test_attention_all_full_precision_is_textbook(ns):
    """With at most R + sink tokens nothing is quantized."""
    L = 128 + ns - 1
    k, v = _cache_inputs(1, 1, L, seed=2)
    c = oracle.OracleCache(1, 1, 256, 2, num_sink=ns)
    c.append(k, v, [L])
    assert c.split(0)[1] == 0
    q = _normal((1, 1, 128), rng=np.random.default_rng(9))
    got = c.attention(q)[0, 0].astype(np.float64)
    want = _textbook_attention(q[0, 0], k[0, 0], v[0, 0], 1 / math.sqrt(128))
    np.testing.assert_allclose(got, want, rtol=2 ** -10, atol=2 ** -24)


def test_attention_single_token_returns_its_value():
    k, v = _cache_inputs(1, 1, 1)
    c = oracle.OracleCache(1, 1, 64, 4)
    c.append(k, v, [1])
    q = _normal((1, 1, 128))
    assert (c.attention(q)[0, 0] == v[0, 0, 0]).all()


def test_attention_equal_keys_gives_mean_value():
    """Identical keys give uniform weights, so the output is mean(v_hat)."""
    T = 300
    row = _normal((128,), rng=np.random.default_rng(11))
    k = np.broadcast_to(row, (1, 1, T, 128)).copy()
    _, v = _cache_inputs(1, 1, T)
    c = oracle.OracleCache(1, 1, 320, 2)
    c.append(k, v, [T])
    K, V = c.keys_values(0, 0)
    assert (K == row.astype(np.float64)).all()      # constant groups: scale 0, x_hat = min
    q = _normal((1, 1, 128))
    np.testing.assert_allclose(c.attention(q)[0, 0].astype(np.float64), V.mean(0),
                               rtol=2 ** -10, atol=2 ** -14)


def test_attention_query_head_mapping():
    """Query head j reads KV head j // (Hq / H)."""
    k, v = _cache_inputs(1, 2, 40)
    v[0, 1] = np.float16(7.0)
    c = oracle.OracleCache(1, 2, 64, 2)
    c.append(k, v, [40])
    out = c.attention(_normal((1, 4, 128)))
    assert (out[0, 2:] == 7.0).all() and (out[0, :2] != 7.0).any()


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("ns", [0, 1])
def test_attention_brute_force_tiny(bits, ns):
    """Attention read from the packed state equals dense attention over values
    re-derived here by nearest-grid-point search and explicit token order."""
    T = 256 + ns + 5
    k, v = _cache_inputs(1, 1, T, seed=21)
    c = oracle.OracleCache(1, 1, 400, bits, num_sink=ns)
    c.append(k, v, [T])
    ns_, Lq, r = c.split(0)
    assert (ns_, Lq, r) == (ns, 256, 5)
    # rebuild K_hat, V_hat independently
    K = [list(map(float, k[0, 0, t])) for t in range(T)]
    V = [list(map(float, v[0, 0, t])) for t in range(T)]
    levels = 2 ** bits - 1
    Ko, Vo = c.keys_values(0, 0)

    def nearest(x, lo, hi, got):
        """The grid point nearest to x; within 1e-6 of a tie either neighbour
        is accepted (the code is decided by fp32 arithmetic there)."""
        sc = float(np.float32((np.float32(hi) - np.float32(lo)) / np.float32(levels)))
        if sc == 0:
            return lo
        y = (x - lo) / sc
        c0 = math.floor(y)
        if abs(y - (c0 + 0.5)) < 1e-6:
            ok = {min(max(cc, 0), levels) * sc + lo for cc in (c0, c0 + 1)}
            assert got in ok
            return got
        return min(max(round(y), 0), levels) * sc + lo

    for g in range(Lq // 32):
        toks = range(ns_ + 32 * g, ns_ + 32 * g + 32)
        for d in range(128):
            col = [K[t][d] for t in toks]
            lo, hi = min(col), max(col)
            for t in toks:
                K[t][d] = nearest(K[t][d], lo, hi, float(Ko[t, d]))
        for t in toks:
            lo, hi = min(V[t]), max(V[t])
            V[t] = [nearest(x, lo, hi, float(Vo[t, d])) for d, x in enumerate(V[t])]
    assert (np.array(K) == Ko).all() and (np.array(V) == Vo).all()
    q = _normal((1, 1, 128), rng=np.random.default_rng(5))
    want = _textbook_attention(q[0, 0], K, V, 1 / math.sqrt(128))
    got = c.attention(q)[0, 0].astype(np.float64)
    np.testing.assert_allclose(got, want, rtol=2 ** -10, atol=2 ** -20)


# ----------------------------------------------------------------------- RoPE

def test_rope_identity_at_zero_and_norm_preserving():
    x = np.random.default_rng(2).standard_normal((5, 128))
    assert (oracle.rope_rotate(x[:1], [0]) == x[:1]).all()
    y = oracle.rope_rotate(x, [1, 7, 100, 4096, 1 << 20])
    n_x = x[:, :64] ** 2 + x[:, 64:] ** 2
    n_y = y[:, :64] ** 2 + y[:, 64:] ** 2
    np.testing.assert_allclose(n_x, n_y, rtol=1e-12)


def test_rope_matches_complex_rotation():
    """Pair (i, i+64) as the complex number x_i + i*x_{i+64}, multiplied by
    exp(i * p * theta^(-2i/D))."""
    x = np.random.default_rng(3).standard_normal(128)
    for p in (1, 33, 16384):
        y = oracle.rope_rotate(x[None], [p])[0]
        for i in range(64):
            z = complex(x[i], x[i + 64]) * cmath.exp(1j * p * 10000.0 ** (-2 * i / 128))
            assert abs(y[i] - z.real) < 1e-9 and abs(y[i + 64] - z.imag) < 1e-9


def test_rope_hand_values_and_relative_position():
    x = np.zeros(128)
    x[0] = 1.0                                   # omega_0 = 1
    y = oracle.rope_rotate(x[None], [1])[0]
    assert abs(y[0] - math.cos(1)) < 1e-15 and abs(y[64] - math.sin(1)) < 1e-15
    x = np.zeros(128)
    x[32] = 1.0                                  # omega_32 = 10000^(-1/2) = 0.01
    y = oracle.rope_rotate(x[None], [50])[0]
    assert abs(y[32] - math.cos(0.5)) < 1e-12 and abs(y[96] - math.sin(0.5)) < 1e-12
    # <R(p) a, R(p') b> depends only on p - p'
    a, b = np.random.default_rng(4).standard_normal((2, 128))
    d1 = oracle.rope_rotate(a[None], [10])[0] @ oracle.rope_rotate(b[None], [3])[0]
    d2 = oracle.rope_rotate(a[None], [1010])[0] @ oracle.rope_rotate(b[None], [1003])[0]
    assert abs(d1 - d2) < 1e-9


def test_pre_rope_attention_equals_rotated_dense():
    """Keys stored pre-RoPE and rotated after dequantization equal dense
    attention over RoPE(x_hat) at absolute positions."""
    T = 200
    k, v = _cache_inputs(1, 1, T, seed=8)
    c = oracle.OracleCache(1, 1, 256, 2, num_sink=1)
    c.append(k, v, [T])
    K, V = c.keys_values(0, 0)
    Kr = oracle.rope_rotate(K, np.arange(T))
    q = _normal((1, 1, 128), rng=np.random.default_rng(6))
    want = oracle.dense_attention(q[0, 0].astype(np.float64), Kr, V, 1 / math.sqrt(128))
    got = c.attention(q, pre_rope=True)[0, 0]
    np.testing.assert_allclose(got.astype(np.float64), want, rtol=2 ** -10, atol=2 ** -24)
    # and rotation changes the answer (it is not silently skipped)
    assert np.abs(c.attention(q, pre_rope=False)[0, 0].astype(np.float64) - want).max() > 1e-3


def test_zero_extremes_are_stored_as_positive_zero():
    """A slice whose min (or max) is a zero stores +0 whichever zero it saw."""
    x = np.zeros((32, 128), np.float16)
    x[:16, :] = np.float16(-0.0)
    x[5, 7] = 1.0
    c, s, m = oracle.quantize_key_group(x, 2)
    assert not np.signbit(m).any() and not np.signbit(s).any()
    c, s, m = oracle.quantize_value_tokens(-x, 2)
    assert not np.signbit(m[16:]).any()


# ------------------------------------------- per-token key ablation (f1)

def test_per_token_key_block_layout_roundtrip():
    """Per-token keys keep one fp32 (scale, min) per token: 2560 B (2-bit)
    and 4608 B (4-bit) per block; packing round-trips."""
    assert oracle.block_bytes(2, key_per_token=True) == 2 * 1024 + 4 * 4 * 32
    assert oracle.block_bytes(4, key_per_token=True) == 2 * 2048 + 4 * 4 * 32
    rng = np.random.default_rng(3)
    for bits in (2, 4):
        kc = rng.integers(0, 1 << bits, (3, 32, 128)).astype(np.uint8)
        vc = rng.integers(0, 1 << bits, (3, 32, 128)).astype(np.uint8)
        ks, km, vs, vm = (rng.standard_normal((3, 32)).astype(np.float32) for _ in range(4))
        blk = oracle.kivi.pack_block(kc, ks, km, vc, vs, vm, bits, key_per_token=True)
        assert blk.shape == (3, oracle.block_bytes(bits, key_per_token=True))
        out = oracle.kivi.unpack_block(blk, bits, key_per_token=True)
        for a, b in zip(out, (kc, ks, km, vc, vs, vm)):
            np.testing.assert_array_equal(a, b)


def test_per_token_key_cache_dequant_and_streaming():
    """A per-token-key cache dequantizes every quantized key as code * s_t +
    m_t with (s_t, m_t) taken over that token's 128 channels, keeps the
    window exact, and prefill equals token-by-token appends."""
    rng = np.random.default_rng(4)
    S, H, T = 2, 2, 200
    k = rng.standard_normal((S, H, T, 128)).astype(np.float16)
    v = rng.standard_normal((S, H, T, 128)).astype(np.float16)
    a = oracle.OracleCache(S, H, 256, 2, residual=64, key_per_token=True)
    a.append(k, v, [T, T - 9])
    b = oracle.OracleCache(S, H, 256, 2, residual=64, key_per_token=True)
    for t in range(T):
        b.append(k[:, :, t:t + 1], v[:, :, t:t + 1], [1, int(t < T - 9)])
    np.testing.assert_array_equal(a.blocks, b.blocks)
    ns, Lq, r = a.split(0)
    kh, _ = a.keys_values(0, 1)
    x = k[0, 1, :Lq].astype(np.float32)
    mn, mx = x.min(-1), x.max(-1)
    sc = ((mx - mn) / np.float32(3)).astype(np.float32)
    c = np.clip(np.rint((x - mn[:, None]) / sc[:, None]), 0, 3)
    np.testing.assert_allclose(kh[:Lq], c * sc[:, None].astype(np.float64) + mn[:, None], rtol=0, atol=1e-6)
    np.testing.assert_array_equal(kh[Lq:], k[0, 1, Lq:Lq + r].astype(np.float64))


def test_ablation_ordering_on_outlier_keys():
    """The pages' qualitative ordering on keys with fixed outlier channels
    (KIVI page, paragraphs 1-3; "KV cache quantization", "Keys are harder
    than values"): per-channel key groups with the 128-token window beat a
    32-token window (the smallest the group storage allows, the reading of
    'no residual'), and both beat per-token key groups, measured as mean
    attention error against exact fp16 attention."""
    rng = np.random.default_rng(11)
    T, Hq = 250, 64
    k = rng.standard_normal((1, 1, T, 128)).astype(np.float32)
    k[..., [3, 17, 64, 101]] *= 20
    k = k.astype(np.float16)
    v = rng.standard_normal((1, 1, T, 128)).astype(np.float16)
    q = rng.standard_normal((1, Hq, 128)).astype(np.float16)
    scale = 1 / np.sqrt(128)
    exact = np.stack([oracle.dense_attention(q[0, j].astype(np.float64), k[0, 0].astype(np.float64),
                                             v[0, 0].astype(np.float64), scale) for j in range(Hq)])
    errs = {}
    for name, R, kpt in (("channel_R128", 128, False), ("channel_R32", 32, False), ("token_R128", 128, True)):
        c = oracle.OracleCache(1, 1, 256, 2, residual=R, key_per_token=kpt)
        c.append(k, v, [T])
        errs[name] = float(np.abs(c.attention(q)[0].astype(np.float64) - exact).mean())
    assert errs["channel_R128"] < errs["channel_R32"] < errs["token_R128"], errs


# ---------------------------------------------------------------- Hadamard


def test_hadamard_matrix_is_symmetric_orthogonal_and_recursive():
    """Without any library: H is symmetric, H H = D I, its entries are +-1,
    and it follows the Sylvester doubling [[H, H], [H, -H]] from H_1 = [1]."""
    for D in (2, 8, 128):
        H = oracle.hadamard_matrix(D)
        assert set(np.unique(H).tolist()) == {-1.0, 1.0}
        np.testing.assert_array_equal(H, H.T)
        np.testing.assert_array_equal(H @ H, D * np.eye(D))
        h = oracle.hadamard_matrix(D // 2) if D > 2 else np.ones((1, 1))
        np.testing.assert_array_equal(H, np.block([[h, h], [h, -h]]))


def test_hadamard_matrix_is_sylvester():
    """The matrix from its definition equals scipy's Sylvester construction."""
    linalg = pytest.importorskip("scipy.linalg")
    for D in (2, 8, 128):
        np.testing.assert_array_equal(oracle.hadamard_matrix(D), linalg.hadamard(D).astype(np.float64))


def test_hadamard_rotate_exact_on_small_integers():
    """Integer inputs of magnitude <= 8 keep every fp32 partial sum exact, and
    H x / 128 is then a multiple of 2^-7 of magnitude <= 8, exact in fp16: the
    fast transform must equal the matrix product bit for bit.  Basis vector
    e_j maps to row j of H times 2^-7."""
    rng = np.random.default_rng(21)
    x = rng.integers(-8, 9, (64, 128)).astype(np.float16)
    want = (x.astype(np.float64) @ oracle.hadamard_matrix(128).T / 128).astype(np.float16)
    np.testing.assert_array_equal(oracle.hadamard_rotate(x).view(np.uint16), want.view(np.uint16))
    eye = np.eye(128, dtype=np.float16)
    np.testing.assert_array_equal(oracle.hadamard_rotate(eye).astype(np.float64),
                                  oracle.hadamard_matrix(128) / 128)


def test_hadamard_rotate_within_one_ulp_of_exact():
    """On fp16 data with outlier channels the fp32 transform then fp16
    rounding lands within one fp16 ulp of the fp64 product rounded once, and
    on it for nearly every element."""
    rng = np.random.default_rng(22)
    x = rng.standard_normal((200, 128)).astype(np.float32)
    x[:, [3, 17, 64, 101]] *= 20
    x = x.astype(np.float16)
    got = oracle.hadamard_rotate(x)
    exact = x.astype(np.float64) @ oracle.hadamard_matrix(128).T / 128
    once = exact.astype(np.float16)
    ulp = np.spacing(np.abs(once).astype(np.float16)).astype(np.float64)
    assert (np.abs(got.astype(np.float64) - once.astype(np.float64)) <= ulp).all()
    assert (got == once).mean() > 0.99
    # the rotation never leaves the input's range
    assert np.abs(got.astype(np.float64)).max() <= np.abs(x.astype(np.float64)).max()


def test_hadamard_unrotate_inverts_rotation():
    """H (H x / D) = x: unrotating the rotated fp16 vectors gives x back
    within the fp16 rounding of the rotated entries (each at most half an
    ulp, summed over D entries of H)."""
    rng = np.random.default_rng(23)
    x = rng.standard_normal((50, 128)).astype(np.float16)
    y = oracle.hadamard_rotate(x)
    back = oracle.hadamard_unrotate(y)
    half_ulp = np.spacing(np.abs(y)).astype(np.float64).max(-1, keepdims=True) / 2
    assert (np.abs(back - x.astype(np.float64)) <= 128 * half_ulp).all()


def test_hadamard_cache_streaming_window_and_error_bound():
    """With the rotation: prefill equals token-by-token appends, the sink and
    the window hold the tokens as given, and the quantized rows come back
    within the rotated-domain half-scale bound carried through the
    orthogonal transform: ||x_hat - x|| <= sqrt(D) (||scale / 2|| + ||fp16
    rounding of the rotated row||)."""
    rng = np.random.default_rng(24)
    S, H, T = 2, 2, 230
    k = rng.standard_normal((S, H, T, 128)).astype(np.float32)
    k[..., [5, 77]] *= 15
    k = k.astype(np.float16)
    v = rng.standard_normal((S, H, T, 128)).astype(np.float16)
    for kpt in (False, True):
        a = oracle.OracleCache(S, H, 256, 2, residual=64, num_sink=1, key_per_token=kpt, hadamard=True)
        a.append(k, v, [T, T - 5])
        b = oracle.OracleCache(S, H, 256, 2, residual=64, num_sink=1, key_per_token=kpt, hadamard=True)
        for t in range(T):
            b.append(k[:, :, t:t + 1], v[:, :, t:t + 1], [1, int(t < T - 5)])
        np.testing.assert_array_equal(a.blocks, b.blocks)
        ns, Lq, r = a.split(1)
        kh, vh = a.keys_values(1, 0)
        np.testing.assert_array_equal(kh[:ns], k[1, 0, :ns].astype(np.float64))
        np.testing.assert_array_equal(kh[ns + Lq:], k[1, 0, ns + Lq:ns + Lq + r].astype(np.float64))
        np.testing.assert_array_equal(vh[ns + Lq:], v[1, 0, ns + Lq:ns + Lq + r].astype(np.float64))
        # value rows (per token in the rotated domain)
        xv = v[1, 0, ns:ns + Lq]
        yv = oracle.hadamard_rotate(xv)
        _, sv, _ = oracle.quantize_value_tokens(yv, 2)
        yexact = xv.astype(np.float64) @ oracle.hadamard_matrix(128).T / 128
        rnd = np.linalg.norm(yv.astype(np.float64) - yexact, axis=-1)
        err = np.linalg.norm(vh[ns:ns + Lq] - xv.astype(np.float64), axis=-1)
        bound = np.sqrt(128) * (np.sqrt(128) * sv.astype(np.float64) / 2 + rnd) * (1 + 1e-6)
        assert (err <= bound).all()
        plain = oracle.OracleCache(S, H, 256, 2, residual=64, num_sink=1, key_per_token=kpt)
        plain.append(k, v, [T, T - 5])
        assert not np.array_equal(a.blocks, plain.blocks)  # the rotation reached the codes


def test_hadamard_attention_in_rotated_domain():
    """Decode over a rotating cache can score the groups with H q against the
    rotated dequantized rows and rotate their value sum back by H: the
    result equals the oracle's attention over the unrotated rows.  A cache
    short enough to stay in full precision is unaffected by the rotation."""
    rng = np.random.default_rng(25)
    T = 200
    k = rng.standard_normal((1, 1, T, 128)).astype(np.float16)
    v = rng.standard_normal((1, 1, T, 128)).astype(np.float16)
    q = rng.standard_normal((1, 3, 128)).astype(np.float16)
    c = oracle.OracleCache(1, 1, 256, 2, residual=64, hadamard=True)
    c.append(k, v, [T])
    ns, Lq, r = c.split(0)
    kc, ks, km, vc, vs, vm = oracle.kivi.unpack_block(c.blocks[0, 0, :Lq // 32], 2)
    ky = oracle.dequantize(kc, ks[:, None, :], km[:, None, :]).reshape(-1, 128)
    vy = oracle.dequantize(vc, vs[:, :, None], vm[:, :, None]).reshape(-1, 128)
    H = oracle.hadamard_matrix(128)
    scale = 1 / np.sqrt(128)
    got = c.attention(q)[0].astype(np.float64)
    for j in range(3):
        qj = q[0, j].astype(np.float64)
        zg = ky @ (H @ qj) * scale
        zw = k[0, 0, Lq:].astype(np.float64) @ qj * scale
        m = max(zg.max(), zw.max())
        pg, pw = np.exp(zg - m), np.exp(zw - m)
        o = H @ (pg @ vy) + pw @ v[0, 0, Lq:].astype(np.float64)
        o /= pg.sum() + pw.sum()
        assert np.abs(got[j] - o).max() <= 1e-3 * np.abs(o).max() + 1e-3
    short = oracle.OracleCache(1, 1, 256, 2, residual=64, hadamard=True)
    plain = oracle.OracleCache(1, 1, 256, 2, residual=64)
    for cc in (short, plain):
        cc.append(k[:, :, :63], v[:, :, :63], [63])
    np.testing.assert_array_equal(short.attention(q), plain.attention(q))


def test_hadamard_helps_per_token_keys_on_outlier_channels():
    """The point of the rotation: spreading fixed outlier channels over all
    channels shrinks per-token key ranges, so per-token key groups after the
    rotation give a smaller mean attention error than without it."""
    rng = np.random.default_rng(26)
    T, Hq = 250, 64
    k = rng.standard_normal((1, 1, T, 128)).astype(np.float32)
    k[..., [3, 17, 64, 101]] *= 20
    k = k.astype(np.float16)
    v = rng.standard_normal((1, 1, T, 128)).astype(np.float16)
    q = rng.standard_normal((1, Hq, 128)).astype(np.float16)
    scale = 1 / np.sqrt(128)
    exact = np.stack([oracle.dense_attention(q[0, j].astype(np.float64), k[0, 0].astype(np.float64),
                                             v[0, 0].astype(np.float64), scale) for j in range(Hq)])
    errs = {}
    for rot in (False, True):
        c = oracle.OracleCache(1, 1, 256, 2, residual=32, key_per_token=True, hadamard=rot)
        c.append(k, v, [T])
        errs[rot] = float(np.abs(c.attention(q)[0].astype(np.float64) - exact).mean())
    assert errs[True] < 0.8 * errs[False], errs


# --------------------------------------------------------- dense-and-sparse


def _first_abs_max(vec):
    """Brute force: the first position of the largest magnitude."""
    best, arg = -1.0, -1
    for i, x in enumerate(vec):
        if abs(float(x)) > best:
            best, arg = abs(float(x)), i
    return arg


@pytest.mark.parametrize("bits", [2, 4])
@pytest.mark.parametrize("axis", [-1, -2])
def test_dense_sparse_reduces_to_plain_quantization(bits, axis):
    """The outlier is the first largest-magnitude element of its slice; the
    other codes, the scale and the min are those of plain asymmetric
    quantization of the slice with the outlier replaced by the min of the
    rest (which leaves the rest's range unchanged); the outlier's code is 0
    and its value is kept exactly."""
    rng = np.random.default_rng(31 + bits)
    x = rng.standard_normal((6, 32, 128)).astype(np.float32)
    x[rng.random(x.shape) < 0.01] *= 40
    x = x.astype(np.float16)
    c, s, m, idx, val = oracle.quantize_dense_sparse(x, axis, bits)
    xs = np.moveaxis(x, axis, -1)
    cs = np.moveaxis(c, axis, -1)
    for b in range(xs.shape[0]):
        for r in range(xs.shape[1]):
            vec = xs[b, r]
            i = _first_abs_max(vec)
            assert idx[b, r] == i and val[b, r] == vec[i]
            rest = np.delete(vec, i)
            rep = vec.copy()
            rep[i] = rest.min()
            pc, ps, pm = oracle.quantize_asymmetric(rep[None, :], -1, bits)
            assert ps[0] == s[b, r] and pm[0] == m[b, r]
            want = pc[0].copy()
            want[i] = 0
            np.testing.assert_array_equal(cs[b, r], want)


def test_dense_sparse_error_bound_and_spike_isolation():
    """Every non-outlier element comes back within half a scale of the
    rest's range, the outlier exactly; a single spike per vector no longer
    inflates the error of the others (plain quantization's error grows with
    the spike, the split's does not)."""
    rng = np.random.default_rng(33)
    x = rng.standard_normal((200, 128)).astype(np.float32)
    spike = rng.integers(0, 128, 200)
    x[np.arange(200), spike] = 60 * np.sign(rng.standard_normal(200))
    x = x.astype(np.float16)
    c, s, m, idx, val = oracle.quantize_dense_sparse(x, -1, 2)
    np.testing.assert_array_equal(idx, spike)
    xh = oracle.dequantize(c, s[:, None], m[:, None])
    xh[np.arange(200), idx] = val
    err = np.abs(xh - x.astype(np.float64))
    assert err[np.arange(200), idx].max() == 0
    assert (err <= s[:, None].astype(np.float64) / 2 * (1 + 1e-6) + 1e-7).all()
    pc, ps, pm = oracle.quantize_asymmetric(x, -1, 2)
    plain = np.abs(oracle.dequantize(pc, ps[:, None], pm[:, None]) - x.astype(np.float64))
    others = np.ones_like(err, bool)
    others[np.arange(200), idx] = False
    assert err[others].mean() < 0.25 * plain[others].mean()


def test_dense_sparse_ties_and_degenerate_slices():
    """Ties go to the first position (+a before -a and the reverse); a
    constant slice keeps its first element as the outlier and the rest has
    scale 0; a zero slice gives index 0, value 0, scale 0."""
    x = np.zeros((4, 8), np.float16)
    x[0] = [1, -3, 2, 3, 0, 0, 0, 0]
    x[1] = [1, 3, 2, -3, 0, 0, 0, 0]
    x[2] = 5
    c, s, m, idx, val = oracle.quantize_dense_sparse(x, -1, 2)
    assert list(idx) == [1, 1, 0, 0]
    assert list(val.astype(np.float64)) == [-3, 3, 5, 0]
    assert s[2] == 0 and m[2] == 5 and (c[2] == 0).all()
    assert s[3] == 0 and m[3] == 0 and not np.signbit(m[3])
    # row 0 without its outlier: rest in [0, 3] -> scale 1, min 0
    assert s[0] == 1 and m[0] == 0 and list(c[0]) == [1, 0, 2, 3, 0, 0, 0, 0]


def test_dense_sparse_block_layout_roundtrip():
    """One 32-bit entry (fp16 bits, then the index at bit 16) per key slice
    and per value token after the metadata: 3968 / 6016 B per block with
    per-channel keys, 2816 / 4864 B with per-token keys; packing
    round-trips."""
    assert oracle.block_bytes(2, outliers=True) == 3328 + 4 * (128 + 32)
    assert oracle.block_bytes(4, outliers=True) == 5376 + 4 * (128 + 32)
    assert oracle.block_bytes(2, key_per_token=True, outliers=True) == 2560 + 4 * 64
    assert oracle.block_bytes(4, key_per_token=True, outliers=True) == 4608 + 4 * 64
    e = oracle.kivi.sparse_entries(np.array([5, 31], np.uint8), np.array([-2.5, 1.0], np.float16))
    assert list(e) == [0xC100 | (5 << 16), 0x3C00 | (31 << 16)]  # -2.5 = 0xC100, 1.0 = 0x3C00
    rng = np.random.default_rng(34)
    for bits, kpt in ((2, False), (4, True)):
        n = 32 if kpt else 128
        kc = rng.integers(0, 1 << bits, (3, 32, 128)).astype(np.uint8)
        vc = rng.integers(0, 1 << bits, (3, 32, 128)).astype(np.uint8)
        ks, km = (rng.standard_normal((3, n)).astype(np.float32) for _ in range(2))
        vs, vm = (rng.standard_normal((3, 32)).astype(np.float32) for _ in range(2))
        ki = rng.integers(0, 32 if not kpt else 128, (3, n)).astype(np.uint8)
        kv = rng.standard_normal((3, n)).astype(np.float16)
        vi = rng.integers(0, 128, (3, 32)).astype(np.uint8)
        vv = rng.standard_normal((3, 32)).astype(np.float16)
        blk = oracle.kivi.pack_block(kc, ks, km, vc, vs, vm, bits, kpt, sparse=(ki, kv, vi, vv))
        out = oracle.kivi.unpack_block(blk, bits, key_per_token=kpt, outliers=True)
        for a, b in zip(out, (kc, ks, km, vc, vs, vm, ki, kv, vi, vv)):
            np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("kpt", [False, True])
def test_dense_sparse_cache_streaming_and_reconstruction(kpt):
    """With the split: prefill equals token-by-token appends; every
    dequantized slice holds its outlier exactly and the rest within half of
    the rest's scale; sink and window exact."""
    rng = np.random.default_rng(35)
    S, H, T = 2, 2, 230
    k = rng.standard_normal((S, H, T, 128)).astype(np.float32)
    k[rng.random(k.shape) < 0.005] *= 50
    k = k.astype(np.float16)
    v = rng.standard_normal((S, H, T, 128)).astype(np.float16)
    a = oracle.OracleCache(S, H, 256, 2, residual=64, num_sink=1, key_per_token=kpt, outliers=True)
    a.append(k, v, [T, T - 11])
    b = oracle.OracleCache(S, H, 256, 2, residual=64, num_sink=1, key_per_token=kpt, outliers=True)
    for t in range(T):
        b.append(k[:, :, t:t + 1], v[:, :, t:t + 1], [1, int(t < T - 11)])
    np.testing.assert_array_equal(a.blocks, b.blocks)
    ns, Lq, r = a.split(0)
    kh, vh = a.keys_values(0, 1)
    np.testing.assert_array_equal(kh[:ns], k[0, 1, :ns].astype(np.float64))
    np.testing.assert_array_equal(kh[ns + Lq:], k[0, 1, ns + Lq:ns + Lq + r].astype(np.float64))
    for got, src, axis, is_key in ((kh, k, -1 if kpt else -2, True), (vh, v, -1, False)):
        x = src[0, 1, ns:ns + Lq].reshape(-1, 32, 128)
        _, s, m, idx, val = oracle.quantize_dense_sparse(x, axis, 2)
        g = got[ns:ns + Lq].reshape(-1, 32, 128)
        err = np.abs(g - x.astype(np.float64))
        if axis == -2:
            assert (err <= s[:, None, :].astype(np.float64) / 2 * (1 + 1e-6) + 1e-7).all()
            gi = np.arange(g.shape[0])[:, None]
            np.testing.assert_array_equal(g[gi, idx, np.arange(128)[None, :]], val.astype(np.float64))
        else:
            assert (err <= s[:, :, None].astype(np.float64) / 2 * (1 + 1e-6) + 1e-7).all()
            gi = np.arange(g.shape[0])[:, None]
            np.testing.assert_array_equal(g[gi, np.arange(32)[None, :], idx], val.astype(np.float64))


def test_dense_sparse_helps_on_per_token_spikes():
    """Outliers at random positions (not fixed channels) skew per-channel key
    groups and per-token value ranges; isolating one per vector lowers the
    mean attention error."""
    rng = np.random.default_rng(36)
    T, Hq = 250, 64
    k = rng.standard_normal((1, 1, T, 128)).astype(np.float32)
    v = rng.standard_normal((1, 1, T, 128)).astype(np.float32)
    for a in (k, v):
        a[rng.random(a.shape) < 0.004] *= 30
    k, v = k.astype(np.float16), v.astype(np.float16)
    q = rng.standard_normal((1, Hq, 128)).astype(np.float16)
    scale = 1 / np.sqrt(128)
    exact = np.stack([oracle.dense_attention(q[0, j].astype(np.float64), k[0, 0].astype(np.float64),
                                             v[0, 0].astype(np.float64), scale) for j in range(Hq)])
    errs = {}
    for sp in (False, True):
        c = oracle.OracleCache(1, 1, 256, 2, residual=32, outliers=sp)
        c.append(k, v, [T])
        errs[sp] = float(np.abs(c.attention(q)[0].astype(np.float64) - exact).mean())
    assert errs[True] < 0.8 * errs[False], errs
