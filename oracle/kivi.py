"""Plain CPU statement of KIVI-style low-bit KV-cache quantization and of decode
attention over the quantized cache (test infrastructure; see package header).

Everything here is numpy.  Quantization decisions are taken in IEEE fp32 (the
precision the packed metadata is stored in); dequantization and attention run
in fp64 and the attention output is rounded once to fp16.

Method, by source (page title, section):

* Asymmetric min/scale codes, x_hat = code * scale + min, codes in
  [0, 2^b - 1]: "KV cache quantization", "What they report" (an asymmetric
  2-bit scheme) and the KIVI page title.
* Keys per channel, each group being 32 tokens of one channel; values per
  token: "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
  second paragraph; "KV cache quantization", "Keys are harder than values".
* The newest tokens (up to R = 128) stay in full precision and are quantized
  in blocks when the window fills: KIVI page, third paragraph; the
  grouped + residual split that attention reads: "KV cache quantization",
  "Keys are harder than values" (streaming bullet).
* Keys stored before RoPE, RoPE applied after dequantization: "KV cache
  quantization", "Keys are harder than values" (RoPE bullet).
* First token kept in fp16 (attention sink): "KV cache quantization",
  "What they report" (KVQuant paragraph).
* Optional per-vector dense-and-sparse split: each vector's outlier is kept
  apart so that it does not skew the vector's quantization range ("KV cache
  quantization", "What they report", KVQuant paragraph).
* Optional Walsh-Hadamard rotation of each key and value vector before it is
  quantized (a training-free rotation named as a design decision of a robust
  low-bit path): "2-Bit KV Cache Quantization: Memory You Save, Recall You
  Risk", "Method map: three ways to shrink the cache".

Readings taken where the pages are silent:
min/max and scale in fp32, scale = (max - min) / (2^b - 1) by one IEEE
division, code = round-half-even of (x - min) / scale by one IEEE
subtraction and one IEEE division, scale == 0 gives code 0; one (scale, min)
per value token over all head_dim channels; the window flushes the moment it
holds R tokens; the sink keeps both K and V of token 0; RoPE is rotate-half
over channel pairs (i, i + D/2) with omega_i = theta^(-2i/D) at absolute
positions; softmax scale defaults to 1/sqrt(D).  The rotation is the
Sylvester-ordered Walsh-Hadamard transform scaled by 1/D, evaluated as the
fast transform in fp32 (strides 1, 2, ..., D/2 in that order) and rounded to
fp16; it applies to the tokens as they are quantized (the sink and the
full-precision window keep the tokens as given), and the dequantized group
rows are rotated back by H (H H = D I).  The dense-and-sparse split takes,
in every quantization slice (a key channel's 32 tokens, or a token's D
channels), the one element of largest magnitude (the first in slice order on
ties) as the outlier: it is kept exactly in fp16 with its index, the slice's
min and max are taken over the other elements, and the outlier's code is 0.
"""

from __future__ import annotations

import math

import numpy as np

GROUP = 32          # tokens per key group (KIVI page, second paragraph)
HEAD_DIM = 128


# --------------------------------------------------------------------------
# Asymmetric uniform quantization
# --------------------------------------------------------------------------

def quantize_asymmetric(x, axis: int, bits: int):
    """Asymmetric b-bit quantization of fp16 `x`, one (scale, min) per slice
    taken along `axis`.

    min/max are exact in fp32 (the inputs are fp16; a zero extreme is stored
    as +0).  scale is
    fl32((max - min) / (2^b - 1)); code = clamp(rne(fl32(fl32(x - min) /
    scale)), 0, 2^b - 1), and a slice with max == min has scale 0 and all
    codes 0.  Returns (codes uint8 shaped like x, scale fp32, min fp32), the
    last two with `axis` removed.
    """
    x32 = np.asarray(x, dtype=np.float16).astype(np.float32)
    # + 0 turns a -0 extreme into +0, so the stored min never depends on
    # which of two equal zeros a reduction happened to return
    mn = x32.min(axis=axis, keepdims=True) + np.float32(0)
    mx = x32.max(axis=axis, keepdims=True) + np.float32(0)
    levels = np.float32(2 ** bits - 1)
    scale = (mx - mn) / levels                      # fp32 / fp32: one IEEE division
    assert scale.dtype == np.float32
    d = x32 - mn                                    # one IEEE fp32 subtraction
    with np.errstate(divide="ignore", invalid="ignore"):
        y = d / scale                               # one IEEE fp32 division
    c = np.rint(y)                                  # round half to even
    c = np.where(scale == 0, np.float32(0), c)
    c = np.clip(c, np.float32(0), levels)
    return (c.astype(np.uint8),
            np.squeeze(scale, axis=axis).astype(np.float32),
            np.squeeze(mn, axis=axis).astype(np.float32))


def quantize_dense_sparse(x, axis: int, bits: int):
    """Dense-and-sparse quantization of fp16 `x`, one slice per position
    along the other axes: the slice's largest-|x| element (the first in
    slice order on ties) is the outlier, kept exactly as (index, fp16 value);
    the other elements are quantized as by `quantize_asymmetric`, with min
    and max taken over them alone; the outlier's code is 0.

    Returns (codes, scale, min, index uint8, value fp16), the last four with
    `axis` removed.
    """
    x16 = np.asarray(x, dtype=np.float16)
    x32 = x16.astype(np.float32)
    idx = np.argmax(np.abs(x32), axis=axis)           # first maximum
    n = x32.shape[axis]
    pos = np.expand_dims(idx, axis) == np.arange(n).reshape([-1 if a == axis % x32.ndim else 1
                                                             for a in range(x32.ndim)])
    mn = np.where(pos, np.float32(np.inf), x32).min(axis=axis, keepdims=True) + np.float32(0)
    mx = np.where(pos, np.float32(-np.inf), x32).max(axis=axis, keepdims=True) + np.float32(0)
    levels = np.float32(2 ** bits - 1)
    scale = (mx - mn) / levels
    d = x32 - mn
    with np.errstate(divide="ignore", invalid="ignore"):
        y = d / scale
    c = np.rint(y)
    c = np.where(scale == 0, np.float32(0), c)
    c = np.clip(c, np.float32(0), levels)
    c = np.where(pos, np.float32(0), c)
    val = np.take_along_axis(x16, np.expand_dims(idx, axis), axis=axis)
    return (c.astype(np.uint8),
            np.squeeze(scale, axis=axis).astype(np.float32),
            np.squeeze(mn, axis=axis).astype(np.float32),
            idx.astype(np.uint8),
            np.squeeze(val, axis=axis))


def quantize_key_group(k_group, bits: int):
    """Per-channel key quantization of one group: k_group is [32 tokens][D]
    fp16; each channel gets its own (scale, min) over the group's 32 tokens
    (KIVI page, second paragraph).  Returns codes [32][D], scale [D], min [D].
    """
    assert k_group.shape[-2] == GROUP
    return quantize_asymmetric(k_group, axis=-2, bits=bits)


def quantize_value_tokens(v_tokens, bits: int):
    """Per-token value quantization: v_tokens is [T][D] fp16; each token gets
    one (scale, min) over its D channels (KIVI page, second paragraph).
    Returns codes [T][D], scale [T], min [T]."""
    return quantize_asymmetric(v_tokens, axis=-1, bits=bits)


def quantize_keys_per_token(k_tokens, bits: int):
    """The per-token round-to-nearest baseline the KIVI page's first paragraph
    contrasts with (used by tests to show what per-channel grouping buys)."""
    return quantize_asymmetric(k_tokens, axis=-1, bits=bits)


def dequantize(codes, scale, mn):
    """x_hat = code * scale + min, in fp64 (scale/min broadcast by caller)."""
    return (codes.astype(np.float64) * np.asarray(scale, np.float64)
            + np.asarray(mn, np.float64))


# --------------------------------------------------------------------------
# Packed format
# --------------------------------------------------------------------------
#
# A code tile has `rows` x `cols` b-bit codes.  Keys use rows = the group's 32
# tokens, cols = the D channels; values use rows = the D channels, cols = the
# group's 32 tokens.  The tile is stored as 32 "lanes" x W 32-bit words
# (W = rows * cols * b / 1024), little-endian.  For element (row, col):
#
#   mt, h, g     = row // 16, (row // 8) % 2, row % 8
#   kt, j, q, e  = col // 16, (col // 8) % 2, (col % 8) // 2, col % 2
#   tau = 2 * (mt % 2) + h ;  P = mt // 2 ;  KT = cols // 16
#   nu  = 8 // b                      (fields per byte)
#   u   = tau % nu
#   w   = (P * KT + kt) * (4 // nu) + tau // nu
#   lane = 4 * g + q
#   word byte offset = ((w // 4) * 32 + lane) * 16 + (w % 4) * 4
#   bit within word  = 16 * e + 8 * j + b * u
#
# The map is a bijection between tile elements and the tile's bits.

def code_location(row: int, col: int, bits: int, rows: int, cols: int):
    """(byte offset, bit in byte) of element (row, col) of a packed tile."""
    assert bits in (2, 4) and rows % 32 == 0 and cols % 16 == 0
    assert 0 <= row < rows and 0 <= col < cols
    nu = 8 // bits
    mt, h, g = row // 16, (row // 8) % 2, row % 8
    kt, j, q, e = col // 16, (col // 8) % 2, (col % 8) // 2, col % 2
    tau = 2 * (mt % 2) + h
    P = mt // 2
    KT = cols // 16
    u = tau % nu
    w = (P * KT + kt) * (4 // nu) + tau // nu
    lane = 4 * g + q
    word_byte = ((w // 4) * 32 + lane) * 16 + (w % 4) * 4
    bit = 16 * e + 8 * j + bits * u
    return word_byte + bit // 8, bit % 8


_LOC_CACHE: dict = {}


def code_location_table(rows: int, cols: int, bits: int):
    """Arrays (byte[rows, cols], bit[rows, cols]) of `code_location`."""
    key = (rows, cols, bits)
    if key not in _LOC_CACHE:
        byte = np.empty((rows, cols), np.int64)
        bit = np.empty((rows, cols), np.int64)
        for r in range(rows):
            for c in range(cols):
                byte[r, c], bit[r, c] = code_location(r, c, bits, rows, cols)
        _LOC_CACHE[key] = (byte, bit)
    return _LOC_CACHE[key]


_INV_CACHE: dict = {}


def _inverse_table(rows: int, cols: int, bits: int):
    """For every packed byte and field: the flat element index stored there.
    Building it asserts that the map is a bijection."""
    key = (rows, cols, bits)
    if key in _INV_CACHE:
        return _INV_CACHE[key]
    byte, bit = code_location_table(rows, cols, bits)
    nu = 8 // bits
    inv = np.full((rows * cols * bits // 8, nu), -1, np.int64)
    for idx, (by, bi) in enumerate(zip(byte.reshape(-1), bit.reshape(-1))):
        assert bi % bits == 0 and inv[by, bi // bits] == -1
        inv[by, bi // bits] = idx
    assert (inv >= 0).all()
    _INV_CACHE[key] = inv
    return inv


def pack_tile(codes, bits: int):
    """Pack codes[..., rows, cols] (uint8, < 2^b) into [..., rows*cols*b/8]
    bytes following the map above."""
    codes = np.asarray(codes, np.uint8)
    rows, cols = codes.shape[-2:]
    assert int(codes.max(initial=0)) < (1 << bits)
    inv = _inverse_table(rows, cols, bits)
    flat = codes.reshape(codes.shape[:-2] + (rows * cols,))
    out = np.zeros(codes.shape[:-2] + (inv.shape[0],), np.uint8)
    for f in range(inv.shape[1]):
        out |= (flat[..., inv[:, f]] << np.uint8(bits * f)).astype(np.uint8)
    return out


def unpack_tile(buf, bits: int, rows: int, cols: int):
    """Inverse of `pack_tile`: bytes [..., rows*cols*b/8] -> codes [..., rows, cols]."""
    buf = np.asarray(buf, np.uint8)
    byte, bit = code_location_table(rows, cols, bits)
    mask = (1 << bits) - 1
    vals = buf[..., byte.reshape(-1)].astype(np.uint32) >> bit.reshape(-1).astype(np.uint32)
    return (vals & mask).astype(np.uint8).reshape(buf.shape[:-1] + (rows, cols))


def block_bytes(bits: int, head_dim: int = HEAD_DIM, key_per_token: bool = False,
                outliers: bool = False) -> int:
    """Bytes of one 32-token group block: K codes, V codes (32*D*b/8 each),
    K scale and K min (fp32 per channel; per token when keys are grouped per
    token), V scale and V min (fp32 per token); with the dense-and-sparse
    split, one 32-bit outlier entry per key slice and per value token."""
    kmeta = GROUP if key_per_token else head_dim
    sparse = 4 * (kmeta + GROUP) if outliers else 0
    return 2 * (GROUP * head_dim * bits // 8) + 2 * 4 * kmeta + 2 * 4 * GROUP + sparse


def sparse_entries(idx, val):
    """32-bit outlier entries: the fp16 value's bits in bits 0-15, the index
    within the slice in bits 16-23."""
    return (np.asarray(val, np.float16).view(np.uint16).astype(np.uint32)
            | (np.asarray(idx, np.uint32) << 16))


def pack_block(kc, ks, km, vc, vs, vm, bits: int, key_per_token: bool = False, sparse=None):
    """One group block.  kc: [32 tok][D] key codes, ks/km: [D] ([32] when
    keys are grouped per token); vc: [32 tok][D] value codes, vs/vm: [32];
    sparse: None, or (key outlier index, key outlier value, value outlier
    index, value outlier value), each per key slice / per value token."""
    D = kc.shape[-1]
    kbytes = GROUP * D * bits // 8
    km_n = GROUP if key_per_token else D
    parts = [
        pack_tile(kc, bits),                                   # rows = tokens
        pack_tile(np.swapaxes(vc, -1, -2), bits),              # rows = channels
        np.asarray(ks, np.float32).view(np.uint8).reshape(ks.shape[:-1] + (4 * km_n,)),
        np.asarray(km, np.float32).view(np.uint8).reshape(km.shape[:-1] + (4 * km_n,)),
        np.asarray(vs, np.float32).view(np.uint8).reshape(vs.shape[:-1] + (4 * GROUP,)),
        np.asarray(vm, np.float32).view(np.uint8).reshape(vm.shape[:-1] + (4 * GROUP,)),
    ]
    if sparse is not None:
        ki, kv, vi, vv = sparse
        parts.append(sparse_entries(ki, kv).view(np.uint8).reshape(ki.shape[:-1] + (4 * km_n,)))
        parts.append(sparse_entries(vi, vv).view(np.uint8).reshape(vi.shape[:-1] + (4 * GROUP,)))
    out = np.concatenate(parts, axis=-1)
    assert out.shape[-1] == block_bytes(bits, D, key_per_token, sparse is not None)
    assert parts[0].shape[-1] == kbytes
    return out


def unpack_block(buf, bits: int, head_dim: int = HEAD_DIM, key_per_token: bool = False,
                 outliers: bool = False):
    """Inverse of `pack_block`: returns (kc [32][D], ks [D], km [D] (both
    [32] for per-token keys), vc [32][D], vs [32], vm [32]), followed with
    outliers by (key index, key value, value index, value value)."""
    D = head_dim
    buf = np.ascontiguousarray(buf, np.uint8)
    cb = GROUP * D * bits // 8
    o = 0
    kc = unpack_tile(buf[..., o:o + cb], bits, GROUP, D); o += cb
    vcT = unpack_tile(buf[..., o:o + cb], bits, D, GROUP); o += cb

    def f32(n):
        nonlocal o
        a = np.ascontiguousarray(buf[..., o:o + 4 * n]).view(np.float32)
        o += 4 * n
        return a
    ks = f32(GROUP if key_per_token else D)
    km = f32(GROUP if key_per_token else D)
    vs = f32(GROUP)
    vm = f32(GROUP)
    dense = (kc, ks, km, np.swapaxes(vcT, -1, -2), vs, vm)
    if not outliers:
        return dense

    def entries(n):
        nonlocal o
        e = np.ascontiguousarray(buf[..., o:o + 4 * n]).view(np.uint32)
        o += 4 * n
        return (e >> 16).astype(np.uint8), (e & 0xFFFF).astype(np.uint16).view(np.float16)
    ki, kv = entries(GROUP if key_per_token else D)
    vi, vv = entries(GROUP)
    return dense + (ki, kv, vi, vv)


# --------------------------------------------------------------------------
# Walsh-Hadamard rotation (applied to tokens as they are quantized)
# --------------------------------------------------------------------------

def hadamard_rotate(x):
    """fp16(H x / D) of each D-vector of fp16 `x` (last axis), H the
    Sylvester Walsh-Hadamard matrix, H[i][j] = (-1)^popcount(i & j).

    Evaluated as the fast transform in fp32: for stride = 1, 2, ..., D/2 in
    that order, every element pair (i, i + stride) with the stride bit of i
    clear becomes (a + b, a - b) (one IEEE fp32 add or subtract each); the
    result is scaled by 1/D (a power of two: exact) and rounded to fp16
    (half to even).  Since every |entry| of H x / D is at most max |x|, the
    result never leaves the fp16 range.
    """
    y = np.asarray(x, np.float16).astype(np.float32)
    D = y.shape[-1]
    assert D & (D - 1) == 0
    lead = y.shape[:-1]
    stride = 1
    while stride < D:
        t = y.reshape(lead + (D // (2 * stride), 2, stride))
        a, b = t[..., 0, :], t[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (D,))
        stride *= 2
    return (y * np.float32(1.0 / D)).astype(np.float16)


def hadamard_matrix(D: int):
    """H[i][j] = (-1)^popcount(i & j) in fp64, from the definition."""
    i = np.arange(D)
    bits = np.bitwise_and(i[:, None], i[None, :])
    par = np.zeros_like(bits)
    while bits.any():
        par ^= bits & 1
        bits >>= 1
    return np.where(par == 1, -1.0, 1.0)


def hadamard_unrotate(y):
    """x = H y in fp64 (the inverse of y = H x / D)."""
    y = np.asarray(y, np.float64)
    return y @ hadamard_matrix(y.shape[-1]).T


# --------------------------------------------------------------------------
# RoPE (applied to dequantized pre-RoPE keys)
# --------------------------------------------------------------------------

def rope_rotate(x, positions, theta: float = 10000.0):
    """Rotate-half RoPE in fp64: channel pairs (i, i + D/2) rotate by angle
    p * theta^(-2i/D) at absolute position p ("KV cache quantization",
    "Keys are harder than values": RoPE rotates between pairs of channels)."""
    x = np.asarray(x, np.float64)
    D = x.shape[-1]
    half = D // 2
    i = np.arange(half, dtype=np.float64)
    omega = np.power(float(theta), -2.0 * i / D)
    ang = np.asarray(positions, np.float64)[:, None] * omega[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


# --------------------------------------------------------------------------
# Streaming cache state
# --------------------------------------------------------------------------

class OracleCache:
    """The cache of S sequences x H KV heads, held in the same byte layout as
    the device buffers:

    blocks [S][H][max_groups][block_bytes] u8, k_res/v_res [S][H][R][D] fp16,
    k_sink/v_sink [S][H][num_sink][D] fp16, seq_len [S] int32.

    Token p of a sequence goes to the sink if p < num_sink; otherwise it
    enters the full-precision window, and whenever the window holds R tokens
    those R tokens are quantized into R/32 group blocks and the window empties
    (KIVI page, third paragraph).  seq_len counts every stored token.

    key_per_token switches keys to the per-token grouping the KIVI page's
    first paragraph describes as the baseline (one scale and min per token
    over its D channels, like values): the ablation of per-channel keys.
    hadamard rotates every key and value token by hadamard_rotate as its
    window is quantized; the blocks then hold the rotated tokens' codes.
    outliers applies the dense-and-sparse split (quantize_dense_sparse) to
    every key slice and value token.
    """

    def __init__(self, num_seqs, num_kv_heads, capacity, bits, residual=128,
                 num_sink=0, head_dim=HEAD_DIM, key_per_token=False, hadamard=False, outliers=False):
        assert bits in (2, 4) and residual % GROUP == 0 and residual > 0
        assert num_sink in (0, 1) and capacity >= 1
        self.S, self.H, self.D = num_seqs, num_kv_heads, head_dim
        self.bits, self.R, self.ns, self.capacity = bits, residual, num_sink, capacity
        self.kpt = bool(key_per_token)
        self.rot = bool(hadamard)
        self.sparse = bool(outliers)
        stream_cap = max(capacity - num_sink, 0)
        self.max_groups = (stream_cap // residual) * residual // GROUP
        self.bb = block_bytes(bits, head_dim, self.kpt, self.sparse)
        self.blocks = np.zeros((num_seqs, num_kv_heads, self.max_groups, self.bb), np.uint8)
        self.k_res = np.zeros((num_seqs, num_kv_heads, residual, head_dim), np.float16)
        self.v_res = np.zeros_like(self.k_res)
        self.k_sink = np.zeros((num_seqs, num_kv_heads, num_sink, head_dim), np.float16)
        self.v_sink = np.zeros_like(self.k_sink)
        self.seq_len = np.zeros(num_seqs, np.int32)

    # -- append ------------------------------------------------------------
    def append(self, k_new, v_new, new_len):
        """Append new_len[s] tokens of k_new/v_new [S][H][max_new][D] fp16 to
        each sequence s, in token order."""
        k_new = np.asarray(k_new, np.float16)
        v_new = np.asarray(v_new, np.float16)
        for s in range(self.S):
            n = int(new_len[s])
            L0 = int(self.seq_len[s])
            assert 0 <= n <= k_new.shape[2] and L0 + n <= self.capacity
            j = 0
            while j < n and L0 + j < self.ns:               # sink slot(s)
                self.k_sink[s, :, L0 + j] = k_new[s, :, j]
                self.v_sink[s, :, L0 + j] = v_new[s, :, j]
                j += 1
            while j < n:                                    # full-precision window
                stored = L0 + j - self.ns                   # stream tokens so far
                r = stored % self.R
                take = min(self.R - r, n - j)
                self.k_res[s, :, r:r + take] = k_new[s, :, j:j + take]
                self.v_res[s, :, r:r + take] = v_new[s, :, j:j + take]
                j += take
                if r + take == self.R:                      # window full: flush
                    self._flush(s, first_group=(stored - r) // GROUP)
            self.seq_len[s] = L0 + n

    def _flush(self, s, first_group):
        """Quantize the R tokens of sequence s's window into R/32 blocks."""
        H, D, R = self.H, self.D, self.R
        kg = self.k_res[s].reshape(H, R // GROUP, GROUP, D)
        vg = self.v_res[s].reshape(H, R // GROUP, GROUP, D)
        if self.rot:
            kg, vg = hadamard_rotate(kg), hadamard_rotate(vg)
        if self.sparse:
            kc, ks, km, ki, kv = quantize_dense_sparse(kg, -1 if self.kpt else -2, self.bits)
            vc, vs, vm, vi, vv = quantize_dense_sparse(vg, -1, self.bits)
            blk = pack_block(kc, ks, km, vc, vs, vm, self.bits, self.kpt, sparse=(ki, kv, vi, vv))
        else:
            if self.kpt:
                kc, ks, km = quantize_keys_per_token(kg, self.bits)  # per token
            else:
                kc, ks, km = quantize_key_group(kg, self.bits)       # per channel
            vc, vs, vm = quantize_value_tokens(vg, self.bits)        # per token
            blk = pack_block(kc, ks, km, vc, vs, vm, self.bits, self.kpt)
        self.blocks[s, :, first_group:first_group + R // GROUP] = blk

    # -- reading the state back -------------------------------------------
    def split(self, s):
        """(sink tokens, quantized tokens Lq, residual tokens r) of sequence s."""
        L = int(self.seq_len[s])
        ns = min(L, self.ns)
        n = L - ns
        r = n % self.R
        return ns, n - r, r

    def keys_values(self, s, h):
        """Dequantized pre-RoPE keys and values of (s, h) in position order,
        fp64 [L][D] each: sink (exact), groups (code*scale+min, rotated back
        by H when the cache rotates), window (exact)."""
        ns, Lq, r = self.split(s)
        ks = [self.k_sink[s, h, :ns].astype(np.float64)]
        vs = [self.v_sink[s, h, :ns].astype(np.float64)]
        ng = Lq // GROUP
        if ng:
            parts = unpack_block(self.blocks[s, h, :ng], self.bits, self.D, self.kpt, self.sparse)
            kc, ksc, kmn, vc, vsc, vmn = parts[:6]
            if self.kpt:
                kd = dequantize(kc, ksc[:, :, None], kmn[:, :, None])
            else:
                kd = dequantize(kc, ksc[:, None, :], kmn[:, None, :])
            vd = dequantize(vc, vsc[:, :, None], vmn[:, :, None])
            if self.sparse:  # outliers exactly as stored: [group][token][channel]
                ki, kv, vi, vv = parts[6:]
                g = np.arange(ng)[:, None]
                sl = np.arange(ki.shape[1])[None, :]
                if self.kpt:
                    kd[g, sl, ki] = kv
                else:
                    kd[g, ki, sl] = kv
                vd[g, np.arange(GROUP)[None, :], vi] = vv
            ks.append(kd.reshape(-1, self.D))
            vs.append(vd.reshape(-1, self.D))
            if self.rot:
                ks[-1], vs[-1] = hadamard_unrotate(ks[-1]), hadamard_unrotate(vs[-1])
        ks.append(self.k_res[s, h, :r].astype(np.float64))
        vs.append(self.v_res[s, h, :r].astype(np.float64))
        return np.concatenate(ks, 0), np.concatenate(vs, 0)

    def dequant_all(self):
        """[S][H][capacity][D] fp64 K_hat (pre-RoPE) and V_hat; NaN past seq_len."""
        K = np.full((self.S, self.H, self.capacity, self.D), np.nan)
        V = np.full_like(K, np.nan)
        for s in range(self.S):
            L = int(self.seq_len[s])
            for h in range(self.H):
                k, v = self.keys_values(s, h)
                K[s, h, :L], V[s, h, :L] = k, v
        return K, V

    def attention(self, q, softmax_scale=None, pre_rope=False, rope_theta=10000.0,
                  heads=None):
        """Decode attention of one query token per (sequence, query head).

        q: [S][Hq][D] fp16 (already rotated by the caller when keys are
        stored pre-RoPE).  Query head j reads KV head j // (Hq / H).  Returns
        fp16 [S][Hq][D]; rows not in `heads` (a list of (s, j)) stay zero.
        """
        q = np.asarray(q, np.float16)
        S, Hq, D = q.shape
        assert S == self.S and Hq % self.H == 0 and D == self.D
        grp = Hq // self.H
        scale = 1.0 / math.sqrt(D) if softmax_scale is None or softmax_scale <= 0 else float(softmax_scale)
        out = np.zeros((S, Hq, D), np.float16)
        todo = heads if heads is not None else [(s, j) for s in range(S) for j in range(Hq)]
        cache = {}
        for s, j in todo:
            h = j // grp
            if (s, h) not in cache:
                k, v = self.keys_values(s, h)
                if pre_rope:
                    k = rope_rotate(k, np.arange(k.shape[0]), rope_theta)
                cache[(s, h)] = (k, v)
            k, v = cache[(s, h)]
            out[s, j] = dense_attention(q[s, j].astype(np.float64), k, v, scale).astype(np.float16)
        return out


def dense_attention(q, K, V, scale):
    """softmax(scale * K q) V in fp64 with max subtraction; zeros if L == 0."""
    if K.shape[0] == 0:
        return np.zeros(q.shape[-1])
    z = (K @ q) * scale
    p = np.exp(z - z.max())
    return (p @ V) / p.sum()
