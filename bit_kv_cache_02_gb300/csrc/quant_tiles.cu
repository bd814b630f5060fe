// Quantize-and-pack of the groups that an append flushes, one tile per warp.
//
// Source: "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
// second paragraph (keys quantized per channel over groups of 32 tokens,
// values per token, asymmetric min/scale codes) and third paragraph (the
// window of newest tokens is quantized in blocks when it fills); keys
// grouped per token are the baseline the first paragraph contrasts with.
//
// Each group block is made of two independent halves: the key tile (32
// tokens x 128 channels, one (scale, min) per channel) and the value tile
// (one (scale, min) per token).  A warp quantizes one tile at a time, with
// no synchronization beyond its own lanes: the line of tiles (key tile,
// value tile, next group, ...) of every (sequence, KV head) is cut into one
// contiguous range per warp.  The 32 token rows of a tile reach shared memory
// through one 256-byte bulk copy per lane (rows from the fp16 window or the
// new tokens alike), into the warp's slot (a ring of one by default), whose
// rows are padded to 272 bytes so that both read patterns below are free of
// bank conflicts.  A warp's next tile is copied once the current one is
// packed; the 20 to 24 warps of an SM hide that latency from one another.
//
//   key tile:   lane L owns channels 4L .. 4L+3 of all 32 tokens: their
//               min/max are lane-local, and the lane packs the codes of its
//               channels into half-words of the mma-fragment layout.
//   value tile: lane L owns tokens 2p, 2p+1 (p = L % 16) over channels
//               64 (L / 16) .. +63: the token statistics take one exchange
//               with lane L ^ 16, and byte permutes pair the two tokens of a
//               channel, which the layout places in the two halves of a word.
//
// A packed word takes codes from two lanes (the two channel octets j of a
// 16-channel tile for keys, the two token octets for values): each lane
// builds its half, one shuffle ORs in the partner's, and one of the two
// stores the word.  Codes use the reciprocal filter with the exact IEEE
// fallback of quant_common.cuh, so they equal the oracle's bit for bit.  The
// lanes store the finished words and the slice scales and mins straight into
// the group block (a tile's code words and metadata together cover whole
// 32-byte sectors, which L2 merges before they reach HBM), so a warp needs
// shared memory only for its ring.
//
// Options, as template flags of the kernel: keys grouped per token
// (key_tile_kpt), the Walsh-Hadamard rotation of the rows in place before a
// tile is quantized (rotate_tile), and dense-and-sparse blocks (an outlier
// pass before the statistics).  Per-token keys with outlier entries, and
// batches of more than kTileFlushMaxSeqs sequences, use the general flush
// kernel.
#include "quant_common.cuh"

namespace kvq {

constexpr int kRowPad = 272;                // bytes per token row in a ring slot (256 + 16)
constexpr int kSlotBytes = kG * kRowPad;    // 8704
// Ring slots per warp, and warps per CTA (one CTA per SM) at each bit width.
// One slot measured fastest: the slot is refilled only once its tile is
// packed, but the smaller shared memory lets 20 (2-bit) or 24 (4-bit) warps
// share an SM, which hide each other's copy latency and fixed-latency
// stalls better than 13 warps with two slots each (the register budget that
// the warp count leaves decides between 20 and 24).
#ifndef KVQ_TILE_RING
#define KVQ_TILE_RING 1
#endif
#ifndef KVQ_TILE_WARPS_2BIT
#define KVQ_TILE_WARPS_2BIT 20
#endif
#ifndef KVQ_TILE_WARPS_4BIT
#define KVQ_TILE_WARPS_4BIT 24
#endif

struct TileSmem {  // one warp's shared memory: the ring, then its mbarriers
  static constexpr int NS = KVQ_TILE_RING;  // ring slots
  static constexpr int BAR = NS * kSlotBytes;
  static constexpr int BYTES = (BAR + 8 * NS + 127) / 128 * 128;
  static_assert(kSlotBytes % 16 == 0 && kRowPad % 16 == 0, "bulk copies need 16-byte alignment");
};

template <int BITS>
struct TileShape {
  static constexpr int WANT = BITS == 2 ? KVQ_TILE_WARPS_2BIT : KVQ_TILE_WARPS_4BIT;
  static constexpr int WARPS = 232448 / TileSmem::BYTES < WANT ? 232448 / TileSmem::BYTES : WANT;
};

// The flush of sequence s in this append: groups ng starting at stream
// index Lq0 (0 when the sequence is skipped: its lengths are reported by the
// tail kernel), the window's first stream index n0 - (n0 % R) = Lq0 and the
// length L0 before the append.
struct SeqFlush {
  int ng, Lq0, n0, L0;
};

__device__ __forceinline__ SeqFlush seq_flush(const Geo &geo, const int *new_len, int max_new, int s) {
  SeqFlush f;
  f.L0 = geo.seq_len[s];
  const int nn = new_len[s];
  f.ng = f.Lq0 = f.n0 = 0;
  if (nn < 0 || nn > max_new || f.L0 < 0 || f.L0 + nn > geo.capacity) return f;
  f.n0 = max(f.L0 - geo.ns, 0);
  const int n1 = max(f.L0 + nn - geo.ns, 0);
  f.Lq0 = f.n0 - f.n0 % geo.R;
  f.ng = (n1 - n1 % geo.R - f.Lq0) / kG;
  return f;
}

// A position on the tile line: sequence s (its flush f), KV head h, group g
// of the flush, kind 0 (keys) or 1 (values).
struct TilePos {
  int s, h, g, kind;
  SeqFlush f;
};

// Next tile of the line (skipping sequences with nothing to flush); false
// past the last sequence.
__device__ __forceinline__ bool next_tile(TilePos &p, const Geo &geo, const int *new_len, int max_new) {
  if (p.kind == 0) {
    p.kind = 1;
    return true;
  }
  p.kind = 0;
  if (++p.g < p.f.ng) return true;
  p.g = 0;
  if (++p.h < geo.H) return true;
  p.h = 0;
  while (++p.s < geo.S) {
    p.f = seq_flush(geo, new_len, max_new, p.s);
    if (p.f.ng > 0) return true;
  }
  return false;
}

// Codes of NF fp16 pairs into one word: pair f holds the fields e = 0 (low
// half) and e = 1 (high half) of one slice pair whose reciprocal filter
// constants are (rcp, c); its codes land at bits pos_f and 16 + pos_f, with
// sc[f] = 2^pos_f.  Each half accumulates 2^23 + sum code * 2^pos exactly in
// fp32 and the low 16 bits of both are joined by one byte permute.  Sets
// `near` when some estimate lies within the filter's tolerance of a rounding
// boundary (thr = 1/2 - tol): the word is then redone exactly.
template <int NF>
__device__ __forceinline__ uint32_t pack_pairs(const uint32_t (&x)[NF], f2x rcp, f2x c, const float (&sc)[NF],
                                               float thr, bool &near) {
  const f2x magic = f2_pack(kMagic, kMagic);
  f2x acc = f2_pack(kPackBase, kPackBase);
  float emax = 0.f;
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const float2 xf = __half22float2(*reinterpret_cast<const __half2 *>(&x[f]));
    const f2x y = f2_fma(f2_pack(xf.x, xf.y), rcp, c);
    const f2x r = f2_sub(f2_add(y, magic), magic);  // rne(y), exact
    const float2 e = f2_unpack(f2_sub(y, r));
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(emax) : "f"(emax), "f"(e.x), "f"(e.y));  // max of |.|
    acc = f2_fma(r, f2_pack(sc[f], sc[f]), acc);
  }
  near = emax > thr;
  const float2 a = f2_unpack(acc);
  return __byte_perm(__float_as_uint(a.x), __float_as_uint(a.y), 0x5410);
}

// The same word by the IEEE subtract and divide of every code (when the
// filter cannot decide one of them; rare, out of line).
template <int BITS, int NF>
__device__ __noinline__ uint32_t pack_pairs_exact(const uint32_t (&x)[NF], float lo0, float sc0, float lo1, float sc1,
                                                  const int (&pos)[NF]) {
  uint32_t w = 0;
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const float2 xf = __half22float2(*reinterpret_cast<const __half2 *>(&x[f]));
    w |= exact_code<BITS>(xf.x, lo0, sc0) << pos[f];
    w |= exact_code<BITS>(xf.y, lo1, sc1) << (16 + pos[f]);
  }
  return w;
}

// Byte offset of packed word w of lane l in a code tile.
__device__ __forceinline__ int word_offset(int w, int l) { return ((w >> 2) * 32 + l) * 16 + (w & 3) * 4; }

// Slice constants of a pair of slices (lo, hi in fp32): scales, the filter
// constants as pairs, and the filter threshold.
struct PairQ {
  float lo0, lo1, sc0, sc1, thr;
  f2x rcp, c;
};

__device__ __forceinline__ PairQ pair_q(float lo0, float hi0, float lo1, float hi1, float levels) {
  PairQ p;
  p.lo0 = lo0;
  p.lo1 = lo1;
  p.sc0 = __fdiv_rn(__fsub_rn(hi0, lo0), levels);
  p.sc1 = __fdiv_rn(__fsub_rn(hi1, lo1), levels);
  const SliceQ a = make_slice(lo0, p.sc0, levels), b = make_slice(lo1, p.sc1, levels);
  p.rcp = f2_pack(a.rcp, b.rcp);
  p.c = f2_pack(a.c, b.c);
  p.thr = 0.5f - fmaxf(a.tol, b.tol);
  return p;
}

// -------------------------------------------------- dense-and-sparse slices
//
// Blocks with outlier entries ("KV cache quantization", "What they report":
// dense-and-sparse quantization isolating outliers per vector): the outlier
// of a slice is its first element of largest magnitude, kept exactly in the
// slice's 32-bit entry (fp16 bits, index at bit 16); min and scale come from
// the other elements and the outlier's code is 0.  Before a tile's
// statistics, the pass below records every slice's outlier and overwrites
// it in the tile with a neighbour of its slice, so the unchanged statistics
// see the other elements only; once the slice's min is known, the owner lane
// writes that min in its place, which the unchanged packing codes 0.  Keys
// are per channel here (per-token keys with outlier entries use the general
// flush kernel).

// First row of largest magnitude per channel as fp16 (2 x 16-bit lanes):
// min over rows of (match ? row : 32), exact in fp16.
__device__ __forceinline__ uint32_t h2_first_match(uint32_t mag, uint32_t best, float pos, uint32_t idx) {
  const __half2 eq = __heq2(*reinterpret_cast<const __half2 *>(&mag), *reinterpret_cast<const __half2 *>(&best));
  const __half2 cand = __hfma2(eq, __float2half2_rn(pos - 32.f), __float2half2_rn(32.f));
  return h2min(idx, h2_as_u32(cand));
}

struct KeyOutliers {
  int row[4];  // outlier row of channels 4L .. 4L+3 of this lane
};

__device__ __forceinline__ KeyOutliers key_outliers_tile(uint8_t *tile, uint8_t *blk, int bits, int lane) {
  uint8_t *col = tile + 8 * lane;
  uint32_t ma = 0u, mb = 0u;  // magnitudes of channels (4L, 4L+1) and (4L+2, 4L+3)
#pragma unroll 8
  for (int t = 0; t < kG; ++t) {
    const uint2 w = *reinterpret_cast<const uint2 *>(col + t * kRowPad);
    ma = h2max(ma, w.x & 0x7FFF7FFFu);
    mb = h2max(mb, w.y & 0x7FFF7FFFu);
  }
  const uint32_t none = h2_as_u32(__float2half2_rn(32.f));
  uint32_t ia = none, ib = none;
#pragma unroll 8
  for (int t = 0; t < kG; ++t) {
    const uint2 w = *reinterpret_cast<const uint2 *>(col + t * kRowPad);
    ia = h2_first_match(w.x & 0x7FFF7FFFu, ma, float(t), ia);
    ib = h2_first_match(w.y & 0x7FFF7FFFu, mb, float(t), ib);
  }
  const float2 fa = __half22float2(*reinterpret_cast<const __half2 *>(&ia));
  const float2 fb = __half22float2(*reinterpret_cast<const __half2 *>(&ib));
  KeyOutliers o;
  o.row[0] = static_cast<int>(fa.x);
  o.row[1] = static_cast<int>(fa.y);
  o.row[2] = static_cast<int>(fb.x);
  o.row[3] = static_cast<int>(fb.y);
  uint32_t e[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint16_t *x = reinterpret_cast<uint16_t *>(col + o.row[c] * kRowPad) + c;
    e[c] = static_cast<uint32_t>(*x) | (static_cast<uint32_t>(o.row[c]) << 16);
    const int nb = o.row[c] < kG - 1 ? o.row[c] + 1 : o.row[c] - 1;
    *x = reinterpret_cast<const uint16_t *>(col + nb * kRowPad)[c];
  }
  if (blk) reinterpret_cast<uint4 *>(blk + off_ksp(bits))[lane] = make_uint4(e[0], e[1], e[2], e[3]);
  return o;
}

struct ValOutliers {
  int ch[2];     // channel (0 .. 127) of the outlier of rows a, b of this lane
  bool own[2];   // whether this lane's channel half holds it
};

// Lane (p, hf) of value_tile: rows a = 2p + j and b = 2p + 1 - j, channels
// 64 hf .. 64 hf + 63; the other channel half is lane L ^ 16's, whose
// channels come later in slice order (it wins only a strictly larger
// magnitude).
__device__ __forceinline__ ValOutliers value_outliers_tile(uint8_t *tile, uint8_t *blk, int bits, int lane) {
  const int p = lane & 15, hf = lane >> 4, j = (p >> 2) & 1;
  const int rows[2] = {2 * p + j, 2 * p + 1 - j};
  const uint32_t none = h2_as_u32(__float2half2_rn(32.f));
  ValOutliers o;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    uint8_t *row = tile + rows[r] * kRowPad + 128 * hf;
    uint32_t m2 = 0u;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 w = reinterpret_cast<const uint4 *>(row)[i];
      m2 = h2max(h2max(m2, w.x & 0x7FFF7FFFu), h2max(w.y & 0x7FFF7FFFu, h2max(w.z & 0x7FFF7FFFu, w.w & 0x7FFF7FFFu)));
    }
    const float2 mf = __half22float2(*reinterpret_cast<const __half2 *>(&m2));
    const float m = fmaxf(mf.x, mf.y);  // this half's largest magnitude
    const uint32_t mh = h2_as_u32(__float2half2_rn(m));
    // first word whose even (low) and whose odd (high) channel matches
    uint32_t iw = none;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint4 w = reinterpret_cast<const uint4 *>(row)[i];
      iw = h2_first_match(w.x & 0x7FFF7FFFu, mh, float(4 * i), iw);
      iw = h2_first_match(w.y & 0x7FFF7FFFu, mh, float(4 * i + 1), iw);
      iw = h2_first_match(w.z & 0x7FFF7FFFu, mh, float(4 * i + 2), iw);
      iw = h2_first_match(w.w & 0x7FFF7FFFu, mh, float(4 * i + 3), iw);
    }
    const float2 wf = __half22float2(*reinterpret_cast<const __half2 *>(&iw));
    const int c_in = min(2 * static_cast<int>(wf.x), 2 * static_cast<int>(wf.y) + 1);  // channel within the half
    const float om = __shfl_xor_sync(0xffffffffu, m, 16);
    o.own[r] = hf == 0 ? m >= om : m > om;
    o.ch[r] = 64 * hf + c_in;
    if (o.own[r]) {
      uint16_t *x = reinterpret_cast<uint16_t *>(row) + c_in;
      if (blk)
        reinterpret_cast<uint32_t *>(blk + off_vsp(bits))[rows[r]] =
            static_cast<uint32_t>(*x) | (static_cast<uint32_t>(64 * hf + c_in) << 16);
      *x = reinterpret_cast<const uint16_t *>(row)[c_in < 63 ? c_in + 1 : c_in - 1];
    }
  }
  return o;
}

// ---------------------------------------------------------------- key tile
//
// Lane L: channels 4L .. 4L+3, i.e. k-tile kt = L / 4, channel octet j =
// (L / 2) % 2 and lane columns qA = 2 (L % 2) (channels 4L, 4L+1) and qB = qA
// + 1 (4L+2, 4L+3); fp16 pair A of token t holds channels 4L, 4L+1 (fields
// e = 0, 1), pair B channels 4L+2, 4L+3.  Word (kt, hw) of lane 4g + q holds
// tokens 8 (hw NU + u) + g at bits 16e + 8j + b u: this lane's half of it,
// OR-ed with lane L ^ 2's (the other octet), is stored by the lane whose
// octet j = g / 4.  The loops stay rolled and re-read the tile from shared
// memory: fully unrolled, the key and value code no longer fit the
// instruction cache.
template <int BITS, bool SP>
__device__ __forceinline__ void key_tile(uint8_t *tile, uint8_t *blk, int lane, const KeyOutliers &ko) {
  constexpr int NU = 8 / BITS, WH = 4 / NU;
  const float levels = float((1 << BITS) - 1);
  const int kt = lane >> 2, j = (lane >> 1) & 1, q0 = 2 * (lane & 1);
  const uint8_t *col = tile + 8 * lane;  // this lane's 8 bytes of token row t at col + t * kRowPad
  uint32_t mnA, mxA, mnB, mxB;
  {
    uint32_t an[4], ax[4], bn[4], bx[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 w = *reinterpret_cast<const uint2 *>(col + i * kRowPad);
      an[i] = ax[i] = w.x;
      bn[i] = bx[i] = w.y;
    }
#pragma unroll 2
    for (int t = 4; t < kG; t += 4) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint2 w = *reinterpret_cast<const uint2 *>(col + (t + i) * kRowPad);
        an[i] = h2min(an[i], w.x);
        ax[i] = h2max(ax[i], w.x);
        bn[i] = h2min(bn[i], w.y);
        bx[i] = h2max(bx[i], w.y);
      }
    }
    mnA = h2min(h2min(an[0], an[1]), h2min(an[2], an[3]));
    mxA = h2max(h2max(ax[0], ax[1]), h2max(ax[2], ax[3]));
    mnB = h2min(h2min(bn[0], bn[1]), h2min(bn[2], bn[3]));
    mxB = h2max(h2max(bx[0], bx[1]), h2max(bx[2], bx[3]));
  }
  PairQ qa, qb;
  {
    const float2 la = h2_to_f2_pos0(mnA), ha = h2_to_f2_pos0(mxA), lb = h2_to_f2_pos0(mnB), hb = h2_to_f2_pos0(mxB);
    qa = pair_q(la.x, ha.x, la.y, ha.y, levels);
    qb = pair_q(lb.x, hb.x, lb.y, hb.y, levels);
  }
  if (blk) {
    reinterpret_cast<float4 *>(blk + off_ks(BITS))[lane] = make_float4(qa.sc0, qa.sc1, qb.sc0, qb.sc1);
    reinterpret_cast<float4 *>(blk + off_km(BITS))[lane] = make_float4(qa.lo0, qa.lo1, qb.lo0, qb.lo1);
  }
  if constexpr (SP) {  // each outlier becomes its channel's min: code 0
    const float lo4[4] = {qa.lo0, qa.lo1, qb.lo0, qb.lo1};
#pragma unroll
    for (int c = 0; c < 4; ++c)
      reinterpret_cast<__half *>(tile + 8 * lane + ko.row[c] * kRowPad)[c] = __float2half_rn(lo4[c]);
  }
  float sc[NU];
  int pos[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    pos[u] = 8 * j + BITS * u;
    sc[u] = __int_as_float((127 + pos[u]) << 23);
  }
#pragma unroll 2
  for (int wg = 0; wg < 8 * WH; ++wg) {  // (hw, g)
    const int hw = wg >> 3, g = wg & 7;
    uint32_t va[NU], vb[NU];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const uint2 w = *reinterpret_cast<const uint2 *>(col + (8 * (hw * NU + u) + g) * kRowPad);
      va[u] = w.x;
      vb[u] = w.y;
    }
    bool na, nb;
    uint32_t pa = pack_pairs<NU>(va, qa.rcp, qa.c, sc, qa.thr, na);
    uint32_t pb = pack_pairs<NU>(vb, qb.rcp, qb.c, sc, qb.thr, nb);
    if (__any_sync(0xffffffffu, na || nb)) {
      if (na) pa = pack_pairs_exact<BITS, NU>(va, qa.lo0, qa.sc0, qa.lo1, qa.sc1, pos);
      if (nb) pb = pack_pairs_exact<BITS, NU>(vb, qb.lo0, qb.sc0, qb.lo1, qb.sc1, pos);
    }
    pa |= __shfl_xor_sync(0xffffffffu, pa, 2);
    pb |= __shfl_xor_sync(0xffffffffu, pb, 2);
    if ((g >> 2) == j && blk) {
      uint8_t *codes = blk + off_kc(BITS);
      const int w = kt * WH + hw;
      *reinterpret_cast<uint32_t *>(codes + word_offset(w, 4 * g + q0)) = pa;
      *reinterpret_cast<uint32_t *>(codes + word_offset(w, 4 * g + q0 + 1)) = pb;
    }
  }
}

// ------------------------------------------------------- rotation pre-pass
//
// Walsh-Hadamard rotation of every token row of a tile in place, fp16(H x /
// 128) ("2-Bit KV Cache Quantization: Memory You Save, Recall You Risk",
// "Method map: three ways to shrink the cache"; H the Sylvester matrix):
// the fast transform in fp32 with strides 1, 2, ..., 64 in that order, one
// IEEE add or subtract per butterfly, the exact scale 1/128 and one fp16
// rounding, before the tile is quantized.  Four lanes share a row, lane r +
// 8 q holding channels 32 q .. 32 q + 31 of row r of each pass of 8 rows:
// strides 1 to 16 are butterflies inside a lane, strides 32 and 64 pair lane
// L with L ^ 8 and L ^ 16.  (A quarter warp reads 8 rows at one offset, so
// the 272-byte row padding keeps the reads and writes conflict free.)
__device__ __forceinline__ void rotate_tile(uint8_t *tile, int lane) {
  const int r = lane & 7, q = lane >> 3;
#pragma unroll 1
  for (int pass = 0; pass < kG / 8; ++pass) {
    uint4 *p = reinterpret_cast<uint4 *>(tile + (8 * pass + r) * kRowPad + 64 * q);
    float f[32];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 w = p[k];
      const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&wv[i]));
        f[8 * k + 2 * i] = t.x;
        f[8 * k + 2 * i + 1] = t.y;
      }
    }
#pragma unroll
    for (int st = 1; st < 32; st <<= 1)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (!(i & st)) {
          const float a = f[i], b = f[i + st];
          f[i] = __fadd_rn(a, b);
          f[i + st] = __fsub_rn(a, b);
        }
#pragma unroll
    for (int m = 8; m <= 16; m <<= 1) {
      const bool upper = (lane & m) != 0;  // this lane holds the b of each butterfly
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, f[i], m);
        f[i] = upper ? __fsub_rn(o, f[i]) : __fadd_rn(f[i], o);
      }
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t wv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        wv[i] = h2_as_u32(__floats2half2_rn(f[8 * k + 2 * i] * 0.0078125f, f[8 * k + 2 * i + 1] * 0.0078125f));
      p[k] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
    }
  }
  __syncwarp();  // the rotated rows are read by other lanes next
}

// ------------------------------------------------------ key tile, per token
//
// Keys grouped per token (the ablation of per-channel keys): the tile's
// slices are its 32 tokens, each over the 128 channels.  Lane L still owns
// channels 4L .. 4L+3 of every token and packs them as key_tile does; a
// token's min and max are reduced across the warp (a reduce-scatter leaves
// token t's with lane t, which forms its scale, min and filter constants),
// and the packing loop fetches each token's constants from its lane.

// Codes of NF fp16 pairs into one word as pack_pairs, with the filter
// constants of pair f's slice in (rcp[f], c[f]) (both halves of a pair lie
// in one slice).
template <int NF>
__device__ __forceinline__ uint32_t pack_pairs_tok(const uint32_t (&x)[NF], const float (&rcp)[NF],
                                                   const float (&c)[NF], const float (&sc)[NF], float thr,
                                                   bool &near) {
  const f2x magic = f2_pack(kMagic, kMagic);
  f2x acc = f2_pack(kPackBase, kPackBase);
  float emax = 0.f;
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const float2 xf = __half22float2(*reinterpret_cast<const __half2 *>(&x[f]));
    const f2x y = f2_fma(f2_pack(xf.x, xf.y), f2_pack(rcp[f], rcp[f]), f2_pack(c[f], c[f]));
    const f2x r = f2_sub(f2_add(y, magic), magic);  // rne(y), exact
    const float2 e = f2_unpack(f2_sub(y, r));
    asm("max.abs.f32 %0, %1, %2, %3;" : "=f"(emax) : "f"(emax), "f"(e.x), "f"(e.y));
    acc = f2_fma(r, f2_pack(sc[f], sc[f]), acc);
  }
  near = emax > thr;
  const float2 a = f2_unpack(acc);
  return __byte_perm(__float_as_uint(a.x), __float_as_uint(a.y), 0x5410);
}

// The same word by the IEEE subtract and divide, pair f in slice (lo[f], scl[f]).
template <int BITS, int NF>
__device__ __noinline__ uint32_t pack_pairs_tok_exact(const uint32_t (&x)[NF], const float (&lo)[NF],
                                                      const float (&scl)[NF], const int (&pos)[NF]) {
  uint32_t w = 0;
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const float2 xf = __half22float2(*reinterpret_cast<const __half2 *>(&x[f]));
    w |= exact_code<BITS>(xf.x, lo[f], scl[f]) << pos[f];
    w |= exact_code<BITS>(xf.y, lo[f], scl[f]) << (16 + pos[f]);
  }
  return w;
}

template <int BITS>
__device__ __forceinline__ void key_tile_kpt(const uint8_t *tile, uint8_t *blk, int lane) {
  constexpr int NU = 8 / BITS, WH = 4 / NU;
  const float levels = float((1 << BITS) - 1);
  const int kt = lane >> 2, j = (lane >> 1) & 1, q0 = 2 * (lane & 1);
  const uint8_t *col = tile + 8 * lane;  // this lane's 8 bytes of token row t at col + t * kRowPad
  // (min, -max) of this lane's four channels of every token as an fp16 pair,
  // then the warp's: after the exchanges at distances 16, 8, 4, 2, 1 lane t
  // holds token t's
  uint32_t part[kG];
#pragma unroll
  for (int t = 0; t < kG; ++t) {
    const uint2 w = *reinterpret_cast<const uint2 *>(col + t * kRowPad);
    const uint32_t mn = h2min(w.x, w.y), nmx = h2max(w.x, w.y) ^ 0x80008000u;  // -max: the sign bits
    part[t] = h2min(__byte_perm(mn, nmx, 0x5410), __byte_perm(mn, nmx, 0x7632));
  }
#pragma unroll
  for (int d = kG / 2; d >= 1; d >>= 1) {
    const bool up = lane & d;
#pragma unroll
    for (int i = 0; i < d; ++i) {
      const uint32_t send = up ? part[i] : part[i + d];
      const uint32_t keep = up ? part[i + d] : part[i];
      part[i] = h2min(keep, __shfl_xor_sync(0xffffffffu, send, d));
    }
  }
  const float2 ex = h2_to_f2_pos0(part[0]);  // (min, -max) of token `lane`
  const float lo = ex.x, hi = __fadd_rn(-ex.y, 0.f);
  const float scale = __fdiv_rn(__fsub_rn(hi, lo), levels);
  const SliceQ sq = make_slice(lo, scale, levels);
  if (blk) {
    reinterpret_cast<float *>(blk + off_ks(BITS))[lane] = scale;
    reinterpret_cast<float *>(blk + off_km(BITS, true))[lane] = lo;
  }
  float sc[NU];
  int pos[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    pos[u] = 8 * j + BITS * u;
    sc[u] = __int_as_float((127 + pos[u]) << 23);
  }
#pragma unroll 2
  for (int wg = 0; wg < 8 * WH; ++wg) {  // (hw, g)
    const int hw = wg >> 3, g = wg & 7;
    uint32_t va[NU], vb[NU];
    float rc[NU], cc[NU];
    float tol = 0.f;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int tok = 8 * (hw * NU + u) + g;
      const uint2 w = *reinterpret_cast<const uint2 *>(col + tok * kRowPad);
      va[u] = w.x;
      vb[u] = w.y;
      rc[u] = __shfl_sync(0xffffffffu, sq.rcp, tok);
      cc[u] = __shfl_sync(0xffffffffu, sq.c, tok);
      tol = fmaxf(tol, __shfl_sync(0xffffffffu, sq.tol, tok));
    }
    bool na, nb;
    uint32_t pa = pack_pairs_tok<NU>(va, rc, cc, sc, 0.5f - tol, na);
    uint32_t pb = pack_pairs_tok<NU>(vb, rc, cc, sc, 0.5f - tol, nb);
    if (__any_sync(0xffffffffu, na || nb)) {
      float lou[NU], scu[NU];
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        const int tok = 8 * (hw * NU + u) + g;
        lou[u] = __shfl_sync(0xffffffffu, lo, tok);
        scu[u] = __shfl_sync(0xffffffffu, scale, tok);
      }
      if (na) pa = pack_pairs_tok_exact<BITS, NU>(va, lou, scu, pos);
      if (nb) pb = pack_pairs_tok_exact<BITS, NU>(vb, lou, scu, pos);
    }
    pa |= __shfl_xor_sync(0xffffffffu, pa, 2);
    pb |= __shfl_xor_sync(0xffffffffu, pb, 2);
    if ((g >> 2) == j && blk) {
      uint8_t *codes = blk + off_kc(BITS);
      const int w = kt * WH + hw;
      *reinterpret_cast<uint32_t *>(codes + word_offset(w, 4 * g + q0)) = pa;
      *reinterpret_cast<uint32_t *>(codes + word_offset(w, 4 * g + q0 + 1)) = pb;
    }
  }
}

// -------------------------------------------------------------- value tile
//
// Lane L: tokens 2p, 2p+1 (p = L % 16) over channels 64 hf .. 64 hf + 63
// (hf = L / 16).  Token octet j = (p / 4) % 2, lane column q = p % 4 and
// k-tile kt = p / 8 of the layout; word (2P + kt) WH + hw of lane 4g + q
// holds channels 32P + 8 (hw NU + u) + g at bits 16e + 8j + b u, e the token
// parity; lane L ^ 4 holds the other token octet.  The two rows are read in
// the order (2p + j, 2p + 1 - j), which spreads each quarter warp's 16-byte
// reads over the eight bank groups; the byte permutes that pair a channel's
// two tokens undo the order.
template <int BITS, bool KPT, bool SP>
__device__ __forceinline__ void value_tile(uint8_t *tile, uint8_t *blk, int lane, const ValOutliers &vo) {
  constexpr int NU = 8 / BITS, WH = 4 / NU;
  const float levels = float((1 << BITS) - 1);
  const int p = lane & 15, hf = lane >> 4;
  const int j = (p >> 2) & 1, q = p & 3, kt = p >> 3;
  const uint8_t *rowa = tile + (2 * p + j) * kRowPad + 128 * hf;
  const uint8_t *rowb = tile + (2 * p + 1 - j) * kRowPad + 128 * hf;
  const uint32_t lo_sel = j ? 0x1054u : 0x5410u, hi_sel = j ? 0x3276u : 0x7632u;
  // (token 2p, token 2p+1) min and max over the 128 channels
  uint32_t mn2, mx2;
  {
    uint32_t an[4], ax[4], bn[4], bx[4];
    {
      const uint4 a = *reinterpret_cast<const uint4 *>(rowa), b = *reinterpret_cast<const uint4 *>(rowb);
      an[0] = ax[0] = a.x; an[1] = ax[1] = a.y; an[2] = ax[2] = a.z; an[3] = ax[3] = a.w;
      bn[0] = bx[0] = b.x; bn[1] = bx[1] = b.y; bn[2] = bx[2] = b.z; bn[3] = bx[3] = b.w;
    }
#pragma unroll 7
    for (int i = 1; i < 8; ++i) {
      const uint4 a = *reinterpret_cast<const uint4 *>(rowa + 16 * i);
      const uint4 b = *reinterpret_cast<const uint4 *>(rowb + 16 * i);
      const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        an[k] = h2min(an[k], av[k]);
        ax[k] = h2max(ax[k], av[k]);
        bn[k] = h2min(bn[k], bv[k]);
        bx[k] = h2max(bx[k], bv[k]);
      }
    }
    const uint32_t amn = h2min(h2min(an[0], an[1]), h2min(an[2], an[3]));
    const uint32_t amx = h2max(h2max(ax[0], ax[1]), h2max(ax[2], ax[3]));
    const uint32_t bmn = h2min(h2min(bn[0], bn[1]), h2min(bn[2], bn[3]));
    const uint32_t bmx = h2max(h2max(bx[0], bx[1]), h2max(bx[2], bx[3]));
    // (row a, row b) of the low halves and of the high halves, then their
    // min: one pair per token; j = 1 swaps the rows back to (2p, 2p + 1)
    mn2 = h2min(__byte_perm(amn, bmn, lo_sel), __byte_perm(amn, bmn, hi_sel));
    mx2 = h2max(__byte_perm(amx, bmx, lo_sel), __byte_perm(amx, bmx, hi_sel));
    mn2 = h2min(mn2, __shfl_xor_sync(0xffffffffu, mn2, 16));  // the other channel half
    mx2 = h2max(mx2, __shfl_xor_sync(0xffffffffu, mx2, 16));
  }
  PairQ pq;
  {
    const float2 lo = h2_to_f2_pos0(mn2), hi = h2_to_f2_pos0(mx2);
    pq = pair_q(lo.x, hi.x, lo.y, hi.y, levels);
  }
  if (hf == 0 && blk) {
    reinterpret_cast<float2 *>(blk + off_vs(BITS, KPT))[p] = make_float2(pq.sc0, pq.sc1);
    reinterpret_cast<float2 *>(blk + off_vm(BITS, KPT))[p] = make_float2(pq.lo0, pq.lo1);
  }
  if constexpr (SP) {  // each outlier this lane holds becomes its token's min: code 0
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int tok = r == 0 ? 2 * p + j : 2 * p + 1 - j;
      if (vo.own[r])
        reinterpret_cast<__half *>(tile + tok * kRowPad)[vo.ch[r]] = __float2half_rn(tok == 2 * p ? pq.lo0 : pq.lo1);
    }
  }
  float sc[NU];
  int pos[NU];
#pragma unroll
  for (int u = 0; u < NU; ++u) {
    pos[u] = 8 * j + BITS * u;
    sc[u] = __int_as_float((127 + pos[u]) << 23);
  }
  // words of channel block (Pl, hw): channel 64 hf + 32 Pl + 8 (hw NU + u) +
  // g sits in pair m = g / 2 of chunk i = 4 Pl + hw NU + u, low half for even g
#pragma unroll 1
  for (int ph = 0; ph < 2 * WH; ++ph) {  // (Pl, hw)
    const int Pl = ph / WH, hw = ph % WH;
    uint32_t xa[NU][4], xb[NU][4];
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int i = 4 * Pl + hw * NU + u;
      const uint4 a = *reinterpret_cast<const uint4 *>(rowa + 16 * i);
      const uint4 b = *reinterpret_cast<const uint4 *>(rowb + 16 * i);
      xa[u][0] = a.x; xa[u][1] = a.y; xa[u][2] = a.z; xa[u][3] = a.w;
      xb[u][0] = b.x; xb[u][1] = b.y; xb[u][2] = b.z; xb[u][3] = b.w;
    }
    const int w = (2 * (2 * hf + Pl) + kt) * WH + hw;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      uint32_t ve[NU], vo[NU];
#pragma unroll
      for (int u = 0; u < NU; ++u) {
        ve[u] = __byte_perm(xa[u][m], xb[u][m], lo_sel);  // channel 2m (+ base): (token 2p, token 2p + 1)
        vo[u] = __byte_perm(xa[u][m], xb[u][m], hi_sel);  // channel 2m + 1
      }
      bool ne, no;
      uint32_t pe = pack_pairs<NU>(ve, pq.rcp, pq.c, sc, pq.thr, ne);
      uint32_t po = pack_pairs<NU>(vo, pq.rcp, pq.c, sc, pq.thr, no);
      if (__any_sync(0xffffffffu, ne || no)) {
        if (ne) pe = pack_pairs_exact<BITS, NU>(ve, pq.lo0, pq.sc0, pq.lo1, pq.sc1, pos);
        if (no) po = pack_pairs_exact<BITS, NU>(vo, pq.lo0, pq.sc0, pq.lo1, pq.sc1, pos);
      }
      pe |= __shfl_xor_sync(0xffffffffu, pe, 4);
      po |= __shfl_xor_sync(0xffffffffu, po, 4);
      // rows g = 2m, 2m + 1 are stored by the lane of octet j = g / 4
      if ((m >> 1) == j && blk) {
        uint8_t *codes = blk + off_vc(BITS);
        *reinterpret_cast<uint32_t *>(codes + word_offset(w, 4 * (2 * m) + q)) = pe;
        *reinterpret_cast<uint32_t *>(codes + word_offset(w, 4 * (2 * m + 1) + q)) = po;
      }
    }
  }
}

// ------------------------------------------------------------------ kernel

// Persistent CTAs of TileShape<BITS>::WARPS independent warps (one CTA per SM).  Warp gw of
// NW takes tiles [gw U / NW, (gw + 1) U / NW) of the line of U = 2 x (groups
// flushed) tiles, ordered (sequence, KV head, group, keys / values).
template <int BITS, bool KPT, bool ROT, bool SP>
__global__ void __launch_bounds__(TileShape<BITS>::WARPS * 32, 1)
    quant_tiles_kernel(Geo geo, const __half *__restrict__ k_new, const __half *__restrict__ v_new,
                       const int *__restrict__ new_len, int max_new) {
  using TS = TileSmem;
  constexpr int NS = TS::NS, BB = block_bytes(BITS, KPT, SP);
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint8_t *base = smem + warp * TS::BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(base + TS::BAR);
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncwarp();
  constexpr int kWarps = TileShape<BITS>::WARPS;
  const int NW = gridDim.x * kWarps, gw = blockIdx.x * kWarps + warp;
  const int S = geo.S, H = geo.H;

  // ---- the line: U tiles in all; the first tile of this warp's range
  long long tot = 0;
  for (int s = lane; s < S; s += 32) tot += seq_flush(geo, new_len, max_new, s).ng;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
  const long long U = 2 * tot * H;
  const long long ua = gw * U / NW, ub = (gw + 1) * U / NW;
  if (ua >= ub) return;
  TilePos cp;
  {
    long long run = 0;  // tiles of the sequences before chunk c
    cp.s = S;
    for (int c = 0; c < S; c += 32) {
      const long long v = c + lane < S ? 2LL * H * seq_flush(geo, new_len, max_new, c + lane).ng : 0;
      long long incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
      }
      const unsigned m = __ballot_sync(0xffffffffu, c + lane < S && run + incl > ua);
      if (m) {
        const int idx = __ffs(m) - 1;
        cp.s = c + idx;
        const long long local = ua - (run + __shfl_sync(0xffffffffu, incl - v, idx));
        cp.f = seq_flush(geo, new_len, max_new, cp.s);
        const long long per_head = 2LL * cp.f.ng;
        cp.h = static_cast<int>(local / per_head);
        const int rem = static_cast<int>(local - cp.h * per_head);
        cp.g = rem >> 1;
        cp.kind = rem & 1;
        break;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
  }

  // ---- fetch: lane r copies token row r of the tile into the ring slot
  TilePos fp = cp;
  long long fu = ua;  // next tile to fetch
  uint32_t fseq = 0, cseq = 0;
  auto top_up = [&]() {
    while (fu < ub && fseq - cseq < static_cast<uint32_t>(NS)) {
      const uint32_t slot = fseq % NS;
      const size_t sh = static_cast<size_t>(fp.s) * H + fp.h;
      const int i = fp.f.Lq0 + kG * fp.g + lane;  // stream index of row `lane`
      const bool from_window = i < fp.f.n0;
      const __half *src = from_window
                              ? (fp.kind ? geo.v_res : geo.k_res) + (sh * geo.R + (i - fp.f.Lq0)) * kD
                              : (fp.kind ? v_new : k_new) + (sh * max_new + (i + geo.ns - fp.f.L0)) * kD;
      fence_proxy_async();  // this lane's reads of the slot, before the copy that overwrites it
      if (lane == 0) mbar_arrive_expect_tx(&full[slot], kG * kD * 2);
      __syncwarp();
      // (a skipped row leaves the tile's wait to give up)
      if (KVQ_IN_BOUNDS(geo.status, from_window ? i - fp.f.Lq0 : i + geo.ns - fp.f.L0, from_window ? geo.R : max_new))
        bulk_g2s(base + slot * kSlotBytes + lane * kRowPad, src, kD * 2, &full[slot]);
      ++fseq;
      ++fu;
      if (fu < ub) next_tile(fp, geo, new_len, max_new);
    }
  };
  top_up();

  // ---- consume
  bool ok = true;
  for (long long u = ua; u < ub; ++u) {
    const uint32_t slot = cseq % NS;
    if (!mbar_wait_bounded(&full[slot], (cseq / NS) & 1)) {
      ok = false;
      break;
    }
    uint8_t *tile = base + slot * kSlotBytes;
    uint8_t *blk = KVQ_IN_BOUNDS(geo.status, cp.f.Lq0 / kG + cp.g, geo.max_groups)
                       ? group_block(geo, cp.s, cp.h, cp.f.Lq0 / kG + cp.g, BB)  // null: a bad table entry
                       : nullptr;
    if (!blk && cp.kind == 0 && lane == 0) set_status(geo.status, KVQ_STATUS_BAD_BLOCK);
    if (ROT) rotate_tile(tile, lane);
    if (cp.kind == 0) {
      KeyOutliers ko = {};
      if constexpr (SP) ko = key_outliers_tile(tile, blk, BITS, lane);
      if constexpr (KPT)
        key_tile_kpt<BITS>(tile, blk, lane);
      else
        key_tile<BITS, SP>(tile, blk, lane, ko);
    } else {
      ValOutliers vo = {};
      if constexpr (SP) vo = value_outliers_tile(tile, blk, BITS, lane);
      value_tile<BITS, KPT, SP>(tile, blk, lane, vo);
    }
    __syncwarp();  // every lane's reads of the slot are done before it is refilled
    ++cseq;
    top_up();
    if (u + 1 < ub) next_tile(cp, geo, new_len, max_new);
  }
  if (!ok) {
    if (lane == 0) set_status(geo.status, KVQ_STATUS_TIMEOUT);
    for (; cseq < fseq; ++cseq) mbar_wait_bounded(&full[cseq % NS], (cseq / NS) & 1);
  }
}

// One CTA per SM (the attribute is set once per instantiation and device).
template <int BITS, bool KPT, bool ROT, bool SP>
static cudaError_t launch_tiles_t(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                                  int max_new, cudaStream_t stream) {
  using TS = TileSmem;
  constexpr int kWarps = TileShape<BITS>::WARPS;
  static int sms[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int n_sm = dev < 64 ? sms[dev] : 0;
  if (n_sm == 0) {
    if ((e = cudaFuncSetAttribute(quant_tiles_kernel<BITS, KPT, ROT, SP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kWarps * TS::BYTES)) != cudaSuccess)
      return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if (dev < 64) sms[dev] = n_sm;
  }
  quant_tiles_kernel<BITS, KPT, ROT, SP><<<n_sm, kWarps * 32, kWarps * TS::BYTES, stream>>>(geo, k_new, v_new,
                                                                                       new_len, max_new);
  return cudaGetLastError();
}

template <int BITS>
static cudaError_t launch_tiles_b(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                                  int max_new, cudaStream_t stream) {
  // (outlier entries come with neither per-token keys here nor the rotation)
  if (geo.sparse) return launch_tiles_t<BITS, false, false, true>(geo, k_new, v_new, new_len, max_new, stream);
  if (geo.kpt)
    return geo.rot ? launch_tiles_t<BITS, true, true, false>(geo, k_new, v_new, new_len, max_new, stream)
                   : launch_tiles_t<BITS, true, false, false>(geo, k_new, v_new, new_len, max_new, stream);
  return geo.rot ? launch_tiles_t<BITS, false, true, false>(geo, k_new, v_new, new_len, max_new, stream)
                 : launch_tiles_t<BITS, false, false, false>(geo, k_new, v_new, new_len, max_new, stream);
}

bool flush_tiles_serves(const Geo &geo) {
  return !(geo.sparse && (geo.kpt || geo.rot)) && geo.S <= kTileFlushMaxSeqs;
}

cudaError_t launch_flush_tiles(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                               int max_new, cudaStream_t stream) {
  return geo.bits == 2 ? launch_tiles_b<2>(geo, k_new, v_new, new_len, max_new, stream)
                       : launch_tiles_b<4>(geo, k_new, v_new, new_len, max_new, stream);
}

}  // namespace kvq
