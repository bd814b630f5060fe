// Split-K decode attention read directly from the quantized cache.
//
// Source: "KV cache quantization", "Keys are harder than values" (the
// grouped part and the full-precision part of the cache are combined when
// computing attention scores; keys stored before RoPE are rotated after
// dequantization); "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV
// Cache", second and third paragraphs (what the groups and the window hold).
//
// The work of every (sequence, KV head) pair -- 32-token passes over its
// fp16 sink + window tokens, then its packed groups -- is laid out as one
// line of units, and each warp of a single wave of persistent CTAs takes an
// equal, contiguous range of that line (stream-K): ranges cross pair
// boundaries, so the split of each pair's token axis follows from the load
// balance rather than from a fixed chunk size.  A warp streams its groups
// through a small ring of shared-memory slots filled by one-dimensional bulk
// copies completing on per-slot mbarriers, fetching across pair boundaries
// so the next pair's first groups are in flight while the current one ends.
// It leaves a partial (max, sum, unnormalized output) per query head for
// each pair it touches; the warp that completes a pair's partial count
// merges them with a log-sum-exp and writes the fp16 output.  No CTA-wide
// synchronization happens after start-up.

// Scores over a group use mma.sync m16n8k16 with the 32 tokens as M, the
// channels as K and the query as N: the A operand comes straight from the
// packed words (an AND mask leaves each code as an fp16 subnormal
// code * 2^(b*u - 24)), and the B operand is q_d * scale_d split into an fp16
// high part and an fp16 low part (columns 2h and 2h+1 for query head h), so
// the fp32 accumulator sees q * scale to about 22 bits.  The per-channel
// minimum enters through beta = sum_d q_d * min_d.  The value side is the
// same with channels as M and tokens as K: o_d = sum_t (p_t scale_t) c_td +
// sum_t p_t min_t.  B columns of query heads that do not exist (a KV head
// with fewer than four query heads) carry arbitrary finite values; their
// accumulator columns are never read.  With keys stored pre-RoPE the scores
// are instead formed per token on the CUDA cores (dequantize, rotate, dot),
// because the rotation differs per token.
#pragma once

#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kRopeOffStride = 65;     // padded row of the in-group rotation table
constexpr unsigned kFull = 0xffffffffu;

struct PlanHeader;

struct DecodeArgs {
  Geo geo;
  int Hq;
  const __half *q;          // [S][Hq][D]
  __half *out;              // [S][Hq][D]
  float zscale;             // softmax scale * log2(e)
  float *part_o;            // [slots][GQ][D] unnormalized partial outputs
  float2 *part_ml;          // [slots][GQ] (max, sum) in log2 units
  int *counters;            // [S][Hkv] partials finished: zero on entry, left zero on exit
  long long *base;          // [S + 1] first work unit of each sequence (plan kernel), or
                            // null when the decode kernel plans by itself
  PlanHeader *plan;         // total work units (plan kernel)
  int nw;                   // warps sharing the work
  size_t pass_slot0;        // first partial slot of the window passes
  int tail_passes;          // window/sink passes per (sequence, KV head) at most, 32 tokens each
  int max_len;              // host bound on seq_len the plan was sized for
  long long wait_limit;     // SM cycles a ring wait may last before it gives up
  int wait_before_fetch;    // test aid: first ring wait before any copy is issued
  size_t n_slots;           // partial slots in the workspace (bounds checks)
  int n_base;               // rows of rope_base (bounds checks)
  const float2 *rope_base;  // [n_base][64]: cos, sin of (num_sink + 32 r) * omega_i
  const float2 *rope_off;   // [32][64]: cos, sin of delta * omega_i
};

// Shared memory of one warp: a ring of NS group blocks, one mbarrier per
// slot, the query of the current pair (fp32, GQ heads), whose space the
// score operand staging reuses once the query sits in registers, (keys
// stored pre-RoPE) the per-group channel-pair coefficients, and
// (dense-and-sparse blocks) the outlier corrections: score corrections of
// two groups [2][GQ][32] and value corrections [GQ][128], fp32.
// Ring slots (group blocks in flight) per warp.
#ifndef KVQ_DECODE_RING_2BIT
#define KVQ_DECODE_RING_2BIT 4
#endif
#ifndef KVQ_DECODE_RING_4BIT
#define KVQ_DECODE_RING_4BIT 2
#endif

// Pre-RoPE keys at 2-bit with one query head per KV head score through a
// per-group table of each channel pair's 16 possible (X, Y) values: rows of
// 16 float2 padded to kTabStride bytes (the padding keeps the table's
// 16-byte stores and its reads conflict free).
constexpr int kTabStride = 136;

template <int BITS, int GQ, bool ROPE, bool KPT, bool SP = false>
struct WarpSmem {
  static constexpr bool TAB = ROPE && BITS == 2 && GQ == 1 && !KPT;
  static constexpr int BB = block_bytes(BITS, KPT, SP);
  static constexpr int NS = TAB ? 2 : ROPE ? (BITS == 2 ? 3 : 2)
                            : SP ? ((BITS == 2 && GQ != 2) ? 3 : 2)
                                 : (BITS == 2 ? KVQ_DECODE_RING_2BIT : KVQ_DECODE_RING_4BIT);
  static constexpr int BAR_OFF = NS * BB;
  static constexpr int Q_OFF = (BAR_OFF + NS * 8 + 15) / 16 * 16;
  static constexpr int COEF_OFF = Q_OFF + GQ * kD * 4;            // [GQ][64] float4, then [GQ][64] float2
  static constexpr int SP_OFF = COEF_OFF + (TAB ? 64 * kTabStride : ROPE ? GQ * 64 * 24 : 0);
  static constexpr int SP_FLOATS = SP ? GQ * (2 * kG + kD) : 0;
  static constexpr int BYTES = (SP_OFF + SP_FLOATS * 4 + 127) / 128 * 128;
  static_assert(BB % 16 == 0, "bulk copies need 16-byte multiples");
};

// Post-scale of a key score row tau (0..3 = token 8*tau + g) and of a value
// output row (channel 16*mt + 8*h + g): undo the code << (b*u) * 2^-24.
template <int BITS>
static __device__ __forceinline__ float key_row_scale(int tau) {
  const int u = BITS == 2 ? tau : (tau & 1);
  return __int_as_float((127 + 24 - BITS * u) << 23);
}
template <int BITS>
static __device__ __forceinline__ float val_row_scale(int mt, int hh) {
  const int u = BITS == 2 ? 2 * (mt & 1) + hh : hh;
  return __int_as_float((127 + 24 - BITS * u) << 23);
}

// fp16 pair of (x0, x1) when lo_sel == 0, or of the rounding remainder
// (x - fp16(x)) when lo_sel == 1: the high and low parts of a two-term split.
static __device__ __forceinline__ uint32_t split_part(float x0, float x1, float lo_sel) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 f = __half22float2(h);
  return h2_as_u32(__floats2half2_rn(fmaf(-lo_sel, f.x, x0), fmaf(-lo_sel, f.y, x1)));
}

// Query side of the score mma.  Per group, lane L forms q_d * scale_d for
// the four channels 16 kt + 8 j + 2 c + {0, 1} (kt = L % 8, c = L / 8,
// j = 0, 1) of every query head, splits each product into an fp16 high part
// and the fp16 rounding remainder, and stages both in shared memory in the
// order of the B fragments: row (2 head + part) * 4 + c holds, for k-tiles
// 0..7 and j = 0, 1, the channel pair (kt, j, c), 64 bytes per row with the
// 16-byte chunks XOR-swizzled by (row / 2) % 4 so that neither the 8-byte
// stores nor the 16-byte fragment loads meet a bank conflict.  Lane (g, q)
// then loads B column g (query head g / 2, high part for even g, low part for
// odd g; columns of heads that do not exist repeat the last head) with four
// 16-byte loads.  beta = sum_d q_d min_d of head q is reduced across the warp.
// Both use the normalized query q / 2^e (e per head, from frexp of its
// largest |q_d|), so the products stay inside the fp16 range; qscale undoes
// it together with the softmax scale.
template <int GQ>
struct QkOperand {
  float qv[GQ][4];  // channels c0, c0 + 1, c0 + 8, c0 + 9 of each head
  float qscale;     // zscale * 2^e of head (lane & 3)

  static __device__ __forceinline__ int chan0(int lane) { return 16 * (lane & 7) + 2 * (lane >> 3); }
  static __device__ __forceinline__ int swz(int row, int chunk) { return row * 16 + 4 * (chunk ^ ((row >> 1) & 3)); }

  __device__ __forceinline__ void init(const float *q_s, int lane, float zscale) {
    const int c0 = chan0(lane);
    int ex_mine = 0;
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      const float2 a = *reinterpret_cast<const float2 *>(q_s + h * kD + c0);
      const float2 b = *reinterpret_cast<const float2 *>(q_s + h * kD + c0 + 8);
      qv[h][0] = a.x;
      qv[h][1] = a.y;
      qv[h][2] = b.x;
      qv[h][3] = b.y;
      float amax = fmaxf(fmaxf(fabsf(a.x), fabsf(a.y)), fmaxf(fabsf(b.x), fabsf(b.y)));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
      int ex;
      frexpf(amax, &ex);  // |q / 2^ex| < 1
#pragma unroll
      for (int i = 0; i < 4; ++i) qv[h][i] = ldexpf(qv[h][i], -ex);
      if (h == min(lane & 3, GQ - 1)) ex_mine = ex;
    }
    qscale = ldexpf(zscale, ex_mine);
  }

  // stage: GQ * 512 bytes of this warp's shared memory, 16-byte aligned.
  __device__ __forceinline__ void build(const float *ks, const float *km, uint32_t *stage, int lane,
                                        uint32_t (&bq)[8][2], float &beta) const {
    const int c0 = chan0(lane), kt = lane & 7, c = lane >> 3;
    const float2 s0 = *reinterpret_cast<const float2 *>(ks + c0);
    const float2 s1 = *reinterpret_cast<const float2 *>(ks + c0 + 8);
    const float2 m0 = *reinterpret_cast<const float2 *>(km + c0);
    const float2 m1 = *reinterpret_cast<const float2 *>(km + c0 + 8);
    float bp[GQ];
    __syncwarp();  // earlier reads of the stage (or of the query it aliases) are done
#pragma unroll
    for (int h = 0; h < GQ; ++h) {
      const float x0 = qv[h][0] * s0.x, x1 = qv[h][1] * s0.y, x2 = qv[h][2] * s1.x, x3 = qv[h][3] * s1.y;
      const __half2 h01 = __floats2half2_rn(x0, x1), h23 = __floats2half2_rn(x2, x3);
      const float2 f01 = __half22float2(h01), f23 = __half22float2(h23);
      const __half2 l01 = __floats2half2_rn(x0 - f01.x, x1 - f01.y), l23 = __floats2half2_rn(x2 - f23.x, x3 - f23.y);
      const int rh = (2 * h) * 4 + c, rl = (2 * h + 1) * 4 + c;
      *reinterpret_cast<uint2 *>(stage + swz(rh, kt >> 1) + 2 * (kt & 1)) = make_uint2(h2_as_u32(h01), h2_as_u32(h23));
      *reinterpret_cast<uint2 *>(stage + swz(rl, kt >> 1) + 2 * (kt & 1)) = make_uint2(h2_as_u32(l01), h2_as_u32(l23));
      bp[h] = fmaf(qv[h][0], m0.x, fmaf(qv[h][1], m0.y, fmaf(qv[h][2], m1.x, qv[h][3] * m1.y)));
    }
    __syncwarp();
    {
      const int g = lane >> 2, q = lane & 3;
      const int row = (2 * min(g >> 1, GQ - 1) + (g & 1)) * 4 + q;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 w = *reinterpret_cast<const uint4 *>(stage + swz(row, i));
        bq[2 * i][0] = w.x;
        bq[2 * i][1] = w.y;
        bq[2 * i + 1][0] = w.z;
        bq[2 * i + 1][1] = w.w;
      }
    }
    // beta of every head summed over the warp: halving exchanges leave one
    // head's total per lane group, then lane (g, q) fetches head q's
    if (GQ == 1) {
      float v = bp[0];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      beta = v * qscale;
    } else if (GQ == 2) {
      const bool up = lane & 16;
      float v = (up ? bp[1] : bp[0]) + __shfl_xor_sync(kFull, up ? bp[0] : bp[1], 16);
#pragma unroll
      for (int off = 8; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      beta = __shfl_sync(kFull, v, 16 * min(lane & 3, 1)) * qscale;  // lanes 0..15: head 0, 16..31: head 1
    } else {
      const bool b4 = lane & 16, b3 = lane & 8;
      const float t0 = __shfl_xor_sync(kFull, b4 ? bp[0] : bp[2 % GQ], 16);
      const float t1 = __shfl_xor_sync(kFull, b4 ? bp[1] : bp[3 % GQ], 16);
      const float k0 = (b4 ? bp[2 % GQ] : bp[0]) + t0, k1 = (b4 ? bp[3 % GQ] : bp[1]) + t1;
      float v = (b3 ? k1 : k0) + __shfl_xor_sync(kFull, b3 ? k0 : k1, 8);
#pragma unroll
      for (int off = 4; off > 0; off >>= 1) v += __shfl_xor_sync(kFull, v, off);
      beta = __shfl_sync(kFull, v, 8 * (lane & 3)) * qscale;  // lane 8h holds head h = 2 b4 + b3
    }
  }
};

// o[mt] += A(value codes) * bp for one group: o rows are channels 16mt+g and
// 16mt+8+g, columns 2q / 2q+1 (high / low part of query head q).
template <int BITS>
static __device__ __forceinline__ void pv_mma(const uint8_t *vc, int lane, const uint32_t (&bp)[2][2], float (&o)[8][4]) {
  if (BITS == 2) {
    const uint4 w0 = *reinterpret_cast<const uint4 *>(vc + (0 * 32 + lane) * 16);
    const uint4 w1 = *reinterpret_cast<const uint4 *>(vc + (1 * 32 + lane) * 16);
    const uint32_t vw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int P = 0; P < 4; ++P)
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        const uint32_t wd = vw[2 * P + kt], wd8 = wd >> 8;
        mma16816(o[2 * P], wd & 0x00030003u, wd & 0x000C000Cu, wd8 & 0x00030003u, wd8 & 0x000C000Cu, bp[kt][0],
                 bp[kt][1]);
        mma16816(o[2 * P + 1], wd & 0x00300030u, wd & 0x00C000C0u, wd8 & 0x00300030u, wd8 & 0x00C000C0u,
                 bp[kt][0], bp[kt][1]);
      }
  } else {
    uint32_t vw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = *reinterpret_cast<const uint4 *>(vc + (i * 32 + lane) * 16);
      vw[4 * i] = w.x;
      vw[4 * i + 1] = w.y;
      vw[4 * i + 2] = w.z;
      vw[4 * i + 3] = w.w;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int kt = 0; kt < 2; ++kt) {
        const uint32_t wd = vw[4 * (mt >> 1) + 2 * kt + (mt & 1)], wd8 = wd >> 8;
        mma16816(o[mt], wd & 0x000F000Fu, wd & 0x00F000F0u, wd8 & 0x000F000Fu, wd8 & 0x00F000F0u, bp[kt][0],
                 bp[kt][1]);
      }
  }
}

// Score accumulators of the group's 32 tokens: acc[mt] rows g / g+8 are
// tokens 16mt + g / 16mt + 8 + g, columns 2q / 2q+1 the parts of head q.
template <int BITS>
static __device__ __forceinline__ void qk_mma(const uint8_t *kc, int lane, const uint32_t (&bq)[8][2], float (&acc)[2][4]) {
#pragma unroll
  for (int i = 0; i < 2; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  if (BITS == 2) {
    const uint4 w0 = *reinterpret_cast<const uint4 *>(kc + (0 * 32 + lane) * 16);
    const uint4 w1 = *reinterpret_cast<const uint4 *>(kc + (1 * 32 + lane) * 16);
    const uint32_t kw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int kt = 0; kt < 8; ++kt) {
      const uint32_t wd = kw[kt], wd8 = kw[kt] >> 8;
      mma16816(acc[0], wd & 0x00030003u, wd & 0x000C000Cu, wd8 & 0x00030003u, wd8 & 0x000C000Cu, bq[kt][0],
               bq[kt][1]);
      mma16816(acc[1], wd & 0x00300030u, wd & 0x00C000C0u, wd8 & 0x00300030u, wd8 & 0x00C000C0u, bq[kt][0],
               bq[kt][1]);
    }
  } else {
    uint32_t kw[16];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint4 w = *reinterpret_cast<const uint4 *>(kc + (i * 32 + lane) * 16);
      kw[4 * i] = w.x;
      kw[4 * i + 1] = w.y;
      kw[4 * i + 2] = w.z;
      kw[4 * i + 3] = w.w;
    }
#pragma unroll
    for (int kt = 0; kt < 8; ++kt)
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const uint32_t wd = kw[2 * kt + mt], wd8 = wd >> 8;
        mma16816(acc[mt], wd & 0x000F000Fu, wd & 0x00F000F0u, wd8 & 0x000F000Fu, wd8 & 0x00F000F0u, bq[kt][0],
                 bq[kt][1]);
      }
  }
}

// Token t's packed key word for channel tile kt and lane-column qq (used by
// the pre-RoPE path, one lane per token).
template <int BITS>
static __device__ __forceinline__ uint32_t key_word(const uint8_t *kc, int t, int kt, int qq) {
  constexpr int NU = 8 / BITS;
  const int tau = t >> 3;
  const int w = kt * (4 / NU) + tau / NU;
  const int lane = 4 * (t & 7) + qq;
  return reinterpret_cast<const uint32_t *>(kc)[((w >> 2) * 32 + lane) * 4 + (w & 3)];
}

// ------------------------------------------------------------ work schedule
//
// The decode work of a (sequence, KV head) pair is a run of units: first
// kPassUnits units per 32-token pass over its fp16 sink + window tokens, then
// one unit per packed group.  (A pass costs about kPassUnits groups' time
// however few tokens it holds: its query, key and value loads are
// dependent global round trips.)  Pairs are laid out sequence-major: sequence s
// starts at unit base[s] = Hkv * (units per head of the sequences before
// it), the line holds W units in all.  Each warp derives base[] and W from
// seq_len itself (warp scans), or, for large batches, reads them from a plan
// kernel.  Warp gw of NW takes units [gw W / NW, (gw + 1) W / NW): equal work, contiguous
// across pair boundaries.  A warp leaves one partial result per pair it
// touches (slot gw + pair) plus one per window pass it runs; the warp that
// completes a pair's count merges them.
#ifndef KVQ_PASS_UNITS
#define KVQ_PASS_UNITS 4
#endif
#ifndef KVQ_DECODE_PREFETCH
#define KVQ_DECODE_PREFETCH 1
#endif
// Ring slots a warp fills before its first group arrives; one more per group
// consumed, up to the ring size (0: the whole ring at once).  Every warp
// starts at the same moment, so filling whole rings at once asks HBM for all
// of them together and a warp's first group waits behind the others' later
// ones; a shallow start lets every warp's first groups arrive first.  At
// least 2: the group loop waits on two slots at a time.
#ifndef KVQ_RING_RAMP
#define KVQ_RING_RAMP 2
#endif
static_assert(KVQ_RING_RAMP == 0 || KVQ_RING_RAMP >= 2, "the group loop consumes two slots at a time");
constexpr int kPassUnits = KVQ_PASS_UNITS;
constexpr int kInlinePlanSeqs = 256;  // larger batches use the plan kernel
#ifndef KVQ_MERGE_BATCH
#define KVQ_MERGE_BATCH 8
#endif
constexpr int kMergeBatch = KVQ_MERGE_BATCH;  // partials a merge loads at once (more: in a loop)

struct PlanHeader {
  long long total;  // W
};

// Units per KV head of a sequence of length L (0 when there is nothing to
// attend), and of sequence s.
static __device__ __forceinline__ int len_units(const DecodeArgs &a, int L, Split &spl, int &tp, int &ng) {
  tp = ng = 0;
  spl.nsink = spl.Lq = spl.r = 0;
  if (L <= 0 || L > a.geo.capacity || L > a.max_len) return 0;
  spl = split_len(L, a.geo.ns, a.geo.R);
  ng = spl.Lq / kG;
  tp = (spl.nsink + spl.r + 31) / 32;
  return kPassUnits * tp + ng;
}
static __device__ __forceinline__ int seq_units(const DecodeArgs &a, int s, Split &spl, int &tp, int &ng) {
  return len_units(a, a.geo.seq_len[s], spl, tp, ng);
}

// L2 prefetch of one line (no register, no wait).
static __device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// The warp whose unit range holds unit x.
static __device__ __forceinline__ int owner_warp(long long x, long long W, int NW) {
  return static_cast<int>(((x + 1) * NW - 1) / W);
}

// The warps with a non-empty unit range that intersect [P0, P1): n of them,
// the i-th given by at().  When every range is non-empty (W >= NW) they are
// the owners of the two ends and every warp between.  Otherwise each range
// holds at most one unit, so they are the owners of the units of [P0, P1),
// all distinct; then W < NW <= kMaxDecodeWarps and the owner of a unit takes
// one 32-bit division (scanning the warp ids between the end owners instead
// would cost a division per warp of the launch).
struct Touching {
  int w0, n, p0, W, NW;
  bool by_unit;
  __device__ __forceinline__ int at(int i) const { return by_unit ? ((p0 + i + 1) * NW - 1) / W : w0 + i; }
};
static __device__ __forceinline__ Touching touching_warps(long long P0, long long P1, long long W, int NW) {
  Touching t;
  t.by_unit = W < NW;
  t.NW = NW;
  if (t.by_unit) {
    t.W = static_cast<int>(W);
    t.p0 = static_cast<int>(P0);
    t.w0 = 0;
    t.n = static_cast<int>(P1 - P0);
  } else {
    t.W = t.p0 = 0;
    t.w0 = owner_warp(P0, W, NW);
    t.n = owner_warp(P1 - 1, W, NW) - t.w0 + 1;
  }
  return t;
}

// Scores of one packed group for this lane: z[tau] = log2-domain logit of
// token 8*tau + g for query head q.
template <int BITS, int GQ>
static __device__ __forceinline__ void group_scores(const uint8_t *blk, const QkOperand<GQ> &qo, const float (&kfac)[4],
                                             uint32_t *stage, int lane, float (&z)[4]) {
  uint32_t bq[8][2];
  float beta;
  qo.build(reinterpret_cast<const float *>(blk + off_ks(BITS)), reinterpret_cast<const float *>(blk + off_km(BITS)),
           stage, lane, bq, beta);
  float acc[2][4];
  qk_mma<BITS>(blk + off_kc(BITS), lane, bq, acc);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) z[2 * mt + hh] = fmaf(acc[mt][2 * hh] + acc[mt][2 * hh + 1], kfac[2 * mt + hh], beta);
}

// Scores of one packed group when keys are grouped per token: the B
// fragments hold the query itself split into fp16 high and low parts
// (column 2h and 2h + 1 of head h; the low part is zero for an fp16 query,
// nonzero for a rotated one), built once per (sequence, KV head), and token t's scale s_t
// and min m_t enter as z = s_t (q . c_t) kf + m_t (zscale sum_d q_d).
template <int BITS>
static __device__ __forceinline__ void group_scores_kpt(const uint8_t *blk, const uint32_t (&bq)[8][2],
                                                 const float (&kfac)[4], float zsq, int lane, float (&z)[4]) {
  float acc[2][4];
  qk_mma<BITS>(blk + off_kc(BITS), lane, bq, acc);
  const float *ks = reinterpret_cast<const float *>(blk + off_ks(BITS));
  const float *km = reinterpret_cast<const float *>(blk + off_km(BITS, true));
  const int g = lane >> 2;
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int tau = 2 * mt + hh, t = 8 * tau + g;
      z[tau] = fmaf(acc[mt][2 * hh] + acc[mt][2 * hh + 1], kfac[tau] * ks[t], zsq * km[t]);
    }
}

// Dense-and-sparse blocks, per-channel keys: each lane adds, for its four
// query channels (those of QkOperand), q_d (x_d - min_d) of every head to
// the score correction of the channel's outlier token t_d (zc[h][t]; one
// outlier per channel, several may share a token, hence the shared-memory
// atomics).  The dense part already holds code 0 there, i.e. min_d.
template <int BITS, int GQ>
static __device__ __forceinline__ void key_outliers(const uint8_t *blk, const QkOperand<GQ> &qo, float *zc, int lane) {
  const int c0 = QkOperand<GQ>::chan0(lane);
  const uint32_t *ksp = reinterpret_cast<const uint32_t *>(blk + off_ksp(BITS));
  const float *km = reinterpret_cast<const float *>(blk + off_km(BITS));
  const uint2 e01 = *reinterpret_cast<const uint2 *>(ksp + c0), e89 = *reinterpret_cast<const uint2 *>(ksp + c0 + 8);
  const float2 m01 = *reinterpret_cast<const float2 *>(km + c0), m89 = *reinterpret_cast<const float2 *>(km + c0 + 8);
  const uint32_t e[4] = {e01.x, e01.y, e89.x, e89.y};
  const float m[4] = {m01.x, m01.y, m89.x, m89.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float dx = __half2float(__ushort_as_half(static_cast<unsigned short>(e[i] & 0xFFFFu))) - m[i];
    const int t = static_cast<int>(e[i] >> 16) & (kG - 1);
#pragma unroll
    for (int h = 0; h < GQ; ++h) atomicAdd(zc + h * kG + t, qo.qv[h][i] * dx);
  }
}

// o += values of one group weighted by ps (score layout: token 8*tau + g,
// head q).  The value mma's B column h (h < 4) carries head h's weights
// p_t * scale_t rounded to fp16 and column 4 + h the fp16 rounding
// remainder, so each weight enters to about 22 bits (the two parts of o are
// summed when the partial is written; o columns 2q and 2q+1 of this lane
// are those of B).  One fp16 weight would carry a 2^-12 relative error into
// code * scale, whose size the min can nearly cancel: a value token whose
// range one large entry stretches (|min| >> |x|), or the rotated value sums
// that the Walsh-Hadamard back-transform concentrates into channel 0, would
// then miss the output tolerance.  Values carry the attention output as a
// weighted sum in which the few heavily weighted tokens decide the result
// ("KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache", second
// paragraph), so their weights must not lose precision.
template <int BITS>
static __device__ __forceinline__ void group_values(const uint8_t *blk, const float (&ps)[4], int lane, float (&o)[8][4]) {
  const int q = lane & 3, gcol = lane >> 2;
  const int src = gcol & 3;
  uint32_t bp[2][2];
#pragma unroll
  for (int kt = 0; kt < 2; ++kt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float v0 = __shfl_sync(kFull, ps[2 * kt + j], (4 * (2 * q) + src) & 31);
      const float v1 = __shfl_sync(kFull, ps[2 * kt + j], (4 * (2 * q + 1) + src) & 31);
      bp[kt][j] = split_part(v0, v1, gcol >= 4 ? 1.f : 0.f);
    }
  pv_mma<BITS>(blk + off_vc(BITS), lane, bp, o);
}

// In-place H v of a query head's 128 fp32 channels in shared memory (H the
// Sylvester Walsh-Hadamard matrix): lane L holds channels L + 32 j; strides
// 1 .. 16 pair lanes, 32 and 64 pair registers.  Kept out of line: it runs
// once per (pair, warp) and must not weigh on the kernel's register budget.
static __device__ __noinline__ void hadamard_q(float *v, int lane) {
  float x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) x[j] = v[lane + 32 * j];
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float o = __shfl_xor_sync(kFull, x[j], m);
      x[j] = upper ? o - x[j] : x[j] + o;
    }
  }
  float y0 = x[0] + x[1], y1 = x[0] - x[1], y2 = x[2] + x[3], y3 = x[2] - x[3];
  x[0] = y0 + y2;
  x[2] = y0 - y2;
  x[1] = y1 + y3;
  x[3] = y1 - y3;
#pragma unroll
  for (int j = 0; j < 4; ++j) v[lane + 32 * j] = x[j];
}

// H v of one head's 128 channels held four per lane (lane L has channels
// 4 L .. 4 L + 3): strides 1 and 2 pair registers, 4 .. 64 pair lanes
// L ^ 1 .. L ^ 16.  Out of line, like hadamard_q.
static __device__ __noinline__ float4 hadamard_lane4(float4 v, int lane) {
  float y0 = v.x + v.y, y1 = v.x - v.y, y2 = v.z + v.w, y3 = v.z - v.w;
  v = make_float4(y0 + y2, y1 + y3, y0 - y2, y1 - y3);
#pragma unroll
  for (int m = 1; m < 32; m <<= 1) {
    const bool upper = (lane & m) != 0;
    const float4 o = make_float4(__shfl_xor_sync(kFull, v.x, m), __shfl_xor_sync(kFull, v.y, m),
                                 __shfl_xor_sync(kFull, v.z, m), __shfl_xor_sync(kFull, v.w, m));
    v = upper ? make_float4(o.x - v.x, o.y - v.y, o.z - v.z, o.w - v.w)
              : make_float4(v.x + o.x, v.y + o.y, v.z + o.z, v.w + o.w);
  }
  return v;
}

// Scale the o columns 2q and 2q+1 by their softmax rescale factors.
static __device__ __forceinline__ void rescale_o(float (&o)[8][4], float a_lo, float a_hi) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    o[i][0] *= a_lo;
    o[i][1] *= a_hi;
    o[i][2] *= a_lo;
    o[i][3] *= a_hi;
  }
}

// Resident CTAs per SM the register budget is cut for (tensor-core path,
// query groups of one or two heads).
#ifndef KVQ_DECODE_MIN_BLOCKS
#define KVQ_DECODE_MIN_BLOCKS 4
#endif
#ifndef KVQ_DECODE_MIN_BLOCKS_GQ4
#define KVQ_DECODE_MIN_BLOCKS_GQ4 3
#endif
// One CTA per SM holding every resident warp, rather than several CTAs of
// four warps.  Warps of CTAs launched later on an SM are scheduled behind
// the older ones and finish up to 12 us later; warps of one CTA start as
// equals (their spread fell to about 3 us).  It helped the million-token
// context (-4%) but not the 4096-token batch, whose tail comes from the
// warps that cross pairs, run window passes or merge, so it is off.
#ifndef KVQ_DECODE_ONE_CTA
#define KVQ_DECODE_ONE_CTA 0
#endif

// Launch shape of one instantiation: warps per CTA and CTAs per SM the
// register budget allows (groups of four warps), warps per CTA capped by
// the shared memory a CTA may hold.
template <int BITS, int GQ, bool ROPE, bool KPT, bool SP>
struct CtaShape {
  using WS = WarpSmem<BITS, GQ, ROPE, KPT, SP>;
  static constexpr int kQuads = ROPE ? 3 : (GQ == 4 ? KVQ_DECODE_MIN_BLOCKS_GQ4 : KVQ_DECODE_MIN_BLOCKS);
  static constexpr int kExtra = ROPE ? kG * kRopeOffStride * 8 : 0;  // the in-group rotation table
  static constexpr int kFit = (232448 - kExtra) / WS::BYTES;         // largest opt-in shared memory
  // the table kernel: two CTAs of six warps share the SM (12 warps, as the
  // other pre-RoPE kernels), each CTA one copy of the rotation table
  static constexpr int W = WS::TAB ? 6 : KVQ_DECODE_ONE_CTA ? (4 * kQuads < kFit ? 4 * kQuads : kFit) : 4;
  static constexpr int MIN_BLOCKS = WS::TAB ? 2 : KVQ_DECODE_ONE_CTA ? 1 : kQuads;
  static constexpr int BYTES = W * WS::BYTES + kExtra;
  static_assert(!WS::TAB || MIN_BLOCKS * (BYTES + 1024) <= 233472, "two table CTAs must fit an SM");
};

// Pre-RoPE score of token t = lane through a per-group table (2-bit codes,
// one query head per KV head).  With (a, b) the query rotated back to the
// group's first position, row i of the table holds for every code pair (c1
// of channel i, c2 of channel i + 64), at entry c1 + 4 c2,
//   X = c1 (a s_i) + c2 (b s_{i+64}) + (a m_i + b m_{i+64}),
//   Y = c1 (b s_i) - c2 (a s_{i+64}) + (b m_i - a m_{i+64}),
// so a token's channel pair costs one 4-bit index, one table load and its
// in-group offset rotation (cos, sin): score += cos X + sin Y.  The values
// and their order of operations are those of the coefficient form.  b0[r]:
// (cos, sin) of the first position's angle for channel pair lane + 32 r.
static __device__ __forceinline__ float tab_group_dot(const uint8_t *blk, const float *q_s, const float2 (&b0)[2],
                                                      float *tab, const float2 *roff_s, int lane) {
  constexpr int RS = kTabStride / 4;  // row stride in floats
  const float *ks = reinterpret_cast<const float *>(blk + off_ks(2));
  const float *km = reinterpret_cast<const float *>(blk + off_km(2));
#pragma unroll
  for (int r2 = 0; r2 < 2; ++r2) {
    const int i = lane + 32 * r2;
    const float s1 = ks[i], s2 = ks[i + 64], m1 = km[i], m2 = km[i + 64];
    const float qa = q_s[i], qb = q_s[i + 64];
    const float av = fmaf(qa, b0[r2].x, qb * b0[r2].y), bv = fmaf(qb, b0[r2].x, -qa * b0[r2].y);
    const float cx = av * s1, cy = bv * s2, cz = bv * s1, cw = -av * s2;
    const float c0x = fmaf(av, m1, bv * m2), c0y = fmaf(bv, m1, -av * m2);
    float2 *row = reinterpret_cast<float2 *>(tab + i * RS);
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2) {
      const float ix = fmaf(float(c2), cy, c0x), iy = fmaf(float(c2), cw, c0y);
#pragma unroll
      for (int c1 = 0; c1 < 4; ++c1) row[c1 + 4 * c2] = make_float2(fmaf(float(c1), cx, ix), fmaf(float(c1), cz, iy));
    }
  }
  __syncwarp();
  const int t = lane, uu = (t >> 3) & 3;
  const uint8_t *kc = blk + off_kc(2);
  float dot = 0.f;
#pragma unroll 1
  for (int qq = 0; qq < 4; ++qq) {
    // this token's words of lane 4 (t % 8) + qq: word kt holds channels
    // 16 kt + 8 j + 2 qq + e at bits 16 e + 8 j + 2 (t / 8)
    const uint4 *lw = reinterpret_cast<const uint4 *>(kc) + (4 * (t & 7) + qq);
    const uint4 w0 = lw[0], w1 = lw[32];
    const uint32_t wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
    for (int kt = 0; kt < 4; ++kt) {
      // byte 2 e + j of comb: the index c1 + 4 c2 of channel pair 16 kt + 8 j + 2 qq + e
      const uint32_t lo = (wv[kt] >> (2 * uu)) & 0x03030303u;
      const uint32_t hi = (wv[kt + 4] >> (2 * uu)) & 0x03030303u;
      const uint32_t comb = lo | (hi << 2);
#pragma unroll
      for (int j = 0; j < 2; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int i = 16 * kt + 8 * j + 2 * qq + e;
          const uint32_t k = (comb >> (8 * (2 * e + j))) & 15u;
          const float2 xy = *reinterpret_cast<const float2 *>(tab + i * RS + 2 * k);
          const float2 cs = roff_s[t * kRopeOffStride + i];
          dot = fmaf(cs.x, xy.x, fmaf(cs.y, xy.y, dot));
        }
    }
  }
  return dot;
}

template <int BITS, int GQ, bool ROPE, bool KPT, bool PAGED, bool ROT, bool SP>
__global__ void __launch_bounds__(CtaShape<BITS, GQ, ROPE, KPT, SP>::W * 32, CtaShape<BITS, GQ, ROPE, KPT, SP>::MIN_BLOCKS)
    decode_kernel(DecodeArgs a) {
  using WS = WarpSmem<BITS, GQ, ROPE, KPT, SP>;
  constexpr int NS = WS::NS, BB = WS::BB, kWarps = CtaShape<BITS, GQ, ROPE, KPT, SP>::W;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  uint8_t *ring = smem + warp * WS::BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + WS::BAR_OFF);
  float *q_s = reinterpret_cast<float *>(ring + WS::Q_OFF);              // [GQ][D]
  uint32_t *stage = reinterpret_cast<uint32_t *>(q_s);                   // score operand staging
  float2 *roff_s = reinterpret_cast<float2 *>(smem + kWarps * WS::BYTES);  // [32][65]
  float *zc_s = reinterpret_cast<float *>(ring + WS::SP_OFF);            // [2][GQ][32] score corrections
  float *oc_s = zc_s + 2 * GQ * kG;                                      // [GQ][128] value corrections
  const Geo &geo = a.geo;
  if (SP) {  // the corrections start at zero; their readers zero them again
    for (int i = lane; i < WS::SP_FLOATS; i += 32) zc_s[i] = 0.f;
  }

  if (ROPE) {
    for (int i = threadIdx.x; i < kG * 64; i += blockDim.x)
      roff_s[(i >> 6) * kRopeOffStride + (i & 63)] = a.rope_off[i];
  }
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();  // the only CTA-wide barrier: from here each warp runs alone

  const int NW = a.nw, gw = blockIdx.x * kWarps + warp;
  if (gw >= NW) return;
  const bool head_valid = q < GQ;
  const int H = geo.H, S = geo.S;

  // ---- the work line: total units W, and the sequence s_first holding this
  // warp's first unit with its first unit sbase.  Small batches plan here,
  // every warp on its own (one coalesced read of seq_len per 32 sequences);
  // large ones read the plan kernel's prefix.
  long long W, ua, ub, sbase = 0;
  int s_first = 0;
  if (a.base == nullptr && S <= 32) {
    // up to 32 sequences: one read of seq_len (lane s holds sequence s)
    // serves the empty rows, the total and the prefix
    const int Ls = lane < S ? geo.seq_len[lane] : 0;
    for (int s2 = gw; s2 < S; s2 += NW) {  // rows of sequences with nothing to attend
      const int L = __shfl_sync(kFull, Ls, s2);
      if (L > 0 && L <= geo.capacity && L <= a.max_len) continue;
      if (lane == 0 && L > a.max_len) set_status(geo.status, KVQ_STATUS_MAX_LEN);
      uint4 *o = reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(s2) * a.Hq * kD);
      for (int i = lane; i < a.Hq * kD / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    Split spl;
    int tp, ng;
    const long long v = lane < S ? len_units(a, Ls, spl, tp, ng) : 0;
    long long incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const long long t = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += t;
    }
    W = __shfl_sync(kFull, incl, 31) * H;
    ua = gw * W / NW;
    ub = (gw + 1) * W / NW;
    if (ua >= ub) return;
    // the first sequence whose units end past ua (one exists: ua < W)
    const int idx = __ffs(__ballot_sync(kFull, lane < S && incl * H > ua)) - 1;
    s_first = idx;
    sbase = __shfl_sync(kFull, incl - v, idx) * H;
  } else if (a.base == nullptr) {
    for (int s2 = gw; s2 < S; s2 += NW) {  // rows of sequences with nothing to attend
      const int L = geo.seq_len[s2];
      if (L > 0 && L <= geo.capacity && L <= a.max_len) continue;
      if (lane == 0 && L > a.max_len) set_status(geo.status, KVQ_STATUS_MAX_LEN);
      uint4 *o = reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(s2) * a.Hq * kD);
      for (int i = lane; i < a.Hq * kD / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    long long tot = 0;
    for (int s2 = lane; s2 < S; s2 += 32) {
      Split spl;
      int tp, ng;
      tot += seq_units(a, s2, spl, tp, ng);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(kFull, tot, off);
    W = tot * H;
    ua = gw * W / NW;
    ub = (gw + 1) * W / NW;
    if (ua >= ub) return;
    long long run = 0;  // units of the sequences before chunk c, per KV head
    for (int c = 0; c < S; c += 32) {
      Split spl;
      int tp, ng;
      const long long v = c + lane < S ? seq_units(a, c + lane, spl, tp, ng) : 0;
      long long incl = v;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long t = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += t;
      }
      const unsigned m = __ballot_sync(kFull, c + lane < S && (run + incl) * H > ua);
      if (m) {
        const int idx = __ffs(m) - 1;
        s_first = c + idx;
        sbase = (run + __shfl_sync(kFull, incl - v, idx)) * H;
        break;
      }
      run += __shfl_sync(kFull, incl, 31);
    }
  } else {
    W = a.plan->total;
    ua = gw * W / NW;
    ub = (gw + 1) * W / NW;
    if (ua >= ub) return;
    // the last s with base[s] <= ua, by a 32-way search (base[0] = 0 <= ua
    // keeps the answer in [lo, lo + n))
    int lo = 0, n = S;
    while (n > 32) {
      const int step = (n + 31) / 32;
      const int idx = lo + lane * step;
      const unsigned m = __ballot_sync(kFull, idx < lo + n && a.base[idx] <= ua);
      const int nlo = lo + (31 - __clz(m)) * step;
      n = min(step, lo + n - nlo);
      lo = nlo;
    }
    const unsigned m = __ballot_sync(kFull, lane < n && a.base[lo + lane] <= ua);
    s_first = lo + 31 - __clz(m);
    sbase = a.base[s_first];
  }

  // ---- fetch cursor: walks the packed groups of [ua, ub) in consumer order
  // (fbase: first unit of sequence fs; its unit counts are re-derived from
  // seq_len at each pair change rather than held in registers)
  uint32_t fseq = 0, cseq = 0;  // ring groups issued / consumed
  int fs = s_first, fh, fg = 0, fg_end = 0;
  long long fbase = sbase;
  bool fdone = false;
  {
    Split spl;
    int tp, ng;
    fh = static_cast<int>((ua - fbase) / max(seq_units(a, fs, spl, tp, ng), 1));
  }
  auto fetch_pair = [&]() {  // the group range of pair (fs, fh); false past ub
    Split spl;
    int tp, ng;
    const int u = seq_units(a, fs, spl, tp, ng);
    const long long P0 = fbase + static_cast<long long>(fh) * u;
    const long long gb = P0 + kPassUnits * tp;
    fg = static_cast<int>(min(max(ua - gb, 0LL), static_cast<long long>(ng)));
    fg_end = static_cast<int>(min(max(ub - gb, 0LL), static_cast<long long>(ng)));
#if KVQ_DECODE_PREFETCH
    // warm L2 with the rows the consumer reads directly when it reaches this
    // pair (several groups from now): the query rows, and the sink and
    // window rows of the passes whose first unit is in this warp's range
    if (u > 0 && P0 < ub) {
      const char *qp = reinterpret_cast<const char *>(a.q + (static_cast<size_t>(fs) * a.Hq + static_cast<size_t>(fh) * GQ) * kD);
      if (lane < 2 * GQ) prefetch_l2(qp + 128 * lane);
      const int T = spl.nsink + spl.r;
      const size_t sh = static_cast<size_t>(fs) * H + fh;
      for (int i = lane; i < 4 * T; i += 32) {  // token i / 4: K or V row, first or second 128 bytes
        const int t = i >> 2;
        if (P0 + kPassUnits * (t >> 5) < ua) continue;
        const __half *row = t < spl.nsink ? ((i & 2) ? geo.v_sink : geo.k_sink) + (sh * geo.ns + t) * kD
                                          : ((i & 2) ? geo.v_res : geo.k_res) + (sh * geo.R + (t - spl.nsink)) * kD;
        prefetch_l2(reinterpret_cast<const char *>(row) + 128 * (i & 1));
      }
    }
#endif
    if (PAGED && fg < fg_end) {  // check this range's table entries once
      const int *te = geo.table + (static_cast<size_t>(fs) * H + fh) * geo.max_groups;
      bool bad = false;
      for (int i = fg + lane; i < fg_end; i += 32)
        bad |= static_cast<unsigned>(te[i]) >= static_cast<unsigned>(geo.num_blocks);
      if (__any_sync(kFull, bad) && lane == 0) set_status(geo.status, KVQ_STATUS_BAD_BLOCK);
    }
    return P0 < ub;
  };
  auto fetch_next_pair = [&]() {
    while (!fdone) {
      if (++fh == H) {
        Split spl;
        int tp, ng;
        fbase += static_cast<long long>(H) * seq_units(a, fs, spl, tp, ng);
        fh = 0;
        if (++fs >= S) {
          fdone = true;
          break;
        }
      }
      if (!fetch_pair()) {
        fdone = true;
        break;
      }
      if (fg < fg_end) break;
    }
  };
  if (a.wait_before_fetch) {
    // test aid: wait on the first ring slot before anything is copied into
    // it, so that the bounded wait runs out (nothing is in flight to drain)
    if (!mbar_wait_bounded(&full[0], 0, a.wait_limit)) {
      if (lane == 0) set_status(geo.status, KVQ_STATUS_TIMEOUT);
      return;
    }
  }
  if (!fetch_pair()) fdone = true;
  if (!fdone && fg >= fg_end) fetch_next_pair();
  auto top_up = [&]() {
    const uint32_t depth = KVQ_RING_RAMP ? min(static_cast<uint32_t>(NS), cseq + KVQ_RING_RAMP)
                                         : static_cast<uint32_t>(NS);
    while (!fdone && fseq - cseq < depth) {
      if (lane == 0) {
        const uint32_t slot = fseq % NS;
        // paged: an entry outside the pool reads pool block 0 (reported when
        // the pair's range was entered)
        size_t blk = (static_cast<size_t>(fs) * H + fh) * geo.max_groups + fg;
        if constexpr (PAGED) {
          const unsigned pb = static_cast<unsigned>(geo.table[blk]);
          blk = pb < static_cast<unsigned>(geo.num_blocks) ? pb : 0u;
        }
        // (a skipped copy leaves its wait to give up: the warp then stops)
        if (KVQ_IN_BOUNDS(geo.status, fg, geo.max_groups) &&
            KVQ_IN_BOUNDS(geo.status, blk, PAGED ? static_cast<size_t>(geo.num_blocks)
                                                 : static_cast<size_t>(S) * H * geo.max_groups)) {
          const uint8_t *src = geo.blocks + blk * BB;
          fence_proxy_async();  // generic reads of the slot before the async write
          mbar_arrive_expect_tx(&full[slot], BB);
          bulk_g2s(ring + slot * BB, src, BB, &full[slot]);
        }
      }
      ++fseq;
      if (++fg >= fg_end) fetch_next_pair();
    }
  };
  top_up();

  // ---- consumer: pairs in order (cbase: first unit of sequence s)
  bool ok = true;
  int s = s_first;
  long long cbase = sbase;
  Split spl;
  int tp, ng;
  int u = seq_units(a, s, spl, tp, ng);
  int h = static_cast<int>((ua - cbase) / max(u, 1));
  while (ok) {
    if (u == 0) {  // sequence with nothing to attend: skip it
      if (++s >= S) break;
      h = 0;
      u = seq_units(a, s, spl, tp, ng);
      continue;
    }
    const long long P0 = cbase + static_cast<long long>(h) * u, P1 = P0 + u;
    if (P0 >= ub) break;
    const long long lo = max(ua, P0), hi = min(ub, P1);
    const int pair = s * H + h;
    const size_t orow0 = (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(h) * GQ) * kD;
    __syncwarp();  // the previous pair's reads of q_s are done
    for (int i = lane; i < GQ * kD; i += 32)
      q_s[i] = KVQ_IN_BOUNDS(geo.status, orow0 + i, static_cast<size_t>(S) * a.Hq * kD) ? __half2float(a.q[orow0 + i])
                                                                                        : 0.f;
    __syncwarp();
    int npart = 0;

    // ------------------ window / sink passes whose first unit is ours
    for (int k = 0; k < tp; ++k) {
      const long long x = P0 + static_cast<long long>(kPassUnits) * k;
      if (x < lo || x >= hi) continue;
      const int T = spl.nsink + spl.r;
      const int t0 = 32 * k;
      const int nt = min(32, T - t0);
      const size_t sh = static_cast<size_t>(pair);
      const int i = t0 + lane;
      const bool valid = lane < nt;
      float dot[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) dot[hh] = 0.f;
      if (valid) {
        int pos;
        const __half *kp;
        if (i < spl.nsink) {
          pos = i;
          kp = geo.k_sink + (KVQ_IN_BOUNDS(geo.status, i, geo.ns) ? (sh * geo.ns + i) * kD : 0);
        } else {
          const int slot = i - spl.nsink;
          pos = spl.nsink + spl.Lq + slot;
          kp = geo.k_res + (KVQ_IN_BOUNDS(geo.status, slot, geo.R) ? (sh * geo.R + slot) * kD : 0);
        }
        const int sidx = pos - geo.ns;  // stream index (negative for the sink)
        // the key row in flight at once (in two halves for four query heads,
        // whose register budget is tighter); two dot chains per head
        constexpr int KH = GQ == 4 ? 2 : 1;  // load rounds
        float dot2[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) dot2[hh] = 0.f;
#pragma unroll
        for (int kh = 0; kh < KH; ++kh) {
        uint4 kr[16 / KH];
#pragma unroll
        for (int c = 0; c < 8 / KH; ++c) {
          kr[c] = *reinterpret_cast<const uint4 *>(kp + 8 * (c + kh * 8 / KH));
          kr[c + 8 / KH] = *reinterpret_cast<const uint4 *>(kp + 64 + 8 * (c + kh * 8 / KH));
        }
#pragma unroll
        for (int cc = 0; cc < 8 / KH; ++cc) {
          const int c = cc + kh * 8 / KH;
          const __half *ha = reinterpret_cast<const __half *>(&kr[cc]);           // channels 8c ..
          const __half *hb = reinterpret_cast<const __half *>(&kr[cc + 8 / KH]);  // channels 64 + 8c ..
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int ch = 8 * c + e;
            float k1 = __half2float(ha[e]), k2 = __half2float(hb[e]);
            if (ROPE && sidx >= 0 && KVQ_IN_BOUNDS(geo.status, sidx >> 5, a.n_base)) {
              const float2 bs = a.rope_base[static_cast<size_t>(sidx >> 5) * 64 + ch];
              const float2 of = roff_s[(sidx & 31) * kRopeOffStride + ch];
              const float cs = bs.x * of.x - bs.y * of.y;
              const float sn = bs.y * of.x + bs.x * of.y;
              const float r1 = k1 * cs - k2 * sn, r2 = k2 * cs + k1 * sn;
              k1 = r1;
              k2 = r2;
            }
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              float &d = (e & 1) ? dot2[hh] : dot[hh];
              d = fmaf(q_s[hh * kD + ch], k1, fmaf(q_s[hh * kD + ch + 64], k2, d));
            }
          }
        }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) dot[hh] += dot2[hh];
      }
      float p[GQ], mh[GQ], lh[GQ], acc[GQ][4];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        const float zz = valid ? dot[hh] * a.zscale : -INFINITY;
        float mx = zz;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
        p[hh] = valid ? fast_exp2(zz - mx) : 0.f;
        float sum = p[hh];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
        mh[hh] = mx;
        lh[hh] = sum;
        acc[hh][0] = acc[hh][1] = acc[hh][2] = acc[hh][3] = 0.f;
      }
      // values: lane holds channels 4*lane .. 4*lane+3; VB rows in flight at once
      constexpr int VB = GQ == 4 ? 8 : 32;
      for (int tb = 0; tb < nt; tb += VB) {
        uint2 raw[VB];
#pragma unroll
        for (int uu = 0; uu < VB; ++uu) {
          const int it = t0 + tb + uu;
          raw[uu] = make_uint2(0u, 0u);
          if (tb + uu < nt) {
            const __half *vp = it < spl.nsink ? geo.v_sink + (sh * geo.ns + it) * kD
                                              : geo.v_res + (sh * geo.R + (it - spl.nsink)) * kD;
            if (KVQ_IN_BOUNDS(geo.status, it < spl.nsink ? it : it - spl.nsink, it < spl.nsink ? geo.ns : geo.R))
              raw[uu] = *reinterpret_cast<const uint2 *>(vp + 4 * lane);
          }
        }
#pragma unroll
        for (int uu = 0; uu < VB; ++uu) {
          const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw[uu].x));
          const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw[uu].y));
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float pt = __shfl_sync(kFull, p[hh], (tb + uu) & 31);
            acc[hh][0] = fmaf(pt, v01.x, acc[hh][0]);
            acc[hh][1] = fmaf(pt, v01.y, acc[hh][1]);
            acc[hh][2] = fmaf(pt, v23.x, acc[hh][2]);
            acc[hh][3] = fmaf(pt, v23.y, acc[hh][3]);
          }
        }
      }
      const size_t slot = a.pass_slot0 + static_cast<size_t>(pair) * a.tail_passes + k;
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        if (!KVQ_IN_BOUNDS(geo.status, slot, a.n_slots)) break;
        float *po = a.part_o + (slot * GQ + hh) * kD;
        *reinterpret_cast<float4 *>(po + 4 * lane) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
        if (lane == 0) a.part_ml[slot * GQ + hh] = make_float2(mh[hh], lh[hh]);
      }
      ++npart;
    }

    // ------------------------------------------- packed groups of our range
    {
      const long long gb = P0 + static_cast<long long>(kPassUnits) * tp;
      const int g_lo = static_cast<int>(min(max(lo - gb, 0LL), static_cast<long long>(ng)));
      const int g_hi = static_cast<int>(min(max(hi - gb, 0LL), static_cast<long long>(ng)));
      float o[8][4];
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
      float m_run = -INFINITY, l_run = 0.f, mu_run = 0.f;
      if (g_lo < g_hi) {
        if (!ROPE) {
          QkOperand<GQ> qo;
          float kfac[4];
          uint32_t bqc[8][2];  // keys per token: the query's B fragments, fixed for the pair
          float zsq = 0.f;     // keys per token: zscale * sum_d q_d of this lane's head
          if (ROT) {  // groups hold y = H x / D: score them with H q (q . x = H q . y)
            __syncwarp();
            for (int hh = 0; hh < GQ; ++hh) hadamard_q(q_s + hh * kD, lane);
            __syncwarp();
          }
          if (!KPT) {
            qo.init(q_s, lane, a.zscale);
#pragma unroll
            for (int tau = 0; tau < 4; ++tau) kfac[tau] = key_row_scale<BITS>(tau) * qo.qscale;
          } else {
            const int hd = min(g >> 1, GQ - 1);
#pragma unroll
            for (int kt = 0; kt < 8; ++kt)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const float2 qv = *reinterpret_cast<const float2 *>(q_s + hd * kD + 16 * kt + 8 * j + 2 * q);
                bqc[kt][j] = split_part(qv.x, qv.y, (g & 1) ? 1.f : 0.f);  // (zero low part for fp16 q)
              }
            float qs[GQ];
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              qs[hh] = q_s[hh * kD + lane] + q_s[hh * kD + lane + 32] + q_s[hh * kD + lane + 64] +
                       q_s[hh * kD + lane + 96];
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) qs[hh] += __shfl_xor_sync(kFull, qs[hh], off);
              if (hh == min(q, GQ - 1)) zsq = qs[hh] * a.zscale;
            }
#pragma unroll
            for (int tau = 0; tau < 4; ++tau) kfac[tau] = key_row_scale<BITS>(tau) * a.zscale;
          }
          // two groups (64 tokens) per iteration: independent score mmas, one
          // softmax update, two value mmas
          for (int gi = g_lo; gi < g_hi; gi += 2) {
            const bool two = gi + 1 < g_hi;
            const uint32_t sa = cseq % NS, sb = (cseq + 1) % NS;
            if (!mbar_wait_bounded(&full[sa], (cseq / NS) & 1, a.wait_limit) ||
                (two && !mbar_wait_bounded(&full[sb], ((cseq + 1) / NS) & 1, a.wait_limit))) {
              ok = false;
              break;
            }
            const uint8_t *ba = ring + sa * BB, *bb = ring + sb * BB;
            float za[4], zb[4];
            if (KPT)
              group_scores_kpt<BITS>(ba, bqc, kfac, zsq, lane, za);
            else
              group_scores<BITS, GQ>(ba, qo, kfac, stage, lane, za);
            if (two) {
              if (KPT)
                group_scores_kpt<BITS>(bb, bqc, kfac, zsq, lane, zb);
              else
                group_scores<BITS, GQ>(bb, qo, kfac, stage, lane, zb);
            } else {
              zb[0] = zb[1] = zb[2] = zb[3] = -INFINITY;
            }
            if (SP) {  // outliers: z_t += zscale q_d (x - min) of each slice's outlier
              if (KPT) {  // one outlier per token: this lane's tokens, query from shared memory
                const float *qh = q_s + min(q, GQ - 1) * kD;
#pragma unroll
                for (int gg = 0; gg < 2; ++gg) {
                  if (gg == 1 && !two) break;
                  const uint8_t *bk = gg ? bb : ba;
                  const uint32_t *ksp = reinterpret_cast<const uint32_t *>(bk + off_ksp(BITS, true));
                  const float *km = reinterpret_cast<const float *>(bk + off_km(BITS, true));
#pragma unroll
                  for (int tau = 0; tau < 4; ++tau) {
                    const uint32_t e = ksp[8 * tau + g];
                    const float dx = __half2float(__ushort_as_half(static_cast<unsigned short>(e & 0xFFFFu))) -
                                     km[8 * tau + g];
                    const float corr = a.zscale * qh[(e >> 16) & (kD - 1)] * dx;
                    if (gg) zb[tau] += corr; else za[tau] += corr;
                  }
                }
              } else {
                key_outliers<BITS, GQ>(ba, qo, zc_s, lane);
                if (two) key_outliers<BITS, GQ>(bb, qo, zc_s + GQ * kG, lane);
                __syncwarp();
                if (head_valid) {
#pragma unroll
                  for (int tau = 0; tau < 4; ++tau) {
                    float *ca = zc_s + q * kG + 8 * tau + g, *cb = ca + GQ * kG;
                    za[tau] = fmaf(*ca, qo.qscale, za[tau]);
                    zb[tau] = fmaf(*cb, qo.qscale, zb[tau]);
                    *ca = 0.f;
                    *cb = 0.f;
                  }
                }
                __syncwarp();
              }
            }
            float mx = fmaxf(fmaxf(fmaxf(za[0], za[1]), fmaxf(za[2], za[3])),
                             fmaxf(fmaxf(zb[0], zb[1]), fmaxf(zb[2], zb[3])));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = fast_exp2(m_run - m_new);
            const float *vsa = reinterpret_cast<const float *>(ba + off_vs(BITS, KPT));
            const float *vma = reinterpret_cast<const float *>(ba + off_vm(BITS, KPT));
            const float *vsb = reinterpret_cast<const float *>(bb + off_vs(BITS, KPT));
            const float *vmb = reinterpret_cast<const float *>(bb + off_vm(BITS, KPT));
            float psa[4], psb[4], psum = 0.f, mus = 0.f;
            float wsp[2][4];  // outliers: p_t (x - min_t) of each token's value outlier
#pragma unroll
            for (int tau = 0; tau < 4; ++tau) {
              const float pa = fast_exp2(za[tau] - m_new);
              psum += pa;
              psa[tau] = pa * vsa[8 * tau + g];
              mus = fmaf(pa, vma[8 * tau + g], mus);
              if (SP) {
                const uint32_t e = reinterpret_cast<const uint32_t *>(ba + off_vsp(BITS, KPT))[8 * tau + g];
                wsp[0][tau] = pa * (__half2float(__ushort_as_half(static_cast<unsigned short>(e & 0xFFFFu))) -
                                    vma[8 * tau + g]);
              }
            }
            if (two) {
#pragma unroll
              for (int tau = 0; tau < 4; ++tau) {
                const float pb = fast_exp2(zb[tau] - m_new);
                psum += pb;
                psb[tau] = pb * vsb[8 * tau + g];
                mus = fmaf(pb, vmb[8 * tau + g], mus);
                if (SP) {
                  const uint32_t e = reinterpret_cast<const uint32_t *>(bb + off_vsp(BITS, KPT))[8 * tau + g];
                  wsp[1][tau] = pb * (__half2float(__ushort_as_half(static_cast<unsigned short>(e & 0xFFFFu))) -
                                      vmb[8 * tau + g]);
                }
              }
            }
            l_run = fmaf(l_run, alpha, psum);
            mu_run = fmaf(mu_run, alpha, mus);
            m_run = m_new;
            const bool rescale = __any_sync(kFull, head_valid && alpha != 1.f);
            if (rescale)
              rescale_o(o, __shfl_sync(kFull, alpha, (2 * q) & 31), __shfl_sync(kFull, alpha, (2 * q + 1) & 31));
            if (SP) {  // value corrections: rescaled with o, then this step's outliers added
              if (rescale) {
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                  const float ah = __shfl_sync(kFull, alpha, hh);
#pragma unroll
                  for (int j = 0; j < 4; ++j) oc_s[hh * kD + lane + 32 * j] *= ah;
                }
              }
              __syncwarp();
              if (head_valid) {
#pragma unroll
                for (int tau = 0; tau < 4; ++tau) {
                  const uint32_t ea = reinterpret_cast<const uint32_t *>(ba + off_vsp(BITS, KPT))[8 * tau + g];
                  atomicAdd(oc_s + q * kD + ((ea >> 16) & (kD - 1)), wsp[0][tau]);
                  if (two) {
                    const uint32_t eb = reinterpret_cast<const uint32_t *>(bb + off_vsp(BITS, KPT))[8 * tau + g];
                    atomicAdd(oc_s + q * kD + ((eb >> 16) & (kD - 1)), wsp[1][tau]);
                  }
                }
              }
            }
            group_values<BITS>(ba, psa, lane, o);
            if (two) group_values<BITS>(bb, psb, lane, o);
            __syncwarp();
            cseq += two ? 2 : 1;
            top_up();
          }
        } else {
          // pre-RoPE keys, one lane per token t.  With (C0, S0) the rotation of
          // the group's first position p0 and (Ct, St) that of the offset t, the
          // query rotated back to p0 (a = q'_i, b = q'_{i+64}) gives
          //   q . R(p0 + t) k = sum_i Ct (a k_i + b k_{i+64}) + St (b k_i - a k_{i+64}),
          // and with k = code * scale + min the per-pair coefficients of
          //   X = c1 (a s_i) + c2 (b s_{i+64}) + (a m_i + b m_{i+64}),
          //   Y = c1 (b s_i) - c2 (a s_{i+64}) + (b m_i - a m_{i+64})
          // are formed once per group (two pairs per lane) for all 32 tokens.
          float4 *coef = reinterpret_cast<float4 *>(ring + WS::COEF_OFF);            // [GQ][64]
          float2 *coef0 = reinterpret_cast<float2 *>(ring + WS::COEF_OFF + GQ * 64 * 16);  // [GQ][64]
          float m_all[GQ];
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) m_all[hh] = -INFINITY;
          for (int gi = g_lo; gi < g_hi; ++gi) {
            const uint32_t slot = cseq % NS;
            if (!mbar_wait_bounded(&full[slot], (cseq / NS) & 1, a.wait_limit)) {
              ok = false;
              break;
            }
            const uint8_t *blk = ring + slot * BB;
            const float *ks = reinterpret_cast<const float *>(blk + off_ks(BITS));
            const float *km = reinterpret_cast<const float *>(blk + off_km(BITS));
            const float *vs = reinterpret_cast<const float *>(blk + off_vs(BITS));
            const float *vm = reinterpret_cast<const float *>(blk + off_vm(BITS));
            const uint8_t *kc = blk + off_kc(BITS);
            const int t = lane;
            const int tau = t >> 3, uu = tau % (8 / BITS);
            float dot[GQ];
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) dot[hh] = 0.f;
            if constexpr (WS::TAB) {
              float2 b0[2];
#pragma unroll
              for (int r2 = 0; r2 < 2; ++r2)  // (cos, sin) of p0 theta_i
                b0[r2] = KVQ_IN_BOUNDS(geo.status, gi, a.n_base)
                             ? a.rope_base[static_cast<size_t>(gi) * 64 + lane + 32 * r2]
                             : make_float2(1.f, 0.f);
              dot[0] = tab_group_dot(blk, q_s, b0, reinterpret_cast<float *>(ring + WS::COEF_OFF), roff_s, lane);
            } else {
#pragma unroll
              for (int r2 = 0; r2 < 2; ++r2) {
                const int i = lane + 32 * r2;
                const float2 b0 = KVQ_IN_BOUNDS(geo.status, gi, a.n_base) ? a.rope_base[static_cast<size_t>(gi) * 64 + i]
                                                                           : make_float2(1.f, 0.f);  // (cos, sin) of p0 theta_i
                const float s1 = ks[i], s2 = ks[i + 64], m1 = km[i], m2 = km[i + 64];
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                  const float qa = q_s[hh * kD + i], qb = q_s[hh * kD + i + 64];
                  const float av = fmaf(qa, b0.x, qb * b0.y), bv = fmaf(qb, b0.x, -qa * b0.y);
                  coef[hh * 64 + i] = make_float4(av * s1, bv * s2, bv * s1, -av * s2);
                  coef0[hh * 64 + i] = make_float2(fmaf(av, m1, bv * m2), fmaf(bv, m1, -av * m2));
                }
              }
              __syncwarp();
#pragma unroll 1
              for (int qq = 0; qq < 4; ++qq) {
                // this token's words of lane 4 (t % 8) + qq: word kt (2-bit) or
                // 2 kt + tau / 2 (4-bit) holds channels 16 kt + 8 j + 2 qq + e
                constexpr int WPL = BITS * 4;  // words per lane
                const uint4 *lw = reinterpret_cast<const uint4 *>(kc) + (4 * (t & 7) + qq);
                uint32_t wv[WPL];
#pragma unroll
                for (int m = 0; m < WPL / 4; ++m) {
                  const uint4 c4 = lw[32 * m];
                  wv[4 * m] = c4.x;
                  wv[4 * m + 1] = c4.y;
                  wv[4 * m + 2] = c4.z;
                  wv[4 * m + 3] = c4.w;
                }
#pragma unroll
                for (int kt = 0; kt < 4; ++kt) {
                  const uint32_t wa = BITS == 2 ? wv[kt] : ((tau >> 1) ? wv[2 * kt + 1] : wv[2 * kt]);
                  const uint32_t wb = BITS == 2 ? wv[kt + 4] : ((tau >> 1) ? wv[2 * (kt + 4) + 1] : wv[2 * (kt + 4)]);
#pragma unroll
                  for (int j = 0; j < 2; ++j)
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                      const int i = 16 * kt + 8 * j + 2 * qq + e;
                      const int sh = 16 * e + 8 * j + BITS * uu;
                      // code -> fp32 on the FMA pipe: the field under 2^23
                      const float c1 = __uint_as_float(((wa >> sh) & ((1u << BITS) - 1u)) | 0x4B000000u) - 8388608.f;
                      const float c2 = __uint_as_float(((wb >> sh) & ((1u << BITS) - 1u)) | 0x4B000000u) - 8388608.f;
                      const float2 cs = roff_s[t * kRopeOffStride + i];
#pragma unroll
                      for (int hh = 0; hh < GQ; ++hh) {
                        const float4 cf = coef[hh * 64 + i];
                        const float2 c0 = coef0[hh * 64 + i];
                        const float X = fmaf(c1, cf.x, fmaf(c2, cf.y, c0.x));
                        const float Y = fmaf(c1, cf.z, fmaf(c2, cf.w, c0.y));
                        dot[hh] = fmaf(cs.x, X, fmaf(cs.y, Y, dot[hh]));
                      }
                    }
                }
              }
            }
            const float vsc = vs[t], vmn = vm[t];
            float ps[GQ];
            float alpha_q = 1.f, psum_q = 0.f, mus_q = 0.f, m_q = m_run, a_lo = 1.f, a_hi = 1.f;
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              const float zz = dot[hh] * a.zscale;
              float mx = zz;
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
              const float m_new = fmaxf(m_all[hh], mx);
              const float alpha = fast_exp2(m_all[hh] - m_new);
              m_all[hh] = m_new;
              const float p = fast_exp2(zz - m_new);
              ps[hh] = p * vsc;
              float pl = p, pm = p * vmn;
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) {
                pl += __shfl_xor_sync(kFull, pl, off);
                pm += __shfl_xor_sync(kFull, pm, off);
              }
              if (hh == q) {
                alpha_q = alpha;
                psum_q = pl;
                mus_q = pm;
                m_q = m_new;
              }
              if (hh == 2 * q) a_lo = alpha;
              if (hh == 2 * q + 1) a_hi = alpha;
            }
            l_run = fmaf(l_run, alpha_q, g == 0 ? psum_q : 0.f);
            mu_run = fmaf(mu_run, alpha_q, g == 0 ? mus_q : 0.f);
            m_run = m_q;
            rescale_o(o, a_lo, a_hi);
            // B column g: head g & 3's weights, fp16 high parts in columns
            // 0..3 and rounding remainders in 4..7 (as group_values)
            uint32_t bp[2][2];
#pragma unroll
            for (int kt = 0; kt < 2; ++kt)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                float v0 = 0.f, v1 = 0.f;
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                  const float a0 = __shfl_sync(kFull, ps[hh], 16 * kt + 8 * j + 2 * q);
                  const float a1 = __shfl_sync(kFull, ps[hh], 16 * kt + 8 * j + 2 * q + 1);
                  if (hh == (g & 3)) {
                    v0 = a0;
                    v1 = a1;
                  }
                }
                bp[kt][j] = split_part(v0, v1, g >= 4 ? 1.f : 0.f);
              }
            pv_mma<BITS>(blk + off_vc(BITS), lane, bp, o);
            __syncwarp();
            ++cseq;
            top_up();
          }
        }
      }
      if (!ok) break;
      // this warp's partial of the pair's packed groups (empty if it had none)
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l_run += __shfl_xor_sync(kFull, l_run, off);
        mu_run += __shfl_xor_sync(kFull, mu_run, off);
      }
      const size_t slot = KVQ_IN_BOUNDS(geo.status, static_cast<size_t>(gw) + pair, a.pass_slot0)
                              ? static_cast<size_t>(gw) + pair : 0;
      const float mu_c[2] = {__shfl_sync(kFull, mu_run, (2 * q) & 31), __shfl_sync(kFull, mu_run, (2 * q + 1) & 31)};
      // the value weights' low parts sit in columns 4 .. 7, two lanes up:
      // fold them in.  (A rotating cache leaves this partial in the rotated
      // value domain; the merge rotates the groups' sum back.)
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[mt][i] += __shfl_down_sync(kFull, o[mt][i], 2);
      if (SP) __syncwarp();  // every value correction of the range is in
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        if (2 * q + c < GQ) {
          float *po = a.part_o + (slot * GQ + 2 * q + c) * kD;
#pragma unroll
          for (int mt = 0; mt < 8; ++mt)
#pragma unroll
            for (int rr = 0; rr < 2; ++rr) {
              float v = fmaf(o[mt][2 * rr + c], val_row_scale<BITS>(mt, rr), mu_c[c]);
              if (SP) {
                float *oc = oc_s + (2 * q + c) * kD + 16 * mt + 8 * rr + g;
                v += *oc;
                *oc = 0.f;
              }
              po[16 * mt + 8 * rr + g] = v;
            }
        }
      }
      if (SP) __syncwarp();
      if (head_valid && g == 0) a.part_ml[slot * GQ + q] = make_float2(m_run, l_run);
      ++npart;
    }

    // ---- the warp completing the pair's count merges its partials; lane
    // 0's acq_rel add publishes this warp's partials (ordered before it by
    // the warp barrier) and observes every other warp's
    __syncwarp();
    const Touching tw = touching_warps(P0, P1, W, NW);
    const int expect = tp + tw.n;
    int last = 0;
    if (lane == 0) last = atom_add_acq_rel(&a.counters[pair], npart) + npart == expect;
    if (__shfl_sync(kFull, last, 0)) {
      __threadfence();
      if (lane == 0) a.counters[pair] = 0;  // ready for the next call
      const size_t pass0 = a.pass_slot0 + static_cast<size_t>(pair) * a.tail_passes;
      for (int hh = 0; hh < GQ; ++hh) {
        float M = -INFINITY;
        float Ls = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f), accg = acc;  // window passes, groups
        auto add = [&](const float2 ml, const float4 ov, float4 &to) {
          const float wgt = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
          Ls = fmaf(ml.y, wgt, Ls);
          to.x = fmaf(ov.x, wgt, to.x);
          to.y = fmaf(ov.y, wgt, to.y);
          to.z = fmaf(ov.z, wgt, to.z);
          to.w = fmaf(ov.w, wgt, to.w);
        };
        auto slot_of = [&](int i) -> size_t { return i < tp ? pass0 + i : static_cast<size_t>(tw.at(i - tp)) + pair; };
        const int np = tp + tw.n;
        if (np <= kMergeBatch) {
          // every partial's loads issued together: one L2 round trip
          float2 ml[kMergeBatch];
          float4 ov[kMergeBatch];
#pragma unroll
          for (int i = 0; i < kMergeBatch; ++i) {
            ml[i] = make_float2(-INFINITY, 0.f);
            ov[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (i < np) {
              const size_t sl = slot_of(i);
              ml[i] = __ldcg(&a.part_ml[sl * GQ + hh]);
              ov[i] = __ldcg(reinterpret_cast<const float4 *>(a.part_o + (sl * GQ + hh) * kD) + lane);
            }
          }
#pragma unroll
          for (int i = 0; i < kMergeBatch; ++i) M = fmaxf(M, ml[i].x);
          if (M != -INFINITY) {
#pragma unroll
            for (int i = 0; i < kMergeBatch; ++i)
              if (i < np) add(ml[i], ov[i], i < tp ? acc : accg);
          }
        } else {
          for (int k = lane; k < tp; k += 32) M = fmaxf(M, __ldcg(&a.part_ml[(pass0 + k) * GQ + hh]).x);
          for (int i = lane; i < tw.n; i += 32)
            M = fmaxf(M, __ldcg(&a.part_ml[(static_cast<size_t>(tw.at(i)) + pair) * GQ + hh]).x);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
          auto add_slot = [&](size_t sl, float4 &to) {
            add(__ldcg(&a.part_ml[sl * GQ + hh]),
                __ldcg(reinterpret_cast<const float4 *>(a.part_o + (sl * GQ + hh) * kD) + lane), to);
          };
          if (M != -INFINITY) {
            for (int k = 0; k < tp; ++k) add_slot(pass0 + k, acc);
#pragma unroll 4
            for (int i = 0; i < tw.n; ++i) add_slot(static_cast<size_t>(tw.at(i)) + pair, accg);
          }
        }
        if (ROT) accg = hadamard_lane4(accg, lane);  // the groups' values back from H x / D: x = H y
        acc = make_float4(acc.x + accg.x, acc.y + accg.y, acc.z + accg.z, acc.w + accg.w);
        const float inv = M == -INFINITY ? 0.f : 1.f / Ls;
        if (!KVQ_IN_BOUNDS(geo.status, orow0 + static_cast<size_t>(hh) * kD, static_cast<size_t>(S) * a.Hq * kD)) break;
        __half2 *op = reinterpret_cast<__half2 *>(a.out + orow0 + static_cast<size_t>(hh) * kD) + 2 * lane;
        op[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
        op[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
      }
    }
    if (P1 >= ub) break;
    if (++h == H) {
      h = 0;
      cbase += static_cast<long long>(H) * u;
      if (++s >= S) break;
      u = seq_units(a, s, spl, tp, ng);
    }
  }
  if (!ok) {
    set_status(geo.status, KVQ_STATUS_TIMEOUT);
    // let this warp's copies still in flight land before it exits: they read
    // valid cache blocks, so they complete; the wait keeps its own default
    // bound (about two seconds) whatever limit gave up above
    for (; cseq < fseq; ++cseq) mbar_wait_bounded(&full[cseq % NS], (cseq / NS) & 1);
  }
}

// ---------------------------------------------------------------- host side

// Defined in decode.cu: the plan kernel's launch, and the warp count set by
// kvq_set_decode_warps (0: every resident warp).
cudaError_t launch_plan(const DecodeArgs &a, cudaStream_t stream);
int decode_warps_override();

// Defined in decode_paged.cu, decode_rot.cu and decode_rot_paged.cu: the
// launches of the paged-layout kernels and of the kernels for caches whose
// tokens are Walsh-Hadamard rotated (contiguous and paged).
cudaError_t launch_paged(const DecodeArgs &a, int gq, cudaStream_t stream);
cudaError_t launch_rot(const DecodeArgs &a, int gq, cudaStream_t stream);
cudaError_t launch_rot_paged(const DecodeArgs &a, int gq, cudaStream_t stream);
// Defined in decode_sparse.cu and decode_sparse_paged.cu: dense-and-sparse blocks.
cudaError_t launch_sparse(const DecodeArgs &a, int gq, cudaStream_t stream);
cudaError_t launch_sparse_paged(const DecodeArgs &a, int gq, cudaStream_t stream);

// Resident CTAs per SM of one instantiation on the current device, and the
// device's SM count (cached per device ordinal).
template <int BITS, int GQ, bool ROPE, bool KPT, bool PAGED, bool ROT, bool SP>
static cudaError_t kernel_slots(int &per_sm, int &n_sm, int &bytes_out) {
  constexpr int bytes = CtaShape<BITS, GQ, ROPE, KPT, SP>::BYTES, kWarps = CtaShape<BITS, GQ, ROPE, KPT, SP>::W;
  auto kern = decode_kernel<BITS, GQ, ROPE, KPT, PAGED, ROT, SP>;
  static int resident[64] = {};
  static int sms[64] = {};
  bytes_out = bytes;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  per_sm = dev < 64 ? resident[dev] : 0;
  n_sm = dev < 64 ? sms[dev] : 0;
  if (per_sm == 0) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kWarps * 32, bytes)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    per_sm = max(per_sm, 1);
    if (dev < 64) {
      resident[dev] = per_sm;
      sms[dev] = n_sm;
    }
  }
  return cudaSuccess;
}

// Warps one launch spreads the work over: every resident warp of the device
// (one wave of persistent CTAs), at most kMaxDecodeWarps, or the override.
template <int BITS, int GQ, bool ROPE, bool KPT, bool PAGED, bool ROT, bool SP>
static cudaError_t launch_t(DecodeArgs a, cudaStream_t stream) {
  constexpr int kWarps = CtaShape<BITS, GQ, ROPE, KPT, SP>::W;
  int per_sm = 0, n_sm = 0, bytes = 0;
  cudaError_t e = kernel_slots<BITS, GQ, ROPE, KPT, PAGED, ROT, SP>(per_sm, n_sm, bytes);
  if (e != cudaSuccess) return e;
  const int over = decode_warps_override();
  int nw = over ? over : min(n_sm * per_sm * kWarps, kMaxDecodeWarps);
  nw = max(nw, 1);
  a.nw = nw;
  if (a.base != nullptr) {
    if ((e = launch_plan(a, stream)) != cudaSuccess) return e;
  }
  decode_kernel<BITS, GQ, ROPE, KPT, PAGED, ROT, SP><<<(nw + kWarps - 1) / kWarps, kWarps * 32, bytes, stream>>>(a);
  return cudaGetLastError();
}

template <int BITS, int GQ, bool PAGED, bool ROT, bool SP>
static cudaError_t launch_g(const DecodeArgs &a, cudaStream_t stream) {
  // keys grouped per token, rotating caches and dense-and-sparse blocks are
  // never stored pre-RoPE (rejected at the boundary)
  if (a.geo.kpt) return launch_t<BITS, GQ, false, true, PAGED, ROT, SP>(a, stream);
  if constexpr (!ROT && !SP) {
    if (a.geo.pre_rope) return launch_t<BITS, GQ, true, false, PAGED, false, false>(a, stream);
  }
  return launch_t<BITS, GQ, false, false, PAGED, ROT, SP>(a, stream);
}

template <int BITS, bool PAGED, bool ROT, bool SP>
static cudaError_t launch_b(const DecodeArgs &a, int gq, cudaStream_t stream) {
  switch (gq) {
    case 1: return launch_g<BITS, 1, PAGED, ROT, SP>(a, stream);
    case 2: return launch_g<BITS, 2, PAGED, ROT, SP>(a, stream);
    default: return launch_g<BITS, 4, PAGED, ROT, SP>(a, stream);
  }
}

}  // namespace kvq
