// Split-K decode attention read directly from the quantized cache.
//
// Source: "KV cache quantization", "Keys are harder than values" (the
// grouped part and the full-precision part of the cache are combined when
// computing attention scores; keys stored before RoPE are rotated after
// dequantization); "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV
// Cache", second and third paragraphs (what the groups and the window hold).
//
// The kernel is persistent and every warp is its own streaming engine: a
// warp takes work items (a run of `chunk` packed groups of one (sequence, KV
// head), or that pair's fp16 sink + window tokens) from a global counter,
// keeps a small ring of group blocks in flight with one-dimensional bulk
// copies completing on per-slot mbarriers, and already fetches the next
// item's first groups while it finishes the current one.  Each item leaves a
// partial (max, sum, unnormalized output) per query head; the warp that
// finishes the last item of a (sequence, KV head) merges them with a
// log-sum-exp and writes the fp16 output.  No CTA-wide synchronization
// happens after start-up.
//
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
#include <math.h>

#include "kvq_internal.cuh"

namespace kvq {

constexpr int kWarps = 4;              // independent warps per CTA
constexpr int kRopeOffStride = 65;     // padded row of the in-group rotation table
constexpr unsigned kFull = 0xffffffffu;

struct DecodeArgs {
  Geo geo;
  int Hq;
  const __half *q;          // [S][Hq][D]
  __half *out;              // [S][Hq][D]
  float zscale;             // softmax scale * log2(e)
  float *part_o;            // [S][Hq][nsp][D]
  float2 *part_ml;          // [S][Hq][nsp] (max, sum) in log2 units
  int *counters;            // [S][Hkv] items finished, zeroed before the launch
  int *work;                // next work item, zeroed before the launch
  int items;                // S * Hkv * nsp
  int nsp;                  // items per (sequence, KV head): window passes + chunks
  int tail_passes;          // window/sink items per (sequence, KV head), 32 tokens each
  int chunk;                // groups per item
  int max_len;              // host bound on seq_len the plan was sized for
  const float2 *rope_base;  // [n_base][64]: cos, sin of (num_sink + 32 r) * omega_i
  const float2 *rope_off;   // [32][64]: cos, sin of delta * omega_i
};

// Shared memory of one warp: a ring of NS group blocks, one mbarrier per
// slot, and the query of the current item (fp32, up to 4 heads).
// Ring slots (group blocks in flight) per warp.
#ifndef KVQ_DECODE_RING_2BIT
#define KVQ_DECODE_RING_2BIT 3
#endif
#ifndef KVQ_DECODE_RING_4BIT
#define KVQ_DECODE_RING_4BIT 2
#endif

template <int BITS>
struct WarpSmem {
  static constexpr int BB = block_bytes(BITS);
  static constexpr int NS = BITS == 2 ? KVQ_DECODE_RING_2BIT : KVQ_DECODE_RING_4BIT;
  static constexpr int BAR_OFF = NS * BB;
  static constexpr int Q_OFF = (BAR_OFF + NS * 8 + 15) / 16 * 16;
  static constexpr int BYTES = (Q_OFF + 4 * kD * 4 + 127) / 128 * 128;
  static_assert(BB % 16 == 0, "bulk copies need 16-byte multiples");
};

// Post-scale of a key score row tau (0..3 = token 8*tau + g) and of a value
// output row (channel 16*mt + 8*h + g): undo the code << (b*u) * 2^-24.
template <int BITS>
__device__ __forceinline__ float key_row_scale(int tau) {
  const int u = BITS == 2 ? tau : (tau & 1);
  return __int_as_float((127 + 24 - BITS * u) << 23);
}
template <int BITS>
__device__ __forceinline__ float val_row_scale(int mt, int hh) {
  const int u = BITS == 2 ? 2 * (mt & 1) + hh : hh;
  return __int_as_float((127 + 24 - BITS * u) << 23);
}

// fp16 pair of (x0, x1) when lo_sel == 0, or of the rounding remainder
// (x - fp16(x)) when lo_sel == 1: the high and low parts of a two-term split.
__device__ __forceinline__ uint32_t split_part(float x0, float x1, float lo_sel) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 f = __half22float2(h);
  return h2_as_u32(__floats2half2_rn(fmaf(-lo_sel, f.x, x0), fmaf(-lo_sel, f.y, x1)));
}

// Query side of the score mma.  build() returns, per group, bq[kt][j] = the
// B-fragment register of this lane (column g: query head g/2, high part for
// even g, low part for odd g; channels 16kt + 8j + 2q + {0,1}) and beta =
// sum_d q_d min_d of head q, both for the normalized query q / 2^e.
template <int GQ>
struct QkOperand {
  // GQ <= 2: the 64 channel pairs x heads x {high, low} are spread over all
  // 32 lanes (lane = pair % PL + PL * part + 2 PL * head) and gathered with
  // one shuffle per fragment register.  GQ == 4: each lane computes exactly
  // the 16 pairs its own fragment holds.
  static constexpr bool kGather = GQ <= 2;
  static constexpr int PL = kGather ? 16 / GQ : 4;
  static constexpr int NR = kGather ? 4 * GQ : 16;
  float qv[2 * NR];
  float lo_sel;
  int pbase;
  int head_lane;
  float qscale;

  __device__ __forceinline__ int channel(int r) const {
    return kGather ? 2 * (pbase + PL * r) : 16 * (r >> 1) + 8 * (r & 1) + 2 * pbase;
  }

  __device__ __forceinline__ void init(const float *q_s, int lane, float zscale) {
    const int g = lane >> 2, q = lane & 3;
    int hd;
    if (kGather) {
      pbase = lane % PL;
      lo_sel = static_cast<float>((lane / PL) & 1);
      hd = min(lane / (2 * PL), GQ - 1);
    } else {
      pbase = q;
      lo_sel = static_cast<float>(g & 1);
      hd = min(g >> 1, GQ - 1);
    }
    float amax = 0.f;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int ch = channel(r);
      qv[2 * r] = q_s[hd * kD + ch];
      qv[2 * r + 1] = q_s[hd * kD + ch + 1];
      amax = fmaxf(amax, fmaxf(fabsf(qv[2 * r]), fabsf(qv[2 * r + 1])));
    }
#pragma unroll
    for (int off = 1; off < (kGather ? PL : 4); off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, off));
    int ex;
    frexpf(amax, &ex);  // |q / 2^ex| < 1 keeps q * scale inside the fp16 range
#pragma unroll
    for (int i = 0; i < 2 * NR; ++i) qv[i] = ldexpf(qv[i], -ex);
    head_lane = kGather ? min(2 * PL * q, 31) : 8 * q;
    qscale = ldexpf(zscale, __shfl_sync(kFull, ex, head_lane));
  }

  __device__ __forceinline__ void build(const float *ks, const float *km, int lane, uint32_t (&bq)[8][2],
                                        float &beta) const {
    const int g = lane >> 2, q = lane & 3;
    uint32_t v[NR];
    float bp = 0.f;
#pragma unroll
    for (int r = 0; r < NR; ++r) {
      const int ch = channel(r);
      const float2 sc = *reinterpret_cast<const float2 *>(ks + ch);
      const float2 mn = *reinterpret_cast<const float2 *>(km + ch);
      v[r] = split_part(qv[2 * r] * sc.x, qv[2 * r + 1] * sc.y, lo_sel);
      bp = fmaf(qv[2 * r], mn.x, fmaf(qv[2 * r + 1], mn.y, bp));
    }
    if (kGather) {
      bp = lo_sel != 0.f ? 0.f : bp;  // each pair counted once, by its high-part lane
#pragma unroll
      for (int off = 1; off < PL; off <<= 1) bp += __shfl_xor_sync(kFull, bp, off);
      const int src_hi = PL * (g & 1) + 2 * PL * (g >> 1);
#pragma unroll
      for (int kt = 0; kt < 8; ++kt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int P = 8 * kt + 4 * j + q;
          bq[kt][j] = __shfl_sync(kFull, v[(8 * kt) / PL], (P % PL + src_hi) & 31);
        }
    } else {
#pragma unroll
      for (int kt = 0; kt < 8; ++kt) {
        bq[kt][0] = v[2 * kt];
        bq[kt][1] = v[2 * kt + 1];
      }
      bp += __shfl_xor_sync(kFull, bp, 1);
      bp += __shfl_xor_sync(kFull, bp, 2);
    }
    beta = __shfl_sync(kFull, bp, head_lane) * qscale;
  }
};

// o[mt] += A(value codes) * bp for one group: o rows are channels 16mt+g and
// 16mt+8+g, columns 2q / 2q+1 (high / low part of query head q).
template <int BITS>
__device__ __forceinline__ void pv_mma(const uint8_t *vc, int lane, const uint32_t (&bp)[2][2], float (&o)[8][4]) {
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
__device__ __forceinline__ void qk_mma(const uint8_t *kc, int lane, const uint32_t (&bq)[8][2], float (&acc)[2][4]) {
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
__device__ __forceinline__ uint32_t key_word(const uint8_t *kc, int t, int kt, int qq) {
  constexpr int NU = 8 / BITS;
  const int tau = t >> 3;
  const int w = kt * (4 / NU) + tau / NU;
  const int lane = 4 * (t & 7) + qq;
  return reinterpret_cast<const uint32_t *>(kc)[((w >> 2) * 32 + lane) * 4 + (w & 3)];
}

// Per-warp decode work item of one (sequence, KV head).  Its items are
// numbered split = 0 .. nsp-1: the first `tail_passes` cover the fp16 sink +
// window tokens 32 at a time (scheduled first: they are the slowest per
// byte), the rest are runs of `chunk` packed groups.  kind: 1 = groups
// [g0, g0+ng); 2 = window/sink tokens [32*split, 32*split + 32); 3 = zero the
// output rows (empty sequence, or length out of range); 0 = nothing to do;
// -1 = past the end.  nparts = partial results the (sequence, KV head)
// produces in total.
struct Item {
  int s, h, split, kind, g0, ng, tparts, nparts;
  Split spl;
};

__device__ __forceinline__ Item item_of(const DecodeArgs &a, int it) {
  Item x;
  x.kind = -1;
  x.s = x.h = x.split = x.g0 = x.ng = x.tparts = x.nparts = 0;
  x.spl.nsink = x.spl.Lq = x.spl.r = 0;
  if (it >= a.items) return x;
  const int per_s = a.geo.H * a.nsp;
  x.s = it / per_s;
  const int rem = it - x.s * per_s;
  x.h = rem / a.nsp;
  x.split = rem - x.h * a.nsp;
  const int L = a.geo.seq_len[x.s];
  x.kind = 0;
  if (L <= 0 || L > a.geo.capacity || L > a.max_len) {
    if (x.split == 0) x.kind = 3;
    return x;
  }
  x.spl = split_len(L, a.geo.ns, a.geo.R);
  const int ng_all = x.spl.Lq / kG;
  const int nchunks = (ng_all + a.chunk - 1) / a.chunk;
  x.tparts = (x.spl.nsink + x.spl.r + 31) / 32;
  x.nparts = x.tparts + nchunks;
  if (x.split < a.tail_passes) {
    if (x.split < x.tparts) x.kind = 2;
  } else {
    const int c = x.split - a.tail_passes;
    if (c < nchunks) {
      x.kind = 1;
      x.g0 = c * a.chunk;
      x.ng = min(a.chunk, ng_all - x.g0);
    }
  }
  return x;
}

// Scores of one packed group for this lane: z[tau] = log2-domain logit of
// token 8*tau + g for query head q.
template <int BITS, int GQ>
__device__ __forceinline__ void group_scores(const uint8_t *blk, const QkOperand<GQ> &qo, const float (&kfac)[4],
                                             int lane, float (&z)[4]) {
  uint32_t bq[8][2];
  float beta;
  qo.build(reinterpret_cast<const float *>(blk + off_ks(BITS)), reinterpret_cast<const float *>(blk + off_km(BITS)),
           lane, bq, beta);
  float acc[2][4];
  qk_mma<BITS>(blk + off_kc(BITS), lane, bq, acc);
#pragma unroll
  for (int mt = 0; mt < 2; ++mt)
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) z[2 * mt + hh] = fmaf(acc[mt][2 * hh] + acc[mt][2 * hh + 1], kfac[2 * mt + hh], beta);
}

// o += values of one group weighted by ps (score layout: token 8*tau + g,
// head q).  The value mma's B column h carries head h's p_t * scale_t as one
// fp16 (its rounding error, at most 2^-11 relative per weight, enters the
// output linearly); o columns 2q and 2q+1 of this lane are heads 2q, 2q+1.
template <int BITS>
__device__ __forceinline__ void group_values(const uint8_t *blk, const float (&ps)[4], int lane, float (&o)[8][4]) {
  const int q = lane & 3, gcol = lane >> 2;
  uint32_t bp[2][2];
#pragma unroll
  for (int kt = 0; kt < 2; ++kt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float v0 = __shfl_sync(kFull, ps[2 * kt + j], (4 * (2 * q) + gcol) & 31);
      const float v1 = __shfl_sync(kFull, ps[2 * kt + j], (4 * (2 * q + 1) + gcol) & 31);
      bp[kt][j] = h2_as_u32(__floats2half2_rn(v0, v1));
    }
  pv_mma<BITS>(blk + off_vc(BITS), lane, bp, o);
}

// Scale the o columns of heads 2q and 2q+1 by their softmax rescale factors.
__device__ __forceinline__ void rescale_o(float (&o)[8][4], float a_lo, float a_hi) {
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    o[i][0] *= a_lo;
    o[i][1] *= a_hi;
    o[i][2] *= a_lo;
    o[i][3] *= a_hi;
  }
}

template <int BITS, int GQ, bool ROPE>
__global__ void __launch_bounds__(kWarps * 32, ROPE ? 2 : (GQ == 4 ? 3 : 4)) decode_kernel(DecodeArgs a) {
  using WS = WarpSmem<BITS>;
  constexpr int NS = WS::NS, BB = WS::BB;
  extern __shared__ __align__(128) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;
  uint8_t *ring = smem + warp * WS::BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + WS::BAR_OFF);
  float *q_s = reinterpret_cast<float *>(ring + WS::Q_OFF);              // [GQ][D]
  float2 *roff_s = reinterpret_cast<float2 *>(smem + kWarps * WS::BYTES);  // [32][65]
  const Geo &geo = a.geo;

  if (ROPE) {
    for (int i = threadIdx.x; i < kG * 64; i += blockDim.x)
      roff_s[(i >> 6) * kRopeOffStride + (i & 63)] = a.rope_off[i];
  }
  if (lane == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(&full[i], 1);
    fence_mbar_init();
  }
  __syncthreads();  // the only CTA-wide barrier: from here each warp runs alone

  const bool head_valid = q < GQ;
    uint32_t fseq = 0, cseq = 0;                     // ring groups issued / consumed
  bool ok = true;

#ifndef KVQ_DECODE_STATIC
#define KVQ_DECODE_STATIC 0
#endif
  int k_static = 0;
  auto grab = [&]() {
    int it = 0;
    if (KVQ_DECODE_STATIC) {
      it = (blockIdx.x * kWarps + warp) + (k_static++) * static_cast<int>(gridDim.x * kWarps);
    } else if (lane == 0) {
      it = atomicAdd(a.work, 1);
    }
    return it;
  };
  Item cur = item_of(a, __shfl_sync(kFull, grab(), 0)), nxt;
  int cur_fetched = 0, nxt_fetched = 0;
  bool have_nxt = false;
  int nid = 0;

  // issue the next group of `it` into the next ring slot (lane 0 issues)
  auto issue = [&](const Item &it, int gidx) {
    if (lane == 0) {
      const uint32_t slot = fseq % NS;
      const uint8_t *src =
          geo.blocks + ((static_cast<size_t>(it.s) * geo.H + it.h) * geo.max_groups + it.g0 + gidx) * BB;
      fence_proxy_async();  // generic reads of the slot before the async write
      mbar_arrive_expect_tx(&full[slot], BB);
      bulk_g2s(ring + slot * BB, src, BB, &full[slot]);
    }
    ++fseq;
  };
  auto top_up = [&]() {
    while (fseq - cseq < static_cast<uint32_t>(NS)) {
      if (cur.kind == 1 && cur_fetched < cur.ng) {
        issue(cur, cur_fetched++);
      } else if (have_nxt && nxt.kind == 1 && nxt_fetched < nxt.ng) {
        issue(nxt, nxt_fetched++);
      } else {
        break;
      }
    }
  };
  top_up();
  // the next item is claimed at the start of the current one and resolved
  // (its lengths read, its first groups fetched) once the first groups of
  // the current item are under way, so the claim's latency stays hidden
  auto resolve = [&]() {
    if (!have_nxt) {
      nxt = item_of(a, __shfl_sync(kFull, nid, 0));
      nxt_fetched = 0;
      have_nxt = true;
      top_up();
    }
  };

  while (cur.kind != -1) {
    nid = grab();
    if (cur.kind != 1 || ROPE) resolve();
    const size_t orow0 = (static_cast<size_t>(cur.s) * a.Hq + static_cast<size_t>(cur.h) * GQ) * kD;
    const size_t prow0 = (static_cast<size_t>(cur.s) * a.Hq + static_cast<size_t>(cur.h) * GQ) * a.nsp + cur.split;
    if (cur.kind == 3) {
      for (int i = lane; i < GQ * kD; i += 32) a.out[orow0 + i] = __float2half_rn(0.f);
      if (lane == 0 && cur.h == 0 && geo.seq_len[cur.s] > a.max_len) set_status(geo.status, KVQ_STATUS_MAX_LEN);
    } else if (cur.kind == 1 || cur.kind == 2) {
      __syncwarp();  // the previous item's reads of q_s are done
      for (int i = lane; i < GQ * kD; i += 32) q_s[i] = __half2float(a.q[orow0 + i]);
      __syncwarp();
      if (cur.kind == 1) {
        // ---------------------------------------------------- quantized groups
        float o[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
        float m_run = -INFINITY, l_run = 0.f, mu_run = 0.f;
        if (!ROPE) {
          QkOperand<GQ> qo;
          qo.init(q_s, lane, a.zscale);
          float kfac[4];
#pragma unroll
          for (int tau = 0; tau < 4; ++tau) kfac[tau] = key_row_scale<BITS>(tau) * qo.qscale;
          // two groups (64 tokens) per iteration: independent score mmas, one
          // softmax update, two value mmas
          for (int gi = 0; gi < cur.ng; gi += 2) {
            const bool two = gi + 1 < cur.ng;
            const uint32_t sa = cseq % NS, sb = (cseq + 1) % NS;
            if (!mbar_wait_bounded(&full[sa], (cseq / NS) & 1) ||
                (two && !mbar_wait_bounded(&full[sb], ((cseq + 1) / NS) & 1))) {
              ok = false;
              break;
            }
            const uint8_t *ba = ring + sa * BB, *bb = ring + sb * BB;
            float za[4], zb[4];
            group_scores<BITS, GQ>(ba, qo, kfac, lane, za);
            if (two) {
              group_scores<BITS, GQ>(bb, qo, kfac, lane, zb);
            } else {
              zb[0] = zb[1] = zb[2] = zb[3] = -INFINITY;
            }
            float mx = fmaxf(fmaxf(fmaxf(za[0], za[1]), fmaxf(za[2], za[3])),
                             fmaxf(fmaxf(zb[0], zb[1]), fmaxf(zb[2], zb[3])));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = fast_exp2(m_run - m_new);
            const float *vsa = reinterpret_cast<const float *>(ba + off_vs(BITS));
            const float *vma = reinterpret_cast<const float *>(ba + off_vm(BITS));
            const float *vsb = reinterpret_cast<const float *>(bb + off_vs(BITS));
            const float *vmb = reinterpret_cast<const float *>(bb + off_vm(BITS));
            float psa[4], psb[4], psum = 0.f, mus = 0.f;
#pragma unroll
            for (int tau = 0; tau < 4; ++tau) {
              const float pa = fast_exp2(za[tau] - m_new);
              psum += pa;
              psa[tau] = pa * vsa[8 * tau + g];
              mus = fmaf(pa, vma[8 * tau + g], mus);
            }
            if (two) {
#pragma unroll
              for (int tau = 0; tau < 4; ++tau) {
                const float pb = fast_exp2(zb[tau] - m_new);
                psum += pb;
                psb[tau] = pb * vsb[8 * tau + g];
                mus = fmaf(pb, vmb[8 * tau + g], mus);
              }
            }
            l_run = fmaf(l_run, alpha, psum);
            mu_run = fmaf(mu_run, alpha, mus);
            m_run = m_new;
            if (__any_sync(kFull, head_valid && alpha != 1.f))
              rescale_o(o, __shfl_sync(kFull, alpha, (2 * q) & 31), __shfl_sync(kFull, alpha, (2 * q + 1) & 31));
            group_values<BITS>(ba, psa, lane, o);
            if (two) group_values<BITS>(bb, psb, lane, o);
            resolve();
            __syncwarp();
            cseq += two ? 2 : 1;
            top_up();
          }
        } else {
          // pre-RoPE keys: one lane per token, dequantize, rotate, dot
          float m_all[GQ];
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) m_all[hh] = -INFINITY;
          for (int gi = 0; gi < cur.ng; ++gi) {
            const uint32_t slot = cseq % NS;
            if (!mbar_wait_bounded(&full[slot], (cseq / NS) & 1)) {
              ok = false;
              break;
            }
            const uint8_t *blk = ring + slot * BB;
            const float *ks = reinterpret_cast<const float *>(blk + off_ks(BITS));
            const float *km = reinterpret_cast<const float *>(blk + off_km(BITS));
            const float *vs = reinterpret_cast<const float *>(blk + off_vs(BITS));
            const float *vm = reinterpret_cast<const float *>(blk + off_vm(BITS));
            const uint8_t *kc = blk + off_kc(BITS);
            const float2 *base = a.rope_base + static_cast<size_t>(cur.g0 + gi) * 64;
            const int t = lane;
            const int u = (t >> 3) % (8 / BITS);
            float dot[GQ];
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) dot[hh] = 0.f;
#pragma unroll 1
            for (int kt = 0; kt < 4; ++kt) {
#pragma unroll
              for (int qq = 0; qq < 4; ++qq) {
                const uint32_t wa = key_word<BITS>(kc, t, kt, qq);
                const uint32_t wb = key_word<BITS>(kc, t, kt + 4, qq);
#pragma unroll
                for (int j = 0; j < 2; ++j)
#pragma unroll
                  for (int e = 0; e < 2; ++e) {
                    const int ch = 16 * kt + 8 * j + 2 * qq + e;
                    const int sh = 16 * e + 8 * j + BITS * u;
                    const float ca = static_cast<float>((wa >> sh) & ((1u << BITS) - 1u));
                    const float cb = static_cast<float>((wb >> sh) & ((1u << BITS) - 1u));
                    const float k1 = fmaf(ca, ks[ch], km[ch]);
                    const float k2 = fmaf(cb, ks[ch + 64], km[ch + 64]);
                    const float2 bs = base[ch];
                    const float2 of = roff_s[t * kRopeOffStride + ch];
                    const float cs = bs.x * of.x - bs.y * of.y;
                    const float sn = bs.y * of.x + bs.x * of.y;
                    const float r1 = k1 * cs - k2 * sn;
                    const float r2 = k2 * cs + k1 * sn;
#pragma unroll
                    for (int hh = 0; hh < GQ; ++hh)
                      dot[hh] = fmaf(q_s[hh * kD + ch], r1, fmaf(q_s[hh * kD + ch + 64], r2, dot[hh]));
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
                  if (hh == g) {
                    v0 = a0;
                    v1 = a1;
                  }
                }
                bp[kt][j] = h2_as_u32(__floats2half2_rn(v0, v1));
              }
            pv_mma<BITS>(blk + off_vc(BITS), lane, bp, o);
            resolve();
            __syncwarp();
            ++cseq;
            top_up();
          }
        }
        if (!ok) break;
        // this item's partial state per query head
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
          l_run += __shfl_xor_sync(kFull, l_run, off);
          mu_run += __shfl_xor_sync(kFull, mu_run, off);
        }
        {
          const float mu_c[2] = {__shfl_sync(kFull, mu_run, (2 * q) & 31), __shfl_sync(kFull, mu_run, (2 * q + 1) & 31)};
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (2 * q + c < GQ) {
              float *po = a.part_o + (prow0 + static_cast<size_t>(2 * q + c) * a.nsp) * kD;
#pragma unroll
              for (int mt = 0; mt < 8; ++mt)
#pragma unroll
                for (int rr = 0; rr < 2; ++rr)
                  po[16 * mt + 8 * rr + g] = fmaf(o[mt][2 * rr + c], val_row_scale<BITS>(mt, rr), mu_c[c]);
            }
          }
          if (head_valid && g == 0) a.part_ml[prow0 + static_cast<size_t>(q) * a.nsp] = make_float2(m_run, l_run);
        }
      } else {
        // ------------------ 32 sink / window tokens, CUDA cores, one per lane
        const int T = cur.spl.nsink + cur.spl.r;
        const int t0 = 32 * cur.split;
        const int nt = min(32, T - t0);
        const size_t sh = static_cast<size_t>(cur.s) * geo.H + cur.h;
        const int i = t0 + lane;
        const bool valid = lane < nt;
        float dot[GQ];
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) dot[hh] = 0.f;
        if (valid) {
          int pos;
          const __half *kp;
          if (i < cur.spl.nsink) {
            pos = i;
            kp = geo.k_sink + (sh * geo.ns + i) * kD;
          } else {
            const int slot = i - cur.spl.nsink;
            pos = cur.spl.nsink + cur.spl.Lq + slot;
            kp = geo.k_res + (sh * geo.R + slot) * kD;
          }
          const int sidx = pos - geo.ns;  // stream index (negative for the sink)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            uint4 ra[4], rb[4];  // channels 32*half + 8c.. and 64 + 32*half + 8c..
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              ra[c] = *reinterpret_cast<const uint4 *>(kp + 32 * half + 8 * c);
              rb[c] = *reinterpret_cast<const uint4 *>(kp + 64 + 32 * half + 8 * c);
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const __half *ha = reinterpret_cast<const __half *>(&ra[c]);
              const __half *hb = reinterpret_cast<const __half *>(&rb[c]);
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                const int ch = 32 * half + 8 * c + e;
                float k1 = __half2float(ha[e]), k2 = __half2float(hb[e]);
                if (ROPE && sidx >= 0) {
                  const float2 bs = a.rope_base[static_cast<size_t>(sidx >> 5) * 64 + ch];
                  const float2 of = roff_s[(sidx & 31) * kRopeOffStride + ch];
                  const float cs = bs.x * of.x - bs.y * of.y;
                  const float sn = bs.y * of.x + bs.x * of.y;
                  const float r1 = k1 * cs - k2 * sn, r2 = k2 * cs + k1 * sn;
                  k1 = r1;
                  k2 = r2;
                }
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh)
                  dot[hh] = fmaf(q_s[hh * kD + ch], k1, fmaf(q_s[hh * kD + ch + 64], k2, dot[hh]));
              }
            }
          }
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
        // values: lane holds channels 4*lane .. 4*lane+3; eight rows in flight
        for (int tb = 0; tb < nt; tb += 8) {
          uint2 raw[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int it = t0 + tb + u;
            raw[u] = make_uint2(0u, 0u);
            if (tb + u < nt) {
              const __half *vp = it < cur.spl.nsink ? geo.v_sink + (sh * geo.ns + it) * kD
                                                    : geo.v_res + (sh * geo.R + (it - cur.spl.nsink)) * kD;
              raw[u] = *reinterpret_cast<const uint2 *>(vp + 4 * lane);
            }
          }
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw[u].x));
            const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw[u].y));
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
              const float pt = __shfl_sync(kFull, p[hh], (tb + u) & 31);
              acc[hh][0] = fmaf(pt, v01.x, acc[hh][0]);
              acc[hh][1] = fmaf(pt, v01.y, acc[hh][1]);
              acc[hh][2] = fmaf(pt, v23.x, acc[hh][2]);
              acc[hh][3] = fmaf(pt, v23.y, acc[hh][3]);
            }
          }
        }
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh) {
          float *po = a.part_o + (prow0 + static_cast<size_t>(hh) * a.nsp) * kD;
          *reinterpret_cast<float4 *>(po + 4 * lane) = make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
          if (lane == 0) a.part_ml[prow0 + static_cast<size_t>(hh) * a.nsp] = make_float2(mh[hh], lh[hh]);
        }
      }
      // the last item of this (sequence, KV head) to finish merges them all;
      // lane 0's acq_rel add publishes the warp's partial (ordered before it
      // by the warp barrier) and observes every earlier item's
      __syncwarp();
      int last = 0;
      if (lane == 0)
        last = atom_add_acq_rel(&a.counters[static_cast<size_t>(cur.s) * geo.H + cur.h], 1) == cur.nparts - 1;
      if (__shfl_sync(kFull, last, 0)) {
        __threadfence();
        for (int hh = 0; hh < GQ; ++hh) {
          const size_t r0 = (static_cast<size_t>(cur.s) * a.Hq + static_cast<size_t>(cur.h) * GQ + hh) * a.nsp;
          // partial i lives at split i (window passes) or tail_passes + i - tparts (chunks)
          auto split_of = [&](int i) { return i < cur.tparts ? i : a.tail_passes + i - cur.tparts; };
          float M = -INFINITY;
          for (int i = lane; i < cur.nparts; i += 32) M = fmaxf(M, __ldcg(&a.part_ml[r0 + split_of(i)]).x);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
          float Ls = 0.f;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          if (M != -INFINITY) {
#pragma unroll 4
            for (int i = 0; i < cur.nparts; ++i) {
              const size_t r = r0 + split_of(i);
              const float2 ml = __ldcg(&a.part_ml[r]);
              const float4 ov = __ldcg(reinterpret_cast<const float4 *>(a.part_o + r * kD) + lane);
              const float wgt = ml.x == -INFINITY ? 0.f : fast_exp2(ml.x - M);
              Ls = fmaf(ml.y, wgt, Ls);
              acc.x = fmaf(ov.x, wgt, acc.x);
              acc.y = fmaf(ov.y, wgt, acc.y);
              acc.z = fmaf(ov.z, wgt, acc.z);
              acc.w = fmaf(ov.w, wgt, acc.w);
            }
          }
          const float inv = M == -INFINITY ? 0.f : 1.f / Ls;
          __half2 *op = reinterpret_cast<__half2 *>(a.out + orow0 + static_cast<size_t>(hh) * kD) + 2 * lane;
          op[0] = __floats2half2_rn(acc.x * inv, acc.y * inv);
          op[1] = __floats2half2_rn(acc.z * inv, acc.w * inv);
        }
      }
    }
    resolve();
    cur = nxt;
    cur_fetched = nxt_fetched;
    have_nxt = false;
  }
  if (!ok) {
    set_status(geo.status, KVQ_STATUS_TIMEOUT);
    // let this warp's copies still in flight land before it exits
    for (; cseq < fseq; ++cseq) mbar_wait_bounded(&full[cseq % NS], (cseq / NS) & 1);
  }
}

// cos/sin tables for on-the-fly RoPE, in fp64 then rounded to fp32:
// base[r][i] at angle (num_sink + 32 r) * omega_i, off[d][i] at d * omega_i,
// omega_i = theta^(-2i/D).
__global__ void rope_table_kernel(float2 *base, int n_base, float2 *off, int ns, float theta) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= (n_base + kG) * 64) return;
  const int r = idx / 64, i = idx % 64;
  const double omega = pow(static_cast<double>(theta), -2.0 * i / kD);
  const double ang = r < n_base ? static_cast<double>(ns + kG * r) * omega : static_cast<double>(r - n_base) * omega;
  double sn, cs;
  sincos(ang, &sn, &cs);
  const float2 v = make_float2(static_cast<float>(cs), static_cast<float>(sn));
  if (r < n_base)
    base[idx] = v;
  else
    off[(r - n_base) * 64 + i] = v;
}

// ---------------------------------------------------------------- host side

template <int BITS, int GQ, bool ROPE>
static cudaError_t launch_t(const DecodeArgs &a, cudaStream_t stream) {
  using WS = WarpSmem<BITS>;
  constexpr int bytes = kWarps * WS::BYTES + (ROPE ? kG * kRopeOffStride * 8 : 0);
  auto kern = decode_kernel<BITS, GQ, ROPE>;
  // per instantiation and device ordinal: attributes set, resident CTAs per SM
  static int resident[64] = {};
  static int sms[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int per_sm = dev < 64 ? resident[dev] : 0, n_sm = dev < 64 ? sms[dev] : 0;
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
  const long long want = (static_cast<long long>(a.items) + kWarps - 1) / kWarps;
  const int grid = static_cast<int>(min(want, static_cast<long long>(n_sm) * per_sm));
  kern<<<grid, kWarps * 32, bytes, stream>>>(a);
  return cudaGetLastError();
}

template <int BITS, int GQ>
static cudaError_t launch_g(const DecodeArgs &a, cudaStream_t stream) {
  return a.geo.pre_rope ? launch_t<BITS, GQ, true>(a, stream) : launch_t<BITS, GQ, false>(a, stream);
}

template <int BITS>
static cudaError_t launch_b(const DecodeArgs &a, int gq, cudaStream_t stream) {
  switch (gq) {
    case 1: return launch_g<BITS, 1>(a, stream);
    case 2: return launch_g<BITS, 2>(a, stream);
    default: return launch_g<BITS, 4>(a, stream);
  }
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

static int g_chunk_override = 0;

int set_decode_chunk(int groups) {
  if (groups != 0 && (groups < 4 || groups > 1024 || groups % 4 != 0)) return -1;
  g_chunk_override = groups;
  return 0;
}

DecodePlan plan_decode(const Geo &geo, int Hq, int max_len) {
  DecodePlan p;
  const Split sp = split_len(max_len, geo.ns, geo.R);
  const long long ng_max = sp.Lq / kG;
  int chunk = g_chunk_override;
  if (chunk == 0) {
    // about six items per warp of a full GB300 (152 SMs x 16 warps) so the
    // dynamic schedule balances, at least 8 groups per item, and at most
    // ~512 items per (sequence, KV head) so the final merge stays short
    const long long total = static_cast<long long>(geo.S) * geo.H * ng_max;
    long long c = (total + 6LL * 152 * 16 - 1) / (6LL * 152 * 16);
    c = max(c, (ng_max + 510) / 511);
    c = min(max(c, 8LL), 1024LL);
    chunk = static_cast<int>((c + 3) / 4 * 4);
  }
  p.chunk = chunk;
  p.tail_passes = (geo.R - 1 + geo.ns + 31) / 32;
  p.nsp = static_cast<int>((ng_max + chunk - 1) / chunk) + p.tail_passes;
  p.items = static_cast<long long>(geo.S) * geo.H * p.nsp;
  p.n_base = geo.pre_rope ? (max(max_len - geo.ns, 1) + kG - 1) / kG : 0;
  const size_t rows = static_cast<size_t>(geo.S) * Hq * p.nsp;
  p.off_ml = align256(rows * kD * sizeof(float));
  p.off_cnt = p.off_ml + align256(rows * sizeof(float2));
  p.cnt_bytes = (static_cast<size_t>(geo.S) * geo.H + 1) * sizeof(int);
  p.off_base = p.off_cnt + align256(p.cnt_bytes);
  p.off_off = p.off_base + align256(static_cast<size_t>(p.n_base) * 64 * sizeof(float2));
  p.bytes = p.off_off + (geo.pre_rope ? align256(kG * 64 * sizeof(float2)) : 0);
  return p;
}

cudaError_t launch_decode(const Geo &geo, int Hq, const __half *q, float softmax_scale, __half *out,
                          void *workspace, const DecodePlan &p, int max_len, cudaStream_t stream,
                          uint64_t *launches) {
  DecodeArgs a;
  a.geo = geo;
  a.Hq = Hq;
  a.q = q;
  a.out = out;
  a.zscale = softmax_scale * 1.4426950408889634f;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  a.part_o = reinterpret_cast<float *>(ws);
  a.part_ml = reinterpret_cast<float2 *>(ws + p.off_ml);
  a.counters = reinterpret_cast<int *>(ws + p.off_cnt);
  a.work = a.counters + static_cast<size_t>(geo.S) * geo.H;
  a.items = static_cast<int>(p.items);
  a.nsp = p.nsp;
  a.tail_passes = p.tail_passes;
  a.chunk = p.chunk;
  a.max_len = max_len;
  a.rope_base = reinterpret_cast<const float2 *>(ws + p.off_base);
  a.rope_off = reinterpret_cast<const float2 *>(ws + p.off_off);
  cudaError_t e = cudaMemsetAsync(a.counters, 0, p.cnt_bytes, stream);
  if (e != cudaSuccess) return e;
  if (geo.pre_rope) {
    const int n = (p.n_base + kG) * 64;
    rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(reinterpret_cast<float2 *>(ws + p.off_base), p.n_base,
                                                           reinterpret_cast<float2 *>(ws + p.off_off), geo.ns,
                                                           geo.theta);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int gq = Hq / geo.H;
  e = geo.bits == 2 ? launch_b<2>(a, gq, stream) : launch_b<4>(a, gq, stream);
  ++*launches;
  return e;
}

}  // namespace kvq
