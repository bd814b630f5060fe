// Split-K decode attention read directly from the quantized cache.
//
// Source: "KV cache quantization", "Keys are harder than values" (the
// grouped part and the full-precision part of the cache are combined when
// computing attention scores; keys stored before RoPE are rotated after
// dequantization); "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV
// Cache", second and third paragraphs (what the groups and the window hold).
//
// One CTA handles one split (a run of `chunk` groups, or the sink + window
// tail) of one (sequence, KV head) for all query heads of that KV head.  A
// producer warp streams the split's blocks into a shared-memory ring with
// bulk copies; four consumer warps take one group each per stage.  The CTA
// that finishes last for a (sequence, KV head) merges every split's
// (max, sum, output) with a log-sum-exp and writes the fp16 output, so one
// call is one kernel (plus a RoPE table kernel for pre-RoPE keys).
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

constexpr int kConsumerWarps = 4;
constexpr int kDecThreads = (kConsumerWarps + 1) * 32;
constexpr int kStageGroups = kConsumerWarps;  // one group per consumer warp per stage
constexpr int kRopeOffStride = 65;            // padded row of the in-group rotation table
constexpr int kMergeChunk = 512;              // split weights staged per pass of the final merge
constexpr unsigned kFull = 0xffffffffu;

struct DecodeArgs {
  Geo geo;
  int Hq;
  const __half *q;          // [S][Hq][D]
  __half *out;              // [S][Hq][D]
  float zscale;             // softmax scale * log2(e)
  float *part_o;            // [S][Hq][nsp][D]
  float2 *part_ml;          // [S][Hq][nsp] (max, sum) in log2 units
  int *counters;            // [S][Hkv] splits finished, zeroed before the launch
  int nsp;
  int chunk;                // groups per split
  int max_len;              // host bound on seq_len the grid and tables were sized for
  const float2 *rope_base;  // [n_base][64]: cos, sin of (num_sink + 32 r) * omega_i
  const float2 *rope_off;   // [32][64]: cos, sin of delta * omega_i
};

template <int BITS>
struct Stages {
  static constexpr int n = BITS == 2 ? 4 : 2;
};

template <int BITS, int NSTAGES>
struct DecSmem {
  static constexpr int BB = block_bytes(BITS);
  static constexpr int STAGE = kStageGroups * BB;
  static constexpr int BAR_OFF = NSTAGES * STAGE;
  static constexpr int Q_OFF = BAR_OFF + 2 * NSTAGES * 8;
  static constexpr int RED_OFF = Q_OFF + 4 * kD * 4;  // q for up to 4 heads
  static constexpr int ROPE_OFF = RED_OFF + 16 * 4;   // block-reduction scratch + flag
  static constexpr int BYTES_NOROPE = ROPE_OFF;
  static constexpr int BYTES_ROPE = ROPE_OFF + kG * kRopeOffStride * 8;
  // aliases of the ring once every stage is consumed: per-warp states, then
  // the merge weights
  static constexpr int MRG_BYTES = kConsumerWarps * 4 * (2 + kD) * 4;
  static_assert(STAGE * NSTAGES >= MRG_BYTES + kMergeChunk * 4, "merge area does not fit the ring");
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

// Block-wide max / sum over the CTA's threads (red: 8 floats of smem).
__device__ __forceinline__ float block_reduce(float v, bool is_max, float *red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float o = __shfl_xor_sync(kFull, v, off);
    v = is_max ? fmaxf(v, o) : v + o;
  }
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  v = red[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

template <int BITS, int GQ, bool ROPE, int NSTAGES>
__global__ void __launch_bounds__(kDecThreads, ROPE ? 2 : (GQ == 4 ? 3 : 4)) decode_split_kernel(DecodeArgs a) {
  using SM = DecSmem<BITS, NSTAGES>;
  constexpr int BB = SM::BB;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t *ring = smem;
  uint64_t *full_bar = reinterpret_cast<uint64_t *>(smem + SM::BAR_OFF);
  uint64_t *empty_bar = full_bar + NSTAGES;
  float *q_s = reinterpret_cast<float *>(smem + SM::Q_OFF);           // [GQ][D]
  float *red = reinterpret_cast<float *>(smem + SM::RED_OFF);         // [16]
  float2 *roff_s = reinterpret_cast<float2 *>(smem + SM::ROPE_OFF);   // [32][65]
  float *mrg_m = reinterpret_cast<float *>(smem);                      // [4][GQ]
  float *mrg_l = mrg_m + kConsumerWarps * GQ;                          // [4][GQ]
  float *mrg_o = mrg_l + kConsumerWarps * GQ;                          // [4][GQ][D]
  float *wts = reinterpret_cast<float *>(smem + SM::MRG_BYTES);        // [kMergeChunk]

  const Geo &geo = a.geo;
  const int s = blockIdx.z, h = blockIdx.y, sp = blockIdx.x;
  const int L = geo.seq_len[s];
  const size_t orow0 = (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(h) * GQ) * kD;
  if (L < 0 || L > geo.capacity || L > a.max_len) {
    if (sp == 0) {
      for (int i = threadIdx.x; i < GQ * kD; i += blockDim.x) a.out[orow0 + i] = __float2half_rn(0.f);
      if (L > a.max_len && h == 0 && threadIdx.x == 0) set_status(geo.status, KVQ_STATUS_MAX_LEN);
    }
    return;
  }
  const Split spl = split_len(L, geo.ns, geo.R);
  const int ng = spl.Lq / kG;
  const int nchunks = (ng + a.chunk - 1) / a.chunk;
  if (sp > nchunks) return;
  const bool tail = (sp == nchunks);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, q = lane & 3;

  for (int i = threadIdx.x; i < GQ * kD; i += blockDim.x) q_s[i] = __half2float(a.q[orow0 + i]);
  if (ROPE) {
    for (int i = threadIdx.x; i < kG * 64; i += blockDim.x)
      roff_s[(i >> 6) * kRopeOffStride + (i & 63)] = a.rope_off[i];
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < NSTAGES; ++i) {
      mbar_init(&full_bar[i], 1);
      mbar_init(&empty_bar[i], kConsumerWarps);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // Running softmax state of this lane: query head q of the output layout.
  float o[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
  float m_run = -INFINITY, l_run = 0.f, mu_run = 0.f;
  const bool head_valid = q < GQ;
  const float col_lo = static_cast<float>(g & 1);  // B column g: low part when odd
  const int hc = g >> 1;                           // B column g: query head

  if (!tail) {
    const int g0 = sp * a.chunk;
    const int ngr = min(ng, g0 + a.chunk) - g0;
    const int nst = (ngr + kStageGroups - 1) / kStageGroups;
    const uint8_t *src = geo.blocks + ((static_cast<size_t>(s) * geo.H + h) * geo.max_groups + g0) * BB;
    if (warp == kConsumerWarps) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        int issued = 0;
        for (int k = 0; k < nst; ++k) {
          const int slot = k % NSTAGES;
          if (k >= NSTAGES && !mbar_wait_bounded(&empty_bar[slot], ((k / NSTAGES) - 1) & 1)) {
            set_status(geo.status, KVQ_STATUS_TIMEOUT);
            break;
          }
          const int cnt = min(kStageGroups, ngr - k * kStageGroups);
          mbar_arrive_expect_tx(&full_bar[slot], cnt * BB);
          bulk_g2s(ring + slot * SM::STAGE, src + static_cast<size_t>(k) * SM::STAGE, cnt * BB, &full_bar[slot]);
          issued = k + 1;
        }
        // let every copy still in flight land before the ring is reused
        for (int k = max(0, issued - NSTAGES); k < issued; ++k)
          if (!mbar_wait_bounded(&full_bar[k % NSTAGES], (k / NSTAGES) & 1)) set_status(geo.status, KVQ_STATUS_TIMEOUT);
      }
    } else if (!ROPE) {
      // ------------------------------------------- consumer, tensor-core path
      QkOperand<GQ> qo;
      qo.init(q_s, lane, a.zscale);
      float kfac[4];
#pragma unroll
      for (int tau = 0; tau < 4; ++tau) kfac[tau] = key_row_scale<BITS>(tau) * qo.qscale;

      for (int k = 0; k < nst; ++k) {
        const int slot = k % NSTAGES;
        const int gi = k * kStageGroups + warp;
        if (gi < ngr) {
          if (!mbar_wait_bounded(&full_bar[slot], (k / NSTAGES) & 1)) {
            set_status(geo.status, KVQ_STATUS_TIMEOUT);
            break;
          }
          const uint8_t *blk = ring + slot * SM::STAGE + warp * BB;
          const float *vs = reinterpret_cast<const float *>(blk + off_vs(BITS));
          const float *vm = reinterpret_cast<const float *>(blk + off_vm(BITS));
          uint32_t bq[8][2];
          float beta;
          qo.build(reinterpret_cast<const float *>(blk + off_ks(BITS)),
                   reinterpret_cast<const float *>(blk + off_km(BITS)), lane, bq, beta);
          float acc[2][4];
          qk_mma<BITS>(blk + off_kc(BITS), lane, bq, acc);
          float z[4];
#pragma unroll
          for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              z[2 * mt + hh] = fmaf(acc[mt][2 * hh] + acc[mt][2 * hh + 1], kfac[2 * mt + hh], beta);

          // online softmax over the group's 32 tokens (8 lanes share head q)
          float mx = fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3]));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
          const float m_new = fmaxf(m_run, mx);
          const float alpha = exp2f(m_run - m_new);
          float ps[4], psum = 0.f, mus = 0.f;
#pragma unroll
          for (int tau = 0; tau < 4; ++tau) {
            const float p = exp2f(z[tau] - m_new);
            psum += p;
            ps[tau] = p * vs[8 * tau + g];
            mus = fmaf(p, vm[8 * tau + g], mus);
          }
          l_run = fmaf(l_run, alpha, psum);
          mu_run = fmaf(mu_run, alpha, mus);
          m_run = m_new;
          if (__any_sync(kFull, head_valid && alpha != 1.f)) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              o[i][0] *= alpha; o[i][1] *= alpha; o[i][2] *= alpha; o[i][3] *= alpha;
            }
          }
          // B operand of the value mma: tokens 16kt + 8j + 2q + e, head hc
          uint32_t bp[2][2];
#pragma unroll
          for (int kt = 0; kt < 2; ++kt)
#pragma unroll
            for (int j = 0; j < 2; ++j) {
              const float v0 = __shfl_sync(kFull, ps[2 * kt + j], (4 * (2 * q) + hc) & 31);
              const float v1 = __shfl_sync(kFull, ps[2 * kt + j], (4 * (2 * q + 1) + hc) & 31);
              bp[kt][j] = split_part(v0, v1, col_lo);
            }
          pv_mma<BITS>(blk + off_vc(BITS), lane, bp, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
      }
    } else {
      // ---------------------------------------- consumer, pre-RoPE keys path
      // one lane per token: dequantize, rotate at the token's position, dot
      float m_all[GQ];
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) m_all[hh] = -INFINITY;
      for (int k = 0; k < nst; ++k) {
        const int slot = k % NSTAGES;
        const int gi = k * kStageGroups + warp;
        if (gi < ngr) {
          if (!mbar_wait_bounded(&full_bar[slot], (k / NSTAGES) & 1)) {
            set_status(geo.status, KVQ_STATUS_TIMEOUT);
            break;
          }
          const uint8_t *blk = ring + slot * SM::STAGE + warp * BB;
          const float *ks = reinterpret_cast<const float *>(blk + off_ks(BITS));
          const float *km = reinterpret_cast<const float *>(blk + off_km(BITS));
          const float *vs = reinterpret_cast<const float *>(blk + off_vs(BITS));
          const float *vm = reinterpret_cast<const float *>(blk + off_vm(BITS));
          const uint8_t *kc = blk + off_kc(BITS);
          const float2 *base = a.rope_base + static_cast<size_t>(g0 + gi) * 64;
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
          float alpha_q = 1.f, psum_q = 0.f, mus_q = 0.f, m_q = m_run;
#pragma unroll
          for (int hh = 0; hh < GQ; ++hh) {
            const float z = dot[hh] * a.zscale;
            float mx = z;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
            const float m_new = fmaxf(m_all[hh], mx);
            const float alpha = exp2f(m_all[hh] - m_new);
            m_all[hh] = m_new;
            const float p = exp2f(z - m_new);
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
          }
          l_run = fmaf(l_run, alpha_q, g == 0 ? psum_q : 0.f);
          mu_run = fmaf(mu_run, alpha_q, g == 0 ? mus_q : 0.f);
          m_run = m_q;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i][0] *= alpha_q; o[i][1] *= alpha_q; o[i][2] *= alpha_q; o[i][3] *= alpha_q;
          }
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
                if (hh == hc) {
                  v0 = a0;
                  v1 = a1;
                }
              }
              bp[kt][j] = split_part(v0, v1, col_lo);
            }
          pv_mma<BITS>(blk + off_vc(BITS), lane, bp, o);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[slot]);
      }
    }
  }
  __syncthreads();  // ring free from here on: the merge area aliases it

  if (!tail) {
    if (warp < kConsumerWarps) {
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        l_run += __shfl_xor_sync(kFull, l_run, off);
        mu_run += __shfl_xor_sync(kFull, mu_run, off);
      }
      if (head_valid) {
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int ch = 16 * mt + 8 * hh + g;
            mrg_o[(warp * GQ + q) * kD + ch] =
                fmaf(o[mt][2 * hh] + o[mt][2 * hh + 1], val_row_scale<BITS>(mt, hh), mu_run);
          }
        if (g == 0) {
          mrg_m[warp * GQ + q] = m_run;
          mrg_l[warp * GQ + q] = l_run;
        }
      }
    }
  } else if (warp < kConsumerWarps) {
    // ------------------------------------------- sink + window, CUDA cores
    const int T = spl.nsink + spl.r;
    const int i = kG * warp + lane;
    const bool valid = i < T;
    const size_t sh = static_cast<size_t>(s) * geo.H + h;
    int pos = 0;
    const __half *kp = nullptr;
    if (valid) {
      if (i < spl.nsink) {
        pos = i;
        kp = geo.k_sink + (sh * geo.ns + i) * kD;
      } else {
        const int slot = i - spl.nsink;
        pos = spl.nsink + spl.Lq + slot;
        kp = geo.k_res + (sh * geo.R + slot) * kD;
      }
    }
    float dot[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) dot[hh] = 0.f;
    if (valid) {
      const int sidx = pos - geo.ns;  // stream index (negative for the sink)
#pragma unroll 1
      for (int c8 = 0; c8 < 8; ++c8) {
        const uint4 ra = *reinterpret_cast<const uint4 *>(kp + c8 * 8);
        const uint4 rb = *reinterpret_cast<const uint4 *>(kp + 64 + c8 * 8);
        const __half *ha = reinterpret_cast<const __half *>(&ra);
        const __half *hb = reinterpret_cast<const __half *>(&rb);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int ch = c8 * 8 + e;
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
    float p[GQ], mh[GQ], lh[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
      const float zz = valid ? dot[hh] * a.zscale : -INFINITY;
      float mx = zz;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
      p[hh] = valid ? exp2f(zz - mx) : 0.f;
      float sum = p[hh];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(kFull, sum, off);
      mh[hh] = mx;
      lh[hh] = sum;
    }
    float acc[GQ][4];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) acc[hh][0] = acc[hh][1] = acc[hh][2] = acc[hh][3] = 0.f;
    const int nt = min(kG, T - kG * warp);
    for (int t = 0; t < nt; ++t) {
      const int it = kG * warp + t;
      const __half *vp = it < spl.nsink ? geo.v_sink + (sh * geo.ns + it) * kD
                                        : geo.v_res + (sh * geo.R + (it - spl.nsink)) * kD;
      const uint2 raw = *reinterpret_cast<const uint2 *>(vp + 4 * lane);
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2 *>(&raw.y));
#pragma unroll
      for (int hh = 0; hh < GQ; ++hh) {
        const float pt = __shfl_sync(kFull, p[hh], t);
        acc[hh][0] = fmaf(pt, v01.x, acc[hh][0]);
        acc[hh][1] = fmaf(pt, v01.y, acc[hh][1]);
        acc[hh][2] = fmaf(pt, v23.x, acc[hh][2]);
        acc[hh][3] = fmaf(pt, v23.y, acc[hh][3]);
      }
    }
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) {
      *reinterpret_cast<float4 *>(&mrg_o[(warp * GQ + hh) * kD + 4 * lane]) =
          make_float4(acc[hh][0], acc[hh][1], acc[hh][2], acc[hh][3]);
      if (lane == 0) {
        mrg_m[warp * GQ + hh] = mh[hh];
        mrg_l[warp * GQ + hh] = lh[hh];
      }
    }
  }
  __syncthreads();

  // this split's (max, sum, unnormalized output) per query head
  const size_t prow0 = (static_cast<size_t>(s) * a.Hq + static_cast<size_t>(h) * GQ) * a.nsp;
  for (int idx = threadIdx.x; idx < GQ * kD; idx += blockDim.x) {
    const int hh = idx / kD, ch = idx % kD;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mrg_m[w * GQ + hh]);
    float Ls = 0.f, Os = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float mw = mrg_m[w * GQ + hh];
        if (mw != -INFINITY) {
          const float f = exp2f(mw - M);
          Ls = fmaf(mrg_l[w * GQ + hh], f, Ls);
          Os = fmaf(mrg_o[(w * GQ + hh) * kD + ch], f, Os);
        }
      }
    }
    const size_t row = prow0 + static_cast<size_t>(hh) * a.nsp + sp;
    a.part_o[row * kD + ch] = Os;
    if (ch == 0) a.part_ml[row] = make_float2(M, Ls);
  }

  // the last split of this (sequence, KV head) to finish merges them all
  __threadfence();
  __syncthreads();
  int *flag = reinterpret_cast<int *>(red + 8);
  if (threadIdx.x == 0) *flag = atomicAdd(&a.counters[static_cast<size_t>(s) * geo.H + h], 1) == nchunks;
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  const int nsplit = nchunks + 1;
  for (int hh = 0; hh < GQ; ++hh) {
    const size_t r0 = prow0 + static_cast<size_t>(hh) * a.nsp;
    float M = -INFINITY;
    for (int i = threadIdx.x; i < nsplit; i += blockDim.x) M = fmaxf(M, __ldcg(&a.part_ml[r0 + i]).x);
    M = block_reduce(M, true, red);
    float lpart = 0.f, acc = 0.f;
    for (int c0 = 0; c0 < nsplit; c0 += kMergeChunk) {
      const int n = min(kMergeChunk, nsplit - c0);
      __syncthreads();  // the previous chunk's weights are consumed
      for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const float2 ml = __ldcg(&a.part_ml[r0 + c0 + i]);
        const float wgt = ml.x == -INFINITY ? 0.f : exp2f(ml.x - M);
        wts[i] = wgt;
        lpart = fmaf(ml.y, wgt, lpart);
      }
      __syncthreads();
      if (threadIdx.x < kD) {
        const float *po = a.part_o + (r0 + c0) * kD + threadIdx.x;
#pragma unroll 4
        for (int i = 0; i < n; ++i) acc = fmaf(__ldcg(po + static_cast<size_t>(i) * kD), wts[i], acc);
      }
    }
    const float Ls = block_reduce(lpart, false, red);
    if (threadIdx.x < kD)
      a.out[orow0 + static_cast<size_t>(hh) * kD + threadIdx.x] = __float2half_rn(M == -INFINITY ? 0.f : acc / Ls);
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
static cudaError_t launch_split_t(const DecodeArgs &a, dim3 grid, cudaStream_t stream) {
  constexpr int NST = Stages<BITS>::n;
  using SM = DecSmem<BITS, NST>;
  constexpr int bytes = ROPE ? SM::BYTES_ROPE : SM::BYTES_NOROPE;
  auto kern = decode_split_kernel<BITS, GQ, ROPE, NST>;
  static unsigned long long attr_set = 0;  // per instantiation: one bit per device ordinal
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !(attr_set >> dev & 1ULL)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (dev < 64) attr_set |= 1ULL << dev;
  }
  kern<<<grid, kDecThreads, bytes, stream>>>(a);
  return cudaGetLastError();
}

template <int BITS, int GQ>
static cudaError_t launch_split_g(const DecodeArgs &a, dim3 grid, cudaStream_t stream) {
  return a.geo.pre_rope ? launch_split_t<BITS, GQ, true>(a, grid, stream)
                        : launch_split_t<BITS, GQ, false>(a, grid, stream);
}

template <int BITS>
static cudaError_t launch_split_b(const DecodeArgs &a, int gq, dim3 grid, cudaStream_t stream) {
  switch (gq) {
    case 1: return launch_split_g<BITS, 1>(a, grid, stream);
    case 2: return launch_split_g<BITS, 2>(a, grid, stream);
    default: return launch_split_g<BITS, 4>(a, grid, stream);
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
  const int ng_max = sp.Lq / kG;
  int chunk = g_chunk_override;
  if (chunk == 0) {
    // about 32 groups (1024 tokens) per split, smaller when the (sequence,
    // head) count alone cannot fill a few waves of the GPU
    chunk = 32;
    const long long pairs = static_cast<long long>(geo.S) * geo.H;
    while (chunk > 8 && pairs * ((ng_max + chunk - 1) / chunk) < 4LL * 152 * 4) chunk /= 2;
  }
  p.chunk = chunk;
  p.nsp = (ng_max + chunk - 1) / chunk + 1;
  p.n_base = geo.pre_rope ? (max(max_len - geo.ns, 1) + kG - 1) / kG : 0;
  const size_t rows = static_cast<size_t>(geo.S) * Hq * p.nsp;
  p.off_ml = align256(rows * kD * sizeof(float));
  p.off_cnt = p.off_ml + align256(rows * sizeof(float2));
  p.off_base = p.off_cnt + align256(static_cast<size_t>(geo.S) * geo.H * sizeof(int));
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
  a.nsp = p.nsp;
  a.chunk = p.chunk;
  a.max_len = max_len;
  a.rope_base = reinterpret_cast<const float2 *>(ws + p.off_base);
  a.rope_off = reinterpret_cast<const float2 *>(ws + p.off_off);
  cudaError_t e = cudaMemsetAsync(a.counters, 0, static_cast<size_t>(geo.S) * geo.H * sizeof(int), stream);
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
  dim3 grid(p.nsp, geo.H, geo.S);
  e = geo.bits == 2 ? launch_split_b<2>(a, gq, grid, stream) : launch_split_b<4>(a, gq, grid, stream);
  ++*launches;
  return e;
}

}  // namespace kvq
