// Quantize-and-pack of full windows (flush) and the fp16 window / sink append.
//
// Source: "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
// second paragraph (keys per channel in 32-token groups, values per token)
// and third paragraph (newest tokens kept in full precision, quantized in
// blocks when the window fills); "KV cache quantization", "What they report"
// (first token kept in fp16).
//
// A CTA of 256 threads quantizes one group at a time: its 32 key and value
// rows are loaded into registers (the next group's while the current one is
// processed), stored to shared tiles laid out so that every later access is
// free of bank conflicts, reduced to per-channel key and per-token value
// min/max, and packed into the block format, which is staged in shared
// memory and written with one bulk copy.
#include "quant_common.cuh"

namespace kvq {

constexpr int kQuantThreads = 256;

// ------------------------------------------------------- shared tiles

// Value tile: the token-pair word (tokens 2 tw, 2 tw + 1) of channel ch.
// Two channels (ch, ch ^ 1) share a 32-word row, XOR-swizzled so that both
// the transposing stores (fixed channel offset, 16 channel blocks x 2 token
// pairs per warp) and the packing loads (fixed field, 8 channels x 4 token
// pairs per warp) touch 32 distinct banks.
__device__ __forceinline__ int vword(int ch, int tw) {
  const int rp = ch >> 1;
  const int swz = (4 * (rp & 3)) ^ (2 * ((rp >> 2) & 15));
  return rp * 32 + ((((ch & 1) << 4) + tw) ^ swz);
}

struct __align__(128) QuantSmem {
  uint32_t k[kG * 64];       // key tile: word (token, channel pair) at token * 64 + pair
  uint32_t v[kD * 16];       // value tile: vword()
  uint32_t kstat[8][64][2];  // per-warp key (min, max) half2 of each channel pair
  SliceQ kq[kD];             // key channel constants
  SliceQ vq[kG];             // value token constants
  uint32_t vstat[kG / 2][2]; // value (min, max) half2 of each token pair
  uint32_t kvst[kG / 2][2];  // key (min, max) half2 of each token pair (keys grouped per token)
  uint32_t vout[kG];         // dense-and-sparse: outlier entry of each value token
  uint32_t kout[kG];         // ... and of each key token (keys grouped per token)
  __align__(128) uint8_t blk[block_bytes(4, false, true)];  // the packed block being built
};

// One group's rows in registers: thread (p, c8) holds the 16-byte chunk c8
// (channels 8 c8 .. 8 c8 + 7) of tokens 2p and 2p + 1 of the keys and values.
struct GroupRegs {
  uint4 k[2], v[2];
};

// Where the 32 tokens of a group come from: stream index i < n0 sits in
// window slot i - Lq0, later ones are new token i + num_sink - L0.
struct GroupSrc {
  int s, h, i0, n0, Lq0, L0;
};

__device__ __forceinline__ void load_group(GroupRegs &r, const Geo &geo, const GroupSrc &g,
                                           const __half *__restrict__ k_new, const __half *__restrict__ v_new,
                                           int max_new) {
  const int p = threadIdx.x >> 4, c8 = threadIdx.x & 15;
  const size_t sh = static_cast<size_t>(g.s) * geo.H + g.h;
  if (g.i0 >= g.n0) {  // the whole group is new input (every prefill group)
    const int j = g.i0 + 2 * p + geo.ns - g.L0;
    if (!KVQ_IN_BOUNDS(geo.status, j + 1, max_new) || !KVQ_IN_BOUNDS(geo.status, j, max_new)) return;
    const __half *pk = k_new + (sh * max_new + j) * kD + c8 * 8;
    const __half *pv = v_new + (sh * max_new + j) * kD + c8 * 8;
    r.k[0] = *reinterpret_cast<const uint4 *>(pk);
    r.k[1] = *reinterpret_cast<const uint4 *>(pk + kD);
    r.v[0] = *reinterpret_cast<const uint4 *>(pv);
    r.v[1] = *reinterpret_cast<const uint4 *>(pv + kD);
    return;
  }
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int i = g.i0 + 2 * p + t;
    const __half *pk, *pv;
    if (i < g.n0) {
      if (!KVQ_IN_BOUNDS(geo.status, i - g.Lq0, geo.R)) continue;
      const size_t off = (sh * geo.R + (i - g.Lq0)) * kD;
      pk = geo.k_res + off;
      pv = geo.v_res + off;
    } else {
      if (!KVQ_IN_BOUNDS(geo.status, i + geo.ns - g.L0, max_new)) continue;
      const size_t off = (sh * max_new + (i + geo.ns - g.L0)) * kD;
      pk = k_new + off;
      pv = v_new + off;
    }
    r.k[t] = *reinterpret_cast<const uint4 *>(pk + c8 * 8);
    r.v[t] = *reinterpret_cast<const uint4 *>(pv + c8 * 8);
  }
}

// Walsh-Hadamard rotation of one token row, fp16(H x / 128) (the rotation
// lever of "2-Bit KV Cache Quantization: Memory You Save, Recall You Risk",
// "Method map: three ways to shrink the cache"; H the Sylvester matrix).
// The 16 threads c8 of a token pair hold its 128 channels, thread c8 the
// channels 8 c8 .. 8 c8 + 7, so strides 1, 2, 4 are butterflies inside a
// thread and strides 8, 16, 32, 64 pair thread c8 with c8 ^ 1, ^ 2, ^ 4, ^ 8.
// Strides run in ascending order and each butterfly (a, b) -> (a + b, a - b)
// is one fp32 add or subtract, so the result is the same fp32 value however
// the channels are spread; the scale 1/128 is exact and fp16 rounds once.
__device__ __forceinline__ uint4 hadamard_row(uint4 x, int c8) {
  float f[8];
  const __half2 *xh = reinterpret_cast<const __half2 *>(&x);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = __half22float2(xh[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
#pragma unroll
  for (int st = 1; st < 8; st <<= 1)
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (!(i & st)) {
        const float a = f[i], b = f[i + st];
        f[i] = __fadd_rn(a, b);
        f[i + st] = __fsub_rn(a, b);
      }
#pragma unroll
  for (int m = 1; m < 16; m <<= 1) {
    const bool upper = (c8 & m) != 0;  // this thread holds the b of each butterfly
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float o = __shfl_xor_sync(0xffffffffu, f[i], m);
      f[i] = upper ? __fsub_rn(o, f[i]) : __fadd_rn(f[i], o);
    }
  }
  uint4 y;
  __half2 *yh = reinterpret_cast<__half2 *>(&y);
#pragma unroll
  for (int i = 0; i < 4; ++i) yh[i] = __floats2half2_rn(f[2 * i] * 0.0078125f, f[2 * i + 1] * 0.0078125f);
  return y;
}

// Dense-and-sparse split of tokens 2p and 2p + 1, whose 128 channels the 16
// threads c8 hold 8 each (channels 8 c8 .. 8 c8 + 7 of ra and rb): the
// outlier is the first channel of largest magnitude; entry[t] holds its fp16
// bits and, at bit 16, its channel; mn2 / mx2 are the (token 2p, token 2p + 1)
// half2 min and max over the other 127 channels (fp16 values, so exact).
// Every thread of the warp calls it.
__device__ __forceinline__ void token_outliers(const uint4 &ra, const uint4 &rb, int c8, int lane,
                                               uint32_t (&entry)[2], uint32_t &mn2, uint32_t &mx2) {
  float lo[2], hi[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const __half *x = reinterpret_cast<const __half *>(t ? &rb : &ra);
    const uint16_t *xb = reinterpret_cast<const uint16_t *>(t ? &rb : &ra);
    float best = -1.f;
    int bi = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float a = fabsf(__half2float(x[c]));
      if (a > best) {
        best = a;
        bi = 8 * c8 + c;
      }
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, o);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ob > best || (ob == best && oi < bi)) {
        best = ob;
        bi = oi;
      }
    }
    float l = INFINITY, u = -INFINITY;
    uint32_t bits = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const float v = __half2float(x[c]);
      if (8 * c8 + c != bi) {
        l = fminf(l, v);
        u = fmaxf(u, v);
      } else {
        bits = xb[c];
      }
    }
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      l = fminf(l, __shfl_xor_sync(0xffffffffu, l, o));
      u = fmaxf(u, __shfl_xor_sync(0xffffffffu, u, o));
    }
    bits = __shfl_sync(0xffffffffu, bits, (lane & 16) | (bi >> 3));  // from the thread holding channel bi
    entry[t] = bits | (static_cast<uint32_t>(bi) << 16);
    lo[t] = l;
    hi[t] = u;
  }
  mn2 = h2_as_u32(__floats2half2_rn(lo[0], lo[1]));
  mx2 = h2_as_u32(__floats2half2_rn(hi[0], hi[1]));
}

// Quantize and pack the group held in `rin` (tokens from stream index i0 of
// (s, h)) and write its block with a bulk copy issued by thread 0.  Before
// the call thread 0 must have waited (bulk_wait_read) for the previous
// block's copy out of sm.blk.  Three CTA barriers inside, the last one after
// every read of the tiles.  KPT: keys grouped per token (scale and min over
// each token's channels, like values) instead of per channel.  ROT: the
// rows are Walsh-Hadamard rotated first (every thread of the CTA calls this).
// SP: dense-and-sparse ("KV cache quantization", "What they report",
// KVQuant paragraph): each slice's first largest-magnitude element leaves
// the statistics, its entry goes to the block, and its tile element is
// replaced by the slice's min so that the packing codes it 0.
template <int BITS, bool KPT, bool ROT, bool SP>
__device__ __forceinline__ void quantize_group(QuantSmem &sm, const GroupRegs &rin, const Geo &geo, int s, int h,
                                               int i0) {
  constexpr int NU = 8 / BITS;  // fields per byte
  constexpr int WH = 4 / NU;    // words per (lane, k-tile)
  const float levels = float((1 << BITS) - 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int p = tid >> 4, c8 = tid & 15;
  float *blkf = reinterpret_cast<float *>(sm.blk);
  uint32_t *blkw = reinterpret_cast<uint32_t *>(sm.blk);
  GroupRegs r = rin;
  if (ROT) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      r.k[t] = hadamard_row(r.k[t], c8);
      r.v[t] = hadamard_row(r.v[t], c8);
    }
  }

  // ---- tiles, partial key statistics, value token statistics
  {
    *reinterpret_cast<uint4 *>(&sm.k[(2 * p) * 64 + 4 * c8]) = r.k[0];
    *reinterpret_cast<uint4 *>(&sm.k[(2 * p + 1) * 64 + 4 * c8]) = r.k[1];
    if (!KPT && !SP) {
      const uint32_t ka[4] = {r.k[0].x, r.k[0].y, r.k[0].z, r.k[0].w};
      const uint32_t kb[4] = {r.k[1].x, r.k[1].y, r.k[1].z, r.k[1].w};
      uint32_t kmn[4], kmx[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kmn[i] = h2min(ka[i], kb[i]);
        kmx[i] = h2max(ka[i], kb[i]);
        kmn[i] = h2min(kmn[i], __shfl_xor_sync(0xffffffffu, kmn[i], 16));  // the warp's other token pair
        kmx[i] = h2max(kmx[i], __shfl_xor_sync(0xffffffffu, kmx[i], 16));
      }
      if (lane < 16) {
        uint4 *ks = reinterpret_cast<uint4 *>(&sm.kstat[warp][4 * c8][0]);
        ks[0] = make_uint4(kmn[0], kmx[0], kmn[1], kmx[1]);
        ks[1] = make_uint4(kmn[2], kmx[2], kmn[3], kmx[3]);
      }
    } else if (KPT && SP) {
      uint32_t e[2], mn2, mx2;
      token_outliers(r.k[0], r.k[1], c8, lane, e, mn2, mx2);
      if (c8 == 0) {
        *reinterpret_cast<uint2 *>(sm.kvst[p]) = make_uint2(mn2, mx2);
        *reinterpret_cast<uint2 *>(&sm.kout[2 * p]) = make_uint2(e[0], e[1]);
      }
    } else if (KPT) {  // per-token keys: (token 2p, token 2p + 1) min/max over the 128 channels
      const __half *ka = reinterpret_cast<const __half *>(&r.k[0]);
      const __half *kb = reinterpret_cast<const __half *>(&r.k[1]);
      __half2 kn2 = __halves2half2(ka[0], kb[0]), kx2 = kn2;
#pragma unroll
      for (int c = 1; c < 8; ++c) {
        const __half2 pr = __halves2half2(ka[c], kb[c]);
        kn2 = __hmin2(kn2, pr);
        kx2 = __hmax2(kx2, pr);
      }
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        const uint32_t a = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t *>(&kn2), o);
        const uint32_t b = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t *>(&kx2), o);
        kn2 = __hmin2(kn2, *reinterpret_cast<const __half2 *>(&a));
        kx2 = __hmax2(kx2, *reinterpret_cast<const __half2 *>(&b));
      }
      if (c8 == 0)
        *reinterpret_cast<uint2 *>(sm.kvst[p]) =
            make_uint2(*reinterpret_cast<uint32_t *>(&kn2), *reinterpret_cast<uint32_t *>(&kx2));
    }
    const __half *va = reinterpret_cast<const __half *>(&r.v[0]);
    const __half *vb = reinterpret_cast<const __half *>(&r.v[1]);
    __half2 mn2 = __halves2half2(va[0], vb[0]), mx2 = mn2;
    if (SP) {
      uint32_t e[2], smn, smx;
      token_outliers(r.v[0], r.v[1], c8, lane, e, smn, smx);
      mn2 = *reinterpret_cast<const __half2 *>(&smn);
      mx2 = *reinterpret_cast<const __half2 *>(&smx);
      if (c8 == 0) *reinterpret_cast<uint2 *>(&sm.vout[2 * p]) = make_uint2(e[0], e[1]);
    }
    // vword(8 c8 + c, p) = 128 c8 + 32 (c / 2) + ((p ^ 2 c8) ^ 16 (c % 2) ^ 4 (c / 2))
    uint32_t *vrow = sm.v + 128 * c8;
    const int vx = p ^ (2 * c8);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const __half2 pr = __halves2half2(va[c], vb[c]);  // (token 2p, token 2p + 1) of channel 8 c8 + c
      vrow[32 * (c >> 1) + (vx ^ ((16 * (c & 1)) ^ (4 * (c >> 1))))] = *reinterpret_cast<const uint32_t *>(&pr);
      if (!SP) {
        mn2 = __hmin2(mn2, pr);
        mx2 = __hmax2(mx2, pr);
      }
    }
    if (!SP) {
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {  // over the 16 lanes holding the tokens' 128 channels
        const uint32_t a = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t *>(&mn2), o);
        const uint32_t b = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t *>(&mx2), o);
        mn2 = __hmin2(mn2, *reinterpret_cast<const __half2 *>(&a));
        mx2 = __hmax2(mx2, *reinterpret_cast<const __half2 *>(&b));
      }
    }
    if (c8 == 0)
      *reinterpret_cast<uint2 *>(sm.vstat[p]) =
          make_uint2(*reinterpret_cast<uint32_t *>(&mn2), *reinterpret_cast<uint32_t *>(&mx2));
  }
  __syncthreads();
  // ---- key channel statistics over the 8 warps' partials (or key token
  // statistics); block scales
  if (KPT && tid < kG) {
    const float2 mnf = h2_to_f2_pos0(sm.kvst[tid >> 1][0]), mxf = h2_to_f2_pos0(sm.kvst[tid >> 1][1]);
    const float lo = tid & 1 ? mnf.y : mnf.x, hi = tid & 1 ? mxf.y : mxf.x;
    const float sc = __fdiv_rn(__fsub_rn(hi, lo), levels);
    sm.kq[tid] = make_slice(lo, sc, levels);
    blkf[off_ks(BITS) / 4 + tid] = sc;
    blkf[off_km(BITS, KPT) / 4 + tid] = lo;
    if (SP) {  // the entry, and the outlier's tile element becomes the min (code 0)
      const uint32_t e = sm.kout[tid];
      blkw[off_ksp(BITS, KPT) / 4 + tid] = e;
      reinterpret_cast<__half *>(sm.k)[kD * tid + (e >> 16)] = __float2half_rn(lo);
    }
  } else if (!KPT && tid < kD) {
    float lo, hi;
    if (SP) {  // channel tid over the group's 32 tokens, from the tile
      const __half *col = reinterpret_cast<const __half *>(sm.k) + tid;  // token t at col[kD * t]
      float best = -1.f;
      int bi = 0;
      for (int t = 0; t < kG; ++t) {
        const float a = fabsf(__half2float(col[kD * t]));
        if (a > best) {
          best = a;
          bi = t;
        }
      }
      lo = INFINITY;
      hi = -INFINITY;
      for (int t = 0; t < kG; ++t) {
        if (t == bi) continue;
        const float v = __half2float(col[kD * t]);
        lo = fminf(lo, v);
        hi = fmaxf(hi, v);
      }
      lo = __fadd_rn(lo, 0.f);
      hi = __fadd_rn(hi, 0.f);
      const uint32_t bits = reinterpret_cast<const uint16_t *>(sm.k)[kD * bi + tid];
      blkw[off_ksp(BITS, KPT) / 4 + tid] = bits | (static_cast<uint32_t>(bi) << 16);
      // the outlier's tile element becomes the min (code 0); the neighbouring
      // channel's thread only ever reads the other half of this word
      reinterpret_cast<__half *>(sm.k)[kD * bi + tid] = __float2half_rn(lo);
    } else {
      const int cp = tid >> 1, e = tid & 1;
      uint32_t mn = sm.kstat[0][cp][0], mx = sm.kstat[0][cp][1];
#pragma unroll
      for (int w = 1; w < 8; ++w) {
        mn = h2min(mn, sm.kstat[w][cp][0]);
        mx = h2max(mx, sm.kstat[w][cp][1]);
      }
      const float2 mnf = h2_to_f2_pos0(mn), mxf = h2_to_f2_pos0(mx);
      lo = e ? mnf.y : mnf.x;
      hi = e ? mxf.y : mxf.x;
    }
    const float sc = __fdiv_rn(__fsub_rn(hi, lo), levels);
    sm.kq[tid] = make_slice(lo, sc, levels);
    blkf[off_ks(BITS) / 4 + tid] = sc;
    blkf[off_km(BITS, KPT) / 4 + tid] = lo;
  } else if (tid >= kD && tid < kD + kG) {  // value tokens
    const int t = tid - kD;
    const float2 mnf = h2_to_f2_pos0(sm.vstat[t >> 1][0]), mxf = h2_to_f2_pos0(sm.vstat[t >> 1][1]);
    const float lo = t & 1 ? mnf.y : mnf.x, hi = t & 1 ? mxf.y : mxf.x;
    const float sc = __fdiv_rn(__fsub_rn(hi, lo), levels);
    sm.vq[t] = make_slice(lo, sc, levels);
    blkf[off_vs(BITS, KPT) / 4 + t] = sc;
    blkf[off_vm(BITS, KPT) / 4 + t] = lo;
    if (SP) {
      const uint32_t e = sm.vout[t];
      blkw[off_vsp(BITS, KPT) / 4 + t] = e;
      reinterpret_cast<__half *>(&sm.v[vword(e >> 16, t >> 1)])[t & 1] = __float2half_rn(lo);
    }
  }
  __syncthreads();

  // ---- pack.  Warps 0-3: key words, warps 4-7: value words.
  if (warp < 4) {
    // word (lane 4g + q, w = kt * WH + hw): tokens 8 tau + g for tau = hw NU
    // + u, channels 16 kt + 8 j + 2 q + e.  Lanes of a warp share g and take
    // the 32 (kt, q); half of them visit j in the other order so that each
    // load instruction covers 32 distinct channel pairs mod 32 (banks).
    const int kt = lane >> 2, q = lane & 3;
    const int jx = kt >> 2;
    f2x rcp[2], cc[2];
    float tol = 0.f;
    if (!KPT) {
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const SliceQ a = sm.kq[16 * kt + 8 * j + 2 * q], b = sm.kq[16 * kt + 8 * j + 2 * q + 1];
        rcp[j] = f2_pack(a.rcp, b.rcp);
        cc[j] = f2_pack(a.c, b.c);
        tol = fmaxf(tol, fmaxf(a.tol, b.tol));
      }
    }
    const float thr_ch = 0.5f - tol;
#pragma unroll
    for (int gi = 0; gi < 2; ++gi) {
      const int g = 2 * warp + gi;
#pragma unroll
      for (int hw = 0; hw < WH; ++hw) {
        uint32_t x[2 * NU];
        f2x fr[2 * NU], fc[2 * NU];
        int pos[2 * NU];
        float thr = thr_ch;
#pragma unroll
        for (int u = 0; u < NU; ++u) {
          f2x tr = 0, tc = 0;
          if (KPT) {  // both fields of a pair belong to token 8 tau + g
            const SliceQ a = sm.kq[8 * (hw * NU + u) + g];
            tr = f2_pack(a.rcp, a.rcp);
            tc = f2_pack(a.c, a.c);
            thr = fminf(thr, 0.5f - a.tol);
          }
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = jj ^ jx, tau = hw * NU + u, f = 2 * u + jj;
            x[f] = sm.k[(8 * tau + g) * 64 + 8 * kt + 4 * j + q];
            fr[f] = KPT ? tr : (jx ? rcp[jj ^ 1] : rcp[jj]);
            fc[f] = KPT ? tc : (jx ? cc[jj ^ 1] : cc[jj]);
            pos[f] = 8 * j + BITS * u;
          }
        }
        bool near;
        uint32_t word = pack_word<2 * NU>(x, fr, fc, pos, thr, near);
        if (__any_sync(0xffffffffu, near) && near) {
          word = 0;
          for (int f = 0; f < 4 * NU; ++f) {
            const int u = f >> 2, j = (f >> 1) & 1, e = f & 1;
            const int tau = hw * NU + u, ch = 16 * kt + 8 * j + 2 * q + e;
            const uint32_t w2 = sm.k[(8 * tau + g) * 64 + (ch >> 1)];
            const float xv = __half2float(reinterpret_cast<const __half *>(&w2)[e]);
            const int sl = KPT ? 8 * tau + g : ch;
            word |= exact_code<BITS>(xv, sm.kq[sl].mn, blkf[off_ks(BITS) / 4 + sl]) << (16 * e + 8 * j + BITS * u);
          }
        }
        const int w = kt * WH + hw, L = 4 * g + q;
        blkw[off_kc(BITS) / 4 + ((w >> 2) * 32 + L) * 4 + (w & 3)] = word;
      }
    }
  } else {
    // word (lane 4g + q, w = (2P + kt) * WH + hw): channels 32 P + 8 tau + g
    // for tau = hw NU + u, tokens 16 kt + 8 j + 2 q + e; warp 4 + P.
    const int P = warp - 4, g = lane >> 2, q = lane & 3;
    // vword(32 P + 8 tau + g, 8 kt + 4 j + q) = vbase + 128 tau
    //   + ((16 (g % 2) + q) ^ 4 (g / 2) ^ 8 kt ^ 8 P ^ 4 j ^ 2 tau)
    const uint32_t *vbase = sm.v + (16 * P + (g >> 1)) * 32;
    const int vy = ((16 * (g & 1)) | q) ^ (4 * (g >> 1));
#pragma unroll
    for (int kt = 0; kt < 2; ++kt) {
      const int vyk = vy ^ (8 * kt) ^ (8 * P);
      f2x rcp[2], cc[2];
      float tol = 0.f;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const SliceQ a = sm.vq[16 * kt + 8 * j + 2 * q], b = sm.vq[16 * kt + 8 * j + 2 * q + 1];
        rcp[j] = f2_pack(a.rcp, b.rcp);
        cc[j] = f2_pack(a.c, b.c);
        tol = fmaxf(tol, fmaxf(a.tol, b.tol));
      }
      const float thr = 0.5f - tol;
#pragma unroll
      for (int hw = 0; hw < WH; ++hw) {
        uint32_t x[2 * NU];
        f2x fr[2 * NU], fc[2 * NU];
        int pos[2 * NU];
#pragma unroll
        for (int u = 0; u < NU; ++u)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int tau = hw * NU + u, f = 2 * u + j;
            x[f] = vbase[128 * tau + (vyk ^ (4 * j) ^ (2 * tau))];
            fr[f] = rcp[j];
            fc[f] = cc[j];
            pos[f] = 8 * j + BITS * u;
          }
        bool near;
        uint32_t word = pack_word<2 * NU>(x, fr, fc, pos, thr, near);
        if (__any_sync(0xffffffffu, near) && near) {
          word = 0;
          for (int f = 0; f < 4 * NU; ++f) {
            const int u = f >> 2, j = (f >> 1) & 1, e = f & 1;
            const int tau = hw * NU + u, tok = 16 * kt + 8 * j + 2 * q + e;
            const uint32_t w2 = sm.v[vword(32 * P + 8 * tau + g, tok >> 1)];
            const float xv = __half2float(reinterpret_cast<const __half *>(&w2)[e]);
            word |= exact_code<BITS>(xv, sm.vq[tok].mn, blkf[off_vs(BITS, KPT) / 4 + tok]) << (16 * e + 8 * j + BITS * u);
          }
        }
        const int w = (2 * P + kt) * WH + hw, L = 4 * g + q;
        blkw[off_vc(BITS) / 4 + ((w >> 2) * 32 + L) * 4 + (w & 3)] = word;
      }
    }
  }
  fence_proxy_async();  // this thread's block writes, before the bulk copy reads them
  __syncthreads();
  if (tid == 0) {
    uint8_t *dst = KVQ_IN_BOUNDS(geo.status, i0 / kG, geo.max_groups) ? group_block(geo, s, h, i0 / kG, block_bytes(BITS, KPT, SP))
                                                                      : nullptr;
    if (dst)
      bulk_s2g(dst, sm.blk, block_bytes(BITS, KPT, SP));
    else
      set_status(geo.status, KVQ_STATUS_BAD_BLOCK);
  }
}

// Length bits of seq_len; while the fused step append runs, the bits above
// count the CTAs of a sequence that have finished with it.
constexpr int kLenBits = 22;
constexpr int kLenMask = (1 << kLenBits) - 1;

// Flush groups of an append, by persistent CTAs.  Task t = group slot
// t % gmax of (sequence, KV head) t / gmax (fewer than 2^31 tasks); CTA b
// takes tasks b, b + grid, ... and loads the next task's rows while it
// quantizes the current one.
template <int BITS, bool KPT, bool ROT, bool SP>
__global__ void __launch_bounds__(kQuantThreads, 4) quant_flush_kernel(Geo geo, const __half *__restrict__ k_new,
                                                                       const __half *__restrict__ v_new,
                                                                       const int *__restrict__ new_len,
                                                                       int max_new, int gmax) {
  __shared__ QuantSmem sm;
  // task = (sequence, KV head) sh, group slot gs; CTA b starts at task b and
  // steps by the grid, i.e. by (dq, dr) in (sh, gs)
  const int nsh = geo.S * geo.H;
  const int dq = static_cast<int>(gridDim.x / static_cast<unsigned>(gmax));
  const int dr = static_cast<int>(gridDim.x % static_cast<unsigned>(gmax));
  int sh = static_cast<int>(blockIdx.x / static_cast<unsigned>(gmax));
  int gs = static_cast<int>(blockIdx.x % static_cast<unsigned>(gmax));
  // advance (sh, gs) to the first task at or after it with a group to flush;
  // false past the last task
  auto find = [&](GroupSrc &g) {
    for (; sh < nsh; gs += dr, sh += dq + (gs >= gmax ? 1 : 0), gs -= gs >= gmax ? gmax : 0) {
      const int s = static_cast<int>(static_cast<unsigned>(sh) / static_cast<unsigned>(geo.H));
      const int L0 = geo.seq_len[s], nn = new_len[s];
      if (nn < 0 || nn > max_new || L0 < 0 || L0 + nn > geo.capacity) continue;  // reported by the tail kernel
      const int n0 = max(L0 - geo.ns, 0), n1 = max(L0 + nn - geo.ns, 0);
      const int Lq0 = n0 - n0 % geo.R, Lq1 = n1 - n1 % geo.R;
      if (gs >= (Lq1 - Lq0) / kG) continue;
      g.s = s;
      g.h = sh - s * geo.H;
      g.i0 = Lq0 + gs * kG;
      g.n0 = n0;
      g.Lq0 = Lq0;
      g.L0 = L0;
      return true;
    }
    return false;
  };
  auto step = [&]() {
    gs += dr;
    sh += dq;
    if (gs >= gmax) {
      gs -= gmax;
      ++sh;
    }
  };
  GroupSrc cur, nxt;
  if (!find(cur)) return;
  GroupRegs rc, rn;
  load_group(rc, geo, cur, k_new, v_new, max_new);
  while (true) {
    step();
    const bool more = find(nxt);
    if (more) load_group(rn, geo, nxt, k_new, v_new, max_new);
    if (threadIdx.x == 0) bulk_wait_read();  // the previous block's copy has left sm.blk
    quantize_group<BITS, KPT, ROT, SP>(sm, rc, geo, cur.s, cur.h, cur.i0);
    if (!more) break;
    cur = nxt;
    rc = rn;
  }
  if (threadIdx.x == 0) bulk_wait_all();
}

// Copy the new tokens of (sequence s, KV heads [h0, h1)) that land in the
// sink or in the window; threads tid = 0 .. nthr-1 of the CTA share the work.
__device__ __forceinline__ void copy_tail(const Geo &geo, int s, int h0, int h1, int L0, int nn,
                                          const __half *__restrict__ k_new, const __half *__restrict__ v_new,
                                          int max_new, int tid, int nthr) {
  const int n1 = max(L0 + nn - geo.ns, 0);
  const int Lq1 = n1 - n1 % geo.R;
  const int j_sink_end = min(max(geo.ns - L0, 0), nn);      // new tokens [0, j_sink_end) -> sink
  const int j_win = max(Lq1 + geo.ns - L0, j_sink_end);      // new tokens [j_win, nn) -> window
  const int n_copy = j_sink_end + max(nn - j_win, 0);
  constexpr int C16 = kD / 8;  // 16-byte chunks per token row
  for (int idx = tid; idx < (h1 - h0) * n_copy * C16; idx += nthr) {
    const int c8 = idx % C16;
    const int k = (idx / C16) % n_copy;
    const int h = h0 + idx / (C16 * n_copy);
    const int j = k < j_sink_end ? k : j_win + (k - j_sink_end);
    const int pos = L0 + j;
    const size_t sh = static_cast<size_t>(s) * geo.H + h;
    __half *dk, *dv;
    if (pos < geo.ns) {
      dk = geo.k_sink + (sh * geo.ns + pos) * kD;
      dv = geo.v_sink + (sh * geo.ns + pos) * kD;
    } else {
      const int slot = pos - geo.ns - Lq1;
      if (!KVQ_IN_BOUNDS(geo.status, slot, geo.R)) continue;
      dk = geo.k_res + (sh * geo.R + slot) * kD;
      dv = geo.v_res + (sh * geo.R + slot) * kD;
    }
    if (!KVQ_IN_BOUNDS(geo.status, j, max_new)) continue;
    const size_t src = (sh * max_new + j) * kD + c8 * 8;
    reinterpret_cast<uint4 *>(dk)[c8] = *reinterpret_cast<const uint4 *>(k_new + src);
    reinterpret_cast<uint4 *>(dv)[c8] = *reinterpret_cast<const uint4 *>(v_new + src);
  }
}

// Append of at most R new tokens per sequence in one kernel, one CTA per
// (KV head, sequence): at most one window fills, and the CTA then quantizes
// its R / 32 groups one after another (loading the next group's rows while
// it quantizes the current one).  Each CTA adds 1 << kLenBits to seq_len[s]
// once it needs seq_len no more; the CTA that completes the count (Hkv
// arrivals) stores the final length (clearing the count) and reports bad
// lengths, and no CTA reads seq_len[s] after that store.  When no window
// fills, a CTA arrives right after reading the length and copies its head's
// new tokens into the window (or sink), prefetched at launch.  When one
// fills, the copy would overwrite window slots the sequence's other CTAs may
// still be quantizing, so the CTAs arrive after quantizing and the last one
// copies the new tokens of every head.
template <int BITS, bool KPT, bool ROT, bool SP>
__global__ void __launch_bounds__(kQuantThreads, 4) step_append_kernel(Geo geo, const __half *__restrict__ k_new,
                                                                    const __half *__restrict__ v_new,
                                                                    const int *__restrict__ new_len, int max_new) {
  __shared__ QuantSmem sm;
  const int s = blockIdx.y, h = blockIdx.x;
  __shared__ int s_last, s_old;
  constexpr int C16 = kD / 8;  // 16-byte chunks per token row
  // thread (pj, pc) prefetches chunk pc of new token pj of this head
  const int pj = threadIdx.x / C16, pc = threadIdx.x % C16;
  const bool pre = pj < min(max_new, kQuantThreads / C16);
  uint4 pk = make_uint4(0u, 0u, 0u, 0u), pv = pk;
  const size_t sh = static_cast<size_t>(s) * geo.H + h;
  if (pre) {
    const size_t src = (sh * max_new + pj) * kD + pc * 8;
    pk = *reinterpret_cast<const uint4 *>(k_new + src);
    pv = *reinterpret_cast<const uint4 *>(v_new + src);
  }
  const int raw = geo.seq_len[s];  // the length, plus arrivals of other CTAs in the high bits
  const int nn = new_len[s];
  if (raw < 0) {  // a negative length: no CTA of the sequence arrives, so it stays as it is
    if (threadIdx.x == 0) set_status(geo.status, KVQ_STATUS_BAD_LEN);
    return;
  }
  const int L0 = raw & kLenMask;
  const bool bad_len = nn < 0 || nn > max_new;
  const bool over = !bad_len && L0 + nn > geo.capacity;
  const int n0 = max(L0 - geo.ns, 0);
  const int Lq0 = n0 - n0 % geo.R;
  const int n1 = max(L0 + nn - geo.ns, 0);
  const int Lq1 = n1 - n1 % geo.R;
  const bool flush = !bad_len && !over && Lq1 != Lq0;

  auto arrive = [&]() {  // thread 0; s_last / s_old valid after the next barrier
    const int old = atomicAdd(&geo.seq_len[s], 1 << kLenBits);
    s_old = old - (geo.H - 1) * (1 << kLenBits);  // seq_len[s] before this kernel
    s_last = (old >> kLenBits) == geo.H - 1;
  };
  if (!flush) {
    if (threadIdx.x == 0) arrive();
    if (!bad_len && !over) {
      if (nn <= kQuantThreads / C16) {
        if (pj < nn) {  // no window fills: every new token goes to the sink or the window
          const int pos = L0 + pj;
          __half *dk, *dv;
          if (pos < geo.ns) {
            dk = geo.k_sink + (sh * geo.ns + pos) * kD;
            dv = geo.v_sink + (sh * geo.ns + pos) * kD;
          } else {
            const int slot = pos - geo.ns - Lq1;
            dk = geo.k_res + (sh * geo.R + (KVQ_IN_BOUNDS(geo.status, slot, geo.R) ? slot : 0)) * kD;
            dv = geo.v_res + (sh * geo.R + (KVQ_IN_BOUNDS(geo.status, slot, geo.R) ? slot : 0)) * kD;
          }
          reinterpret_cast<uint4 *>(dk)[pc] = pk;
          reinterpret_cast<uint4 *>(dv)[pc] = pv;
        }
      } else {
        copy_tail(geo, s, h, h + 1, L0, nn, k_new, v_new, max_new, threadIdx.x, blockDim.x);
      }
    }
    __syncthreads();
  } else {
    GroupSrc g;
    g.s = s;
    g.h = h;
    g.i0 = Lq0;
    g.n0 = n0;
    g.Lq0 = Lq0;
    g.L0 = L0;
    GroupRegs rc, rn;
    load_group(rc, geo, g, k_new, v_new, max_new);
    for (int i0 = Lq0; i0 < Lq1; i0 += kG) {
      if (i0 + kG < Lq1) {
        g.i0 = i0 + kG;
        load_group(rn, geo, g, k_new, v_new, max_new);
      }
      if (threadIdx.x == 0) bulk_wait_read();
      quantize_group<BITS, KPT, ROT, SP>(sm, rc, geo, s, h, i0);
      rc = rn;
    }
    // quantize_group ends with a barrier: every read of the window is done
    if (threadIdx.x == 0) arrive();
    __syncthreads();
    if (s_last) copy_tail(geo, s, 0, geo.H, L0, nn, k_new, v_new, max_new, threadIdx.x, blockDim.x);
    if (threadIdx.x == 0) bulk_wait_all();
  }
  if (s_last && threadIdx.x == 0) {
    if (bad_len) set_status(geo.status, KVQ_STATUS_BAD_LEN);
    if (over) set_status(geo.status, KVQ_STATUS_CAPACITY);
    geo.seq_len[s] = bad_len || over ? s_old : L0 + nn;
  }
}

// One CTA per sequence: copy the new tokens that land in the sink or in the
// window, then advance seq_len (one CTA owns a sequence, so no other CTA
// reads seq_len[s] after it is written).
__global__ void __launch_bounds__(256) append_tail_kernel(Geo geo, const __half *__restrict__ k_new,
                                                          const __half *__restrict__ v_new,
                                                          const int *__restrict__ new_len, int max_new) {
  const int s = blockIdx.x;
  const int L0 = geo.seq_len[s];
  const int nn = new_len[s];
  if (nn < 0 || nn > max_new || L0 < 0) {
    if (threadIdx.x == 0) set_status(geo.status, KVQ_STATUS_BAD_LEN);
    return;
  }
  if (L0 + nn > geo.capacity) {
    if (threadIdx.x == 0) set_status(geo.status, KVQ_STATUS_CAPACITY);
    return;
  }
  copy_tail(geo, s, 0, geo.H, L0, nn, k_new, v_new, max_new, threadIdx.x, blockDim.x);
  __syncthreads();
  if (threadIdx.x == 0) geo.seq_len[s] = L0 + nn;
}

// The same as append_tail_kernel with one CTA per (KV head, sequence), for
// long appends whose tails (up to R - 1 window tokens per head) a single CTA
// per sequence copies too slowly.  Every CTA reads seq_len[s], then adds
// 1 << kLenBits to it; the CTA completing the count (Hkv arrivals) stores
// the new length (or the old one for a bad length, reported by head 0's
// CTA), so no CTA reads seq_len[s] after it changes.  A negative length
// makes every CTA leave the sequence untouched.  Each thread moves up to four
// 16-byte chunks of K and of V per round, loads before stores.
__global__ void __launch_bounds__(256) append_tail_split_kernel(Geo geo, const __half *__restrict__ k_new,
                                                                const __half *__restrict__ v_new,
                                                                const int *__restrict__ new_len, int max_new) {
  const int s = blockIdx.y, h = blockIdx.x;
  __shared__ int s_last, s_old;
  const int raw = geo.seq_len[s];
  const int nn = new_len[s];
  if (raw < 0) {
    if (threadIdx.x == 0 && h == 0) set_status(geo.status, KVQ_STATUS_BAD_LEN);
    return;
  }
  __syncthreads();  // every thread has read seq_len[s]
  if (threadIdx.x == 0) {
    const int old = atomicAdd(&geo.seq_len[s], 1 << kLenBits);
    s_old = old - (geo.H - 1) * (1 << kLenBits);  // seq_len[s] before this kernel (valid for the last)
    s_last = (old >> kLenBits) == geo.H - 1;
  }
  const int L0 = raw & kLenMask;
  const bool bad_len = nn < 0 || nn > max_new;
  const bool over = !bad_len && L0 + nn > geo.capacity;
  if (!bad_len && !over) {
    const int n1 = max(L0 + nn - geo.ns, 0);
    const int Lq1 = n1 - n1 % geo.R;
    const int j_sink_end = min(max(geo.ns - L0, 0), nn);  // new tokens [0, j_sink_end) -> sink
    const int j_win = max(Lq1 + geo.ns - L0, j_sink_end);  // new tokens [j_win, nn) -> window
    const int n_copy = j_sink_end + max(nn - j_win, 0);
    constexpr int C16 = kD / 8;  // 16-byte chunks per token row
    const int total = n_copy * C16;
    const size_t sh = static_cast<size_t>(s) * geo.H + h;
    for (int base = threadIdx.x; base < total; base += 4 * blockDim.x) {
      uint4 kr[4], vr[4];
      uint4 *dk[4], *dv[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = base + u * blockDim.x;
        dk[u] = dv[u] = nullptr;
        if (idx >= total) continue;
        const int k = idx / C16, c8 = idx % C16;
        const int j = k < j_sink_end ? k : j_win + (k - j_sink_end);
        const int pos = L0 + j;
        if (!KVQ_IN_BOUNDS(geo.status, pos < geo.ns ? pos : pos - geo.ns - Lq1, pos < geo.ns ? geo.ns : geo.R) ||
            !KVQ_IN_BOUNDS(geo.status, j, max_new))
          continue;
        const size_t row = pos < geo.ns ? sh * geo.ns + pos : sh * geo.R + (pos - geo.ns - Lq1);
        dk[u] = reinterpret_cast<uint4 *>((pos < geo.ns ? geo.k_sink : geo.k_res) + row * kD) + c8;
        dv[u] = reinterpret_cast<uint4 *>((pos < geo.ns ? geo.v_sink : geo.v_res) + row * kD) + c8;
        const size_t src = (sh * max_new + j) * kD + c8 * 8;
        kr[u] = *reinterpret_cast<const uint4 *>(k_new + src);
        vr[u] = *reinterpret_cast<const uint4 *>(v_new + src);
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (dk[u]) {
          *dk[u] = kr[u];
          *dv[u] = vr[u];
        }
    }
  }
  __syncthreads();  // s_last / s_old
  if (s_last && threadIdx.x == 0) {
    if (bad_len) set_status(geo.status, KVQ_STATUS_BAD_LEN);
    if (over) set_status(geo.status, KVQ_STATUS_CAPACITY);
    geo.seq_len[s] = bad_len || over ? s_old : L0 + nn;
  }
}

// Upper bound on groups quantized per (sequence, head) by one append of at
// most max_new tokens: a window holding R-1 tokens plus max_new new ones.
int max_flush_groups(int R, int max_new) { return ((R - 1 + max_new) / R) * (R / kG); }

using FlushKernel = void (*)(Geo, const __half *, const __half *, const int *, int, int);
using StepKernel = void (*)(Geo, const __half *, const __half *, const int *, int);

// Instantiations by (bits, keys per token, plain / rotated / dense-and-sparse).
static int variant(const Geo &geo) {
  return ((geo.bits == 4 ? 2 : 0) + (geo.kpt ? 1 : 0)) * 3 + (geo.rot ? 1 : geo.sparse ? 2 : 0);
}
#define KVQ_QUANT_SET(K, B, P)                                                                  \
  K<B, P, false, false>, K<B, P, true, false>, K<B, P, false, true>
static const FlushKernel kFlushKernels[12] = {
    KVQ_QUANT_SET(quant_flush_kernel, 2, false), KVQ_QUANT_SET(quant_flush_kernel, 2, true),
    KVQ_QUANT_SET(quant_flush_kernel, 4, false), KVQ_QUANT_SET(quant_flush_kernel, 4, true)};
static const StepKernel kStepKernels[12] = {
    KVQ_QUANT_SET(step_append_kernel, 2, false), KVQ_QUANT_SET(step_append_kernel, 2, true),
    KVQ_QUANT_SET(step_append_kernel, 4, false), KVQ_QUANT_SET(step_append_kernel, 4, true)};
#undef KVQ_QUANT_SET

// Persistent CTAs of flush kernel variant v on the current device: every
// resident slot (cached per variant and device ordinal).
static cudaError_t flush_grid(int v, int &ctas) {
  static int cache[12][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 64 && cache[v][dev]) {
    ctas = cache[v][dev];
    return cudaSuccess;
  }
  int per_sm = 0, n_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kFlushKernels[v], kQuantThreads, 0)) !=
      cudaSuccess)
    return e;
  if ((e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  ctas = max(per_sm, 1) * n_sm;
  if (dev < 64) cache[v][dev] = ctas;
  return cudaSuccess;
}

cudaError_t launch_quant_append(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                                int max_new, cudaStream_t stream, uint64_t *launches) {
  const int v = variant(geo);
  // a decode-sized append (at most one window fills): one kernel
  if (max_new <= geo.R && geo.capacity <= kLenMask && geo.H < (1 << (31 - kLenBits))) {
    dim3 grid(geo.H, geo.S);
    kStepKernels[v]<<<grid, kQuantThreads, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
    ++*launches;
    return cudaGetLastError();
  }
  const int gmax = max_flush_groups(geo.R, max_new);
  if (gmax > 0 && flush_tiles_serves(geo)) {
    cudaError_t e = launch_flush_tiles(geo, k_new, v_new, new_len, max_new, stream);
    ++*launches;
    if (e != cudaSuccess) return e;
  } else if (gmax > 0) {
    int ctas = 0;
    cudaError_t e = flush_grid(v, ctas);
    if (e != cudaSuccess) return e;
    const long long ntask = static_cast<long long>(gmax) * geo.H * geo.S;
    if (ntask > 2147483647LL) return cudaErrorInvalidValue;
    const int grid = static_cast<int>(min(static_cast<long long>(ctas), ntask));
    kFlushKernels[v]<<<grid, kQuantThreads, 0, stream>>>(geo, k_new, v_new, new_len, max_new, gmax);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (geo.capacity <= kLenMask && geo.H < (1 << (31 - kLenBits)))
    append_tail_split_kernel<<<dim3(geo.H, geo.S), 256, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
  else
    append_tail_kernel<<<geo.S, 256, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace kvq
