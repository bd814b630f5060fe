// Quantize-and-pack of full windows (flush) and the fp16 window / sink append.
//
// Source: "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
// second paragraph (keys per channel in 32-token groups, values per token)
// and third paragraph (newest tokens kept in full precision, quantized in
// blocks when the window fills); "KV cache quantization", "What they report"
// (first token kept in fp16).
#include "kvq_internal.cuh"

namespace kvq {

constexpr int kQuantThreads = 256;
constexpr float kMagic = 12582912.f;  // 1.5 * 2^23: x + kMagic rounds x to an integer (half to even)

// Per-slice (one key channel of a group, or one value token) constants of
// the code computation.  The code is rne(fl(fl(x - min) / scale)) clamped
// to [0, 2^b - 1], scale == 0 giving 0.  It is first evaluated from
// y' = fma(x, rcp, c) with rcp = fl(1/scale) and c = fl(-min * rcp), which
// differs from both the exact quotient (x - min) / scale and the IEEE
// result fl(fl(x - min) / scale) by less than half of `tol`
// ((2^b) * 2^-23 + |c| * 2^-24 each, from the three roundings); when y'
// lies farther than `tol` from every rounding boundary k + 1/2, all three
// round to the same integer.  Otherwise the IEEE subtract and divide decide.
struct SliceQ {
  float rcp, c, tol, mn;
};

__device__ __forceinline__ SliceQ make_slice(float mn, float scale, float levels) {
  SliceQ q;
  q.mn = mn;
  q.rcp = scale > 0.f ? __frcp_rn(scale) : 0.f;
  q.c = __fmul_rn(-mn, q.rcp);
  q.tol = (levels + 1.f) * 4.76837158203125e-07f + fabsf(q.c) * 2.384185791015625e-07f;  // 2^-21, 2^-22
  return q;
}

// Fast code of x; `near` is set when y' is within tol of a rounding boundary.
__device__ __forceinline__ uint32_t fast_code(float x, const SliceQ &q, bool &near) {
  const float y = fmaf(x, q.rcp, q.c);
  const float t = y + kMagic;
  near = fabsf(fabsf(y - (t - kMagic)) - 0.5f) <= q.tol;
  return __float_as_uint(t) - __float_as_uint(kMagic);
}

// The code by the IEEE subtract and divide (rarely needed, kept out of line).
template <int BITS>
__device__ __noinline__ uint32_t exact_code(float x, float mn, float scale) {
  const float r = rintf(__fdiv_rn(__fsub_rn(x, mn), scale));
  return static_cast<uint32_t>(fminf(fmaxf(r, 0.f), float((1 << BITS) - 1)));
}

constexpr int kVStride = kG + 2;  // padded row (in halves) of the transposed value tile

// The CTA (kQuantThreads threads) quantizes the 32-token group of (sequence
// s, KV head h) starting at stream index i0.  Its tokens come from the old
// window (stream index < n0, window slot i - Lq0) or from the new input
// (new token i + num_sink - L0).
template <int BITS>
__device__ __forceinline__ void flush_group(const Geo &geo, int s, int h, int i0, int n0, int Lq0, int L0,
                                            const __half *__restrict__ k_new, const __half *__restrict__ v_new,
                                            int max_new) {
  __shared__ __align__(16) __half sk[kG][kD];         // keys, token rows
  __shared__ __align__(16) __half svT[kD][kVStride];  // values, channel rows
  __shared__ __align__(16) SliceQ kq[kD];
  __shared__ __align__(16) SliceQ vq[kG];
  __shared__ float k_sc[kD], v_sc[kG];

  const float levels = float((1 << BITS) - 1);
  const size_t sh = static_cast<size_t>(s) * geo.H + h;
  uint8_t *blk = geo.blocks + (sh * geo.max_groups + i0 / kG) * static_cast<size_t>(block_bytes(BITS));
  {
    // thread (p, c8): tokens 2p and 2p+1, channels 8 c8 .. 8 c8 + 7
    const int p = threadIdx.x >> 4, c8 = threadIdx.x & 15;
    uint4 kr[2], vr[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int i = i0 + 2 * p + r;
      const __half *pk, *pv;
      if (i < n0) {
        const size_t off = (sh * geo.R + (i - Lq0)) * kD;
        pk = geo.k_res + off;
        pv = geo.v_res + off;
      } else {
        const size_t off = (sh * max_new + (i + geo.ns - L0)) * kD;
        pk = k_new + off;
        pv = v_new + off;
      }
      kr[r] = *reinterpret_cast<const uint4 *>(pk + c8 * 8);
      vr[r] = *reinterpret_cast<const uint4 *>(pv + c8 * 8);
    }
    *reinterpret_cast<uint4 *>(&sk[2 * p][c8 * 8]) = kr[0];
    *reinterpret_cast<uint4 *>(&sk[2 * p + 1][c8 * 8]) = kr[1];
    const __half *va = reinterpret_cast<const __half *>(&vr[0]);
    const __half *vb = reinterpret_cast<const __half *>(&vr[1]);
    __half2 mn2 = __halves2half2(va[0], vb[0]), mx2 = mn2;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const __half2 pair = __halves2half2(va[c], vb[c]);  // (token 2p, token 2p+1) of channel 8 c8 + c
      *reinterpret_cast<__half2 *>(&svT[c8 * 8 + c][2 * p]) = pair;
      mn2 = __hmin2(mn2, pair);
      mx2 = __hmax2(mx2, pair);
    }
    // per-token min/max over the 16 lanes holding the token's 128 channels
#pragma unroll
    for (int o = 1; o < 16; o <<= 1) {
      const uint32_t a = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t *>(&mn2), o);
      const uint32_t b = __shfl_xor_sync(0xffffffffu, *reinterpret_cast<uint32_t *>(&mx2), o);
      mn2 = __hmin2(mn2, *reinterpret_cast<const __half2 *>(&a));
      mx2 = __hmax2(mx2, *reinterpret_cast<const __half2 *>(&b));
    }
    if (c8 < 2) {  // lane 0 of the pair finishes token 2p, lane 1 token 2p+1
      const float2 mnf = __half22float2(mn2), mxf = __half22float2(mx2);
      // + 0 stores a zero extreme as +0 whichever zero the reduction kept
      const float mn = __fadd_rn(c8 == 0 ? mnf.x : mnf.y, 0.f), mx = __fadd_rn(c8 == 0 ? mxf.x : mxf.y, 0.f);
      const int t = 2 * p + c8;
      const float sc = __fdiv_rn(__fsub_rn(mx, mn), levels);
      vq[t] = make_slice(mn, sc, levels);
      v_sc[t] = sc;
      reinterpret_cast<float *>(blk + off_vs(BITS))[t] = sc;
      reinterpret_cast<float *>(blk + off_vm(BITS))[t] = mn;
    }
  }
  __syncthreads();
  if (threadIdx.x < kD / 2) {  // keys: channels 2d, 2d+1, min/max over the 32 tokens (exact in fp16)
    const int d = 2 * threadIdx.x;
    __half2 mn2 = *reinterpret_cast<const __half2 *>(&sk[0][d]), mx2 = mn2;
#pragma unroll 8
    for (int t = 1; t < kG; ++t) {
      const __half2 x = *reinterpret_cast<const __half2 *>(&sk[t][d]);
      mn2 = __hmin2(mn2, x);
      mx2 = __hmax2(mx2, x);
    }
    float2 mnf = __half22float2(mn2), mxf = __half22float2(mx2);
    mnf.x = __fadd_rn(mnf.x, 0.f);
    mnf.y = __fadd_rn(mnf.y, 0.f);
    mxf.x = __fadd_rn(mxf.x, 0.f);
    mxf.y = __fadd_rn(mxf.y, 0.f);
    const float sc0 = __fdiv_rn(__fsub_rn(mxf.x, mnf.x), levels);
    const float sc1 = __fdiv_rn(__fsub_rn(mxf.y, mnf.y), levels);
    kq[d] = make_slice(mnf.x, sc0, levels);
    kq[d + 1] = make_slice(mnf.y, sc1, levels);
    k_sc[d] = sc0;
    k_sc[d + 1] = sc1;
    reinterpret_cast<float2 *>(blk + off_ks(BITS))[threadIdx.x] = make_float2(sc0, sc1);
    reinterpret_cast<float2 *>(blk + off_km(BITS))[threadIdx.x] = make_float2(mnf.x, mnf.y);
  }
  __syncthreads();

  // Pack: each thread builds whole 32-bit words.  Word index t' of a tile is
  // stored at byte 4t' (coalesced), i.e. word w = 4(t'/128) + t'%4 of lane
  // (t'/4)%32; its fields are (e, j, u) at bit 16e + 8j + b*u holding
  // element (row, col) = (16 mt + 8 (tau%2) + g, 16 kt + 8 j + 2 q + e).
  // Both tiles read their element pairs (e = 0, 1) as one half2: keys from
  // token rows, values from the transposed channel rows.
  constexpr int NU = 8 / BITS;                // fields per byte
  constexpr int WPL = kG * kD * BITS / 1024;  // words per lane
  for (int widx = threadIdx.x; widx < 2 * 32 * WPL; widx += kQuantThreads) {
    const bool keys = widx < 32 * WPL;
    const int t = keys ? widx : widx - 32 * WPL;
    const int w = (t >> 7) * 4 + (t & 3);
    const int lane = (t >> 2) & 31;
    const int g = lane >> 2, q = lane & 3;
    const int pk = w / (4 / NU);
    const int kt = keys ? pk : (pk & 1);
    const int mt0 = keys ? 0 : 2 * (pk >> 1);
    const SliceQ *sq = keys ? kq : vq;
    const float *ssc = keys ? k_sc : v_sc;
    SliceQ sl[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) sl[j][e] = sq[16 * kt + 8 * j + 2 * q + e];
    uint32_t word = 0;
    bool near = false;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int tau = (w % (4 / NU)) * NU + u;
      const int row = 16 * (mt0 + (tau >> 1)) + 8 * (tau & 1) + g;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int col = 16 * kt + 8 * j + 2 * q;
        const float2 x = __half22float2(keys ? *reinterpret_cast<const __half2 *>(&sk[row][col])
                                             : *reinterpret_cast<const __half2 *>(&svT[row][col]));
        bool n0f, n1f;
        word |= fast_code(x.x, sl[j][0], n0f) << (8 * j + BITS * u);
        word |= fast_code(x.y, sl[j][1], n1f) << (16 + 8 * j + BITS * u);
        near |= n0f | n1f;
      }
    }
    if (__any_sync(0xffffffffu, near) && near) {
      // some field's fast code could differ from the IEEE one: redo the word
      word = 0;
      for (int f = 0; f < 4 * NU; ++f) {
        const int u = f >> 2, j = (f >> 1) & 1, e = f & 1;
        const int tau = (w % (4 / NU)) * NU + u;
        const int row = 16 * (mt0 + (tau >> 1)) + 8 * (tau & 1) + g;
        const int col = 16 * kt + 8 * j + 2 * q + e;
        const float x = __half2float(keys ? sk[row][col] : svT[row][col]);
        word |= exact_code<BITS>(x, sl[j][e].mn, ssc[col]) << (16 * e + 8 * j + BITS * u);
      }
    }
    reinterpret_cast<uint32_t *>(blk + (keys ? off_kc(BITS) : off_vc(BITS)))[t] = word;
  }
}

// Length bits of seq_len; while the fused step append runs, the bits above
// count the CTAs of a sequence that have finished with it.
constexpr int kLenBits = 22;
constexpr int kLenMask = (1 << kLenBits) - 1;

// One CTA quantizes one 32-token group of one (sequence, KV head).
// grid = (group slot, KV head, sequence).
template <int BITS>
__global__ void __launch_bounds__(kQuantThreads) quant_flush_kernel(Geo geo, const __half *__restrict__ k_new,
                                                                    const __half *__restrict__ v_new,
                                                                    const int *__restrict__ new_len, int max_new) {
  const int s = blockIdx.z, h = blockIdx.y, gslot = blockIdx.x;
  const int L0 = geo.seq_len[s];
  const int nn = new_len[s];
  if (nn < 0 || nn > max_new || L0 + nn > geo.capacity || L0 < 0) return;  // reported by the tail kernel
  const int n0 = max(L0 - geo.ns, 0);
  const int Lq0 = n0 - n0 % geo.R;
  const int n1 = max(L0 + nn - geo.ns, 0);
  const int Lq1 = n1 - n1 % geo.R;
  if (gslot >= (Lq1 - Lq0) / kG) return;
  flush_group<BITS>(geo, s, h, Lq0 + gslot * kG, n0, Lq0, L0, k_new, v_new, max_new);
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
      dk = geo.k_res + (sh * geo.R + slot) * kD;
      dv = geo.v_res + (sh * geo.R + slot) * kD;
    }
    const size_t src = (sh * max_new + j) * kD + c8 * 8;
    reinterpret_cast<uint4 *>(dk)[c8] = *reinterpret_cast<const uint4 *>(k_new + src);
    reinterpret_cast<uint4 *>(dv)[c8] = *reinterpret_cast<const uint4 *>(v_new + src);
  }
}

// Append of at most R new tokens per sequence in one kernel, one CTA per
// (KV head, sequence): at most one window fills, and the CTA then quantizes
// its R / 32 groups one after another.  Each CTA adds 1 << kLenBits to
// seq_len[s] once it needs seq_len no more; the CTA that completes the count
// (Hkv arrivals) stores the final length (clearing the count) and reports
// bad lengths, and no CTA reads seq_len[s] after that store.  When no window
// fills, a CTA arrives right after reading the length and copies its head's
// new tokens into the window (or sink), prefetched at launch.  When one
// fills, the copy would overwrite window slots the sequence's other CTAs may
// still be quantizing, so the CTAs arrive after quantizing and the last one
// copies the new tokens of every head.
template <int BITS>
__global__ void __launch_bounds__(kQuantThreads) step_append_kernel(Geo geo, const __half *__restrict__ k_new,
                                                                    const __half *__restrict__ v_new,
                                                                    const int *__restrict__ new_len, int max_new) {
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
            dk = geo.k_res + (sh * geo.R + slot) * kD;
            dv = geo.v_res + (sh * geo.R + slot) * kD;
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
    for (int i0 = Lq0; i0 < Lq1; i0 += kG) {
      flush_group<BITS>(geo, s, h, i0, n0, Lq0, L0, k_new, v_new, max_new);
      __syncthreads();  // the group's reads are done and its shared tiles free again
    }
    if (threadIdx.x == 0) arrive();
    __syncthreads();
    if (s_last) copy_tail(geo, s, 0, geo.H, L0, nn, k_new, v_new, max_new, threadIdx.x, blockDim.x);
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

// Upper bound on groups quantized per (sequence, head) by one append of at
// most max_new tokens: a window holding R-1 tokens plus max_new new ones.
int max_flush_groups(int R, int max_new) { return ((R - 1 + max_new) / R) * (R / kG); }

cudaError_t launch_quant_append(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                                int max_new, cudaStream_t stream, uint64_t *launches) {
  // a decode-sized append (at most one window fills): one kernel
  if (max_new <= geo.R && geo.capacity <= kLenMask && geo.H < (1 << (31 - kLenBits))) {
    dim3 grid(geo.H, geo.S);
    if (geo.bits == 2)
      step_append_kernel<2><<<grid, kQuantThreads, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
    else
      step_append_kernel<4><<<grid, kQuantThreads, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
    ++*launches;
    return cudaGetLastError();
  }
  const int gmax = max_flush_groups(geo.R, max_new);
  if (gmax > 0) {
    dim3 grid(gmax, geo.H, geo.S);
    if (geo.bits == 2)
      quant_flush_kernel<2><<<grid, kQuantThreads, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
    else
      quant_flush_kernel<4><<<grid, kQuantThreads, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
    ++*launches;
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  append_tail_kernel<<<geo.S, 256, 0, stream>>>(geo, k_new, v_new, new_len, max_new);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace kvq
