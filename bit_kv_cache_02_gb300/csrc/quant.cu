// Quantize-and-pack of full windows (flush) and the fp16 window / sink append.
//
// Source: "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
// second paragraph (keys per channel in 32-token groups, values per token)
// and third paragraph (newest tokens kept in full precision, quantized in
// blocks when the window fills); "KV cache quantization", "What they report"
// (first token kept in fp16).
#include "kvq_internal.cuh"

namespace kvq {

// Code of one element: clamp(rne((x - mn) / scale), 0, 2^b - 1), each step an
// IEEE fp32 operation; scale == 0 gives 0.
template <int BITS>
__device__ __forceinline__ uint32_t quant_code(float x, float mn, float scale) {
  if (scale == 0.f) return 0u;
  float y = __fdiv_rn(__fsub_rn(x, mn), scale);
  float c = rintf(y);  // round half to even
  c = fminf(fmaxf(c, 0.f), float((1 << BITS) - 1));
  return static_cast<uint32_t>(c);
}

constexpr int kQuantThreads = 256;

// One CTA quantizes one 32-token group of one (sequence, KV head).
// grid = (group slot, KV head, sequence).  Tokens of the group come from the
// old window (stream index < n0) or from the new input.
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
  const int i0 = Lq0 + gslot * kG;  // first stream index of this group

  __shared__ __align__(16) __half sk[kG][kD];
  __shared__ __align__(16) __half sv[kG][kD];
  __shared__ float k_sc[kD], k_mn[kD], v_sc[kG], v_mn[kG];

  const size_t sh = static_cast<size_t>(s) * geo.H + h;
  for (int idx = threadIdx.x; idx < kG * kD / 8; idx += kQuantThreads) {
    const int t = idx / (kD / 8), c8 = idx % (kD / 8);
    const int i = i0 + t;
    const __half *pk, *pv;
    if (i < n0) {
      const size_t off = (sh * geo.R + (i - Lq0)) * kD;
      pk = geo.k_res + off;
      pv = geo.v_res + off;
    } else {
      const int j = i + geo.ns - L0;
      const size_t off = (sh * max_new + j) * kD;
      pk = k_new + off;
      pv = v_new + off;
    }
    *reinterpret_cast<uint4 *>(&sk[t][c8 * 8]) = *reinterpret_cast<const uint4 *>(pk + c8 * 8);
    *reinterpret_cast<uint4 *>(&sv[t][c8 * 8]) = *reinterpret_cast<const uint4 *>(pv + c8 * 8);
  }
  __syncthreads();

  const float levels = float((1 << BITS) - 1);
  uint8_t *blk = geo.blocks + (sh * geo.max_groups + i0 / kG) * static_cast<size_t>(block_bytes(BITS));
  if (threadIdx.x < kD) {  // keys: one channel per thread, min/max over the 32 tokens
    const int d = threadIdx.x;
    float mn = __half2float(sk[0][d]), mx = mn;
#pragma unroll 8
    for (int t = 1; t < kG; ++t) {
      const float x = __half2float(sk[t][d]);
      mn = fminf(mn, x);
      mx = fmaxf(mx, x);
    }
    const float sc = __fdiv_rn(__fsub_rn(mx, mn), levels);
    k_sc[d] = sc;
    k_mn[d] = mn;
    reinterpret_cast<float *>(blk + off_ks(BITS))[d] = sc;
    reinterpret_cast<float *>(blk + off_km(BITS))[d] = mn;
  } else {  // values: warp w' takes tokens 8w'..8w'+7, min/max over 128 channels
    const int w = (threadIdx.x - kD) >> 5, lane = threadIdx.x & 31;
    for (int tt = 0; tt < kG / 4; ++tt) {
      const int t = w * (kG / 4) + tt;
      float mn = __half2float(sv[t][lane * 4]), mx = mn;
#pragma unroll
      for (int c = 1; c < 4; ++c) {
        const float x = __half2float(sv[t][lane * 4 + c]);
        mn = fminf(mn, x);
        mx = fmaxf(mx, x);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      }
      if (lane == 0) {
        const float sc = __fdiv_rn(__fsub_rn(mx, mn), levels);
        v_sc[t] = sc;
        v_mn[t] = mn;
        reinterpret_cast<float *>(blk + off_vs(BITS))[t] = sc;
        reinterpret_cast<float *>(blk + off_vm(BITS))[t] = mn;
      }
    }
  }
  __syncthreads();

  // Pack: word index t of a tile lives at byte 4t; t = (w/4)*128 + lane*4 + w%4.
  constexpr int NU = 8 / BITS;           // fields per byte
  constexpr int WPL = kG * kD * BITS / 1024;  // words per lane
  for (int widx = threadIdx.x; widx < 2 * 32 * WPL; widx += kQuantThreads) {
    const int tile = widx / (32 * WPL);  // 0: keys, 1: values
    const int t = widx % (32 * WPL);
    const int w = (t >> 7) * 4 + (t & 3);
    const int lane = (t >> 2) & 31;
    const int g = lane >> 2, q = lane & 3;
    const int KT = tile == 0 ? kD / 16 : kG / 16;
    uint32_t word = 0;
#pragma unroll
    for (int u = 0; u < NU; ++u) {
      const int tau = (w % (4 / NU)) * NU + u;
      const int pk = w / (4 / NU);
      const int P = pk / KT, kt = pk % KT;
      const int row = 16 * (2 * P + (tau >> 1)) + 8 * (tau & 1) + g;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int col = 16 * kt + 8 * j + 2 * q + e;
          uint32_t c;
          if (tile == 0) {  // row = token, col = channel
            c = quant_code<BITS>(__half2float(sk[row][col]), k_mn[col], k_sc[col]);
          } else {  // row = channel, col = token
            c = quant_code<BITS>(__half2float(sv[col][row]), v_mn[col], v_sc[col]);
          }
          word |= c << (16 * e + 8 * j + BITS * u);
        }
      }
    }
    reinterpret_cast<uint32_t *>(blk + (tile == 0 ? off_kc(BITS) : off_vc(BITS)))[t] = word;
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
  const int n1 = max(L0 + nn - geo.ns, 0);
  const int Lq1 = n1 - n1 % geo.R;
  const int j_sink_end = min(max(geo.ns - L0, 0), nn);      // new tokens [0, j_sink_end) -> sink
  const int j_win = max(Lq1 + geo.ns - L0, j_sink_end);      // new tokens [j_win, nn) -> window
  const int n_copy = j_sink_end + (nn - j_win);
  constexpr int C16 = kD / 8;  // 16-byte chunks per token row
  for (int idx = threadIdx.x; idx < geo.H * n_copy * C16; idx += blockDim.x) {
    const int c8 = idx % C16;
    const int k = (idx / C16) % n_copy;
    const int h = idx / (C16 * n_copy);
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
  __syncthreads();
  if (threadIdx.x == 0) geo.seq_len[s] = L0 + nn;
}

// Upper bound on groups quantized per (sequence, head) by one append of at
// most max_new tokens: a window holding R-1 tokens plus max_new new ones.
int max_flush_groups(int R, int max_new) { return ((R - 1 + max_new) / R) * (R / kG); }

cudaError_t launch_quant_append(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                                int max_new, cudaStream_t stream, uint64_t *launches) {
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
