// Dequantization of the whole cache into fp32 (test aid).
//
// Source: asymmetric codes x_hat = code * scale + min ("KV cache
// quantization", "What they report"); keys per channel / values per token
// (KIVI page, second paragraph).  Keys are returned pre-RoPE.  When the
// cache rotates its tokens (Walsh-Hadamard, include/kvq.h) the group rows
// are rotated back, x_hat = H y_hat, in fp32.  Dense-and-sparse blocks
// return each slice's outlier as its stored fp16 value.
#include "kvq_internal.cuh"

namespace kvq {

// Code of element (row, col) of a packed tile with `cols` columns.
template <int BITS>
__device__ __forceinline__ uint32_t tile_code(const uint8_t *tile, int row, int col, int cols) {
  constexpr int NU = 8 / BITS;
  const int mt = row >> 4, h = (row >> 3) & 1, g = row & 7;
  const int kt = col >> 4, j = (col >> 3) & 1, q = (col & 7) >> 1, e = col & 1;
  const int tau = 2 * (mt & 1) + h;
  const int P = mt >> 1;
  const int w = (P * (cols >> 4) + kt) * (4 / NU) + tau / NU;
  const int lane = 4 * g + q;
  const uint32_t word = reinterpret_cast<const uint32_t *>(tile)[((w >> 2) * 32 + lane) * 4 + (w & 3)];
  return (word >> (16 * e + 8 * j + BITS * (tau % NU))) & ((1u << BITS) - 1u);
}

// grid = (group slot + 1, KV head, sequence); the last slot converts the
// sink and the window.  KPT: key scale and min per token instead of per
// channel.
template <int BITS, bool KPT>
__global__ void __launch_bounds__(256) dequant_kernel(Geo geo, float *__restrict__ k_out, float *__restrict__ v_out) {
  const int s = blockIdx.z, h = blockIdx.y, gi = blockIdx.x;
  const int L = geo.seq_len[s];
  if (L < 0 || L > geo.capacity) return;
  const Split sp = split_len(L, geo.ns, geo.R);
  const size_t sh = static_cast<size_t>(s) * geo.H + h;
  float *ko = k_out + sh * geo.capacity * kD;
  float *vo = v_out + sh * geo.capacity * kD;
  if (gi < geo.max_groups) {
    if (gi >= sp.Lq / kG) return;
    const uint8_t *blk = group_block(geo, s, h, gi, block_bytes(BITS, KPT, geo.sparse != 0));
    if (!blk) {
      if (threadIdx.x == 0) set_status(geo.status, KVQ_STATUS_BAD_BLOCK);
      return;
    }
    const float *ks = reinterpret_cast<const float *>(blk + off_ks(BITS));
    const float *km = reinterpret_cast<const float *>(blk + off_km(BITS, KPT));
    const float *vs = reinterpret_cast<const float *>(blk + off_vs(BITS, KPT));
    const float *vm = reinterpret_cast<const float *>(blk + off_vm(BITS, KPT));
    const uint32_t *ksp = reinterpret_cast<const uint32_t *>(blk + off_ksp(BITS, KPT));
    const uint32_t *vsp = reinterpret_cast<const uint32_t *>(blk + off_vsp(BITS, KPT));
    const int p0 = sp.nsink + gi * kG;
    __shared__ float rows[2 * kG][kD];  // rotated layout: key rows, then value rows
    for (int idx = threadIdx.x; idx < kG * kD; idx += blockDim.x) {
      const int t = idx / kD, d = idx % kD;
      const uint32_t ck = tile_code<BITS>(blk + off_kc(BITS), t, d, kD);
      const uint32_t cv = tile_code<BITS>(blk + off_vc(BITS), d, t, kG);
      float kx = fmaf(static_cast<float>(ck), ks[KPT ? t : d], km[KPT ? t : d]);
      float vx = fmaf(static_cast<float>(cv), vs[t], vm[t]);
      if (geo.sparse) {  // entry: fp16 bits, index within the slice at bit 16
        const uint32_t ek = ksp[KPT ? t : d], ev = vsp[t];
        if (static_cast<int>(ek >> 16) == (KPT ? d : t)) kx = __half2float(__ushort_as_half(ek & 0xFFFFu));
        if (static_cast<int>(ev >> 16) == d) vx = __half2float(__ushort_as_half(ev & 0xFFFFu));
      }
      if (geo.rot) {
        rows[t][d] = kx;
        rows[kG + t][d] = vx;
      } else if (KVQ_IN_BOUNDS(geo.status, p0 + t, geo.capacity)) {
        ko[static_cast<size_t>(p0 + t) * kD + d] = kx;
        vo[static_cast<size_t>(p0 + t) * kD + d] = vx;
      }
    }
    if (geo.rot) {  // x = H y: butterflies (a, b) -> (a + b, a - b) per stride
      for (int st = 1; st < kD; st <<= 1) {
        __syncthreads();
        for (int i = threadIdx.x; i < 2 * kG * (kD / 2); i += blockDim.x) {
          const int row = i / (kD / 2), b = i % (kD / 2);
          const int lo = (b / st) * 2 * st + b % st;
          const float x0 = rows[row][lo], x1 = rows[row][lo + st];
          rows[row][lo] = x0 + x1;
          rows[row][lo + st] = x0 - x1;
        }
      }
      __syncthreads();
      for (int idx = threadIdx.x; idx < kG * kD; idx += blockDim.x) {
        const int t = idx / kD, d = idx % kD;
        if (!KVQ_IN_BOUNDS(geo.status, p0 + t, geo.capacity)) continue;
        ko[static_cast<size_t>(p0 + t) * kD + d] = rows[t][d];
        vo[static_cast<size_t>(p0 + t) * kD + d] = rows[kG + t][d];
      }
    }
  } else {
    const int n = sp.nsink + sp.r;
    for (int idx = threadIdx.x; idx < n * kD; idx += blockDim.x) {
      const int t = idx / kD, d = idx % kD;
      int pos;
      const __half *kp, *vp;
      if (t < sp.nsink) {
        pos = t;
        kp = geo.k_sink + (sh * geo.ns + t) * kD;
        vp = geo.v_sink + (sh * geo.ns + t) * kD;
      } else {
        const int slot = t - sp.nsink;
        pos = sp.nsink + sp.Lq + slot;
        kp = geo.k_res + (sh * geo.R + slot) * kD;
        vp = geo.v_res + (sh * geo.R + slot) * kD;
      }
      if (!KVQ_IN_BOUNDS(geo.status, pos, geo.capacity)) continue;
      ko[static_cast<size_t>(pos) * kD + d] = __half2float(kp[d]);
      vo[static_cast<size_t>(pos) * kD + d] = __half2float(vp[d]);
    }
  }
}

cudaError_t launch_dequant(const Geo &geo, float *k_out, float *v_out, cudaStream_t stream, uint64_t *launches) {
  dim3 grid(geo.max_groups + 1, geo.H, geo.S);
  if (geo.bits == 2)
    (geo.kpt ? dequant_kernel<2, true> : dequant_kernel<2, false>)<<<grid, 256, 0, stream>>>(geo, k_out, v_out);
  else
    (geo.kpt ? dequant_kernel<4, true> : dequant_kernel<4, false>)<<<grid, 256, 0, stream>>>(geo, k_out, v_out);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace kvq
