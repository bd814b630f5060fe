// Decode attention: the plan kernel, the RoPE tables, the workspace plan and
// the launch of the contiguous-layout kernels (the paged-layout, the
// rotating-cache and the dense-and-sparse kernels are instantiated in
// decode_paged.cu, decode_rot*.cu and decode_sparse*.cu).  The kernel itself
// is in decode_kernel.cuh.
#include "decode_kernel.cuh"

namespace kvq {

// Per-sequence unit prefix (exclusive) times Hkv, the total, and zero output
// rows for sequences with nothing to attend, for batches too large to plan
// inside the decode kernel.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) decode_plan_kernel(DecodeArgs a) {
  __shared__ long long warp_sum[32];
  const int S = a.geo.S, H = a.geo.H;
  const int per = (S + blockDim.x - 1) / blockDim.x;
  const int s0 = threadIdx.x * per, s1 = min(S, s0 + per);
  long long mine = 0;
  for (int s = s0; s < s1; ++s) {
    Split spl;
    int tp, ng;
    mine += seq_units(a, s, spl, tp, ng);
  }
  // exclusive block scan of `mine`
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long v = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) warp_sum[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    long long ws = lane < static_cast<int>(blockDim.x >> 5) ? warp_sum[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long v = __shfl_up_sync(kFull, ws, o);
      if (lane >= o) ws += v;
    }
    warp_sum[lane] = ws;  // inclusive over warps
  }
  __syncthreads();
  long long run = incl - mine + (warp > 0 ? warp_sum[warp - 1] : 0);
  for (int s = s0; s < s1; ++s) {
    a.base[s] = run * H;
    Split spl;
    int tp, ng;
    run += seq_units(a, s, spl, tp, ng);
  }
  if (threadIdx.x == blockDim.x - 1) {
    a.base[S] = run * H;
    a.plan->total = run * H;
  }
  // sequences with nothing to attend (empty, or longer than the cache or the
  // planned bound) get zero output rows, one warp per sequence
  for (int s = warp; s < S; s += blockDim.x >> 5) {
    const int L = a.geo.seq_len[s];
    if (L > 0 && L <= a.geo.capacity && L <= a.max_len) continue;
    if (lane == 0 && L > a.max_len) set_status(a.geo.status, KVQ_STATUS_MAX_LEN);
    uint4 *o = reinterpret_cast<uint4 *>(a.out + static_cast<size_t>(s) * a.Hq * kD);
    for (int i = lane; i < a.Hq * kD / 8; i += 32) o[i] = make_uint4(0u, 0u, 0u, 0u);
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

static int g_warps_override = 0;
static long long g_wait_limit = 0;
static int g_wait_before_fetch = 0;

int decode_warps_override() { return g_warps_override; }

int set_wait_test(long long cycles, int wait_before_fetch) {
  if (cycles < 0 || cycles > kWaitLimitCycles || (wait_before_fetch != 0 && wait_before_fetch != 1)) return -1;
  if (wait_before_fetch && cycles == 0) return -1;  // a wait that nothing completes needs a short limit
  g_wait_limit = cycles;
  g_wait_before_fetch = wait_before_fetch;
  return 0;
}

cudaError_t launch_plan(const DecodeArgs &a, cudaStream_t stream) {
  decode_plan_kernel<<<1, 1024, 0, stream>>>(a);
  return cudaGetLastError();
}

int set_decode_warps(int warps) {
  if (warps < 0 || warps > kMaxDecodeWarps) return -1;
  g_warps_override = warps;
  return 0;
}

static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

DecodePlan plan_decode(const Geo &geo, int Hq, int max_len) {
  DecodePlan p;
  const int gq = Hq / geo.H;
  const size_t pairs = static_cast<size_t>(geo.S) * geo.H;
  p.tail_passes = (geo.R - 1 + geo.ns + 31) / 32;
  p.n_base = geo.pre_rope ? (max(max_len - geo.ns, 1) + kG - 1) / kG : 0;
  // group partial slots gw + pair (gw < kMaxDecodeWarps), then the window
  // pass slots pair * tail_passes + k
  p.pass_slot0 = kMaxDecodeWarps + pairs;
  const size_t slots = p.pass_slot0 + pairs * p.tail_passes;
  p.off_ml = align256(slots * gq * kD * sizeof(float));
  p.off_cnt = p.off_ml + align256(slots * gq * sizeof(float2));
  p.off_base = p.off_cnt + align256(pairs * sizeof(int));
  p.off_hdr = p.off_base + align256((static_cast<size_t>(geo.S) + 1) * sizeof(long long));
  p.off_rope = p.off_hdr + 256;
  p.off_off = p.off_rope + align256(static_cast<size_t>(p.n_base) * 64 * sizeof(float2));
  p.bytes = geo.pre_rope ? p.off_off + align256(kG * 64 * sizeof(float2)) : p.off_rope;
  return p;
}

cudaError_t launch_decode(const Geo &geo, int Hq, const __half *q, float softmax_scale, __half *out,
                          void *workspace, const DecodePlan &p, int max_len, bool zero_counters,
                          cudaStream_t stream, uint64_t *launches) {
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
  // batches of up to kInlinePlanSeqs sequences are planned inside the decode
  // kernel; larger ones by a one-CTA plan kernel
  const bool inline_plan = geo.S <= kInlinePlanSeqs;
  a.base = inline_plan ? nullptr : reinterpret_cast<long long *>(ws + p.off_base);
  a.plan = reinterpret_cast<PlanHeader *>(ws + p.off_hdr);
  a.nw = 0;
  a.pass_slot0 = p.pass_slot0;
  a.tail_passes = p.tail_passes;
  a.max_len = max_len;
  a.wait_limit = g_wait_limit ? g_wait_limit : kWaitLimitCycles;
  a.wait_before_fetch = g_wait_before_fetch;
  a.n_slots = p.pass_slot0 + static_cast<size_t>(geo.S) * geo.H * p.tail_passes;
  a.n_base = p.n_base;
  a.rope_base = reinterpret_cast<const float2 *>(ws + p.off_rope);
  a.rope_off = reinterpret_cast<const float2 *>(ws + p.off_off);
  cudaError_t e = cudaSuccess;
  if (zero_counters &&
      (e = cudaMemsetAsync(a.counters, 0, static_cast<size_t>(geo.S) * geo.H * sizeof(int), stream)) != cudaSuccess)
    return e;
  if (geo.pre_rope) {
    const int n = (p.n_base + kG) * 64;
    rope_table_kernel<<<(n + 255) / 256, 256, 0, stream>>>(reinterpret_cast<float2 *>(ws + p.off_rope), p.n_base,
                                                           reinterpret_cast<float2 *>(ws + p.off_off), geo.ns,
                                                           geo.theta);
    ++*launches;
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  const int gq = Hq / geo.H;
  if (geo.sparse)
    e = geo.table ? launch_sparse_paged(a, gq, stream) : launch_sparse(a, gq, stream);
  else if (geo.rot)
    e = geo.table ? launch_rot_paged(a, gq, stream) : launch_rot(a, gq, stream);
  else if (geo.table)
    e = launch_paged(a, gq, stream);
  else
    e = geo.bits == 2 ? launch_b<2, false, false, false>(a, gq, stream) : launch_b<4, false, false, false>(a, gq, stream);
  *launches += inline_plan ? 1 : 2;
  return e;
}

}  // namespace kvq
