// Internal definitions shared by the kernels of the low-bit KV-cache library.
//
// Packed block (one group of 32 tokens of one (sequence, KV head)):
//   [K codes 32*D*b/8][V codes 32*D*b/8][K scale f32 D][K min f32 D]
//   [V scale f32 32][V min f32 32]
// A code tile is 32 lanes x W 32-bit words.  Element (row, col) (keys: row =
// token, col = channel; values: row = channel, col = token) sits in lane
// 4*(row%8) + (col%8)/2, word w = (P*KT + kt)*(4/nu) + tau/nu, bit
// 16*(col%2) + 8*((col/8)%2) + b*(tau%nu), where mt = row/16, tau =
// 2*(mt%2) + (row/8)%2, P = mt/2, kt = col/16, KT = cols/16, nu = 8/b.  Word
// w of lane l is at byte ((w/4)*32 + l)*16 + (w%4)*4.  With this order one
// 32-bit word yields, under a single AND mask, a half2 register of the
// m16n8k16 A fragment whose two fp16 values are (code << b*u) * 2^-24 (fp16
// subnormals), which the tensor core multiplies exactly.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kD = 128;       // head dimension
constexpr int kG = 32;        // tokens per group

// Key metadata holds one (scale, min) per channel, or per token when keys
// are grouped per token (kpt).
__host__ __device__ constexpr int code_tile_bytes(int bits) { return kG * kD * bits / 8; }
__host__ __device__ constexpr int kmeta_n(bool kpt) { return kpt ? kG : kD; }
// sp: dense-and-sparse blocks add one 32-bit outlier entry per key slice and
// per value token (fp16 value bits 0-15, index within the slice at bit 16).
__host__ __device__ constexpr int block_bytes(int bits, bool kpt = false, bool sp = false) {
  return 2 * code_tile_bytes(bits) + 8 * kmeta_n(kpt) + 8 * kG + (sp ? 4 * (kmeta_n(kpt) + kG) : 0);
}
__host__ __device__ constexpr int off_kc(int) { return 0; }
__host__ __device__ constexpr int off_vc(int bits) { return code_tile_bytes(bits); }
__host__ __device__ constexpr int off_ks(int bits) { return 2 * code_tile_bytes(bits); }
__host__ __device__ constexpr int off_km(int bits, bool kpt = false) { return off_ks(bits) + 4 * kmeta_n(kpt); }
__host__ __device__ constexpr int off_vs(int bits, bool kpt = false) { return off_km(bits, kpt) + 4 * kmeta_n(kpt); }
__host__ __device__ constexpr int off_vm(int bits, bool kpt = false) { return off_vs(bits, kpt) + 4 * kG; }
__host__ __device__ constexpr int off_ksp(int bits, bool kpt = false) { return off_vm(bits, kpt) + 4 * kG; }
__host__ __device__ constexpr int off_vsp(int bits, bool kpt = false) { return off_ksp(bits, kpt) + 4 * kmeta_n(kpt); }

// Cache geometry and buffers as the kernels see them.
struct Geo {
  int S, H, R, ns, bits, pre_rope;
  int kpt;  // keys grouped per token
  int rot;  // tokens Walsh-Hadamard rotated before quantization
  int sparse;  // dense-and-sparse: each slice's largest-magnitude element kept apart
  float theta;
  int capacity;
  int max_groups;
  uint8_t *blocks;
  __half *k_res, *v_res, *k_sink, *v_sink;
  int *seq_len;
  int *status;
  const int *table;  // paged layout: logical group -> pool block (null: contiguous)
  int num_blocks;    // pool blocks when paged
};

// Block of logical group g of (s, h) (bb bytes per block), or null when the
// block table sends it outside the pool.
__device__ __forceinline__ uint8_t *group_block(const Geo &geo, int s, int h, int g, int bb) {
  const size_t lg = (static_cast<size_t>(s) * geo.H + h) * geo.max_groups + g;
  if (!geo.table) return geo.blocks + lg * bb;
  const int pb = geo.table[lg];
  if (pb < 0 || pb >= geo.num_blocks) return nullptr;
  return geo.blocks + static_cast<size_t>(pb) * bb;
}

// Stream bookkeeping of a sequence holding L tokens.
struct Split {
  int nsink;  // tokens in the sink
  int Lq;     // quantized stream tokens
  int r;      // tokens in the window
};

__host__ __device__ inline Split split_len(int L, int ns, int R) {
  Split sp;
  sp.nsink = L < ns ? L : ns;
  int n = L - sp.nsink;
  sp.r = n % R;
  sp.Lq = n - sp.r;
  return sp;
}

// atomicAdd with acquire-release semantics at GPU scope; returns the old value.
__device__ inline int atom_add_acq_rel(int *p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

__device__ inline void set_status(int *status, int bit) {
  if (status) atomicOr(status, bit);
}

// Index checks of debug builds (compiled with -DKVQ_DEBUG_BOUNDS): an index
// outside [0, n) records KVQ_STATUS_BOUNDS and the guarded access is skipped,
// without a trap; release builds compile the checks away.  They cover the
// index arithmetic the kernels do on the device (block, window, sink,
// partial-slot, query, output and table rows), the part no host-side
// validation can see.
__device__ inline bool in_bounds(int *status, long long i, long long n) {
  if (i >= 0 && i < n) return true;
  set_status(status, KVQ_STATUS_BOUNDS);
  return false;
}
#ifdef KVQ_DEBUG_BOUNDS
#define KVQ_IN_BOUNDS(status, i, n) ::kvq::in_bounds((status), static_cast<long long>(i), static_cast<long long>(n))
#else
#define KVQ_IN_BOUNDS(status, i, n) true
#endif

// ---------------------------------------------------------------- PTX helpers

__device__ inline uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ inline void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ inline void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ inline void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ inline void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ inline bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait that lets the hardware suspend the warp for up to `ns`
// nanoseconds while the phase is incomplete (no spinning in the meantime).
__device__ inline bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of phase `parity` of `bar`.
__device__ inline bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// SM clock cycles a pipeline wait may last before it gives up (about two
// seconds).
constexpr long long kWaitLimitCycles = 4000000000LL;

// Wait for phase `parity` of `bar`, giving up once `limit` SM clock cycles
// have passed; returns false (and the caller records KVQ_STATUS_TIMEOUT) on
// timeout.  At the default limit the polls are try_waits, which suspend the
// warp while the phase is incomplete (up to a system-dependent time, then up
// to 100 us per poll); a shorter limit polls without suspending, so it holds
// to within one poll.
__device__ inline bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, long long limit = kWaitLimitCycles) {
  if (limit < kWaitLimitCycles) {
    const long long start = clock64();
    while (!mbar_test_wait(bar, parity)) {
      if (clock64() - start > limit) return false;
    }
    return true;
  }
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait_hint(bar, parity, 100000u)) {
    if (clock64() - start > limit) return false;
  }
  return true;
}

// 2^x on the special-function unit (approximate, flushes subnormal results
// to zero; softmax weights that small do not matter).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Orders this thread's earlier generic-proxy accesses of shared memory
// before its later async-proxy (bulk copy) accesses.
__device__ inline void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// One-dimensional bulk copy global -> shared, completing on `bar`.
__device__ inline void bulk_g2s(void *dst_smem, const void *src_gmem, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// D = A * B + D, m16n8k16, fp16 inputs, fp32 accumulators.
__device__ inline void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ inline uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }

// Split (x0, x1) into fp16 hi + lo parts: hi = fp16(x), lo = fp16(x - hi).
// Returns lo when `want_lo`, else hi.
__device__ inline uint32_t hi_or_lo(float x0, float x1, bool want_lo) {
  __half2 hi = __floats2half2_rn(x0, x1);
  float2 hf = __half22float2(hi);
  __half2 lo = __floats2half2_rn(x0 - hf.x, x1 - hf.y);
  return want_lo ? h2_as_u32(lo) : h2_as_u32(hi);
}

// ------------------------------------------------------- host-side launchers

// Warps one decode launch spreads its work over, at most (sizes the
// workspace's partial-result slots).
constexpr int kMaxDecodeWarps = 2560;

// Workspace plan of one decode call: window passes per (sequence, KV head)
// at most, RoPE base rows, and the byte offsets of the workspace regions
// (partial outputs, partial (max, sum), merge counters, per-sequence work
// prefix, plan header, RoPE tables), each 256-byte aligned.
struct DecodePlan {
  int tail_passes, n_base;
  size_t pass_slot0;
  size_t off_ml, off_cnt, off_base, off_hdr, off_rope, off_off, bytes;
};

cudaError_t launch_quant_append(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                                int max_new, cudaStream_t stream, uint64_t *launches);
// The flush of appends longer than the window by warps that each quantize
// whole key or value tiles (quant_tiles.cu): caches with per-channel keys,
// no rotation and no outlier entries, of at most kTileFlushMaxSeqs sequences
// (each warp plans its range from the lengths of all of them).
constexpr int kTileFlushMaxSeqs = 2048;
bool flush_tiles_serves(const Geo &geo);
cudaError_t launch_flush_tiles(const Geo &geo, const __half *k_new, const __half *v_new, const int *new_len,
                               int max_new, cudaStream_t stream);
cudaError_t launch_dequant(const Geo &geo, float *k_out, float *v_out, cudaStream_t stream, uint64_t *launches);
DecodePlan plan_decode(const Geo &geo, int Hq, int max_len);
cudaError_t launch_decode(const Geo &geo, int Hq, const __half *q, float softmax_scale, __half *out,
                          void *workspace, const DecodePlan &p, int max_len, bool zero_counters,
                          cudaStream_t stream, uint64_t *launches);
// kv_decode_attn that first clears the workspace's merge counters (for
// scratch shared by calls of different geometries).
int decode_attn_clearing(const kvq_cache *cache, int32_t num_q_heads, const uint16_t *q, float softmax_scale,
                         uint16_t *out, void *workspace, size_t workspace_bytes, int32_t max_len, void *stream);
int set_decode_warps(int warps);
// Test aid: cycle limit of the decode kernel's pipeline waits (0: the
// default) and whether each warp's first wait comes before its first copy.
int set_wait_test(long long cycles, int wait_before_fetch);

}  // namespace kvq
