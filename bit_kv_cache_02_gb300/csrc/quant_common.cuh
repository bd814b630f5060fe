// Arithmetic shared by the quantize kernels: the exact code of a value in
// its slice (fast reciprocal filter with an IEEE fallback), paired fp32
// operations, fp16 pair min/max, and the shared -> global bulk store.
//
// Source: "KIVI: A Tuning-Free Asymmetric 2bit Quantization for KV Cache",
// second paragraph (asymmetric min/scale codes per slice); the code of x is
// clamp(rne(fl(fl(x - min) / scale)), 0, 2^b - 1) with scale 0 giving 0.
#pragma once

#include "kvq_internal.cuh"

namespace kvq {

constexpr float kMagic = 12582912.f;    // 1.5 * 2^23: x + kMagic rounds x to an integer (half to even)
constexpr float kPackBase = 8388608.f;  // 2^23: the low bits of 2^23 + n hold the integer n < 2^23

// Per-slice (one key channel of a group, or one value token) constants of
// the code computation.  The code is rne(fl(fl(x - min) / scale)) clamped
// to [0, 2^b - 1], scale == 0 giving 0.  It is first evaluated from
// y' = fma(x, rcp, c) with rcp = 1/scale to 2^-22 relative (the hardware
// approximate reciprocal) and c = fl(-min * rcp).  With Q = (x - min) /
// scale <= 2^b - 1 (to 2^-24), y' - Q stays below (2^b - 1) (2^-22 + 2^-24)
// + |c| 2^-24 and the IEEE result fl(fl(x - min) / scale) - Q below (2^b -
// 1) 2^-23, both under tol / 2 = 2^b 2^-21 + |c| 2^-23; when y' lies
// farther than tol from every rounding boundary k + 1/2, all three round to
// the same integer.  Otherwise the IEEE subtract and divide decide.
struct SliceQ {
  float rcp, c, tol, mn;
};

__device__ __forceinline__ SliceQ make_slice(float mn, float scale, float levels) {
  SliceQ q;
  q.mn = mn;
  float rcp;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(rcp) : "f"(scale));
  q.rcp = scale > 0.f ? rcp : 0.f;
  q.c = __fmul_rn(-mn, q.rcp);
  q.tol = (levels + 1.f) * 9.5367431640625e-07f + fabsf(q.c) * 2.384185791015625e-07f;  // 2^-20, 2^-22
  return q;
}

// The code by the IEEE subtract and divide (rarely needed, kept out of line).
template <int BITS>
__device__ __noinline__ uint32_t exact_code(float x, float mn, float scale) {
  const float r = rintf(__fdiv_rn(__fsub_rn(x, mn), scale));
  return static_cast<uint32_t>(fminf(fmaxf(r, 0.f), float((1 << BITS) - 1)));
}

// ------------------------------------------------- paired fp32 arithmetic

typedef unsigned long long f2x;  // two fp32 lanes in one 64-bit register

__device__ __forceinline__ f2x f2_pack(float a, float b) {
  f2x u;
  asm("mov.b64 %0, {%1, %2};" : "=l"(u) : "f"(a), "f"(b));
  return u;
}
__device__ __forceinline__ float2 f2_unpack(f2x u) {
  float2 f;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(f.x), "=f"(f.y) : "l"(u));
  return f;
}
__device__ __forceinline__ f2x f2_fma(f2x a, f2x b, f2x c) {
  f2x d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ f2x f2_add(f2x a, f2x b) {
  f2x d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ f2x f2_sub(f2x a, f2x b) {
  f2x d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ uint32_t h2min(uint32_t a, uint32_t b) {
  const __half2 m = __hmin2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
  return *reinterpret_cast<const uint32_t *>(&m);
}
__device__ __forceinline__ uint32_t h2max(uint32_t a, uint32_t b) {
  const __half2 m = __hmax2(*reinterpret_cast<const __half2 *>(&a), *reinterpret_cast<const __half2 *>(&b));
  return *reinterpret_cast<const uint32_t *>(&m);
}
// fp16 pair -> fp32, + 0 so that a zero extreme is stored as +0 whichever
// zero the reduction kept
__device__ __forceinline__ float2 h2_to_f2_pos0(uint32_t a) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&a));
  return make_float2(__fadd_rn(f.x, 0.f), __fadd_rn(f.y, 0.f));
}

// One-dimensional bulk copy shared -> global as its own bulk group.
__device__ __forceinline__ void bulk_s2g(void *dst_gmem, const void *src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
               "r"(static_cast<uint32_t>(__cvta_generic_to_shared(src_smem))), "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// the shared source of every committed bulk copy has been read
__device__ __forceinline__ void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// every committed bulk copy has completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Codes of one packed word from NF fp16 pairs: pair f holds the fields e = 0
// and e = 1 of one (u, j), placed at bits pos[f] and 16 + pos[f].  The two
// lanes of the paired arithmetic are the e = 0 and e = 1 halves of the word;
// each accumulates its codes as 2^23 + sum code * 2^pos, exact in fp32, and
// the low 16 bits of both are joined by one byte permute.  Sets `near` when
// some y' lies farther than thr = 1/2 - tol from its rounded value, i.e.
// within tol of a rounding boundary (the word is then redone exactly).
template <int NF>
__device__ __forceinline__ uint32_t pack_word(const uint32_t (&x)[NF], const f2x (&rcp)[NF], const f2x (&c)[NF],
                                              const int (&pos)[NF], float thr, bool &near) {
  const f2x magic = f2_pack(kMagic, kMagic);
  f2x acc = f2_pack(kPackBase, kPackBase);
  float emax = 0.f;
#pragma unroll
  for (int f = 0; f < NF; ++f) {
    const float2 xf = __half22float2(*reinterpret_cast<const __half2 *>(&x[f]));
    const f2x y = f2_fma(f2_pack(xf.x, xf.y), rcp[f], c[f]);
    const f2x r = f2_sub(f2_add(y, magic), magic);  // rne(y'), exact
    const float2 e = f2_unpack(f2_sub(y, r));
    emax = fmaxf(emax, fmaxf(fabsf(e.x), fabsf(e.y)));
    const float sc = __int_as_float((127 + pos[f]) << 23);  // 2^pos
    acc = f2_fma(r, f2_pack(sc, sc), acc);
  }
  near = emax > thr;
  const float2 a = f2_unpack(acc);
  return __byte_perm(__float_as_uint(a.x), __float_as_uint(a.y), 0x5410);
}

}  // namespace kvq
