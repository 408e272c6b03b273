// Device helpers for the selection kernel: order-preserving keys, inline PTX
// for mbarriers, TMA bulk copies and thread-block clusters (sm_90+ forms that
// sm_103a keeps), and compensated fp32 sums.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace qrita {
namespace dev {

// ---------------------------------------------------------------------------
// Order-preserving 32-bit keys. key(a) < key(b) iff a < b for non-NaN floats,
// with -0 mapped to the key of +0 so the two tie (the stable-sort contract
// treats them as equal). Keys below key(-inf) or above key(+inf) are NaNs.
// ---------------------------------------------------------------------------
constexpr uint32_t kKeyNegInf = 0x007FFFFFu;
constexpr uint32_t kKeyPosInf = 0xFF800000u;
constexpr uint32_t kKeyNegZero = 0x7FFFFFFFu;  // never produced by f2key

__device__ __forceinline__ uint32_t f2key(float x) {
  uint32_t b = __float_as_uint(x + 0.0f);  // -0 + 0 = +0; every other value unchanged
  uint32_t m = static_cast<uint32_t>(static_cast<int32_t>(b) >> 31) | 0x80000000u;
  return b ^ m;
}

__device__ __forceinline__ float key2f(uint32_t k) {
  uint32_t b = (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
  return __uint_as_float(b);
}

// Float a pivot key compares against: "x > pivot_f(q)" counts exactly the
// elements with key(x) > q. The one key with no canonical element, -0's raw
// key, is moved one step down (both keys count the same set).
__device__ __forceinline__ float pivot_f(uint32_t q) {
  return key2f(q == kKeyNegZero ? kKeyNegZero - 1u : q);
}

// NaN-propagating max (max.NaN): a NaN anywhere makes the result NaN.
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float r;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
  return r;
}

// ---------------------------------------------------------------------------
// Packed bf16 pairs (one 32-bit word holds elements 2i (low half) and 2i+1).
// ---------------------------------------------------------------------------
// Per-half NaN-propagating max and NaN-ignoring min.
__device__ __forceinline__ uint32_t bf2_max_nan(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t bf2_min(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// 0xFFFF in each half where a >= b (false for NaN), else 0.
__device__ __forceinline__ uint32_t bf2_ge_mask(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.ge.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t bf2_gt_mask(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.gt.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

__device__ __forceinline__ uint32_t bf2_eq_mask(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.eq.u32.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// The smallest bf16 value c >= t (t finite fp32), as raw bits: for bf16 x,
// x >= t exactly when x >= c. Truncating t's low half moves it toward zero:
// up for negative t, down for positive t, so only a positive inexact t steps
// to the next bf16.
__device__ __forceinline__ uint32_t bf16_ceil_bits(float t) {
  uint32_t tb = __float_as_uint(t) >> 16;
  if (__uint_as_float(tb << 16) < t) tb += 1u;
  return tb;
}

// ---------------------------------------------------------------------------
// Compensated fp32 sums: a value is hi + lo with |lo| <= ulp(hi)/2.
// two_sum is Knuth's error-free addition (6 flops, no ordering condition).
// ---------------------------------------------------------------------------
struct F2 {
  float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = a + b;
  float bb = s - a;
  e = (a - (s - bb)) + (b - bb);
}

__device__ __forceinline__ void f2_add(F2& acc, float w) {
  float s, e;
  two_sum(acc.hi, w, s, e);
  acc.hi = s;
  acc.lo += e;
}

__device__ __forceinline__ F2 f2_merge(F2 a, F2 b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e += a.lo + b.lo;
  F2 r;
  r.hi = s + e;
  r.lo = e - (r.hi - s);
  return r;
}

__device__ __forceinline__ F2 f2_make(float hi, float lo) {
  F2 r;
  r.hi = hi;
  r.lo = lo;
  return r;
}

// a - b
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
  F2 nb;
  nb.hi = -b.hi;
  nb.lo = -b.lo;
  return f2_merge(a, nb);
}

// p * a (FMA gives the exact error of the leading product)
__device__ __forceinline__ F2 f2_mul(F2 a, float p) {
  const float hi = p * a.hi;
  const float e = fmaf(p, a.hi, -hi) + p * a.lo;
  F2 r;
  r.hi = hi + e;
  r.lo = e - (r.hi - hi);
  return r;
}

// n * w as a pair (exact for integers n below 2^24)
__device__ __forceinline__ F2 f2_prod(float n, float w) {
  F2 r;
  r.hi = n * w;
  r.lo = fmaf(n, w, -r.hi);
  return r;
}

// a >= b, decided on the pair difference (sign exact to about 2^-48 relative)
__device__ __forceinline__ bool f2_ge(F2 a, F2 b) {
  const F2 d = f2_sub(a, b);
  return d.hi > 0.f || (d.hi == 0.f && d.lo >= 0.f);
}

__device__ __forceinline__ float f2_float(F2 a) { return a.hi + a.lo; }

// round(v), ties to even, for a float 0 <= v < 2^63: the value a 64-bit
// round-to-nearest conversion gives, from two 32-bit conversions (64-bit
// conversions issue on this GPU's narrow fp64 pipe). With h = floor(v / 2^32),
// r = v - h 2^32 is exact in fp32 (v mod 2^32 keeps at most v's 24
// significant bits), so round(v) = h 2^32 + round(r), and round(r) < 2^32.
__device__ __forceinline__ unsigned long long round_u64(float v) {
  const float hf = truncf(v * 0x1p-32f);
  const float r = fmaf(-hf, 0x1p32f, v);
  return (static_cast<unsigned long long>(static_cast<uint32_t>(hf)) << 32) | __float2uint_rn(r);
}

// Exact conversion of a fixed-point integer (< 2^63) to a pair, and back.
__device__ __forceinline__ F2 f2_from_u64(unsigned long long v) {
  const float hi = __ull2float_rz(v);
  const unsigned long long h = static_cast<unsigned long long>(hi);
  F2 r;
  r.hi = hi;
  r.lo = __ull2float_rn(v - h);  // v >= h by round-toward-zero
  return r;
}

__device__ __forceinline__ unsigned long long f2_to_u64(F2 a) {
  if (!(a.hi > 0.f)) return 0ull;
  const unsigned long long h = __float2ull_rz(a.hi);
  const long long l = __float2ll_rn(a.lo + (a.hi - static_cast<float>(h)));
  return l < 0 ? h - static_cast<unsigned long long>(-l) : h + static_cast<unsigned long long>(l);
}

// ---------------------------------------------------------------------------
// Shared-memory addressing, mbarriers and TMA bulk copies.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

// One 1-D bulk copy global -> this CTA's shared memory, completing on bar.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Orders this thread's generic-proxy accesses to shared memory before later
// async-proxy (bulk copy) accesses.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t phase) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(phase)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait for phase `phase` of bar: gives up after `limit_ns` of wall
// time (checked every 64 polls) and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t phase, uint64_t limit_ns) {
  if (mbar_try_wait(bar, phase)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, phase)) return true;
    if ((it & 63u) == 0u && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------------------
// Thread-block clusters and distributed shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Full cluster barrier: every thread of every CTA of the cluster arrives
// (release) and waits (acquire). The non-.aligned forms are used so that a
// warp need not be converged when it reaches the barrier.
// The two halves of a cluster barrier, for work between them that touches
// no other CTA's memory.
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}

// Shared-memory add of 1, predicated in the instruction itself (no branch).
__device__ __forceinline__ void red_inc_shared_if(uint32_t* p, bool cond) {
  asm volatile(
      "{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t@q red.shared.add.u32 [%0], 1;\n\t}" ::"r"(
          static_cast<uint32_t>(__cvta_generic_to_shared(p))),
      "r"(cond ? 1u : 0u)
      : "memory");
}

// The same two on a 32-bit shared-window address (a base from smem_u32 plus
// a byte offset), so hot loops form no 64-bit generic address per update.
__device__ __forceinline__ void red_inc_shared_at_if(uint32_t saddr, bool cond) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.u32 q, %1, 0;\n\t@q red.shared.add.u32 [%0], 1;\n\t}" ::"r"(saddr),
               "r"(cond ? 1u : 0u)
               : "memory");
}

__device__ __forceinline__ void red_add_shared_at(uint32_t saddr, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(saddr), "r"(v) : "memory");
}

// Shared-memory add without a returned value.
__device__ __forceinline__ void red_add_shared_u32(uint32_t* p, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(p))), "r"(v)
               : "memory");
}

// Arrive without release ordering: for a CTA whose earlier accesses to other
// CTAs' memory were loads whose values it has used already.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}

__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release;\n\t"
      "barrier.cluster.wait.acquire;" ::
          : "memory");
}

__device__ __forceinline__ uint32_t map_rank(uint32_t local_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ uint32_t ld_dsmem_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void st_dsmem_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void st_dsmem_u8(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u8 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ float ld_dsmem_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ double ld_dsmem_f64(uint32_t addr) {
  double v;
  asm volatile("ld.shared::cluster.f64 %0, [%1];" : "=d"(v) : "r"(addr) : "memory");
  return v;
}

}  // namespace dev
}  // namespace qrita
