// Outputs beyond the keep-mask: the top-k ids in stable order, and the kept
// ids with renormalised probabilities plus one token drawn from them.
//
// Qrita technical summary (gist.science, paper 2602.01518), "Problem
// statement": the full candidate set is what speculative-decoding
// verification and reinforcement learning consume. Both kernels read a row's
// keep-mask (from the selection kernel) and its logits; one CTA per row.

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "qrita_device.cuh"
#include "qrita_internal.h"

namespace qrita {
namespace {

using namespace dev;

constexpr int kOutThreads = 256;
constexpr int kOutWarps = kOutThreads / 32;
constexpr uint32_t kFullMask = 0xffffffffu;

template <int DT>
__device__ __forceinline__ float logit_at(const void* logits, int64_t off) {
  if constexpr (DT == QRITA_DTYPE_F32) {
    return __ldg(static_cast<const float*>(logits) + off);
  } else {
    const uint32_t b = __ldg(static_cast<const unsigned short*>(logits) + off);
    return __uint_as_float(b << 16);
  }
}

// Exclusive scan of one 32-bit count per thread, in thread order.
__device__ __forceinline__ uint32_t out_excl_scan(uint32_t v, uint32_t* warp_tot, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  uint32_t base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kOutWarps; ++w) {
    const uint32_t s = *reinterpret_cast<volatile uint32_t*>(&warp_tot[w]);
    base += w < warp ? s : 0u;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return base + incl - v;
}

__device__ __forceinline__ unsigned long long out_excl_scan_u64(unsigned long long v, unsigned long long* warp_tot,
                                                                unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  unsigned long long base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kOutWarps; ++w) {
    const unsigned long long s = *reinterpret_cast<volatile unsigned long long*>(&warp_tot[w]);
    base += w < warp ? s : 0ull;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return base + incl - v;
}

// Thread t's contiguous segment of a row of V bytes: [lo, hi).
__device__ __forceinline__ void segment(int64_t V, int64_t& lo, int64_t& hi) {
  const int64_t per = (V + kOutThreads - 1) / kOutThreads;
  lo = min(V, static_cast<int64_t>(threadIdx.x) * per);
  hi = min(V, lo + per);
}

// ---------------------------------------------------------------------------
// Top-k ids in stable order: the kept ids of the row's top-k mask, sorted by
// (logit descending, id ascending) with a bitonic sort of 64-bit keys in
// shared memory: high word the complement of the logit's order key (so
// ascending keys run from the largest logit down), low word the id.
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kOutThreads) ids_kernel(const void* logits, int64_t V, const int32_t* k, int32_t kmax,
                                                          const uint8_t* mask, int32_t* out_ids) {
  extern __shared__ __align__(16) unsigned long long keys[];  // [pow2 >= kmax]
  __shared__ uint32_t warp_tot[kOutWarps];
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x;
  const int32_t kr = k[r];
  int32_t* orow = out_ids + r * static_cast<int64_t>(kmax);
  const uint8_t* mrow = mask + r * V;
  const bool ok = kr >= 1 && kr <= kmax;
  int64_t lo, hi;
  segment(V, lo, hi);
  uint32_t cnt = 0;
  if (ok)
    for (int64_t i = lo; i < hi; ++i) cnt += mrow[i] != 0 ? 1u : 0u;
  uint32_t total = 0;
  uint32_t pos = out_excl_scan(cnt, warp_tot, &total);
  const uint32_t n = ok ? min(total, static_cast<uint32_t>(kmax)) : 0u;
  uint32_t np2 = 1;
  while (np2 < n) np2 <<= 1;
  if (ok) {
    const void* lrow = static_cast<const unsigned char*>(logits) + r * V * (DT == QRITA_DTYPE_F32 ? 4 : 2);
    for (int64_t i = lo; i < hi && pos < n; ++i) {
      if (mrow[i] != 0) {
        const uint32_t key = f2key(logit_at<DT>(lrow, i));
        keys[pos++] = (static_cast<unsigned long long>(~key) << 32) | static_cast<uint32_t>(i);
      }
    }
  }
  for (uint32_t i = n + tid; i < np2; i += kOutThreads) keys[i] = ~0ull;  // padding sorts last
  __syncthreads();
  // bitonic sort, ascending
  for (uint32_t size = 2; size <= np2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t t = tid; t < np2 / 2; t += kOutThreads) {
        const uint32_t a = 2 * stride * (t / stride) + (t % stride);
        const uint32_t b = a + stride;
        const bool up = (a & size) == 0;
        const unsigned long long ka = keys[a], kb = keys[b];
        if ((ka > kb) == up) {
          keys[a] = kb;
          keys[b] = ka;
        }
      }
      __syncthreads();
    }
  }
  for (int32_t i = tid; i < kmax; i += kOutThreads)
    orow[i] = static_cast<uint32_t>(i) < n ? static_cast<int32_t>(keys[i] & 0xFFFFFFFFull) : -1;
}

// ---------------------------------------------------------------------------
// Candidate lists and one draw: the kept ids in id order, their
// probabilities renormalised over the kept set, and the first kept id whose
// cumulative probability exceeds the row's uniform. Weights are the
// selection kernel's: 2^((x - m) log2 e) by the hardware base-2 exponential,
// in 64-bit fixed point for the cumulative sums (exact and order-free).
// ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kOutThreads) cand_kernel(const void* logits, int64_t V, const uint8_t* mask,
                                                           int32_t cap, int32_t* out_ids, float* out_probs,
                                                           int32_t* out_count, const float* u, int32_t* out_sample) {
  __shared__ uint32_t warp_tot[kOutWarps];
  __shared__ unsigned long long warp_tot64[kOutWarps];
  __shared__ float warp_max[kOutWarps];
  __shared__ int32_t sample_at;
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint8_t* mrow = mask + r * V;
  const void* lrow = static_cast<const unsigned char*>(logits) + r * V * (DT == QRITA_DTYPE_F32 ? 4 : 2);
  int64_t lo, hi;
  segment(V, lo, hi);
  // pass 1: count and largest kept logit
  uint32_t cnt = 0;
  float m = -INFINITY;
  for (int64_t i = lo; i < hi; ++i) {
    if (mrow[i] != 0) {
      ++cnt;
      m = fmaxf(m, logit_at<DT>(lrow, i));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
  if (lane == 0) warp_max[warp] = m;
  uint32_t total = 0;
  const uint32_t pos0 = out_excl_scan(cnt, warp_tot, &total);  // (its barriers publish warp_max)
  float rm = -INFINITY;
  for (int w = 0; w < kOutWarps; ++w) rm = fmaxf(rm, *reinterpret_cast<volatile float*>(&warp_max[w]));
  if (tid == 0) {
    out_count[r] = static_cast<int32_t>(total);
    sample_at = -1;
  }
  const bool m_neginf = rm == -INFINITY;  // every kept logit is -inf: equal weights
  const float scale = exp2f(static_cast<float>(62 - (32 - __clz(static_cast<uint32_t>(V)))));
  auto wfx = [&](float x) -> unsigned long long {
    float w = 1.0f;
    if (!m_neginf) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(w) : "f"((x - rm) * 1.4426950408889634f));
    return round_u64(w * scale);
  };
  // pass 2: fixed-point mass of this segment and of the row
  unsigned long long mass = 0ull;
  for (int64_t i = lo; i < hi; ++i)
    if (mrow[i] != 0) mass += wfx(logit_at<DT>(lrow, i));
  unsigned long long z = 0ull;
  const unsigned long long before = out_excl_scan_u64(mass, warp_tot64, &z);
  // the draw: cumulative mass of the first ids exceeds u Z
  unsigned long long target = ~0ull;
  const bool draw = u != nullptr && out_sample != nullptr && total > 0u;
  if (draw) {
    const float uf = u[r];
    const F2 t = f2_mul(f2_from_u64(z), uf);
    target = uf > 0.f ? f2_to_u64(t) : 0ull;
  }
  const float zf = static_cast<float>(z);
  // pass 3: ids and probabilities in id order; the thread whose segment
  // crosses the target draws
  uint32_t pos = pos0;
  unsigned long long acc = before;
  for (int64_t i = lo; i < hi; ++i) {
    if (mrow[i] == 0) continue;
    const unsigned long long w = wfx(logit_at<DT>(lrow, i));
    if (pos < static_cast<uint32_t>(cap)) {
      out_ids[r * cap + pos] = static_cast<int32_t>(i);
      out_probs[r * cap + pos] = static_cast<float>(w) / zf;
    }
    if (draw && acc <= target && target < acc + w) sample_at = static_cast<int32_t>(i);
    acc += w;
    ++pos;
  }
  __syncthreads();
  if (draw && tid == 0) {
    // rounding can leave the target at or past the last cumulative sum: the
    // last kept id then (the oracle does the same), found by last_kept_kernel
    out_sample[r] = *reinterpret_cast<volatile int32_t*>(&sample_at);
  }
  if (!draw && out_sample != nullptr && tid == 0) out_sample[r] = -1;
}

// ---------------------------------------------------------------------------
// Vector forms of both kernels, for rows whose mask and logits start on a
// 16-byte boundary (V a multiple of 16 and aligned base pointers): the row is
// read in units of 16 elements (16 mask bytes, 64 or 32 logit bytes), warp w
// owning a contiguous run of units and its lanes taking 32 consecutive units
// a step, so every load is coalesced. Kept ids keep their order: a warp's
// positions come from a warp scan per step and the warps' totals from one
// block scan.
// ---------------------------------------------------------------------------
constexpr int kUnit = 16;  // elements per unit

// Kept bits of one unit of 16 mask bytes: bit e for byte e nonzero. A byte
// is nonzero exactly when its low seven bits plus 0x7F carry into bit 7 or
// its own bit 7 is set; the four bit-7 flags of a word are then gathered by
// one multiply (bytes 0..3 to bits 0..3).
__device__ __forceinline__ uint32_t unit_kept_bits(const uint4 m) {
  if ((m.x | m.y | m.z | m.w) == 0u) return 0u;  // (most units of a sparse mask)
  const uint32_t w[4] = {m.x, m.y, m.z, m.w};
  uint32_t bits = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t nz = ((((w[i] & 0x7F7F7F7Fu) + 0x7F7F7F7Fu) | w[i]) >> 7) & 0x01010101u;
    bits |= ((nz * 0x01020408u) >> 24) << (4 * i);
  }
  return bits;
}

// The 16 logits of unit u of the row, widened to fp32.
template <int DT>
__device__ __forceinline__ void unit_logits(const void* lrow, int64_t u, float (&x)[kUnit]) {
  if constexpr (DT == QRITA_DTYPE_F32) {
    const uint4* p = static_cast<const uint4*>(lrow) + u * 4;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint4 v = __ldg(p + q);
      x[4 * q] = __uint_as_float(v.x);
      x[4 * q + 1] = __uint_as_float(v.y);
      x[4 * q + 2] = __uint_as_float(v.z);
      x[4 * q + 3] = __uint_as_float(v.w);
    }
  } else {
    const uint4* p = static_cast<const uint4*>(lrow) + u * 2;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 v = __ldg(p + q);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
        x[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }
}

// Warp w's run of units [u_lo, u_hi) of a row of nu units.
__device__ __forceinline__ void warp_units(int64_t nu, int64_t& u_lo, int64_t& u_hi) {
  const int64_t per = (nu + kOutWarps - 1) / kOutWarps;
  u_lo = min(nu, static_cast<int64_t>(threadIdx.x >> 5) * per);
  u_hi = min(nu, u_lo + per);
}

// Exclusive warp scans (lane order) of a 32-bit and a 64-bit value; the
// inclusive total comes back in *tot.
__device__ __forceinline__ uint32_t warp_excl_u32(uint32_t v, uint32_t* tot) {
  const int lane = threadIdx.x & 31;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  *tot = __shfl_sync(kFullMask, incl, 31);
  return incl - v;
}

__device__ __forceinline__ unsigned long long warp_excl_u64(unsigned long long v, unsigned long long* tot) {
  const int lane = threadIdx.x & 31;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  *tot = __shfl_sync(kFullMask, incl, 31);
  return incl - v;
}

// Exclusive scan over the warps of one value per warp (lane 0's), and the
// block total; every thread gets its warp's base.
template <typename T>
__device__ __forceinline__ T warps_excl(T v, T* slots, T* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) slots[warp] = v;
  __syncthreads();
  T base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kOutWarps; ++w) {
    const T s = *reinterpret_cast<volatile T*>(&slots[w]);
    base += w < warp ? s : T(0);
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return base;
}

// Steps of pass 2 whose masses a warp of the candidate kernel records.
constexpr int kCandSteps = 32;

// Units a lane takes per step, and the 16-byte words of one unit's logits:
// every load of a step (its masks, then the logits of its units that keep
// anything, predicated) is issued before any result is used.
template <int DT>
struct StepShape {
  static constexpr int kWords = DT == QRITA_DTYPE_F32 ? 4 : 2;
  static constexpr int kUnits = DT == QRITA_DTYPE_F32 ? 2 : 4;
};

// Units u_first + j * stride (j < kUnits, below u_hi): kept bits and raw logits.
template <int DT>
__device__ __forceinline__ void load_step(const uint4* mrow, const void* lrow, int64_t u_first, int64_t stride,
                                          int64_t u_hi, uint32_t (&bits)[StepShape<DT>::kUnits],
                                          uint4 (&raw)[StepShape<DT>::kUnits][StepShape<DT>::kWords]) {
  constexpr int NU = StepShape<DT>::kUnits, NW = StepShape<DT>::kWords;
  uint4 mv[NU];
#pragma unroll
  for (int j = 0; j < NU; ++j) {
    const int64_t uu = u_first + j * stride;
    mv[j] = uu < u_hi ? __ldg(mrow + uu) : make_uint4(0u, 0u, 0u, 0u);
  }
#pragma unroll
  for (int j = 0; j < NU; ++j) bits[j] = unit_kept_bits(mv[j]);
  const uint4* lp = static_cast<const uint4*>(lrow);
#pragma unroll
  for (int j = 0; j < NU; ++j) {
    const int64_t uu = u_first + j * stride;
#pragma unroll
    for (int q = 0; q < NW; ++q) raw[j][q] = bits[j] != 0u ? __ldg(lp + uu * NW + q) : make_uint4(0u, 0u, 0u, 0u);
  }
}

template <int DT>
__device__ __forceinline__ void widen_unit(const uint4 (&raw)[StepShape<DT>::kWords], float (&x)[kUnit]) {
  if constexpr (DT == QRITA_DTYPE_F32) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      x[4 * q] = __uint_as_float(raw[q].x);
      x[4 * q + 1] = __uint_as_float(raw[q].y);
      x[4 * q + 2] = __uint_as_float(raw[q].z);
      x[4 * q + 3] = __uint_as_float(raw[q].w);
    }
  } else {
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t w[4] = {raw[q].x, raw[q].y, raw[q].z, raw[q].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * q + 2 * i] = __uint_as_float(w[i] << 16);
        x[8 * q + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
      }
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(kOutThreads) ids_kernel_vec(const void* logits, int64_t V, const int32_t* k,
                                                              int32_t kmax, const uint8_t* mask, int32_t* out_ids) {
  constexpr int NU = StepShape<DT>::kUnits, NW = StepShape<DT>::kWords;
  extern __shared__ __align__(16) unsigned long long keys[];  // [pow2 >= kmax]
  __shared__ uint32_t fill;
  const int64_t r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int32_t kr = k[r];
  int32_t* orow = out_ids + r * static_cast<int64_t>(kmax);
  const bool ok = kr >= 1 && kr <= kmax;
  const int64_t nu = V / kUnit;
  const uint4* mrow = reinterpret_cast<const uint4*>(mask + r * V);
  const void* lrow = static_cast<const unsigned char*>(logits) + r * V * (DT == QRITA_DTYPE_F32 ? 4 : 2);
  int64_t u_lo, u_hi;
  warp_units(nu, u_lo, u_hi);
  if (tid == 0) fill = 0u;
  __syncthreads();
  // one pass: every kept id with its order key, in any order (the sort
  // orders them), a lane claiming its slots with one shared atomic; the mask
  // is the row's top-k mask, so it keeps min(k, V) <= kmax ids
  if (ok) {
    for (int64_t ub = u_lo; ub < u_hi; ub += 32 * NU) {
      uint32_t bits[NU];
      uint4 raw[NU][NW];
      load_step<DT>(mrow, lrow, ub + lane, 32, u_hi, bits, raw);
      uint32_t c = 0;
#pragma unroll
      for (int j = 0; j < NU; ++j) c += __popc(bits[j]);
      if (c == 0u) continue;
      uint32_t slot = atomicAdd(&fill, c);
#pragma unroll
      for (int j = 0; j < NU; ++j) {
        if (bits[j] != 0u) {
          const int64_t uu = ub + lane + 32 * j;
          float x[kUnit];
          widen_unit<DT>(raw[j], x);
#pragma unroll
          for (int e = 0; e < kUnit; ++e) {
            if ((bits[j] >> e) & 1u) {
              if (slot < static_cast<uint32_t>(kmax)) {
                const uint32_t key = f2key(x[e]);
                keys[slot] = (static_cast<unsigned long long>(~key) << 32) | static_cast<uint32_t>(uu * kUnit + e);
              }
              ++slot;
            }
          }
        }
      }
    }
  }
  __syncthreads();
  const uint32_t n = ok ? min(*reinterpret_cast<volatile uint32_t*>(&fill), static_cast<uint32_t>(kmax)) : 0u;
  uint32_t np2 = 1;
  while (np2 < n) np2 <<= 1;
  for (uint32_t i = n + tid; i < np2; i += kOutThreads) keys[i] = ~0ull;  // padding sorts last
  __syncthreads();
  // bitonic sort, ascending
  for (uint32_t size = 2; size <= np2; size <<= 1) {
    for (uint32_t stride = size >> 1; stride > 0; stride >>= 1) {
      for (uint32_t t = tid; t < np2 / 2; t += kOutThreads) {
        const uint32_t a = 2 * stride * (t / stride) + (t % stride);
        const uint32_t b = a + stride;
        const bool up = (a & size) == 0;
        const unsigned long long ka = keys[a], kb = keys[b];
        if ((ka > kb) == up) {
          keys[a] = kb;
          keys[b] = ka;
        }
      }
      __syncthreads();
    }
  }
  for (int32_t i = tid; i < kmax; i += kOutThreads)
    orow[i] = static_cast<uint32_t>(i) < n ? static_cast<int32_t>(keys[i] & 0xFFFFFFFFull) : -1;
}

// Candidate lists, vector form: a row is split over a cluster of C CTAs
// (contiguous runs of units, rank order = id order), merged through
// distributed shared memory, in two passes over the row: (1) the kept count
// and the largest kept logit; (2) in id order, the ids and their fixed-point
// weights (written as floats up to cap), and each CTA's mass. Then the one
// warp whose mass range holds the draw's target walks its run again to find
// the token, and the written weights are divided by the total.
struct alignas(16) CandPub {  // what one CTA publishes to its cluster
  unsigned long long mass;
  uint32_t cnt;
  float mx;
};

template <int DT>
__global__ void __launch_bounds__(kOutThreads, 3) cand_kernel_vec(const void* logits, int64_t V, const uint8_t* mask,
                                                                  int32_t cap, int32_t* out_ids, float* out_probs,
                                                                  int32_t* out_count, const float* u,
                                                                  int32_t* out_sample) {
  constexpr int NU = StepShape<DT>::kUnits, NW = StepShape<DT>::kWords;
  __shared__ uint32_t warp_slots[kOutWarps];
  __shared__ unsigned long long warp_slots64[kOutWarps];
  __shared__ float warp_max[kOutWarps];
  __shared__ CandPub pub;
  // each warp's mass per step of pass 2 (its first kCandSteps steps), so the
  // draw recomputes one step instead of walking the warp's whole run
  __shared__ unsigned long long step_mass[kOutWarps][kCandSteps];
  uint32_t C;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(C));
  const uint32_t cr = cluster_rank();
  const int64_t r = blockIdx.x / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t nu = V / kUnit;
  const uint4* mrow = reinterpret_cast<const uint4*>(mask + r * V);
  const void* lrow = static_cast<const unsigned char*>(logits) + r * V * (DT == QRITA_DTYPE_F32 ? 4 : 2);
  // this CTA's run of units, then its warp's
  const int64_t per_cta = (nu + C - 1) / C;
  const int64_t c_lo = min(nu, static_cast<int64_t>(cr) * per_cta), c_hi = min(nu, c_lo + per_cta);
  const int64_t per_w = (c_hi - c_lo + kOutWarps - 1) / kOutWarps;
  const int64_t u_lo = min(c_hi, c_lo + warp * per_w), u_hi = min(c_hi, u_lo + per_w);
  // pass 1: kept count and largest kept logit (units ub + lane + 32 j)
  uint32_t cnt = 0;
  float m = -INFINITY;
  for (int64_t ub = u_lo; ub < u_hi; ub += 32 * NU) {
    uint32_t bits[NU];
    uint4 raw[NU][NW];
    load_step<DT>(mrow, lrow, ub + lane, 32, u_hi, bits, raw);
#pragma unroll
    for (int j = 0; j < NU; ++j) {
      if (bits[j] == 0u) continue;
      cnt += __popc(bits[j]);
      float x[kUnit];
      widen_unit<DT>(raw[j], x);
#pragma unroll
      for (int e = 0; e < kUnit; ++e) m = ((bits[j] >> e) & 1u) ? fmaxf(m, x[e]) : m;
    }
  }
  cnt = __reduce_add_sync(kFullMask, cnt);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(kFullMask, m, o));
  if (lane == 0) warp_max[warp] = m;
  uint32_t cta_cnt = 0;
  const uint32_t wbase = warps_excl<uint32_t>(cnt, warp_slots, &cta_cnt);  // (its barriers publish warp_max)
  if (tid == 0) {
    float cm = -INFINITY;
    for (int w = 0; w < kOutWarps; ++w) cm = fmaxf(cm, *reinterpret_cast<volatile float*>(&warp_max[w]));
    pub.cnt = cta_cnt;
    pub.mx = cm;
    if (cr == 0u && out_sample != nullptr) out_sample[r] = -1;  // a draw below overwrites it
  }
  cluster_sync_all();  // every CTA's count and max are published
  uint32_t total = 0, cbase = 0;
  float rm = -INFINITY;
  for (uint32_t q = 0; q < C; ++q) {
    const uint32_t a = map_rank(smem_u32(&pub), q);
    const uint32_t n = ld_dsmem_u32(a + offsetof(CandPub, cnt));
    total += n;
    cbase += q < cr ? n : 0u;
    rm = fmaxf(rm, ld_dsmem_f32(a + offsetof(CandPub, mx)));
  }
  if (cr == 0u && tid == 0) out_count[r] = static_cast<int32_t>(total);
  const bool m_neginf = rm == -INFINITY;  // every kept logit is -inf: equal weights
  const float scale = exp2f(static_cast<float>(62 - (32 - __clz(static_cast<uint32_t>(V)))));
  auto wfx = [&](float x) -> unsigned long long {
    float w = 1.0f;
    if (!m_neginf) asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(w) : "f"((x - rm) * 1.4426950408889634f));
    return round_u64(w * scale);
  };
  // pass 2: ids and weights in id order (units ub + NU lane + j), this
  // warp's mass, and its mass per step
  unsigned long long wmass = 0ull;
  {
    uint32_t run = cbase + wbase;
    int step = 0;
    for (int64_t ub = u_lo; ub < u_hi; ub += 32 * NU, ++step) {
      const unsigned long long before = wmass;
      uint32_t bits[NU];
      uint4 raw[NU][NW];
      load_step<DT>(mrow, lrow, ub + NU * lane, 1, u_hi, bits, raw);
      uint32_t c = 0;
#pragma unroll
      for (int j = 0; j < NU; ++j) c += __popc(bits[j]);
      uint32_t step_n = 0;
      uint32_t pos = run + warp_excl_u32(c, &step_n);
#pragma unroll
      for (int j = 0; j < NU; ++j) {
        if (bits[j] != 0u) {
          const int64_t uu = ub + NU * lane + j;
          float x[kUnit];
          widen_unit<DT>(raw[j], x);
#pragma unroll
          for (int e = 0; e < kUnit; ++e) {
            if ((bits[j] >> e) & 1u) {
              const unsigned long long w = wfx(x[e]);
              wmass += w;
              if (pos < static_cast<uint32_t>(cap)) {
                out_ids[r * cap + pos] = static_cast<int32_t>(uu * kUnit + e);
                out_probs[r * cap + pos] = static_cast<float>(w);
              }
              ++pos;
            }
          }
        }
      }
      run += step_n;
      if (step < kCandSteps) {
        unsigned long long sm = wmass - before;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sm += __shfl_xor_sync(kFullMask, sm, o);
        if (lane == 0) step_mass[warp][step] = sm;
      }
    }
  }
  const int64_t n_steps = (u_hi - u_lo + 32 * NU - 1) / (32 * NU);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wmass += __shfl_xor_sync(kFullMask, wmass, o);
  unsigned long long cta_mass = 0ull;
  const unsigned long long wmbase = warps_excl<unsigned long long>(wmass, warp_slots64, &cta_mass);
  if (tid == 0) pub.mass = cta_mass;
  cluster_sync_all();  // every CTA's mass is published (and its writes done)
  unsigned long long z = 0ull, mcbase = 0ull;
  for (uint32_t q = 0; q < C; ++q) {
    const uint32_t a = map_rank(smem_u32(&pub), q) + offsetof(CandPub, mass);
    const unsigned long long v = static_cast<unsigned long long>(ld_dsmem_u32(a)) |
                                 (static_cast<unsigned long long>(ld_dsmem_u32(a + 4u)) << 32);
    z += v;
    mcbase += q < cr ? v : 0ull;
  }
  const unsigned long long mbase = mcbase + wmbase;
  const bool draw = u != nullptr && out_sample != nullptr && total > 0u;
  if (draw) {
    const float uf = u[r];
    const F2 t = f2_mul(f2_from_u64(z), uf);
    const unsigned long long target = uf > 0.f ? f2_to_u64(t) : 0ull;
    // the warp whose mass range holds the target finds the step that holds
    // it from its step masses and recomputes that step alone (a run of more
    // than kCandSteps steps walks on from the last recorded one)
    if (mbase <= target && target < mbase + wmass) {
      unsigned long long acc = mbase;
      int64_t ub0 = u_lo;
      const int rec = n_steps < kCandSteps ? static_cast<int>(n_steps) : kCandSteps;
      for (int q = 0; q < rec; ++q) {
        const unsigned long long sm = *reinterpret_cast<volatile unsigned long long*>(&step_mass[warp][q]);
        if (target < acc + sm || q == rec - 1) break;  // (warp-uniform)
        acc += sm;
        ub0 += 32 * NU;
      }
      for (int64_t ub = ub0; ub < u_hi; ub += 32 * NU) {
        uint32_t bits[NU];
        uint4 raw[NU][NW];
        load_step<DT>(mrow, lrow, ub + NU * lane, 1, u_hi, bits, raw);
        unsigned long long lm = 0ull;
#pragma unroll
        for (int j = 0; j < NU; ++j) {
          float x[kUnit];
          widen_unit<DT>(raw[j], x);
#pragma unroll
          for (int e = 0; e < kUnit; ++e)
            if ((bits[j] >> e) & 1u) lm += wfx(x[e]);
        }
        unsigned long long step_m = 0ull;
        unsigned long long a = acc + warp_excl_u64(lm, &step_m);
        if (a <= target && target < a + lm) {
          // this lane holds the token: walk its kept ids again (reloaded:
          // one lane of the row does this)
          for (int j = 0; j < NU; ++j) {
            const int64_t uu = ub + NU * lane + j;
            if (uu >= u_hi) break;
            const uint32_t bj = unit_kept_bits(__ldg(mrow + uu));
            if (bj == 0u) continue;
            float x[kUnit];
            unit_logits<DT>(lrow, uu, x);
#pragma unroll
            for (int e = 0; e < kUnit; ++e) {
              if ((bj >> e) & 1u) {
                const unsigned long long w = wfx(x[e]);
                if (a <= target && target < a + w) out_sample[r] = static_cast<int32_t>(uu * kUnit + e);
                a += w;
              }
            }
          }
        }
        acc += step_m;
        if (acc > target) break;  // (warp-uniform)
      }
    }
  }
  // this CTA's written weights to probabilities
  const float zf = static_cast<float>(z);
  const uint32_t w_lo = min(cbase, static_cast<uint32_t>(cap));
  const uint32_t w_hi = min(cbase + cta_cnt, static_cast<uint32_t>(cap));
  for (uint32_t i = w_lo + tid; i < w_hi; i += kOutThreads) out_probs[r * cap + i] = out_probs[r * cap + i] / zf;
  cluster_sync_all();  // no CTA leaves while another may read its published values
}

// The last kept id of the row (for a target past every cumulative sum).
__global__ void __launch_bounds__(kOutThreads) last_kept_kernel(int64_t V, const uint8_t* mask, int32_t* out_sample) {
  const int64_t r = blockIdx.x;
  if (out_sample[r] >= 0) return;
  const uint8_t* mrow = mask + r * V;
  int64_t best = -1;
  for (int64_t i = threadIdx.x; i < V; i += kOutThreads)
    if (mrow[i] != 0) best = i > best ? i : best;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const long long y = __shfl_xor_sync(kFullMask, static_cast<long long>(best), o);
    best = y > best ? y : best;
  }
  __shared__ long long wb[kOutWarps];
  if ((threadIdx.x & 31) == 0) wb[threadIdx.x >> 5] = best;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long b = -1;
    for (int w = 0; w < kOutWarps; ++w) b = wb[w] > b ? wb[w] : b;
    out_sample[r] = static_cast<int32_t>(b);
  }
}

}  // namespace

size_t ids_smem_bytes(int32_t kmax) {
  size_t np2 = 1;
  while (np2 < static_cast<size_t>(kmax)) np2 <<= 1;
  return np2 * sizeof(unsigned long long);
}

// The vector kernels' condition: every row of the mask and of the logits
// starts on a 16-byte boundary.
static bool vec_rows(const void* logits, const uint8_t* mask, int64_t V) {
  return V % kUnit == 0 && reinterpret_cast<uintptr_t>(logits) % 16u == 0u &&
         reinterpret_cast<uintptr_t>(mask) % 16u == 0u;
}

template <int DT>
static cudaError_t launch_ids_t(const void* logits, int64_t B, int64_t V, const int32_t* k, int32_t kmax, const uint8_t* mask,
                         int32_t* out_ids, size_t smem, cudaStream_t st) {
  const bool vec = vec_rows(logits, mask, V);
  const void* fn = vec ? reinterpret_cast<const void*>(&ids_kernel_vec<DT>) : reinterpret_cast<const void*>(&ids_kernel<DT>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (vec) ids_kernel_vec<DT><<<static_cast<unsigned>(B), kOutThreads, smem, st>>>(logits, V, k, kmax, mask, out_ids);
  else ids_kernel<DT><<<static_cast<unsigned>(B), kOutThreads, smem, st>>>(logits, V, k, kmax, mask, out_ids);
  return cudaGetLastError();
}

int launch_ids(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k, int32_t kmax,
               const uint8_t* mask, int32_t* out_ids, qrita_stream_t stream) {
  const size_t smem = ids_smem_bytes(kmax);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e = dtype == QRITA_DTYPE_F32
                            ? launch_ids_t<QRITA_DTYPE_F32>(logits, B, V, k, kmax, mask, out_ids, smem, st)
                            : launch_ids_t<QRITA_DTYPE_BF16>(logits, B, V, k, kmax, mask, out_ids, smem, st);
  return static_cast<int>(e);
}

int launch_candidates(const void* logits, int dtype, int64_t B, int64_t V, const uint8_t* mask, int32_t cap,
                      int32_t* out_ids, float* out_probs, int32_t* out_count, const float* u, int32_t* out_sample,
                      qrita_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool vec = vec_rows(logits, mask, V);
  const unsigned g = static_cast<unsigned>(B);
  cudaError_t e = cudaSuccess;
  if (vec) {
    // rows of at least 8192 units per CTA split over a cluster (a dense row
    // is the longest work of the launch), up to 4 CTAs
    const int64_t nu = V / kUnit;
    unsigned C = 1;
    while (C < 4 && nu / (2 * C) >= 512) C *= 2;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g * C, 1, 1);
    cfg.blockDim = dim3(kOutThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == QRITA_DTYPE_F32)
      e = cudaLaunchKernelEx(&cfg, cand_kernel_vec<QRITA_DTYPE_F32>, logits, V, mask, cap, out_ids, out_probs, out_count,
                             u, out_sample);
    else
      e = cudaLaunchKernelEx(&cfg, cand_kernel_vec<QRITA_DTYPE_BF16>, logits, V, mask, cap, out_ids, out_probs,
                             out_count, u, out_sample);
  } else if (dtype == QRITA_DTYPE_F32) {
    cand_kernel<QRITA_DTYPE_F32><<<g, kOutThreads, 0, st>>>(logits, V, mask, cap, out_ids, out_probs, out_count, u,
                                                            out_sample);
  } else {
    cand_kernel<QRITA_DTYPE_BF16><<<g, kOutThreads, 0, st>>>(logits, V, mask, cap, out_ids, out_probs, out_count, u,
                                                             out_sample);
  }
  if (e != cudaSuccess) return static_cast<int>(e);
  e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  if (u != nullptr && out_sample != nullptr) {
    last_kept_kernel<<<g, kOutThreads, 0, st>>>(V, mask, out_sample);
    e = cudaGetLastError();
  }
  return static_cast<int>(e);
}

}  // namespace qrita
