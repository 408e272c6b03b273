// Outputs beyond the keep-mask: the top-k ids in stable order, and the kept
// ids with renormalised probabilities plus one token drawn from them.
//
// Qrita technical summary (gist.science, paper 2602.01518), "Problem
// statement": the full candidate set is what speculative-decoding
// verification and reinforcement learning consume. Both kernels read a row's
// keep-mask (from the selection kernel) and its logits; one CTA per row.

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

int launch_ids(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k, int32_t kmax,
               const uint8_t* mask, int32_t* out_ids, qrita_stream_t stream) {
  const size_t smem = ids_smem_bytes(kmax);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == QRITA_DTYPE_F32) {
    e = cudaFuncSetAttribute(ids_kernel<QRITA_DTYPE_F32>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return static_cast<int>(e);
    ids_kernel<QRITA_DTYPE_F32><<<static_cast<unsigned>(B), kOutThreads, smem, st>>>(logits, V, k, kmax, mask, out_ids);
  } else {
    e = cudaFuncSetAttribute(ids_kernel<QRITA_DTYPE_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return static_cast<int>(e);
    ids_kernel<QRITA_DTYPE_BF16><<<static_cast<unsigned>(B), kOutThreads, smem, st>>>(logits, V, k, kmax, mask, out_ids);
  }
  return static_cast<int>(cudaGetLastError());
}

int launch_candidates(const void* logits, int dtype, int64_t B, int64_t V, const uint8_t* mask, int32_t cap,
                      int32_t* out_ids, float* out_probs, int32_t* out_count, const float* u, int32_t* out_sample,
                      qrita_stream_t stream) {
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == QRITA_DTYPE_F32) {
    cand_kernel<QRITA_DTYPE_F32><<<static_cast<unsigned>(B), kOutThreads, 0, st>>>(logits, V, mask, cap, out_ids,
                                                                                   out_probs, out_count, u, out_sample);
  } else {
    cand_kernel<QRITA_DTYPE_BF16><<<static_cast<unsigned>(B), kOutThreads, 0, st>>>(logits, V, mask, cap, out_ids,
                                                                                    out_probs, out_count, u, out_sample);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  if (u != nullptr && out_sample != nullptr) {
    last_kept_kernel<<<static_cast<unsigned>(B), kOutThreads, 0, st>>>(V, mask, out_sample);
    e = cudaGetLastError();
  }
  return static_cast<int>(e);
}

}  // namespace qrita
