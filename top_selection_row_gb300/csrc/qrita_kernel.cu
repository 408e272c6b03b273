// Fused exact top-k / top-p selection kernel for GB300 (sm_103a).
//
// Method: Qrita technical summary (gist.science, paper 2602.01518),
// "Methodology" parts 1-2 and "Implementation details" (pipeline).
//
// One thread-block cluster of C CTAs handles one row; CTA c owns a contiguous
// chunk of the row. The row is streamed from HBM once:
//
//   A2  mu, sigma (and a reference max) from one sample block of the row,
//       read identically by every CTA of the cluster (no exchange needed);
//   A3  delta from the normal-quantile tables, t = mu + delta * sigma;
//   A4  one streaming pass over the chunk keeps Z_t = {x >= t} (value and
//       index) in a shared-memory list, and tracks max / min / NaN / +inf and,
//       for top-p without top-k, the softmax mass of the row and of Z_t;
//   --  one cluster merge through distributed shared memory;
//   A5  hit: every CTA gathers the whole Z_t into its shared memory;
//       fallback (miss, or too many candidates): distributed narrowing passes
//       evaluate two quaternary levels (15 pivots) per cluster merge until the
//       range that holds the boundary fits, then that range is gathered;
//   A6  quaternary pivot search over the gathered candidates with
//       z_mn / N_zmn duplicate tracking, inside each CTA (block barriers only);
//   A7  the same search by softmax mass for top-p;
//   A8  boundary duplicates kept by lowest token id: per-rank counts from the
//       gathered set, then an index cut inside the one straddling CTA;
//   A9  mask emission: hit rows write zeros and scatter the kept ids of the
//       CTA's own list (no second read of the logits); fallback rows stream
//       the chunk again.
//
// Every decision that steers a barrier is taken from merged values that are
// identical in every CTA of the cluster and published through shared memory,
// so control flow, and with it every barrier, is uniform.

#include <cfloat>
#include <cmath>
#include <cstdint>

#include <cuda_runtime.h>

#include "qrita_device.cuh"
#include "qrita_internal.h"

namespace qrita {
namespace {

using namespace dev;

constexpr int kWarps = kThreads / 32;
constexpr uint32_t kFull = 0xffffffffu;
constexpr int kSampleBlocks = 16;
constexpr int kSampleBlock = 64;  // 16 x 64 = 1024 sampled logits per row
constexpr int kBins = kNarrowPivots + 1;
constexpr int kTagShift = 28;  // gathered tag = rank << 28 | index in chunk
// Pinned narrowing (from below only) gives up after this many passes and
// narrows from both ends (a tie group at the boundary larger than the lists).
constexpr int kPinnedPasses = 12;

template <int DT>
struct Elem;
template <>
struct Elem<QRITA_DTYPE_F32> {
  static constexpr int kBytes = 4;
  static constexpr int kPerUnit = 4;  // elements per 16-byte unit
};
template <>
struct Elem<QRITA_DTYPE_BF16> {
  static constexpr int kBytes = 2;
  static constexpr int kPerUnit = 8;
};

template <int DT>
__device__ __forceinline__ void unpack(const uint4 v, float (&x)[Elem<DT>::kPerUnit]) {
  if constexpr (DT == QRITA_DTYPE_F32) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  } else {
    // bf16 is the upper half of binary32: widening is a shift (exact).
    x[0] = __uint_as_float(v.x << 16);
    x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16);
    x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    x[4] = __uint_as_float(v.z << 16);
    x[5] = __uint_as_float(v.z & 0xFFFF0000u);
    x[6] = __uint_as_float(v.w << 16);
    x[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
}

template <int DT>
__device__ __forceinline__ float load_elem(const unsigned char* p) {
  if constexpr (DT == QRITA_DTYPE_F32) {
    return __ldg(reinterpret_cast<const float*>(p));
  } else {
    return __uint_as_float(static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(p))) << 16);
  }
}

__device__ __forceinline__ uint4 ldg16(const unsigned char* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

// Read of shared state another thread wrote before a barrier. Every such read
// goes through a volatile shared load so the compiler can neither reuse an
// earlier load of the same word nor move the load across the barrier.
template <typename T>
__device__ __forceinline__ T vld(const T& r) {
  return *reinterpret_cast<const volatile T*>(&r);
}

// Softmax weight of x for row max m. A row whose max is -inf holds only
// -inf, and equal logits get equal weight 1.
__device__ __forceinline__ float weight(float x, float m, bool m_neginf) {
  return m_neginf ? 1.0f : expf(x - m);
}

// ---------------------------------------------------------------------------
// Shared-memory layout
// ---------------------------------------------------------------------------
struct alignas(16) Slot {  // what one CTA publishes for one cluster merge
  unsigned long long mass[kBins + 1];  // narrowing: per-bin fixed-point mass; [kBins] above hi
  uint32_t cnt[kBins + 1];             // narrowing: per-bin counts; [kBins] above hi
  float f[4];
  uint32_t u[4];
  double d[2];
};

struct alignas(16) Bcast {  // written by one thread / warp 0 before a block barrier
  double d[8];
  float f[12];
  uint32_t u[24];
  uint32_t q[16];  // pivot keys, increasing
  float qf[16];    // pivot floats (+inf padding)
};

struct alignas(16) PAccS {  // per-warp pivot partial (block reduction scratch)
  uint32_t cnt;
  float z;
  uint32_t nz;
  float mhi, mlo;
  uint32_t pad[3];
};

struct alignas(16) Fixed {
  Slot slots[2];
  Bcast bc;
  PAccS red[kWarps][3];
  float redf[kWarps][8];
  uint32_t redu[kWarps][kBins];
  uint32_t bin_cnt[kWarps][kBins];
  unsigned long long bin_mass[kWarps][kBins];
  uint32_t rank_bins[kMaxCluster][kBins + 1];  // latest narrowing merge, per rank
  uint32_t rank_n[kMaxCluster];   // per-rank entries to gather
  uint32_t rank_lo[kMaxCluster];  // per-rank count above the narrowing lo
  uint32_t rank_hi[kMaxCluster];  // per-rank count above the narrowing hi
  uint32_t ties[kMaxCluster];     // per-rank count of boundary-valued elements
  uint32_t scan[kWarps];
  uint32_t own_n;
  uint32_t g_n;
};

// Names of the broadcast slots
enum : int {
  // floats
  BF_MU = 0, BF_SIGMA, BF_MREF, BF_T, BF_MAX, BF_MIN, BF_SMIN, BF_LOF, BF_HIF,
  // uints
  BU_TRUNC = 0, BU_SMIN_N, BU_S, BU_OVF, BU_LO, BU_HI, BU_CLO, BU_CHI, BU_DONE, BU_TAU,
  BU_NKEEP, BU_CABOVE, BU_NP, BU_USED_VALUE, BU_VMODE, BU_MAXR, BU_BELOW,
  // doubles
  BD_ZR = 0, BD_MR, BD_MLO, BD_MHI, BD_TARGET, BD_TOTAL,
};

// ---------------------------------------------------------------------------
// Pivot accumulators of the local search
// ---------------------------------------------------------------------------
struct PAcc {
  uint32_t cnt;
  float z;
  uint32_t nz;
  F2 m;
};

__device__ __forceinline__ void pacc_init(PAcc& a) {
  a.cnt = 0;
  a.z = INFINITY;
  a.nz = 0;
  a.m.hi = 0.f;
  a.m.lo = 0.f;
}

template <bool MASS>
__device__ __forceinline__ void pacc_combine(PAcc& a, const PAcc& b) {
  a.cnt += b.cnt;
  if (b.z < a.z) {
    a.z = b.z;
    a.nz = b.nz;
  } else if (b.z == a.z) {
    a.nz += b.nz;
  }
  if (MASS) a.m = f2_merge(a.m, b.m);
}

template <bool MASS>
__device__ __forceinline__ PAcc pacc_shfl_xor(const PAcc& a, int off) {
  PAcc o;
  o.cnt = __shfl_xor_sync(kFull, a.cnt, off);
  o.z = __shfl_xor_sync(kFull, a.z, off);
  o.nz = __shfl_xor_sync(kFull, a.nz, off);
  if (MASS) {
    o.m.hi = __shfl_xor_sync(kFull, a.m.hi, off);
    o.m.lo = __shfl_xor_sync(kFull, a.m.lo, off);
  } else {
    o.m.hi = 0.f;
    o.m.lo = 0.f;
  }
  return o;
}

// Per-element update of three pivots: count above, softmax mass above, and
// z_mn / N_zmn (smallest element above the pivot and its multiplicity).
// Unused pivots are +inf. Predicated, so the warp never diverges here.
template <bool MASS>
__device__ __forceinline__ void pacc_update(PAcc (&acc)[3], const float (&qf)[3], float x, float w) {
#pragma unroll
  for (int j = 0; j < 3; ++j) {
    const bool g = x > qf[j];
    acc[j].cnt += g ? 1u : 0u;
    if (MASS) f2_add(acc[j].m, g ? w : 0.f);
    const bool lt = g && (x < acc[j].z);
    const bool eq = (x == acc[j].z);
    acc[j].nz = lt ? 1u : (acc[j].nz + (eq ? 1u : 0u));
    acc[j].z = lt ? x : acc[j].z;
  }
}

// ---------------------------------------------------------------------------
// Warp / block helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ uint32_t warp_sum_u(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Exclusive scan of a per-thread count over the block, in thread order.
__device__ __forceinline__ uint32_t block_excl_scan(Fixed& F, uint32_t v, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) F.scan[warp] = incl;
  __syncthreads();
  uint32_t wbase = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t s = vld(F.scan[w]);
    wbase += (w < warp) ? s : 0u;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return wbase + incl - v;
}

// Warp-aggregated append of the flagged values of a unit (value and index)
// to a shared list. Every lane of the warp must call it (convergent).
template <int E>
__device__ __forceinline__ void warp_append(uint32_t* counter, float* vals, uint32_t* idxs,
                                            uint32_t cap, const float (&xs)[E], uint32_t idx0,
                                            uint32_t bits) {
  const int lane = threadIdx.x & 31;
  const uint32_t c = __popc(bits);
  if (__ballot_sync(kFull, c != 0) == 0) return;
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  const uint32_t total = __shfl_sync(kFull, incl, 31);
  uint32_t base = 0;
  if (lane == 31) base = atomicAdd(counter, total);
  base = __shfl_sync(kFull, base, 31);
  uint32_t pos = base + incl - c;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((bits >> e) & 1u) {
      if (pos < cap) {
        vals[pos] = xs[e];
        idxs[pos] = idx0 + e;
      }
      ++pos;
    }
  }
}

// ---------------------------------------------------------------------------
// Pivots: 25/50/75 % of a key range (lo, hi]
// ---------------------------------------------------------------------------
// Value-space quartiles (the pages' reading of "25/50/75 % of the search
// range") when value_ok and both ends are finite floats; otherwise quartiles
// of the 32-bit key range, which always shrink it fourfold. Writes up to 3
// strictly increasing keys inside (lo, hi) and returns how many.
__device__ int quartile_pivots(uint32_t lo, uint32_t hi, bool value_ok, uint32_t* q, bool* used_value) {
  const uint32_t span = hi - lo;
  *used_value = false;
  if (span <= 1u) return 0;
  if (span <= 4u) {
    const int np = static_cast<int>(span) - 1;
    for (int j = 0; j < np; ++j) q[j] = lo + 1u + static_cast<uint32_t>(j);
    return np;
  }
  if (value_ok) {
    const float vlo = key2f(lo), vhi = key2f(hi);
    if (isfinite(vlo) && isfinite(vhi)) {
      const double dl = vlo, dh = vhi;
      const uint32_t a = f2key(static_cast<float>(dl + 0.25 * (dh - dl)));
      const uint32_t b = f2key(static_cast<float>(dl + 0.50 * (dh - dl)));
      const uint32_t c = f2key(static_cast<float>(dl + 0.75 * (dh - dl)));
      if (lo < a && a < b && b < c && c < hi) {
        q[0] = a;
        q[1] = b;
        q[2] = c;
        *used_value = true;
        return 3;
      }
    }
  }
  for (int j = 0; j < 3; ++j) q[j] = lo + static_cast<uint32_t>((static_cast<uint64_t>(span) * (j + 1)) >> 2);
  return 3;
}

// Two quaternary levels at once: the quartile pivots of (lo, hi] and of each
// of the four sub-ranges they cut. Returns the count (<= 15), keys sorted.
__device__ int two_level_pivots(uint32_t lo, uint32_t hi, bool value_ok, uint32_t* q, bool* used_value) {
  uint32_t l1[3];
  const int n1 = quartile_pivots(lo, hi, value_ok, l1, used_value);
  int n = 0;
  uint32_t a = lo;
  for (int s = 0; s <= n1; ++s) {
    const uint32_t b = (s < n1) ? l1[s] : hi;
    uint32_t l2[3];
    bool uv = false;
    const int n2 = quartile_pivots(a, b, value_ok, l2, &uv);
    for (int j = 0; j < n2; ++j) q[n++] = l2[j];
    if (s < n1) q[n++] = l1[s];
    a = b;
  }
  return n;
}

// ---------------------------------------------------------------------------
// Per-CTA context
// ---------------------------------------------------------------------------
template <int DT>
struct Ctx {
  static constexpr int E = Elem<DT>::kPerUnit;
  static constexpr int S = Elem<DT>::kBytes;
  Fixed* F;
  float* own_val;
  uint32_t* own_idx;
  uint32_t ocap;
  float* g_val;
  uint32_t* g_tag;
  uint32_t gcap;
  const unsigned char* gx;     // chunk start in global memory
  const unsigned char* gbody;  // first 16-byte aligned unit of the chunk
  uint8_t* gmask;              // chunk start in the mask
  int n, head_n, body_units, tail_n;
  uint32_t C, crank;
  int ph;           // cluster merge counter (slot parity)
  float m;          // row max (softmax shift)
  bool m_neginf;
  float fix_scale;  // fixed-point scale of weights in [0, 1]
};

// Stream the chunk from global memory: kUnroll 16-byte units per thread in
// flight, then the head / tail elements (fewer than 2E, one per thread).
// unit_fn(xs, idx0, valid) and scalar_fn(x, idx, valid) are called by every
// thread the same number of times (convergent), valid or not.
template <int DT, typename UnitFn, typename ScalarFn>
__device__ __forceinline__ void stream_chunk(const Ctx<DT>& c, UnitFn&& unit_fn, ScalarFn&& scalar_fn) {
  constexpr int E = Ctx<DT>::E;
  constexpr int S = Ctx<DT>::S;
  const int tid = threadIdx.x;
  const int nb = c.body_units;
  for (int base = 0; base < nb; base += kThreads * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int u = base + j * kThreads + tid;
      v[j] = (u < nb) ? ldg16(c.gbody + 16 * static_cast<size_t>(u)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int j = 0; j < kUnroll; ++j) {
      const int u = base + j * kThreads + tid;
      float xs[E];
      unpack<DT>(v[j], xs);
      unit_fn(xs, static_cast<uint32_t>(c.head_n + u * E), u < nb);
    }
  }
  float x = 0.f;
  uint32_t idx = 0;
  const bool valid = tid < c.head_n + c.tail_n;
  if (valid) {
    if (tid < c.head_n) {
      x = load_elem<DT>(c.gx + tid * S);
      idx = static_cast<uint32_t>(tid);
    } else {
      const int j = tid - c.head_n;
      x = load_elem<DT>(c.gbody + 16 * static_cast<size_t>(nb) + j * S);
      idx = static_cast<uint32_t>(c.head_n + nb * E + j);
    }
  }
  scalar_fn(x, idx, valid);
}

// ---------------------------------------------------------------------------
// Distributed narrowing (fallback search over the lists or the chunk)
// ---------------------------------------------------------------------------
struct Range {
  uint32_t lo, hi;      // count/mass(> lo) >= target > count/mass(> hi)
  uint32_t c_lo, c_hi;  // row counts above lo / hi
  double m_lo, m_hi;    // row masses above lo / hi (fixed-point units)
  bool lo_all;          // lo lies below key(-inf): every element is above it
  bool pin_hi;          // narrow from below only: gather everything above lo
  bool fits;            // the range fits the lists: gather it
  bool exact;           // hi - lo <= 1: the boundary value is hi
  bool below;           // the target exceeds everything above lo: the boundary is lo itself
  int passes;
};

// One narrowing pass: up to 15 pivots (two quaternary levels) cut (lo, hi]
// into bins; every CTA bins its elements (from its list, or by streaming its
// chunk again), the bins merge across the cluster in rank order, and warp 0
// keeps the bin that holds the boundary. Counts are exact integers and
// masses exact sums of fixed-point weights, so the merge is deterministic.
// target < 0 means "p_frac times (the pass's total mass + extra)": the pass
// then also measures the softmax denominator.
template <int DT, bool MASS>
__device__ void narrow_pass(Ctx<DT>& c, Range& R, double& target, double p_frac, double extra,
                            bool from_chunk, bool value_ok, bool* used_value_out) {
  constexpr int E = Ctx<DT>::E;
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    uint32_t q[kNarrowPivots];
    bool used_value = false;
    const int np = two_level_pivots(R.lo, R.hi, value_ok, q, &used_value);
    for (int j = 0; j < 16; ++j) {
      F.bc.q[j] = (j < np) ? q[j] : R.hi;
      F.bc.qf[j] = (j < np) ? pivot_f(q[j]) : INFINITY;
    }
    F.bc.u[BU_NP] = static_cast<uint32_t>(np);
    F.bc.u[BU_USED_VALUE] = used_value ? 1u : 0u;
    F.bc.f[BF_LOF] = R.lo_all ? -INFINITY : pivot_f(R.lo);
    F.bc.f[BF_HIF] = pivot_f(R.hi);
  }
  for (int i = tid; i < kWarps * kBins; i += kThreads) {
    (&F.bin_cnt[0][0])[i] = 0u;
    (&F.bin_mass[0][0])[i] = 0ull;
  }
  __syncthreads();
  const float lo_f = vld(F.bc.f[BF_LOF]);
  const float hi_f = vld(F.bc.f[BF_HIF]);
  const bool lo_all = R.lo_all;
  const float scale = c.fix_scale;
  uint32_t above_c = 0;
  unsigned long long above_m = 0ull;
  auto bin_one = [&](float x) {
    if (!(lo_all || x > lo_f)) return;
    unsigned long long wf = 0ull;
    if (MASS) wf = __float2ull_rn(weight(x, c.m, c.m_neginf) * scale);
    if (x > hi_f) {
      ++above_c;
      above_m += wf;
      return;
    }
    // bin = number of pivots below x (pivots increasing, +inf padded)
    int b = 0;
    b += (x > vld(F.bc.qf[b + 7])) ? 8 : 0;
    b += (x > vld(F.bc.qf[b + 3])) ? 4 : 0;
    b += (x > vld(F.bc.qf[b + 1])) ? 2 : 0;
    b += (x > vld(F.bc.qf[b])) ? 1 : 0;
    atomicAdd(&F.bin_cnt[warp][b], 1u);
    if (MASS) atomicAdd(&F.bin_mass[warp][b], wf);
  };
  if (from_chunk) {
    stream_chunk<DT>(
        c,
        [&](const float (&xs)[E], uint32_t, bool valid) {
          if (!valid) return;
#pragma unroll
          for (int e = 0; e < E; ++e) bin_one(xs[e]);
        },
        [&](float x, uint32_t, bool valid) {
          if (valid) bin_one(x);
        });
  } else {
    const uint32_t n = min(vld(F.own_n), c.ocap);
    for (uint32_t i = tid; i < n; i += kThreads) bin_one(c.own_val[i]);
  }
  above_c = warp_sum_u(above_c);
  above_m = warp_sum_u64(above_m);
  if (lane == 0) {
    F.redu[warp][0] = above_c;
    F.redu[warp][1] = static_cast<uint32_t>(above_m);
    F.redu[warp][2] = static_cast<uint32_t>(above_m >> 32);
  }
  __syncthreads();
  Slot& my = F.slots[c.ph & 1];
  if (tid < kBins) {
    uint32_t s = 0;
    unsigned long long sm = 0ull;
    for (int w = 0; w < kWarps; ++w) {
      s += vld(F.bin_cnt[w][tid]);
      sm += vld(F.bin_mass[w][tid]);
    }
    my.cnt[tid] = s;
    my.mass[tid] = sm;
  } else if (tid == kBins) {
    uint32_t s = 0;
    unsigned long long sm = 0ull;
    for (int w = 0; w < kWarps; ++w) {
      s += vld(F.redu[w][0]);
      sm += static_cast<unsigned long long>(vld(F.redu[w][1])) |
            (static_cast<unsigned long long>(vld(F.redu[w][2])) << 32);
    }
    my.cnt[kBins] = s;
    my.mass[kBins] = sm;
  }
  cluster_sync_all();
  if (warp == 0) {
    // lane b sums bin b over the ranks in rank order and keeps per-rank counts
    uint32_t tot_c = 0;
    unsigned long long tot_m = 0ull;
    if (lane <= kBins) {
      const uint32_t cnt_addr = smem_u32(&my.cnt[lane]);
      const uint32_t mass_addr = smem_u32(&my.mass[lane]);
      for (uint32_t r = 0; r < c.C; ++r) {
        const uint32_t cr = ld_dsmem_u32(map_rank(cnt_addr, r));
        F.rank_bins[r][lane] = cr;
        tot_c += cr;
        if (MASS) {
          const uint32_t ma = map_rank(mass_addr, r);
          tot_m += static_cast<unsigned long long>(ld_dsmem_u32(ma)) |
                   (static_cast<unsigned long long>(ld_dsmem_u32(ma + 4)) << 32);
        }
      }
    }
    const int np = static_cast<int>(vld(F.bc.u[BU_NP]));
    uint32_t bc_all[kBins + 1];
    unsigned long long bm_all[kBins + 1];
#pragma unroll
    for (int b = 0; b <= kBins; ++b) {
      bc_all[b] = __shfl_sync(kFull, tot_c, b);
      bm_all[b] = __shfl_sync(kFull, tot_m, b);
    }
    __syncwarp();  // per-rank bins visible to the whole warp
    int lo_j = -1, hi_j = -1;
    if (lane == 0) {
      // cum[b] = elements above pivot b-1 (cum[0]: above lo); top: above hi
      uint32_t cum_c[kBins + 1];
      double cum_m[kBins + 1];
      uint32_t cc = bc_all[kBins];
      double cm = static_cast<double>(bm_all[kBins]);
      for (int b = np; b >= 0; --b) {
        cc += bc_all[b];
        cm += static_cast<double>(bm_all[b]);
        cum_c[b] = cc;
        cum_m[b] = cm;
      }
      double tgt = target;
      if (tgt < 0.0) {
        tgt = p_frac * (cum_m[0] + extra);
        F.bc.d[BD_TOTAL] = cum_m[0];
      }
      F.bc.d[BD_TARGET] = tgt;
      F.bc.u[BU_BELOW] = ((MASS ? cum_m[0] : static_cast<double>(cum_c[0])) < tgt) ? 1u : 0u;
      for (int j = 0; j < np; ++j) {
        const double above = MASS ? cum_m[j + 1] : static_cast<double>(cum_c[j + 1]);
        if (above >= tgt) {
          lo_j = j;
        } else {
          hi_j = j;
          break;
        }
      }
      if (R.pin_hi) hi_j = -1;
      uint32_t nlo = R.lo, nhi = R.hi;
      uint32_t nclo = cum_c[0], nchi = bc_all[kBins];
      double nmlo = cum_m[0], nmhi = static_cast<double>(bm_all[kBins]);
      if (lo_j >= 0) {
        nlo = vld(F.bc.q[lo_j]);
        nclo = cum_c[lo_j + 1];
        nmlo = cum_m[lo_j + 1];
      }
      if (hi_j >= 0) {
        nhi = vld(F.bc.q[hi_j]);
        nchi = cum_c[hi_j + 1];
        nmhi = cum_m[hi_j + 1];
      }
      F.bc.u[BU_LO] = nlo;
      F.bc.u[BU_HI] = nhi;
      F.bc.u[BU_CLO] = nclo;
      F.bc.u[BU_CHI] = nchi;
      F.bc.d[BD_MLO] = nmlo;
      F.bc.d[BD_MHI] = nmhi;
    }
    lo_j = __shfl_sync(kFull, lo_j, 0);
    hi_j = __shfl_sync(kFull, hi_j, 0);
    // per-rank counts above the new lo / hi, from that rank's bins
    uint32_t maxr = 0;
    if (lane < static_cast<int>(c.C)) {
      const uint32_t top = vld(F.rank_bins[lane][kBins]);
      uint32_t above_lo = top, above_hi = top;
      const int lo_first = lo_j >= 0 ? lo_j + 1 : 0;
      for (int b = np; b >= lo_first; --b) above_lo += vld(F.rank_bins[lane][b]);
      if (hi_j >= 0)
        for (int b = np; b > hi_j; --b) above_hi += vld(F.rank_bins[lane][b]);
      F.rank_lo[lane] = above_lo;
      F.rank_hi[lane] = above_hi;
      maxr = R.pin_hi ? above_lo : above_lo - above_hi;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) maxr = max(maxr, __shfl_xor_sync(kFull, maxr, o));
    if (lane == 0) F.bc.u[BU_MAXR] = maxr;
  }
  __syncthreads();
  ++c.ph;
  target = vld(F.bc.d[BD_TARGET]);
  R.lo = vld(F.bc.u[BU_LO]);
  R.hi = vld(F.bc.u[BU_HI]);
  R.c_lo = vld(F.bc.u[BU_CLO]);
  R.c_hi = vld(F.bc.u[BU_CHI]);
  R.m_lo = vld(F.bc.d[BD_MLO]);
  R.m_hi = vld(F.bc.d[BD_MHI]);
  R.lo_all = R.lo < kKeyNegInf;
  const uint32_t maxr = vld(F.bc.u[BU_MAXR]);
  const uint32_t in_range = R.pin_hi ? R.c_lo : R.c_lo - R.c_hi;
  R.fits = in_range <= c.gcap && maxr <= c.ocap;
  R.exact = !R.pin_hi && (R.hi - R.lo <= 1u);
  R.below = vld(F.bc.u[BU_BELOW]) != 0u;
  ++R.passes;
  *used_value_out = vld(F.bc.u[BU_USED_VALUE]) != 0u;
}

template <int DT, bool MASS>
__device__ void narrow(Ctx<DT>& c, Range& R, double& target, double p_frac, double extra, bool from_chunk) {
  bool value_ok = true;
  R.passes = 0;
  R.fits = false;
  R.exact = false;
  R.below = false;
  while (true) {
    const uint32_t span_before = R.hi - R.lo;
    bool used_value = false;
    narrow_pass<DT, MASS>(c, R, target, p_frac, extra, from_chunk, value_ok, &used_value);
    if (R.below || R.fits || R.exact) break;
    if (R.passes >= kMaxRounds) break;
    if (R.pin_hi && R.passes >= kPinnedPasses) R.pin_hi = false;
    // a value-space split that failed to halve the key range hands the next
    // pass to key-space quartiles
    value_ok = !(used_value && (R.hi - R.lo) > span_before / 2u);
  }
}

// Re-read the chunk and keep its elements in (lo, hi] in the own list.
template <int DT>
__device__ void extract_range(Ctx<DT>& c, const Range& R) {
  constexpr int E = Ctx<DT>::E;
  Fixed& F = *c.F;
  if (threadIdx.x == 0) F.own_n = 0;
  __syncthreads();
  const float lo_f = R.lo_all ? -INFINITY : pivot_f(R.lo);
  const float hi_f = R.pin_hi ? INFINITY : pivot_f(R.hi);
  const bool lo_all = R.lo_all;
  stream_chunk<DT>(
      c,
      [&](const float (&xs)[E], uint32_t idx0, bool valid) {
        uint32_t bits = 0;
        if (valid) {
#pragma unroll
          for (int e = 0; e < E; ++e)
            if ((lo_all || xs[e] > lo_f) && !(xs[e] > hi_f)) bits |= 1u << e;
        }
        warp_append<E>(&F.own_n, c.own_val, c.own_idx, c.ocap, xs, idx0, bits);
      },
      [&](float x, uint32_t idx, bool valid) {
        const float xs[1] = {x};
        const uint32_t bits = (valid && (lo_all || x > lo_f) && !(x > hi_f)) ? 1u : 0u;
        warp_append<1>(&F.own_n, c.own_val, c.own_idx, c.ocap, xs, idx, bits);
      });
  __syncthreads();
}

// Copy every rank's own-list entries in (lo, hi] into this CTA's gathered set
// (value, rank << 28 | index). F.rank_n[r] holds rank r's list length.
// sync_first: the lists were rewritten since the last cluster barrier. The
// barrier at the end is the last access to another CTA's memory.
template <int DT>
__device__ void gather(Ctx<DT>& c, float lo_f, float hi_f, bool lo_all, bool sync_first) {
  Fixed& F = *c.F;
  if (threadIdx.x == 0) F.g_n = 0;
  if (sync_first) cluster_sync_all();
  __syncthreads();
  const uint32_t val_base = smem_u32(c.own_val);
  const uint32_t idx_base = smem_u32(c.own_idx);
  for (uint32_t r = 0; r < c.C; ++r) {
    const uint32_t n = min(vld(F.rank_n[r]), c.ocap);
    const uint32_t rv = map_rank(val_base, r);
    const uint32_t ri = map_rank(idx_base, r);
    for (uint32_t b = 0; b < n; b += kThreads) {
      const uint32_t i = b + threadIdx.x;
      float xs[1] = {0.f};
      uint32_t idx = 0, bits = 0;
      if (i < n) {
        xs[0] = ld_dsmem_f32(rv + 4u * i);
        idx = ld_dsmem_u32(ri + 4u * i);
        bits = ((lo_all || xs[0] > lo_f) && !(xs[0] > hi_f)) ? 1u : 0u;
      }
      warp_append<1>(&F.g_n, c.g_val, c.g_tag, c.gcap, xs, (r << kTagShift) | idx, bits);
    }
  }
  cluster_sync_all();
}

// ---------------------------------------------------------------------------
// Local quaternary search over the gathered set (block barriers only)
// ---------------------------------------------------------------------------
struct Local {
  uint32_t lo, hi, c_lo, c_hi;  // row counts above lo / hi
  double m_lo, m_hi;            // row masses above lo / hi (mass search)
  uint32_t c_above;             // row count above the gathered range
  double m_above;               // row mass above the gathered range
  // result
  uint32_t tau, n_keep, count_above;
  int rounds;
  bool capped;
};

// Quaternary search (A6 for counts, A7 for mass) over g_val[0..g_n). The
// search keeps count/mass(> lo) >= target > count/mass(> hi); each round
// evaluates three pivots at 25/50/75 % of the range and stops at the first
// pivot whose z_mn is the boundary (above(q) reaches the target and above(q)
// minus the N_zmn copies of z_mn does not): tau = z_mn and the number of
// kept copies follows. Thread 0 takes every decision and broadcasts it.
template <int DT, bool MASS>
__device__ void local_search(Ctx<DT>& c, Local& s, double target, bool value_pivots) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t gn = min(vld(F.g_n), c.gcap);
  if (tid == 0) {
    F.bc.u[BU_LO] = s.lo;
    F.bc.u[BU_HI] = s.hi;
    F.bc.u[BU_CLO] = s.c_lo;
    F.bc.u[BU_CHI] = s.c_hi;
    F.bc.d[BD_MLO] = s.m_lo;
    F.bc.d[BD_MHI] = s.m_hi;
    F.bc.u[BU_DONE] = 0;
    F.bc.u[BU_VMODE] = value_pivots ? 1u : 0u;
  }
  int rounds = 0;
  for (;;) {
    // thread 0: stop when (lo, hi] holds one key, else pick the pivots
    if (tid == 0) {
      const uint32_t lo = F.bc.u[BU_LO], hi = F.bc.u[BU_HI];
      if (hi - lo <= 1u) {
        const uint32_t c_hi = F.bc.u[BU_CHI], c_lo = F.bc.u[BU_CLO];
        const uint32_t N = c_lo - c_hi;
        F.bc.u[BU_TAU] = hi;
        F.bc.u[BU_CABOVE] = c_hi;
        if (MASS) {
          const double wz = weight(key2f(hi), c.m, c.m_neginf);
          double nk = ceil((target - F.bc.d[BD_MHI]) / wz);
          nk = fmin(fmax(nk, 1.0), static_cast<double>(N));
          F.bc.u[BU_NKEEP] = static_cast<uint32_t>(nk);
        } else {
          F.bc.u[BU_NKEEP] = static_cast<uint32_t>(target) - c_hi;
        }
        F.bc.u[BU_DONE] = 1;
      } else if (rounds >= kMaxRounds) {
        F.bc.u[BU_DONE] = 2;
      } else {
        uint32_t q[3];
        bool used_value = false;
        const int np = quartile_pivots(lo, hi, F.bc.u[BU_VMODE] != 0u, q, &used_value);
        for (int j = 0; j < 3; ++j) {
          F.bc.q[j] = (j < np) ? q[j] : hi;
          F.bc.qf[j] = (j < np) ? pivot_f(q[j]) : INFINITY;
        }
        F.bc.u[BU_NP] = static_cast<uint32_t>(np);
        F.bc.u[BU_USED_VALUE] = used_value ? 1u : 0u;
      }
    }
    __syncthreads();
    const uint32_t done0 = vld(F.bc.u[BU_DONE]);
    if (done0 != 0u) break;
    float qf[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) qf[j] = vld(F.bc.qf[j]);
    PAcc acc[3];
#pragma unroll
    for (int j = 0; j < 3; ++j) pacc_init(acc[j]);
    for (uint32_t i = tid; i < gn; i += kThreads) {
      const float x = c.g_val[i];
      const float w = MASS ? weight(x, c.m, c.m_neginf) : 0.f;
      pacc_update<MASS>(acc, qf, x, w);
    }
#pragma unroll
    for (int j = 0; j < 3; ++j) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const PAcc t = pacc_shfl_xor<MASS>(acc[j], o);
        pacc_combine<MASS>(acc[j], t);
      }
      if (lane == 0) {
        F.red[warp][j].cnt = acc[j].cnt;
        F.red[warp][j].z = acc[j].z;
        F.red[warp][j].nz = acc[j].nz;
        F.red[warp][j].mhi = acc[j].m.hi;
        F.red[warp][j].mlo = acc[j].m.lo;
      }
    }
    __syncthreads();
    ++rounds;
    if (warp == 0) {
      PAcc tot[3];
#pragma unroll
      for (int j = 0; j < 3; ++j) {
        PAcc a;
        pacc_init(a);
        if (lane < kWarps) {
          a.cnt = vld(F.red[lane][j].cnt);
          a.z = vld(F.red[lane][j].z);
          a.nz = vld(F.red[lane][j].nz);
          a.m.hi = vld(F.red[lane][j].mhi);
          a.m.lo = vld(F.red[lane][j].mlo);
        }
#pragma unroll
        for (int o = kWarps / 2; o > 0; o >>= 1) {
          const PAcc t = pacc_shfl_xor<MASS>(a, o);
          pacc_combine<MASS>(a, t);
        }
        tot[j] = a;
      }
      if (lane == 0) {
        const int np = static_cast<int>(F.bc.u[BU_NP]);
        int done_j = -1, lo_j = -1, hi_j = -1;
        double above_j[3] = {0.0, 0.0, 0.0};
        for (int j = 0; j < np; ++j) {
          const double above = MASS ? (f2_value(tot[j].m) + s.m_above)
                                    : static_cast<double>(tot[j].cnt + s.c_above);
          above_j[j] = above;
          if (above >= target) {
            const double wz = MASS ? static_cast<double>(weight(tot[j].z, c.m, c.m_neginf)) : 1.0;
            const double below_z = above - static_cast<double>(tot[j].nz) * wz;
            if (below_z < target) {
              done_j = j;
              break;
            }
            lo_j = j;
          } else {
            hi_j = j;
            break;
          }
        }
        if (done_j >= 0) {
          const PAcc& t = tot[done_j];
          const uint32_t cnt_above = t.cnt + s.c_above - t.nz;
          F.bc.u[BU_TAU] = f2key(t.z);
          F.bc.u[BU_CABOVE] = cnt_above;
          if (MASS) {
            const double wz = weight(t.z, c.m, c.m_neginf);
            double nk = ceil((target - (above_j[done_j] - static_cast<double>(t.nz) * wz)) / wz);
            nk = fmin(fmax(nk, 1.0), static_cast<double>(t.nz));
            F.bc.u[BU_NKEEP] = static_cast<uint32_t>(nk);
          } else {
            F.bc.u[BU_NKEEP] = static_cast<uint32_t>(target) - cnt_above;
          }
          F.bc.u[BU_DONE] = 1;
        } else {
          const uint32_t old_span = F.bc.u[BU_HI] - F.bc.u[BU_LO];
          if (lo_j >= 0) {
            F.bc.u[BU_LO] = F.bc.q[lo_j];
            F.bc.u[BU_CLO] = tot[lo_j].cnt + s.c_above;
            F.bc.d[BD_MLO] = above_j[lo_j];
          }
          if (hi_j >= 0) {
            F.bc.u[BU_HI] = F.bc.q[hi_j];
            F.bc.u[BU_CHI] = tot[hi_j].cnt + s.c_above;
            F.bc.d[BD_MHI] = above_j[hi_j];
          }
          // after a value-space split that failed to halve the key range,
          // the next round splits the key range
          const uint32_t new_span = F.bc.u[BU_HI] - F.bc.u[BU_LO];
          const bool bad = F.bc.u[BU_USED_VALUE] != 0u && new_span > old_span / 2u;
          F.bc.u[BU_VMODE] = (value_pivots && !bad) ? 1u : 0u;
        }
      }
    }
    __syncthreads();
    if (vld(F.bc.u[BU_DONE]) != 0u) break;
  }
  s.tau = vld(F.bc.u[BU_TAU]);
  s.n_keep = vld(F.bc.u[BU_NKEEP]);
  s.count_above = vld(F.bc.u[BU_CABOVE]);
  s.rounds = rounds;
  s.capped = vld(F.bc.u[BU_DONE]) == 2u;
  __syncthreads();
}

// Per-rank counts of gathered entries equal to tau (into F.ties).
template <int DT>
__device__ void count_ties_gathered(Ctx<DT>& c, float tau_f) {
  Fixed& F = *c.F;
  if (threadIdx.x < kMaxCluster) F.ties[threadIdx.x] = 0u;
  __syncthreads();
  const uint32_t gn = min(vld(F.g_n), c.gcap);
  for (uint32_t i = threadIdx.x; i < gn; i += kThreads)
    if (c.g_val[i] == tau_f) atomicAdd(&F.ties[c.g_tag[i] >> kTagShift], 1u);
  __syncthreads();
}

// The index below which exactly `keep` of this CTA's own-list entries equal
// to tau lie (the own list holds every such element of the chunk). 16-way
// splits of the index range; invariant count(idx < lo) < keep <= count(idx < hi).
template <int DT>
__device__ uint32_t tie_index_cut(Ctx<DT>& c, float tau_f, uint32_t keep) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t n = min(vld(F.own_n), c.ocap);
  uint32_t lo = 0, hi = static_cast<uint32_t>(c.n);
  for (int round = 0; round < 32 && hi - lo > 1u; ++round) {
    const uint32_t span = hi - lo;
    uint32_t piv[15];
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      uint32_t p = (span <= 16u) ? lo + 1u + static_cast<uint32_t>(j)
                                 : lo + static_cast<uint32_t>((static_cast<uint64_t>(span) * (j + 1)) >> 4);
      piv[j] = p < hi ? p : hi;  // pivots at hi are inert
    }
    uint32_t cnt[15];
#pragma unroll
    for (int j = 0; j < 15; ++j) cnt[j] = 0;
    for (uint32_t i = tid; i < n; i += kThreads) {
      if (c.own_val[i] == tau_f) {
        const uint32_t ix = c.own_idx[i];
#pragma unroll
        for (int j = 0; j < 15; ++j) cnt[j] += (ix < piv[j]) ? 1u : 0u;
      }
    }
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      const uint32_t v = warp_sum_u(cnt[j]);
      if (lane == 0) F.redu[warp][j] = v;
    }
    __syncthreads();
    uint32_t nlo = lo, nhi = hi;
#pragma unroll
    for (int j = 0; j < 15; ++j) {
      uint32_t s = 0;
      for (int w = 0; w < kWarps; ++w) s += vld(F.redu[w][j]);
      if (piv[j] <= lo || piv[j] >= hi) continue;
      if (s < keep) nlo = max(nlo, piv[j]);
      else nhi = min(nhi, piv[j]);
    }
    lo = nlo;
    hi = nhi;
    __syncthreads();
  }
  return hi;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 4) select_kernel(const __grid_constant__ Params P) {
  constexpr int E = Ctx<DT>::E;
  constexpr int S = Ctx<DT>::S;
  extern __shared__ __align__(128) unsigned char smem[];
  Fixed& F = *reinterpret_cast<Fixed*>(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  Ctx<DT> c;
  c.F = &F;
  c.ocap = static_cast<uint32_t>(P.ocap);
  c.gcap = static_cast<uint32_t>(P.gcap);
  c.own_val = reinterpret_cast<float*>(smem + sizeof(Fixed));
  c.own_idx = reinterpret_cast<uint32_t*>(c.own_val + P.ocap);
  c.g_val = reinterpret_cast<float*>(c.own_idx + P.ocap);
  c.g_tag = reinterpret_cast<uint32_t*>(c.g_val + P.gcap);
  c.C = static_cast<uint32_t>(P.C);
  c.crank = cluster_rank();
  c.ph = 0;
  c.m = 0.f;
  c.m_neginf = false;
  c.fix_scale = 0.f;

  const int64_t r = blockIdx.x / P.C;
  const int32_t V = P.V;
  const int64_t c0 = static_cast<int64_t>(c.crank) * P.chunk;
  const int64_t rem = static_cast<int64_t>(V) - c0;
  c.n = static_cast<int>(rem <= 0 ? 0 : (rem < P.chunk ? rem : P.chunk));
  const int64_t c0c = c0 < V ? c0 : V;
  const unsigned char* grow = static_cast<const unsigned char*>(P.logits) + static_cast<size_t>(r) * V * S;
  c.gx = grow + static_cast<size_t>(c0c) * S;
  c.gmask = P.mask + static_cast<size_t>(r) * V + c0c;
  {
    const uintptr_t ga = reinterpret_cast<uintptr_t>(c.gx);
    const int h = static_cast<int>(((16u - (ga & 15u)) & 15u) / S);
    c.head_n = h < c.n ? h : c.n;
    c.body_units = (c.n - c.head_n) * S / 16;
    c.tail_n = c.n - c.head_n - c.body_units * E;
  }
  c.gbody = c.gx + c.head_n * S;

  // ---- row parameters (uniform)
  int32_t kr = P.k ? P.k[r] : 0;
  const float pr = P.p ? P.p[r] : 1.0f;
  bool k_on = kr >= 1 && kr < V;
  bool p_on = pr < 1.0f;  // NaN compares false: off
  if (p_on && !(pr > 0.0f)) {
    // p <= 0 keeps exactly one token: the same set as k = 1
    p_on = false;
    if (V > 1) {
      k_on = true;
      kr = 1;
    }
  }
  const bool keep_all = !k_on && !p_on;
  const bool p_only = p_on && !k_on;

  // ---- A2: statistics of one sample block of the row (identical in every CTA)
  {
    float sn = 0.f, sx = 0.f, sxx = 0.f, smax = -INFINITY;
#pragma unroll
    for (int j = 0; j < (kSampleBlocks * kSampleBlock) / kThreads; ++j) {
      const int sidx = tid + j * kThreads;
      int64_t pos;
      if (V <= kSampleBlocks * kSampleBlock) {
        pos = sidx;
      } else {
        pos = static_cast<int64_t>(sidx / kSampleBlock) * (V / kSampleBlocks) + (sidx % kSampleBlock);
      }
      if (pos < V) {
        const float x = load_elem<DT>(grow + static_cast<size_t>(pos) * S);
        if (isfinite(x)) {
          sn += 1.f;
          sx += x;
          sxx += x * x;
          smax = fmaxf(smax, x);
        }
      }
    }
    sn = warp_sum_f(sn);
    sx = warp_sum_f(sx);
    sxx = warp_sum_f(sxx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) smax = fmaxf(smax, __shfl_xor_sync(kFull, smax, o));
    if (lane == 0) {
      F.redf[warp][0] = sn;
      F.redf[warp][1] = sx;
      F.redf[warp][2] = sxx;
      F.redf[warp][3] = smax;
    }
    if (tid == 0) F.own_n = 0;
    __syncthreads();
    if (tid == 0) {
      float a = 0.f, b = 0.f, d = 0.f, mx = -INFINITY;
      for (int w = 0; w < kWarps; ++w) {
        a += vld(F.redf[w][0]);
        b += vld(F.redf[w][1]);
        d += vld(F.redf[w][2]);
        mx = fmaxf(mx, vld(F.redf[w][3]));
      }
      const double mean = a > 0.f ? static_cast<double>(b) / a : 0.0;
      const double var = a > 0.f ? fmax(static_cast<double>(d) / a - mean * mean, 0.0) : 0.0;
      const float mu = static_cast<float>(mean);
      const float sigma = static_cast<float>(sqrt(var));
      F.bc.f[BF_MU] = mu;
      F.bc.f[BF_SIGMA] = sigma;
      F.bc.f[BF_MREF] = a > 0.f ? mx : 0.f;
      // ---- A3: delta from the normal-quantile tables, threshold t
      bool trunc = false;
      float t = -INFINITY;
      if (!(P.flags & QRITA_FLAG_NO_TRUNCATION) && a > 0.f && !keep_all) {
        if (k_on) {
          const float u = P.alpha_k * static_cast<float>(kr) / static_cast<float>(V);
          if (u <= P.u_max_k) {
            int i = static_cast<int>(floorf(-2.0f * log2f(u)));
            i = i < 0 ? 0 : (i > kLutK - 1 ? kLutK - 1 : i);
            t = mu + P.lut_k[i] * sigma;
            trunc = true;
          }
        } else {
          const float qv = 1.0f - pr;
          int i = static_cast<int>(ceilf(-4.0f * log2f(qv)));
          if (i <= kLutP - 1) {
            i = i < 0 ? 0 : i;
            t = mu + (sigma + P.lut_p[i] - P.margin_p) * sigma;
            trunc = true;
          }
        }
        if (!isfinite(t)) trunc = false;
      }
      F.bc.f[BF_T] = trunc ? t : -INFINITY;
      F.bc.u[BU_TRUNC] = trunc ? 1u : 0u;
    }
    __syncthreads();
  }
  const float mu = vld(F.bc.f[BF_MU]);
  const float sigma = vld(F.bc.f[BF_SIGMA]);
  const float m_ref = vld(F.bc.f[BF_MREF]);
  const float t = vld(F.bc.f[BF_T]);
  const bool trunc = vld(F.bc.u[BU_TRUNC]) != 0u;

  // ---- A4: the streaming pass (the one HBM read of the row)
  {
    float vmax = -INFINITY, vmin = INFINITY, smin = INFINITY;
    uint32_t smin_n = 0;
    F2 zs = {0.f, 0.f}, ms = {0.f, 0.f};
    auto elem = [&](float x) -> bool {
      vmax = fmax_nan(vmax, x);
      vmin = fminf(vmin, x);
      const bool surv = trunc && x >= t;
      if (surv) {
        if (x < smin) {
          smin = x;
          smin_n = 1;
        } else if (x == smin) {
          ++smin_n;
        }
      }
      if (p_only) {
        const float w = expf(x - m_ref);
        f2_add(zs, w);
        f2_add(ms, surv ? w : 0.f);
      }
      return surv;
    };
    stream_chunk<DT>(
        c,
        [&](const float (&xs)[E], uint32_t idx0, bool valid) {
          uint32_t bits = 0;
          if (valid) {
#pragma unroll
            for (int e = 0; e < E; ++e) bits |= elem(xs[e]) ? (1u << e) : 0u;
          }
          if (trunc) warp_append<E>(&F.own_n, c.own_val, c.own_idx, c.ocap, xs, idx0, bits);
        },
        [&](float x, uint32_t idx, bool valid) {
          const uint32_t bits = (valid && elem(x)) ? 1u : 0u;
          const float xs[1] = {x};
          if (trunc) warp_append<1>(&F.own_n, c.own_val, c.own_idx, c.ocap, xs, idx, bits);
        });
    // block reduce
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      vmax = fmax_nan(vmax, __shfl_xor_sync(kFull, vmax, o));
      vmin = fminf(vmin, __shfl_xor_sync(kFull, vmin, o));
      const float s2 = __shfl_xor_sync(kFull, smin, o);
      const uint32_t n2 = __shfl_xor_sync(kFull, smin_n, o);
      if (s2 < smin) {
        smin = s2;
        smin_n = n2;
      } else if (s2 == smin) {
        smin_n += n2;
      }
      if (p_only) {
        F2 a, b;
        a.hi = __shfl_xor_sync(kFull, zs.hi, o);
        a.lo = __shfl_xor_sync(kFull, zs.lo, o);
        b.hi = __shfl_xor_sync(kFull, ms.hi, o);
        b.lo = __shfl_xor_sync(kFull, ms.lo, o);
        zs = f2_merge(zs, a);
        ms = f2_merge(ms, b);
      }
    }
    if (lane == 0) {
      F.redf[warp][0] = vmax;
      F.redf[warp][1] = vmin;
      F.redf[warp][2] = smin;
      F.redf[warp][3] = zs.hi;
      F.redf[warp][4] = zs.lo;
      F.redf[warp][5] = ms.hi;
      F.redf[warp][6] = ms.lo;
      F.redu[warp][0] = smin_n;
    }
    __syncthreads();
    Slot& my = F.slots[c.ph & 1];
    if (tid == 0) {
      float a = -INFINITY, b = INFINITY, s = INFINITY;
      uint32_t sn = 0;
      F2 z = {0.f, 0.f}, mm = {0.f, 0.f};
      for (int w = 0; w < kWarps; ++w) {
        a = fmax_nan(a, vld(F.redf[w][0]));
        b = fminf(b, vld(F.redf[w][1]));
        const float s2 = vld(F.redf[w][2]);
        const uint32_t n2 = vld(F.redu[w][0]);
        if (s2 < s) {
          s = s2;
          sn = n2;
        } else if (s2 == s) {
          sn += n2;
        }
        const F2 za = {vld(F.redf[w][3]), vld(F.redf[w][4])};
        const F2 ma = {vld(F.redf[w][5]), vld(F.redf[w][6])};
        z = f2_merge(z, za);
        mm = f2_merge(mm, ma);
      }
      my.f[0] = a;
      my.f[1] = b;
      my.f[2] = s;
      my.u[0] = sn;
      my.u[1] = vld(F.own_n);
      my.d[0] = f2_value(z);
      my.d[1] = f2_value(mm);
    }
    cluster_sync_all();
    if (warp == 0) {
      float a = -INFINITY, b = INFINITY, s = INFINITY;
      uint32_t sn = 0, surv = 0, ovf = 0;
      double z = 0.0, mm = 0.0;
      if (lane < static_cast<int>(c.C)) {
        const uint32_t fb = map_rank(smem_u32(&my.f[0]), lane);
        a = ld_dsmem_f32(fb);
        b = ld_dsmem_f32(fb + 4);
        s = ld_dsmem_f32(fb + 8);
        const uint32_t ub = map_rank(smem_u32(&my.u[0]), lane);
        sn = ld_dsmem_u32(ub);
        surv = ld_dsmem_u32(ub + 4);
        const uint32_t db = map_rank(smem_u32(&my.d[0]), lane);
        z = ld_dsmem_f64(db);
        mm = ld_dsmem_f64(db + 8);
        ovf = surv > c.ocap ? 1u : 0u;
        F.rank_n[lane] = surv;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        a = fmax_nan(a, __shfl_xor_sync(kFull, a, o));
        b = fminf(b, __shfl_xor_sync(kFull, b, o));
        const float s2 = __shfl_xor_sync(kFull, s, o);
        const uint32_t n2 = __shfl_xor_sync(kFull, sn, o);
        if (s2 < s) {
          s = s2;
          sn = n2;
        } else if (s2 == s) {
          sn += n2;
        }
        surv += __shfl_xor_sync(kFull, surv, o);
        ovf |= __shfl_xor_sync(kFull, ovf, o);
        z += __shfl_xor_sync(kFull, z, o);
        mm += __shfl_xor_sync(kFull, mm, o);
      }
      if (lane == 0) {
        F.bc.f[BF_MAX] = a;
        F.bc.f[BF_MIN] = b;
        F.bc.f[BF_SMIN] = s;
        F.bc.u[BU_SMIN_N] = sn;
        F.bc.u[BU_S] = surv;
        F.bc.u[BU_OVF] = ovf;
        F.bc.d[BD_ZR] = z;
        F.bc.d[BD_MR] = mm;
      }
    }
    __syncthreads();
    ++c.ph;
  }
  const float row_max = vld(F.bc.f[BF_MAX]);
  const float row_min = vld(F.bc.f[BF_MIN]);
  const float surv_min = vld(F.bc.f[BF_SMIN]);
  const uint32_t surv_min_n = vld(F.bc.u[BU_SMIN_N]);
  const uint32_t survivors = vld(F.bc.u[BU_S]);
  const bool overflow = vld(F.bc.u[BU_OVF]) != 0u;
  const bool invalid = isnan(row_max) || row_max == INFINITY;
  const double Zr = vld(F.bc.d[BD_ZR]);
  const double Mr = vld(F.bc.d[BD_MR]);
  c.m = row_max;
  c.m_neginf = (row_max == -INFINITY);
  // weights exp(x - m) lie in [0, 1]: fixed point with headroom for V terms
  c.fix_scale = exp2f(static_cast<float>(62 - (32 - __clz(static_cast<uint32_t>(V)))));

  uint32_t path = (k_on ? QRITA_PATH_TOPK : 0u) | (p_on ? QRITA_PATH_TOPP : 0u) |
                  (trunc ? QRITA_PATH_TRUNC : 0u) | (overflow ? QRITA_PATH_OVERFLOW : 0u) |
                  (keep_all ? QRITA_PATH_KEEP_ALL : 0u);
  const bool force_fb = (P.flags & QRITA_FLAG_FORCE_FALLBACK) != 0u;
  const bool value_pivots = (P.flags & QRITA_FLAG_KEY_PIVOTS) == 0u;

  // Selection: keep key > tau, plus the n_keep lowest-id elements equal to
  // tau; F.ties[rank] counts the elements equal to tau in each rank's chunk.
  uint32_t tau = 0, n_keep = 0, count_above = 0;
  uint32_t rounds_k = 0, rounds_p = 0, passes = 0;
  uint32_t row_status = invalid ? QRITA_ROW_NONFINITE : QRITA_ROW_OK;
  double z_used = 0.0;
  bool sel_all = keep_all && !invalid;
  bool sel_none = invalid;
  bool remote_done = false;   // the last access to another CTA's memory is behind a barrier
  bool list_emit = false;     // every kept element is in this CTA's own list
  bool ties_in_list = false;  // every element equal to tau is in this CTA's own list
  bool ties_known = false;    // F.ties holds the per-rank tie counts

  if (!invalid && !keep_all) {
    const double pd = static_cast<double>(pr);
    // the streaming pass summed exp(x - m_ref); shift m is exp(m_ref - m) away
    const bool ref_ok = !c.m_neginf && isfinite(Zr) && isfinite(Mr) && Zr > 0.0 &&
                        static_cast<double>(row_max) - m_ref < 80.0;
    const double cf = ref_ok ? exp(static_cast<double>(m_ref) - row_max) : 0.0;
    const double Zm = Zr * cf, Mm = Mr * cf;

    bool k_full = false;  // the gathered set holds the whole top-k set S_k
    uint32_t tau_k = 0, nk_k = 0, above_k = 0;
    if (k_on) {
      const double target = static_cast<double>(kr);
      const bool hit = trunc && !overflow && !force_fb && survivors >= static_cast<uint32_t>(kr);
      path |= hit ? QRITA_PATH_HIT : QRITA_PATH_FALLBACK;
      Local s;
      s.c_above = 0;
      s.m_above = 0.0;
      s.m_lo = s.m_hi = 0.0;
      bool have_exact = false;
      if (hit && survivors <= c.gcap) {
        // gather Z_t whole: the candidates are (key(t) - 1, max]
        gather<DT>(c, -INFINITY, INFINITY, true, false);
        remote_done = true;
        s.lo = f2key(t) - 1u;
        s.c_lo = survivors;
        s.hi = f2key(row_max);
        s.c_hi = 0;
        k_full = true;
        list_emit = true;
        ties_in_list = true;
        if (survivors - surv_min_n < static_cast<uint32_t>(kr)) {
          // z_mn of the initial lo is the smallest survivor: it is the boundary
          s.tau = f2key(surv_min);
          s.count_above = survivors - surv_min_n;
          s.n_keep = static_cast<uint32_t>(kr) - s.count_above;
          s.rounds = 0;
          s.capped = false;
        } else {
          local_search<DT, false>(c, s, target, value_pivots);
        }
      } else {
        // narrow: over the survivor lists on a hit, over the chunk otherwise
        Range R;
        R.pin_hi = p_on && static_cast<uint32_t>(kr) <= c.gcap;
        R.m_lo = R.m_hi = 0.0;
        double tg = target;
        if (hit) {
          R.lo = f2key(t) - 1u;
          R.c_lo = survivors;
          R.hi = f2key(row_max);
          R.c_hi = 0;
        } else {
          R.lo = f2key(row_min) - 1u;
          R.c_lo = static_cast<uint32_t>(V);
          const bool miss_t = trunc && !overflow && survivors < static_cast<uint32_t>(kr);
          R.hi = (!R.pin_hi && miss_t) ? f2key(t) - 1u : f2key(row_max);
          R.c_hi = (!R.pin_hi && miss_t) ? survivors : 0u;
        }
        R.lo_all = R.lo < kKeyNegInf;
        narrow<DT, false>(c, R, tg, 0.0, 0.0, !hit);
        passes += static_cast<uint32_t>(R.passes);
        if (R.exact) {
          s.tau = R.hi;
          s.count_above = R.c_hi;
          s.n_keep = static_cast<uint32_t>(kr) - R.c_hi;
          s.rounds = 0;
          s.capped = false;
          have_exact = true;
          if (warp == 0 && lane < static_cast<int>(c.C))
            F.ties[lane] = vld(F.rank_lo[lane]) - vld(F.rank_hi[lane]);
          __syncthreads();
          ties_known = true;
        } else if (!R.fits) {
          s.capped = true;
          s.rounds = 0;
        } else {
          if (!hit) {
            extract_range<DT>(c, R);
            // an extraction leaves exactly each rank's range in its list
            if (warp == 0 && lane < static_cast<int>(c.C))
              F.rank_n[lane] = R.pin_hi ? vld(F.rank_lo[lane]) : vld(F.rank_lo[lane]) - vld(F.rank_hi[lane]);
            __syncthreads();
          }
          const float glo = R.lo_all ? -INFINITY : pivot_f(R.lo);
          const float ghi = R.pin_hi ? INFINITY : pivot_f(R.hi);
          gather<DT>(c, glo, ghi, R.lo_all, !hit);
          remote_done = true;
          s.lo = R.lo;
          s.c_lo = R.c_lo;
          if (R.pin_hi) {
            // everything above lo is gathered
            s.hi = f2key(row_max);
            s.c_hi = 0;
            s.c_above = 0;
          } else {
            s.hi = R.hi;
            s.c_hi = R.c_hi;
            s.c_above = R.c_hi;  // elements above hi exceed every pivot
          }
          k_full = R.pin_hi;
          list_emit = hit;
          ties_in_list = true;
          local_search<DT, false>(c, s, target, value_pivots);
        }
      }
      rounds_k = static_cast<uint32_t>(s.rounds);
      if (s.capped) {
        sel_none = true;
        row_status = QRITA_ROW_SEARCH_CAP;
      }
      tau_k = s.tau;
      nk_k = s.n_keep;
      above_k = s.count_above;
      tau = tau_k;
      n_keep = nk_k;
      count_above = above_k;
      if (!sel_none && !have_exact) {
        count_ties_gathered<DT>(c, key2f(tau));
        ties_known = true;
      }
    }

    if (p_on && !sel_none) {
      if (k_on && k_full) {
        // top-p over S_k, all of it gathered: Z_k = mass(> tau_k) + n_keep_k w(tau_k)
        const float tk = key2f(tau_k);
        F2 acc = {0.f, 0.f};
        const uint32_t gn = min(vld(F.g_n), c.gcap);
        for (uint32_t i = tid; i < gn; i += kThreads) {
          const float x = c.g_val[i];
          f2_add(acc, x > tk ? weight(x, c.m, c.m_neginf) : 0.f);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          F2 b;
          b.hi = __shfl_xor_sync(kFull, acc.hi, o);
          b.lo = __shfl_xor_sync(kFull, acc.lo, o);
          acc = f2_merge(acc, b);
        }
        if (lane == 0) {
          F.redf[warp][0] = acc.hi;
          F.redf[warp][1] = acc.lo;
        }
        __syncthreads();
        if (tid == 0) {
          F2 a = {0.f, 0.f};
          for (int w = 0; w < kWarps; ++w) {
            const F2 b = {vld(F.redf[w][0]), vld(F.redf[w][1])};
            a = f2_merge(a, b);
          }
          F.bc.d[BD_TOTAL] = f2_value(a);
        }
        __syncthreads();
        const double M_gt = vld(F.bc.d[BD_TOTAL]);
        const double w_tau = weight(tk, c.m, c.m_neginf);
        const double Zk = M_gt + static_cast<double>(nk_k) * w_tau;
        const double target = pd * Zk;
        z_used = Zk;
        if (M_gt < target) {
          // the boundary lies in the tau_k tie group: keep fewer of them
          double nk = ceil((target - M_gt) / w_tau);
          nk = fmin(fmax(nk, 1.0), static_cast<double>(nk_k));
          n_keep = static_cast<uint32_t>(nk);
          count_above = above_k;
        } else {
          Local s;
          s.lo = tau_k;
          s.c_lo = above_k;
          s.m_lo = M_gt;
          s.hi = f2key(row_max);
          s.c_hi = 0;
          s.m_hi = 0.0;
          s.c_above = 0;
          s.m_above = 0.0;
          local_search<DT, true>(c, s, target, value_pivots);
          rounds_p = static_cast<uint32_t>(s.rounds);
          if (s.capped) {
            sel_none = true;
            row_status = QRITA_ROW_SEARCH_CAP;
          }
          tau = s.tau;
          n_keep = s.n_keep;
          count_above = s.count_above;
          count_ties_gathered<DT>(c, key2f(tau));
        }
      } else {
        // top-p only, or top-p over an S_k too large to gather
        const bool hit = !k_on && trunc && !overflow && !force_fb && ref_ok && Mm >= pd * Zm * (1.0 + 1e-5);
        if (!k_on) path |= hit ? QRITA_PATH_HIT : QRITA_PATH_FALLBACK;
        Local s;
        s.c_above = 0;
        s.m_above = 0.0;
        bool have_exact = false;
        double target = pd * Zm;
        if (hit && survivors <= c.gcap) {
          gather<DT>(c, -INFINITY, INFINITY, true, false);
          remote_done = true;
          z_used = Zm;
          s.lo = f2key(t) - 1u;
          s.c_lo = survivors;
          s.m_lo = Mm;
          s.hi = f2key(row_max);
          s.c_hi = 0;
          s.m_hi = 0.0;
          list_emit = true;
          ties_in_list = true;
          local_search<DT, true>(c, s, target, value_pivots);
        } else {
          // narrow by mass in fixed point (shift m); a pass over the chunk
          // measures the denominator (Z, or mass(> tau_k) for S_k) itself
          Range R;
          R.pin_hi = false;
          const float scale = c.fix_scale;
          double extra = 0.0;
          if (k_on) {
            R.lo = tau_k;
            R.c_lo = above_k;
            extra = static_cast<double>(nk_k) * static_cast<double>(weight(key2f(tau_k), c.m, c.m_neginf)) *
                    static_cast<double>(scale);
          } else if (hit) {
            R.lo = f2key(t) - 1u;
            R.c_lo = survivors;
          } else {
            R.lo = f2key(row_min) - 1u;
            R.c_lo = static_cast<uint32_t>(V);
          }
          R.lo_all = R.lo < kKeyNegInf;
          R.hi = f2key(row_max);
          R.c_hi = 0;
          R.m_lo = R.m_hi = 0.0;
          double tg = hit ? pd * Zm * static_cast<double>(scale) : -1.0;
          narrow<DT, true>(c, R, tg, pd, extra, !hit);
          passes += static_cast<uint32_t>(R.passes);
          target = tg / static_cast<double>(scale);
          z_used = target / pd;
          // the emission streams the chunk unless a gather below says otherwise
          list_emit = false;
          if (R.below) {
            // only after top-k: mass(> tau_k) < p Z_k, so the boundary lies in
            // the tau_k tie group (whose per-rank counts F.ties still holds)
            const double M_gt = R.m_lo / scale;
            const double w_tau = weight(key2f(tau_k), c.m, c.m_neginf);
            double nk = ceil((target - M_gt) / w_tau);
            nk = fmin(fmax(nk, 1.0), static_cast<double>(nk_k));
            s.tau = tau_k;
            s.n_keep = static_cast<uint32_t>(nk);
            s.count_above = above_k;
            s.rounds = 0;
            s.capped = false;
            have_exact = true;  // ties already known from top-k
          } else if (R.exact) {
            const double wz = weight(key2f(R.hi), c.m, c.m_neginf);
            double nk = ceil((target - R.m_hi / scale) / wz);
            const uint32_t N = R.c_lo - R.c_hi;
            nk = fmin(fmax(nk, 1.0), static_cast<double>(N));
            s.tau = R.hi;
            s.n_keep = static_cast<uint32_t>(nk);
            s.count_above = R.c_hi;
            s.rounds = 0;
            s.capped = false;
            have_exact = true;
            ties_in_list = false;  // the own list may not hold this tie group
            if (warp == 0 && lane < static_cast<int>(c.C))
              F.ties[lane] = vld(F.rank_lo[lane]) - vld(F.rank_hi[lane]);
            __syncthreads();
            ties_known = true;
          } else if (!R.fits) {
            s.capped = true;
            s.rounds = 0;
          } else {
            if (!hit) {
              extract_range<DT>(c, R);
              if (warp == 0 && lane < static_cast<int>(c.C))
                F.rank_n[lane] = vld(F.rank_lo[lane]) - vld(F.rank_hi[lane]);
              __syncthreads();
            }
            gather<DT>(c, R.lo_all ? -INFINITY : pivot_f(R.lo), pivot_f(R.hi), R.lo_all, !hit);
            remote_done = true;
            s.lo = R.lo;
            s.hi = R.hi;
            s.c_lo = R.c_lo;
            s.c_hi = R.c_hi;
            s.c_above = R.c_hi;
            s.m_lo = R.m_lo / scale;
            s.m_hi = R.m_hi / scale;
            s.m_above = R.m_hi / scale;
            list_emit = hit;
            ties_in_list = true;
            local_search<DT, true>(c, s, target, value_pivots);
          }
        }
        rounds_p = static_cast<uint32_t>(s.rounds);
        if (s.capped) {
          sel_none = true;
          row_status = QRITA_ROW_SEARCH_CAP;
        }
        tau = s.tau;
        n_keep = s.n_keep;
        count_above = s.count_above;
        if (!sel_none && !have_exact) {
          count_ties_gathered<DT>(c, key2f(tau));
          ties_known = true;
        }
      }
    }
  }
  if (!remote_done) {
    cluster_sync_all();  // no CTA leaves while another may read its memory
    remote_done = true;
  }

  // ---- A8: boundary ties by lowest token id
  const float tau_f = key2f(tau);
  uint32_t my_first = 0, my_ties = 0;
  if (!sel_all && !sel_none && ties_known) {
    for (uint32_t l = 0; l < c.crank; ++l) my_first += vld(F.ties[l]);
    my_ties = vld(F.ties[c.crank]);
  }
  // tie_mode 0: none kept, 1: all kept, 2: the lowest-index keep_local
  int tie_mode = 0;
  if (!sel_all && !sel_none && my_ties > 0) {
    if (my_first + my_ties <= n_keep) tie_mode = 1;
    else if (my_first < n_keep) tie_mode = 2;
  }
  const uint32_t keep_local = (tie_mode == 2) ? (n_keep - my_first) : 0u;
  uint32_t idx_cut = 0;
  bool ordered_ties = false;
  if (tie_mode == 2) {
    if (ties_in_list) {
      idx_cut = tie_index_cut<DT>(c, tau_f, keep_local);
    } else {
      ordered_ties = true;
    }
  }

  // ---- A9: mask emission
  if (sel_all || sel_none || list_emit) {
    // fill the chunk's mask, then scatter the kept ids of the own list
    const uint8_t fill = sel_all ? 1 : 0;
    const uint32_t fill4 = sel_all ? 0x01010101u : 0u;
    const uintptr_t ma = reinterpret_cast<uintptr_t>(c.gmask);
    const int mh0 = static_cast<int>((16u - (ma & 15u)) & 15u);
    const int mh = mh0 < c.n ? mh0 : c.n;
    const int mb = (c.n - mh) / 16;
    const int mt = c.n - mh - mb * 16;
    if (tid < mh) c.gmask[tid] = fill;
    for (int i = tid; i < mb; i += kThreads)
      reinterpret_cast<uint4*>(c.gmask + mh)[i] = make_uint4(fill4, fill4, fill4, fill4);
    if (tid < mt) c.gmask[mh + mb * 16 + tid] = fill;
    if (list_emit && !sel_all && !sel_none) {
      __syncthreads();  // the fill is ordered before the scatter
      const uint32_t n = min(vld(F.own_n), c.ocap);
      for (uint32_t i = tid; i < n; i += kThreads) {
        const float x = c.own_val[i];
        bool keep = x > tau_f;
        if (x == tau_f) keep = (tie_mode == 1) || (tie_mode == 2 && c.own_idx[i] < idx_cut);
        if (keep) c.gmask[c.own_idx[i]] = 1;
      }
    }
  } else {
    // stream the chunk again: x > tau kept, ties by the rule above
    const uintptr_t mbp = reinterpret_cast<uintptr_t>(c.gmask + c.head_n);
    const bool vec_ok = (mbp % E) == 0;
    uint32_t running = 0;  // ties seen so far in index order (ordered_ties)
    auto byte_of = [&](float x, uint32_t idx, uint32_t& rank) -> uint8_t {
      if (x > tau_f) return 1;
      if (x == tau_f) {
        if (tie_mode == 1) return 1;
        if (tie_mode == 2) {
          if (ordered_ties) return (rank++ < keep_local) ? 1 : 0;
          return idx < idx_cut ? 1 : 0;
        }
      }
      return 0;
    };
    if (tid == 0) {
      for (int i = 0; i < c.head_n; ++i) {
        const float x = load_elem<DT>(c.gx + i * S);
        c.gmask[i] = byte_of(x, static_cast<uint32_t>(i), running);
      }
    }
    if (ordered_ties) {
      if (tid == 0) F.scan[0] = running;
      __syncthreads();
      running = vld(F.scan[0]);
      __syncthreads();
    }
    const int nb = c.body_units;
    for (int base = 0; base < nb; base += kThreads) {
      const int u = base + tid;
      const bool valid = u < nb;
      float xs[E];
      if (valid) {
        unpack<DT>(ldg16(c.gbody + 16 * static_cast<size_t>(u)), xs);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) xs[e] = -INFINITY;
      }
      uint32_t rank = 0;
      if (ordered_ties) {
        uint32_t mine = 0;
        if (valid) {
#pragma unroll
          for (int e = 0; e < E; ++e) mine += (xs[e] == tau_f) ? 1u : 0u;
        }
        uint32_t tot;
        const uint32_t ex = block_excl_scan(F, mine, &tot);
        rank = running + ex;
        running += tot;
      }
      if (!valid) continue;
      uint8_t bytes[E];
#pragma unroll
      for (int e = 0; e < E; ++e) bytes[e] = byte_of(xs[e], static_cast<uint32_t>(c.head_n + u * E + e), rank);
      uint8_t* dst = c.gmask + c.head_n + static_cast<size_t>(u) * E;
      if (vec_ok) {
        if constexpr (E == 4) {
          *reinterpret_cast<uint32_t*>(dst) =
              bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (static_cast<uint32_t>(bytes[3]) << 24);
        } else {
          const uint32_t w0 = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (static_cast<uint32_t>(bytes[3]) << 24);
          const uint32_t w1 = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (static_cast<uint32_t>(bytes[7]) << 24);
          *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = bytes[e];
      }
    }
    if (tid == 0) {
      for (int j = 0; j < c.tail_n; ++j) {
        const uint32_t idx = static_cast<uint32_t>(c.head_n + nb * E + j);
        const float x = load_elem<DT>(c.gbody + 16 * static_cast<size_t>(nb) + j * S);
        c.gmask[idx] = byte_of(x, idx, running);
      }
    }
  }

  // ---- row outputs (rank 0)
  if (c.crank == 0 && tid == 0) {
    if (P.row_status) P.row_status[r] = static_cast<int32_t>(row_status);
    if (P.row_info) {
      qrita_row_info_t info;
      info.mu = mu;
      info.sigma = sigma;
      info.threshold = trunc ? t : -INFINITY;
      info.row_max = row_max;
      info.survivors = trunc ? survivors : 0u;
      info.path = path;
      info.rounds_k = rounds_k;
      info.rounds_p = rounds_p;
      uint32_t kept;
      if (sel_none) kept = 0;
      else if (sel_all) kept = static_cast<uint32_t>(V);
      else kept = count_above + n_keep;
      info.boundary = sel_none ? NAN : (sel_all ? row_min : tau_f);
      info.n_boundary = (sel_none || sel_all) ? 0u : n_keep;
      info.kept = kept;
      info.status = row_status;
      info.z = z_used;
      info.passes = passes;
      info.reserved = 0u;
      P.row_info[r] = info;
    }
  }
}

}  // namespace

size_t smem_bytes(int ocap, int gcap) {
  size_t b = sizeof(Fixed);
  b += static_cast<size_t>(ocap) * 8u;  // own list: value + index
  b += static_cast<size_t>(gcap) * 8u;  // gathered set: value + tag
  return (b + 127u) & ~static_cast<size_t>(127u);
}

int max_smem_per_block() {
  int dev = 0;
  cudaGetDevice(&dev);
  int v = 0;
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return v;
}

int launch_select(const Params& prm, int dtype, size_t smem, qrita_stream_t stream) {
  const void* fn = dtype == QRITA_DTYPE_F32 ? reinterpret_cast<const void*>(&select_kernel<QRITA_DTYPE_F32>)
                                            : reinterpret_cast<const void*>(&select_kernel<QRITA_DTYPE_BF16>);
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return static_cast<int>(e);
  if (prm.C > 8) {
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return static_cast<int>(e);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(prm.B * prm.C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = reinterpret_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(prm.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == QRITA_DTYPE_F32) {
    e = cudaLaunchKernelEx(&cfg, select_kernel<QRITA_DTYPE_F32>, prm);
  } else {
    e = cudaLaunchKernelEx(&cfg, select_kernel<QRITA_DTYPE_BF16>, prm);
  }
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace qrita
