// Fused exact top-k / top-p selection kernel for GB300 (sm_103a).
//
// Method: Qrita technical summary (gist.science, paper 2602.01518),
// "Methodology" parts 1-2 and "Implementation details" (pipeline). One
// thread-block cluster handles one row: each of its C CTAs owns a contiguous
// chunk of the row, staged once from HBM into its shared memory with TMA bulk
// copies and kept there for every later pass, so the logits are read from HBM
// exactly once and the mask is written exactly once. Per-stage partial
// results are merged across the cluster through distributed shared memory.
//
// Stages (each ends with one cluster-wide merge):
//   A2  sample-block statistics mu, sigma (8 blocks of 64 logits per chunk)
//   A3  delta from the normal-quantile tables, t = mu + delta*sigma
//   A4  truncation pass: Z_t = {x >= t} compacted into a shared-memory list,
//       row max / min, NaN / +inf detection
//       (top-p rows without top-k: one more pass for Z = sum exp(x - m))
//   A5  hit / fallback decision (|Z_t| >= k, or mass(Z_t) >= p Z (1 + 1e-5))
//   A6  quaternary top-k pivot search over Z_t (hit) or the resident chunk
//       (fallback), tracking z_mn / N_zmn per pivot
//   A7  the same search with softmax mass in place of counts, for top-p
//   A8  boundary ties kept by lowest token id (prefix count across the
//       cluster ranks, then in index order inside the one straddling CTA)
//   A9  mask emission: one coalesced pass over the resident chunk
//
// Every decision is computed identically by every thread of the cluster
// from merged values, so control flow, and with it every cluster barrier, is
// uniform. The only waits are bounded mbarrier waits (an expired wait marks
// the row QRITA_ROW_TIMEOUT) and hardware cluster barriers.

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
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;  // 200 ms
constexpr int kSampleBlocks = 8;
constexpr int kSampleBlock = 64;  // kSampleBlocks * kSampleBlock == 2 * kThreads

#ifdef QRITA_TRACE
// Debug-only record of the search rounds of row 0 (built with -DQRITA_TRACE).
__device__ double g_trace[4096];
__device__ unsigned g_trace_n;
__device__ void trace_put(double a, double b, double c, double d, double e, double f, double g, double h,
                          double i, double j) {
  const unsigned n = g_trace_n;
  if (n + 10 > 4096) return;
  const double v[10] = {a, b, c, d, e, f, g, h, i, j};
  for (int t = 0; t < 10; ++t) g_trace[n + t] = v[t];
  g_trace_n = n + 10;
}
#endif

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
    return *reinterpret_cast<const float*>(p);
  } else {
    return __uint_as_float(static_cast<uint32_t>(*reinterpret_cast<const uint16_t*>(p)) << 16);
  }
}

template <int DT>
__device__ __forceinline__ void copy_elem(unsigned char* dst, const unsigned char* src) {
  if constexpr (DT == QRITA_DTYPE_F32) {
    *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
  } else {
    *reinterpret_cast<uint16_t*>(dst) = *reinterpret_cast<const uint16_t*>(src);
  }
}

// ---------------------------------------------------------------------------
// Shared-memory layout
// ---------------------------------------------------------------------------
struct alignas(16) PivotPart {  // one pivot's partial (exchanged between ranks)
  double mass;                  // softmax mass of the elements above the pivot
  uint32_t cnt;                 // elements above the pivot
  float z;                      // z_mn: smallest element above the pivot
  uint32_t nz;                  // N_zmn: how many elements equal z
  uint32_t pad;
};

struct alignas(16) Slot {  // what one CTA publishes for one merge
  PivotPart pv[3];
  double d[2];
  float f[4];
  uint32_t u[4];
};

struct alignas(16) PAccS {  // per-warp pivot partial (block reduction scratch)
  uint32_t cnt;
  float z;
  uint32_t nz;
  float mhi, mlo;
  uint32_t pad[3];
};

struct alignas(16) Fixed {
  uint64_t bars[kMaxPieces];
  Slot slots[2];
  Slot mg;  // merged result of the latest merge
  PAccS red[kWarps][3];
  float redf[kWarps][8];
  uint32_t redu[kWarps][4];
  uint32_t rank_cnt[3][kMaxCluster];  // latest round, per rank and pivot
  float rank_z[3][kMaxCluster];
  uint32_t rank_nz[3][kMaxCluster];
  uint32_t rank_surv[kMaxCluster];   // survivors per rank
  uint32_t cnt_lo[kMaxCluster];      // per-rank count above the search's lo
  uint32_t cnt_hi[kMaxCluster];      // per-rank count above the search's hi
  uint32_t ties[kMaxCluster];        // per-rank count of boundary-valued elements
  uint32_t scan[kWarps];
  uint32_t list_n;
  uint32_t err;
};

// Read of shared state another thread wrote before a barrier. Every such read
// goes through a volatile shared load so the compiler can neither reuse an
// earlier load of the same word nor move the load across the barrier.
template <typename T>
__device__ __forceinline__ T vld(const T& r) {
  return *reinterpret_cast<const volatile T*>(&r);
}

// ---------------------------------------------------------------------------
// Pivot accumulators
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

// Per-element update of the three pivots. Unused pivots are +inf (nothing
// exceeds them). Predicated, so the warp never diverges here.
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

// Softmax weight of x for row max m. A row whose max is -inf holds only
// -inf, and equal logits get equal weight 1.
__device__ __forceinline__ float weight(float x, float m, bool m_neginf) {
  return m_neginf ? 1.0f : expf(x - m);
}

// ---------------------------------------------------------------------------
// Warp / block helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

// Exclusive scan of a per-thread count over the block, in thread order.
// Returns the exclusive prefix; *total receives the block total.
__device__ __forceinline__ uint32_t block_excl_scan(Fixed& F, uint32_t v, uint32_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(kFull, incl, o);
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

// Warp-aggregated append of up to E flagged values to the shared list.
// Every lane of the warp must call it (convergent).
template <int E>
__device__ __forceinline__ void warp_append(Fixed& F, float* list_x, float* list_w, uint32_t cap,
                                            const float (&xs)[E], const float (&ws)[E],
                                            uint32_t bits, bool with_w) {
  const int lane = threadIdx.x & 31;
  const uint32_t c = __popc(bits);
  if (__ballot_sync(kFull, c != 0) == 0) return;
  uint32_t incl = c;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    uint32_t t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  const uint32_t total = __shfl_sync(kFull, incl, 31);
  uint32_t base = 0;
  if (lane == 31) base = atomicAdd(&F.list_n, total);
  base = __shfl_sync(kFull, base, 31);
  uint32_t pos = base + incl - c;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    if ((bits >> e) & 1u) {
      if (pos < cap) {
        list_x[pos] = xs[e];
        if (with_w) list_w[pos] = ws[e];
      }
      ++pos;
    }
  }
}

// ---------------------------------------------------------------------------
// Pivot choice: 25/50/75 % of the current range (lo, hi] of keys
// ---------------------------------------------------------------------------
// Value-space quartiles (the pages' reading of "25/50/75 % of the search
// range") when both ends are finite floats and the previous value-space
// round shrank the key range at least by half; otherwise quartiles of the
// 32-bit key range, which always shrink it fourfold. Returns how many
// pivots are set (1..3); unused pivots are +inf.
__device__ __forceinline__ int choose_pivots(uint32_t lo, uint32_t hi, bool value_ok,
                                             uint32_t (&q)[3], float (&qf)[3], bool* used_value) {
  const uint32_t span = hi - lo;  // >= 2
  int np;
  *used_value = false;
  if (span <= 4u) {
    np = static_cast<int>(span) - 1;
    for (int j = 0; j < 3; ++j) q[j] = lo + 1u + static_cast<uint32_t>(j < np ? j : np - 1);
  } else {
    np = 3;
    bool done = false;
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
          done = true;
          *used_value = true;
        }
      }
    }
    if (!done) {
      for (int j = 0; j < 3; ++j)
        q[j] = lo + static_cast<uint32_t>((static_cast<uint64_t>(span) * (j + 1)) >> 2);
    }
  }
  for (int j = 0; j < 3; ++j) qf[j] = (j < np) ? pivot_f(q[j]) : INFINITY;
  return np;
}

// ---------------------------------------------------------------------------
// The kernel
// ---------------------------------------------------------------------------
template <int DT>
struct Ctx {
  static constexpr int E = Elem<DT>::kPerUnit;
  static constexpr int S = Elem<DT>::kBytes;
  Fixed* F;
  float* list_x;
  float* list_w;
  const unsigned char* sbody;  // shared: first 16-byte unit of the chunk body
  uint32_t cap;
  int n, head_n, body_units, tail_n;
  uint32_t C, crank;
  float m;
  bool m_neginf;
  int ph;  // merge counter (slot parity)
};

// Element e of the chunk in shared memory, by chunk-local index class.
template <int DT>
__device__ __forceinline__ float head_elem(const Ctx<DT>& c, int i) {
  return load_elem<DT>(c.sbody - (c.head_n - i) * Ctx<DT>::S);
}
template <int DT>
__device__ __forceinline__ float tail_elem(const Ctx<DT>& c, int j) {
  return load_elem<DT>(c.sbody + 16 * c.body_units + j * Ctx<DT>::S);
}

// Publish pivot partials, cluster barrier, merge all ranks (warp 0), and
// broadcast through F->mg. above_cnt / above_mass account for this CTA's
// elements above its list's range (list mode), which exceed every pivot.
template <int DT, bool MASS>
__device__ __forceinline__ void reduce_merge_pivots(Ctx<DT>& c, PAcc (&acc)[3], uint32_t above_cnt,
                                                    double above_mass) {
  Fixed& F = *c.F;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int j = 0; j < 3; ++j) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      PAcc t = pacc_shfl_xor<MASS>(acc[j], o);
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
  Slot& my = F.slots[c.ph & 1];
  if (warp == 0) {
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
        PAcc t = pacc_shfl_xor<MASS>(a, o);
        pacc_combine<MASS>(a, t);
      }
      if (lane == 0) {
        my.pv[j].cnt = a.cnt + above_cnt;
        my.pv[j].z = a.z;
        my.pv[j].nz = a.nz;
        my.pv[j].mass = MASS ? (f2_value(a.m) + above_mass) : 0.0;
      }
    }
  }
  cluster_sync_all();
  if (warp == 0) {
    const uint32_t base = smem_u32(&my);
#pragma unroll
    for (int j = 0; j < 3; ++j) {
      uint32_t cnt = 0, nz = 0;
      float z = INFINITY;
      double mass = 0.0;
      if (lane < static_cast<int>(c.C)) {
        const uint32_t a = map_rank(base + j * static_cast<uint32_t>(sizeof(PivotPart)), lane);
        mass = ld_dsmem_f64(a);
        cnt = ld_dsmem_u32(a + 8);
        z = ld_dsmem_f32(a + 12);
        nz = ld_dsmem_u32(a + 16);
        F.rank_cnt[j][lane] = cnt;
        F.rank_z[j][lane] = z;
        F.rank_nz[j][lane] = nz;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const uint32_t cnt2 = __shfl_xor_sync(kFull, cnt, o);
        const float z2 = __shfl_xor_sync(kFull, z, o);
        const uint32_t nz2 = __shfl_xor_sync(kFull, nz, o);
        const double m2 = __shfl_xor_sync(kFull, mass, o);
        cnt += cnt2;
        if (z2 < z) {
          z = z2;
          nz = nz2;
        } else if (z2 == z) {
          nz += nz2;
        }
        mass += m2;
      }
      if (lane == 0) {
        F.mg.pv[j].cnt = cnt;
        F.mg.pv[j].z = z;
        F.mg.pv[j].nz = nz;
        F.mg.pv[j].mass = mass;
      }
    }
  }
  __syncthreads();
  ++c.ph;
}

// One quaternary round's scan. List mode scans the shared list (values and,
// for MASS, cached weights); chunk mode scans the resident chunk and, when
// `compact` is set, also appends the elements in (clo, chi] (and their
// weights) to the list, which then covers that range. lo_all means the lower
// end lies below key(-inf): every element passes it (its float is a NaN).
template <int DT, bool MASS>
__device__ __forceinline__ void scan_round(Ctx<DT>& c, bool list_mode, uint32_t list_len,
                                           const float (&qf)[3], PAcc (&acc)[3], bool compact,
                                           float clo_f, float chi_f, bool lo_all = false) {
  constexpr int E = Ctx<DT>::E;
  Fixed& F = *c.F;
  const int tid = threadIdx.x;
#pragma unroll
  for (int j = 0; j < 3; ++j) pacc_init(acc[j]);
  if (list_mode) {
    for (uint32_t i = tid; i < list_len; i += kThreads) {
      const float x = c.list_x[i];
      const float w = MASS ? c.list_w[i] : 0.f;
      pacc_update<MASS>(acc, qf, x, w);
    }
    return;
  }
  const int iters = (c.body_units + kThreads - 1) / kThreads;
  for (int it = 0; it < iters; ++it) {
    const int u = it * kThreads + tid;
    float xs[E], ws[E];
    uint32_t bits = 0;
    if (u < c.body_units) {
      const uint4 v = *reinterpret_cast<const uint4*>(c.sbody + 16 * u);
      unpack<DT>(v, xs);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        ws[e] = MASS ? weight(xs[e], c.m, c.m_neginf) : 0.f;
        pacc_update<MASS>(acc, qf, xs[e], ws[e]);
        if (compact && (lo_all || xs[e] > clo_f) && !(xs[e] > chi_f)) bits |= 1u << e;
      }
    } else {
#pragma unroll
      for (int e = 0; e < E; ++e) {
        xs[e] = 0.f;
        ws[e] = 0.f;
      }
    }
    if (compact) warp_append<E>(F, c.list_x, c.list_w, c.cap, xs, ws, bits, MASS);
  }
  // head and tail elements (fewer than 2E): one element per thread
  {
    float xs[1], ws[1];
    uint32_t bits = 0;
    const int h = tid;
    xs[0] = 0.f;
    ws[0] = 0.f;
    if (h < c.head_n + c.tail_n) {
      xs[0] = (h < c.head_n) ? head_elem(c, h) : tail_elem(c, h - c.head_n);
      ws[0] = MASS ? weight(xs[0], c.m, c.m_neginf) : 0.f;
      pacc_update<MASS>(acc, qf, xs[0], ws[0]);
      if (compact && (lo_all || xs[0] > clo_f) && !(xs[0] > chi_f)) bits = 1u;
    }
    if (compact) warp_append<1>(F, c.list_x, c.list_w, c.cap, xs, ws, bits, MASS);
  }
}

// Search state shared by the top-k (count) and top-p (mass) searches.
struct Search {
  uint32_t lo, hi;     // keys: count(> lo) >= target > count(> hi) (or mass)
  uint32_t C_lo, C_hi; // row-level counts above lo / hi
  double M_lo, M_hi;   // row-level masses above lo / hi (MASS only)
  double myM_hi;       // this CTA's mass above hi (MASS only)
  // list coverage: the list holds exactly this CTA's elements in (list_lo, list_hi]
  bool list_mode;
  uint32_t list_len;
  uint32_t above_cnt;  // this CTA's elements above list_hi
  double above_mass;
  // result
  uint32_t tau;        // boundary key
  uint32_t n_keep;     // boundary duplicates kept
  uint32_t count_above;  // row-level count strictly above tau
  int rounds;
  bool capped;
};

// Quaternary pivot search (A6 for counts, A7 for mass). On return F->ties
// holds every rank's count of elements equal to the boundary and s.tau,
// s.n_keep, s.count_above are set. target is k (counts) or p*Z (mass).
template <int DT, bool MASS>
__device__ void quaternary_search(Ctx<DT>& c, Search& s, double target, bool value_pivots) {
  Fixed& F = *c.F;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  bool value_ok = value_pivots;
  s.rounds = 0;
  s.capped = false;
  for (;;) {
    __syncthreads();  // cnt_lo / cnt_hi saved by warp 0 last round are visible
    if (s.hi - s.lo <= 1u) {
      // (lo, hi] holds one key, so the boundary value is hi.
      s.tau = s.hi;
      s.count_above = s.C_hi;
      const uint32_t N = s.C_lo - s.C_hi;
      if (MASS) {
        const double wz = weight(key2f(s.hi), c.m, c.m_neginf);
        double nk = ceil((target - s.M_hi) / wz);
        nk = fmin(fmax(nk, 1.0), static_cast<double>(N));
        s.n_keep = static_cast<uint32_t>(nk);
      } else {
        s.n_keep = static_cast<uint32_t>(target) - s.C_hi;
      }
      if (warp == 0 && lane < static_cast<int>(c.C)) F.ties[lane] = vld(F.cnt_lo[lane]) - vld(F.cnt_hi[lane]);
      break;
    }
    if (s.rounds >= kMaxRounds) {
      s.capped = true;
      s.tau = s.hi;
      s.n_keep = 0;
      s.count_above = 0;
      if (warp == 0 && lane < static_cast<int>(c.C)) F.ties[lane] = 0;
      break;
    }
    uint32_t q[3];
    float qf[3];
    bool used_value = false;
    const int np = choose_pivots(s.lo, s.hi, value_ok, q, qf, &used_value);
    const uint32_t old_span = s.hi - s.lo;

    // Chunk-mode CTAs compact the current range once it fits the list.
    bool compact = false, lo_all = false;
    float clo_f = 0.f, chi_f = 0.f;
    if (!s.list_mode) {
      const uint32_t in_range = vld(F.cnt_lo[c.crank]) - vld(F.cnt_hi[c.crank]);
      if (in_range <= c.cap) {
        compact = true;
        lo_all = s.lo < kKeyNegInf;
        clo_f = lo_all ? -INFINITY : pivot_f(s.lo);
        chi_f = pivot_f(s.hi);
        if (threadIdx.x == 0) F.list_n = 0;
        __syncthreads();
      }
    }
    PAcc acc[3];
    scan_round<DT, MASS>(c, s.list_mode, s.list_len, qf, acc, compact, clo_f, chi_f, lo_all);
    const uint32_t add_cnt = s.list_mode ? s.above_cnt : 0u;
    const double add_mass = s.list_mode ? s.above_mass : 0.0;
    reduce_merge_pivots<DT, MASS>(c, acc, add_cnt, add_mass);
    if (compact) {
      s.list_mode = true;
      s.list_len = vld(F.list_n);  // a barrier separates it from the appends
      s.above_cnt = vld(F.cnt_hi[c.crank]);
      s.above_mass = MASS ? s.myM_hi : 0.0;
    }
    ++s.rounds;

#ifdef QRITA_TRACE
    if (c.crank == 0 && threadIdx.x == 0 && blockIdx.x < c.C) {
      for (int j = 0; j < np; ++j) {
        const double wz = MASS ? static_cast<double>(weight(F.mg.pv[j].z, c.m, c.m_neginf)) : 1.0;
        trace_put(static_cast<double>(s.rounds), static_cast<double>(s.lo), static_cast<double>(s.hi),
                  static_cast<double>(q[j]), static_cast<double>(F.mg.pv[j].cnt), F.mg.pv[j].z,
                  static_cast<double>(F.mg.pv[j].nz), F.mg.pv[j].mass, target, wz);
      }
    }
#endif
    // Walk the pivots upward: terminate at the first pivot whose z_mn is the
    // boundary (the condition as read in the design notes: above(q) reaches
    // the target and above(q) minus the z_mn duplicates does not), else move
    // lo up while the pivot still reaches the target, else set hi.
    int done_j = -1, lo_j = -1, hi_j = -1;
    for (int j = 0; j < np; ++j) {
      PivotPart pv;
      pv.mass = vld(F.mg.pv[j].mass);
      pv.cnt = vld(F.mg.pv[j].cnt);
      pv.z = vld(F.mg.pv[j].z);
      pv.nz = vld(F.mg.pv[j].nz);
      const double above = MASS ? pv.mass : static_cast<double>(pv.cnt);
      if (above >= target) {
        const double wz = MASS ? static_cast<double>(weight(pv.z, c.m, c.m_neginf)) : 1.0;
        const double below_z = above - static_cast<double>(pv.nz) * wz;
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
#ifdef QRITA_TRACE
    if (c.crank == 0 && threadIdx.x == 0 && blockIdx.x < c.C)
      trace_put(-1.0, static_cast<double>(done_j), static_cast<double>(lo_j), static_cast<double>(hi_j), 0, 0, 0, 0, 0, 0);
#endif
    if (done_j >= 0) {
      PivotPart pv;
      pv.mass = vld(F.mg.pv[done_j].mass);
      pv.cnt = vld(F.mg.pv[done_j].cnt);
      pv.z = vld(F.mg.pv[done_j].z);
      pv.nz = vld(F.mg.pv[done_j].nz);
      s.tau = f2key(pv.z);
      s.count_above = pv.cnt - pv.nz;
      if (MASS) {
        const double wz = weight(pv.z, c.m, c.m_neginf);
        double nk = ceil((target - (pv.mass - static_cast<double>(pv.nz) * wz)) / wz);
        nk = fmin(fmax(nk, 1.0), static_cast<double>(pv.nz));
        s.n_keep = static_cast<uint32_t>(nk);
      } else {
        s.n_keep = static_cast<uint32_t>(target) - s.count_above;
      }
      if (warp == 0 && lane < static_cast<int>(c.C))
        F.ties[lane] = (vld(F.rank_z[done_j][lane]) == pv.z) ? vld(F.rank_nz[done_j][lane]) : 0u;
      break;
    }
    if (lo_j >= 0) {
      s.lo = q[lo_j];
      s.C_lo = vld(F.mg.pv[lo_j].cnt);
      s.M_lo = vld(F.mg.pv[lo_j].mass);
      if (warp == 0 && lane < static_cast<int>(c.C)) F.cnt_lo[lane] = vld(F.rank_cnt[lo_j][lane]);
    }
    if (hi_j >= 0) {
      s.hi = q[hi_j];
      s.C_hi = vld(F.mg.pv[hi_j].cnt);
      s.M_hi = vld(F.mg.pv[hi_j].mass);
      if (warp == 0 && lane < static_cast<int>(c.C)) F.cnt_hi[lane] = vld(F.rank_cnt[hi_j][lane]);
    }
    // myM_hi needs this CTA's own mass at the new hi: it is the value this
    // CTA published, still in its slot of the merge just done.
    if (MASS && hi_j >= 0) s.myM_hi = vld(F.slots[(c.ph - 1) & 1].pv[hi_j].mass);
    if (used_value) {
      value_ok = (s.hi - s.lo) <= old_span / 2u;
    } else {
      value_ok = value_pivots;
    }
  }
  __syncthreads();  // F.ties visible
}

template <int DT>
__global__ void __launch_bounds__(kThreads) select_kernel(const __grid_constant__ Params P) {
  constexpr int E = Ctx<DT>::E;
  constexpr int S = Ctx<DT>::S;
  extern __shared__ __align__(128) unsigned char smem[];
  Fixed& F = *reinterpret_cast<Fixed*>(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  Ctx<DT> c;
  c.F = &F;
  c.cap = static_cast<uint32_t>(P.cap);
  c.list_x = reinterpret_cast<float*>(smem + sizeof(Fixed));
  c.list_w = c.list_x + P.cap;
  unsigned char* sdata = reinterpret_cast<unsigned char*>(c.list_w + P.cap);
  unsigned char* sbody = sdata + 16;
  c.sbody = sbody;
  c.C = static_cast<uint32_t>(P.C);
  c.crank = cluster_rank();
  c.ph = 0;

  const int64_t r = blockIdx.x / P.C;
  const int32_t V = P.V;
  const int64_t c0 = static_cast<int64_t>(c.crank) * P.chunk;
  const int64_t rem = static_cast<int64_t>(V) - c0;
  c.n = static_cast<int>(rem <= 0 ? 0 : (rem < P.chunk ? rem : P.chunk));
  const unsigned char* gx =
      static_cast<const unsigned char*>(P.logits) + (static_cast<size_t>(r) * V + c0) * S;
  uint8_t* gmask = P.mask + static_cast<size_t>(r) * V + c0;

  // Chunk geometry: head elements up to the first 16-byte boundary of the
  // global row, whole 16-byte units, tail elements.
  {
    const uintptr_t ga = reinterpret_cast<uintptr_t>(gx);
    int h = static_cast<int>(((16u - (ga & 15u)) & 15u) / S);
    c.head_n = h < c.n ? h : c.n;
    c.body_units = (c.n - c.head_n) * S / 16;
    c.tail_n = c.n - c.head_n - c.body_units * E;
  }
  const unsigned char* gbody = gx + c.head_n * S;
  const int piece_units = kPieceBytes / 16;
  const int npieces = (c.body_units + piece_units - 1) / piece_units;

  // ---- stage loads: TMA bulk copies of the body, plain loads of head/tail
  if (tid == 0) {
    F.list_n = 0;
    F.err = 0;
    for (int pc = 0; pc < npieces; ++pc) mbar_init(smem_u32(&F.bars[pc]), 1);
    fence_mbar_init();
    for (int pc = 0; pc < npieces; ++pc) {
      const int u0 = pc * piece_units;
      const int nu = min(piece_units, c.body_units - u0);
      const uint32_t bytes = static_cast<uint32_t>(nu) * 16u;
      const uint32_t bar = smem_u32(&F.bars[pc]);
      mbar_expect_tx(bar, bytes);
      bulk_g2s(smem_u32(sbody + 16 * u0), gbody + 16 * u0, bytes, bar);
    }
  }
  if (tid < c.head_n) copy_elem<DT>(sbody - (c.head_n - tid) * S, gx + tid * S);
  if (tid < c.tail_n)
    copy_elem<DT>(sbody + 16 * c.body_units + tid * S, gbody + 16 * c.body_units + tid * S);

  // ---- row parameters (uniform)
  int32_t kr = P.k ? P.k[r] : 0;
  const float pr = P.p ? P.p[r] : 1.0f;
  bool k_on = kr >= 1 && kr < V;
  bool p_on = pr < 1.0f;  // NaN compares false: off
  if (p_on && !(pr > 0.0f)) {
    // p <= 0 keeps exactly one token: the same set as k = 1.
    p_on = false;
    if (V > 1) {
      k_on = true;
      kr = 1;
    }
  }
  const bool keep_all = !k_on && !p_on;

  // ---- A2: sample-block statistics (plain global loads, overlapping the copies)
  {
    float sn = 0.f, sx = 0.f, sxx = 0.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int sidx = tid + j * kThreads;  // 0 .. 511
      int idx;
      if (c.n <= kSampleBlocks * kSampleBlock) {
        idx = sidx;
      } else {
        idx = (sidx / kSampleBlock) * (c.n / kSampleBlocks) + (sidx % kSampleBlock);
      }
      if (idx < c.n) {
        const float x = load_elem<DT>(gx + static_cast<size_t>(idx) * S);
        if (isfinite(x)) {
          sn += 1.f;
          sx += x;
          sxx += x * x;
        }
      }
    }
    sn = warp_sum_f(sn);
    sx = warp_sum_f(sx);
    sxx = warp_sum_f(sxx);
    if (lane == 0) {
      F.redf[warp][0] = sn;
      F.redf[warp][1] = sx;
      F.redf[warp][2] = sxx;
    }
  }
  __syncthreads();  // also: barriers initialised, head/tail stored, list_n zeroed
  if (warp == 0) {
    float a = lane < kWarps ? vld(F.redf[lane][0]) : 0.f;
    float b = lane < kWarps ? vld(F.redf[lane][1]) : 0.f;
    float d = lane < kWarps ? vld(F.redf[lane][2]) : 0.f;
    a = warp_sum_f(a);
    b = warp_sum_f(b);
    d = warp_sum_f(d);
    if (lane == 0) {
      Slot& my = F.slots[c.ph & 1];
      my.f[0] = a;
      my.f[1] = b;
      my.f[2] = d;
    }
  }
  cluster_sync_all();  // first cluster barrier: every CTA of the cluster is running
  if (warp == 0) {
    double a = 0.0, b = 0.0, d = 0.0;
    if (lane < static_cast<int>(c.C)) {
      const uint32_t base = map_rank(smem_u32(&F.slots[c.ph & 1].f[0]), lane);
      a = ld_dsmem_f32(base);
      b = ld_dsmem_f32(base + 4);
      d = ld_dsmem_f32(base + 8);
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) {
      a += __shfl_xor_sync(kFull, a, o);
      b += __shfl_xor_sync(kFull, b, o);
      d += __shfl_xor_sync(kFull, d, o);
    }
    if (lane == 0) {
      // a = finite samples, b = their sum, d = their sum of squares
      const double mean = a > 0.0 ? b / a : 0.0;
      const double var = a > 0.0 ? fmax(d / a - mean * mean, 0.0) : 0.0;
      F.mg.f[1] = static_cast<float>(mean);
      F.mg.f[2] = static_cast<float>(sqrt(var));
      F.mg.u[0] = a > 0.0 ? 1u : 0u;
    }
  }
  __syncthreads();
  ++c.ph;
  const float mu = vld(F.mg.f[1]);
  const float sigma = vld(F.mg.f[2]);
  const bool have_sample = vld(F.mg.u[0]) != 0u;

  // ---- A3: delta from the normal-quantile tables, threshold t
  bool trunc = false;
  float t = -INFINITY;
  if (!(P.flags & QRITA_FLAG_NO_TRUNCATION) && have_sample && !keep_all) {
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

  // ---- A4: truncation pass over the resident chunk (waits for the copies)
  {
    float vmax = -INFINITY, vmin = INFINITY, smin = INFINITY;
    uint32_t smin_n = 0;
    bool timed_out = false;
    const int it_per_piece = piece_units / kThreads;
    const int iters = (c.body_units + kThreads - 1) / kThreads;
    for (int it = 0; it < iters; ++it) {
      if (it % it_per_piece == 0) {
        if (!mbar_wait_bounded(smem_u32(&F.bars[it / it_per_piece]), 0, kWaitLimitNs)) timed_out = true;
      }
      const int u = it * kThreads + tid;
      float xs[E], ws[E];
      uint32_t bits = 0;
      if (u < c.body_units) {
        const uint4 v = *reinterpret_cast<const uint4*>(sbody + 16 * u);
        unpack<DT>(v, xs);
#pragma unroll
        for (int e = 0; e < E; ++e) {
          vmax = fmax_nan(vmax, xs[e]);
          vmin = fminf(vmin, xs[e]);
          if (trunc && xs[e] >= t) {
            bits |= 1u << e;
            if (xs[e] < smin) {
              smin = xs[e];
              smin_n = 1;
            } else if (xs[e] == smin) {
              ++smin_n;
            }
          }
          ws[e] = 0.f;
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          xs[e] = 0.f;
          ws[e] = 0.f;
        }
      }
      if (trunc) warp_append<E>(F, c.list_x, c.list_w, c.cap, xs, ws, bits, false);
    }
    {
      float xs[1] = {0.f}, ws[1] = {0.f};
      uint32_t bits = 0;
      if (tid < c.head_n + c.tail_n) {
        xs[0] = (tid < c.head_n) ? head_elem(c, tid) : tail_elem(c, tid - c.head_n);
        vmax = fmax_nan(vmax, xs[0]);
        vmin = fminf(vmin, xs[0]);
        if (trunc && xs[0] >= t) {
          bits = 1u;
          if (xs[0] < smin) {
            smin = xs[0];
            smin_n = 1;
          } else if (xs[0] == smin) {
            ++smin_n;
          }
        }
      }
      if (trunc) warp_append<1>(F, c.list_x, c.list_w, c.cap, xs, ws, bits, false);
    }
    if (timed_out) atomicOr(&F.err, 1u);
    // block reduce: max (NaN-propagating), min, (smin, smin_n)
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
    }
    if (lane == 0) {
      F.redf[warp][0] = vmax;
      F.redf[warp][1] = vmin;
      F.redf[warp][2] = smin;
      F.redu[warp][0] = smin_n;
    }
    __syncthreads();
    if (warp == 0) {
      float a = lane < kWarps ? vld(F.redf[lane][0]) : -INFINITY;
      float b = lane < kWarps ? vld(F.redf[lane][1]) : INFINITY;
      float s = lane < kWarps ? vld(F.redf[lane][2]) : INFINITY;
      uint32_t sn = lane < kWarps ? vld(F.redu[lane][0]) : 0u;
#pragma unroll
      for (int o = kWarps / 2; o > 0; o >>= 1) {
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
      }
      if (lane == 0) {
        Slot& my = F.slots[c.ph & 1];
        my.f[0] = a;
        my.f[1] = b;
        my.f[2] = s;
        my.u[0] = sn;
        my.u[1] = vld(F.list_n);
        my.u[2] = F.err;
      }
    }
    cluster_sync_all();
    if (warp == 0) {
      float a = -INFINITY, b = INFINITY, s = INFINITY;
      uint32_t sn = 0, surv = 0, err = 0, ovf = 0;
      if (lane < static_cast<int>(c.C)) {
        const uint32_t base = map_rank(smem_u32(&F.slots[c.ph & 1].f[0]), lane);
        a = ld_dsmem_f32(base);
        b = ld_dsmem_f32(base + 4);
        s = ld_dsmem_f32(base + 8);
        const uint32_t ub = map_rank(smem_u32(&F.slots[c.ph & 1].u[0]), lane);
        sn = ld_dsmem_u32(ub);
        surv = ld_dsmem_u32(ub + 4);
        err = ld_dsmem_u32(ub + 8);
        ovf = surv > c.cap ? 1u : 0u;
        F.rank_surv[lane] = surv;
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
        err |= __shfl_xor_sync(kFull, err, o);
        ovf |= __shfl_xor_sync(kFull, ovf, o);
      }
      if (lane == 0) {
        F.mg.f[0] = a;
        F.mg.f[1] = b;
        F.mg.f[2] = s;
        F.mg.u[0] = sn;
        F.mg.u[1] = surv;
        F.mg.u[2] = err;
        F.mg.u[3] = ovf;
      }
    }
    __syncthreads();
    ++c.ph;
  }
  const float row_max = vld(F.mg.f[0]);
  const float row_min = vld(F.mg.f[1]);
  const float surv_min = vld(F.mg.f[2]);
  const uint32_t surv_min_n = vld(F.mg.u[0]);
  const uint32_t survivors = vld(F.mg.u[1]);
  const bool timed_out = vld(F.mg.u[2]) != 0u;
  const bool overflow = vld(F.mg.u[3]) != 0u;
  const bool nonfinite = isnan(row_max) || row_max == INFINITY;
  const bool invalid = nonfinite || timed_out;
  c.m = row_max;
  c.m_neginf = (row_max == -INFINITY);
  const uint32_t my_surv = vld(F.list_n);

  uint32_t path = (k_on ? QRITA_PATH_TOPK : 0u) | (p_on ? QRITA_PATH_TOPP : 0u) |
                  (trunc ? QRITA_PATH_TRUNC : 0u) | (overflow ? QRITA_PATH_OVERFLOW : 0u) |
                  (keep_all ? QRITA_PATH_KEEP_ALL : 0u);
  const bool force_fb = (P.flags & QRITA_FLAG_FORCE_FALLBACK) != 0u;
  const bool value_pivots = (P.flags & QRITA_FLAG_KEY_PIVOTS) == 0u;

  // Final selection: keep key > tau, plus the n_keep lowest-id elements equal
  // to tau. F.ties[rank] = elements equal to tau in that rank's chunk.
  uint32_t tau = 0, n_keep = 0, count_above = 0;
  uint32_t rounds_k = 0, rounds_p = 0;
  uint32_t row_status = QRITA_ROW_OK;
  double z_used = 0.0;
  bool sel_all = keep_all;
  bool sel_none = false;

  // list coverage of the survivor list: (key(t) - 1, +inf)
  Search s;
  s.list_mode = false;
  s.list_len = 0;
  s.above_cnt = 0;
  s.above_mass = 0.0;
  s.myM_hi = 0.0;

  double Z = 0.0, Mt = 0.0;
  if (invalid) {
    sel_none = true;
    sel_all = false;
    row_status = nonfinite ? QRITA_ROW_NONFINITE : QRITA_ROW_TIMEOUT;
  } else if (!keep_all) {
    // ---- top-p rows without top-k: Z = sum exp(x - m), and the survivors' mass
    if (p_on && !k_on) {
      F2 zs = {0.f, 0.f}, ms = {0.f, 0.f};
      const int iters = (c.body_units + kThreads - 1) / kThreads;
      for (int it = 0; it < iters; ++it) {
        const int u = it * kThreads + tid;
        if (u < c.body_units) {
          float xs[E];
          unpack<DT>(*reinterpret_cast<const uint4*>(sbody + 16 * u), xs);
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const float w = weight(xs[e], c.m, c.m_neginf);
            f2_add(zs, w);
            f2_add(ms, (trunc && xs[e] >= t) ? w : 0.f);
          }
        }
      }
      if (tid < c.head_n + c.tail_n) {
        const float x = (tid < c.head_n) ? head_elem(c, tid) : tail_elem(c, tid - c.head_n);
        const float w = weight(x, c.m, c.m_neginf);
        f2_add(zs, w);
        f2_add(ms, (trunc && x >= t) ? w : 0.f);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        F2 a, b;
        a.hi = __shfl_xor_sync(kFull, zs.hi, o);
        a.lo = __shfl_xor_sync(kFull, zs.lo, o);
        b.hi = __shfl_xor_sync(kFull, ms.hi, o);
        b.lo = __shfl_xor_sync(kFull, ms.lo, o);
        zs = f2_merge(zs, a);
        ms = f2_merge(ms, b);
      }
      if (lane == 0) {
        F.redf[warp][0] = zs.hi;
        F.redf[warp][1] = zs.lo;
        F.redf[warp][2] = ms.hi;
        F.redf[warp][3] = ms.lo;
      }
      __syncthreads();
      if (warp == 0) {
        F2 a = {0.f, 0.f}, b = {0.f, 0.f};
        if (lane < kWarps) {
          a.hi = vld(F.redf[lane][0]);
          a.lo = vld(F.redf[lane][1]);
          b.hi = vld(F.redf[lane][2]);
          b.lo = vld(F.redf[lane][3]);
        }
#pragma unroll
        for (int o = kWarps / 2; o > 0; o >>= 1) {
          F2 a2, b2;
          a2.hi = __shfl_xor_sync(kFull, a.hi, o);
          a2.lo = __shfl_xor_sync(kFull, a.lo, o);
          b2.hi = __shfl_xor_sync(kFull, b.hi, o);
          b2.lo = __shfl_xor_sync(kFull, b.lo, o);
          a = f2_merge(a, a2);
          b = f2_merge(b, b2);
        }
        if (lane == 0) {
          F.slots[c.ph & 1].d[0] = f2_value(a);
          F.slots[c.ph & 1].d[1] = f2_value(b);
        }
      }
      cluster_sync_all();
      if (warp == 0) {
        double a = 0.0, b = 0.0;
        if (lane < static_cast<int>(c.C)) {
          const uint32_t base = map_rank(smem_u32(&F.slots[c.ph & 1].d[0]), lane);
          a = ld_dsmem_f64(base);
          b = ld_dsmem_f64(base + 8);
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) {
          a += __shfl_xor_sync(kFull, a, o);
          b += __shfl_xor_sync(kFull, b, o);
        }
        if (lane == 0) {
          F.mg.d[0] = a;
          F.mg.d[1] = b;
        }
      }
      __syncthreads();
      ++c.ph;
      Z = vld(F.mg.d[0]);
      Mt = vld(F.mg.d[1]);
    }

    // ---- A5 + A6: top-k search
    uint32_t tau_k = 0, nk_k = 0, above_k = 0;
    if (k_on) {
      const bool hit = trunc && !overflow && !force_fb && survivors >= static_cast<uint32_t>(kr);
      path |= hit ? QRITA_PATH_HIT : QRITA_PATH_FALLBACK;
      s.rounds = 0;
      bool done0 = false;
      if (hit) {
        s.list_mode = true;
        s.list_len = my_surv;
        s.above_cnt = 0;
        s.lo = f2key(t) - 1u;
        s.C_lo = survivors;
        s.hi = f2key(row_max);
        s.C_hi = 0;
        if (warp == 0 && lane < static_cast<int>(c.C)) {
          F.cnt_lo[lane] = vld(F.rank_surv[lane]);
          F.cnt_hi[lane] = 0;
        }
        // z_mn of the initial lo is the smallest survivor: check it first.
        if (survivors - surv_min_n < static_cast<uint32_t>(kr)) {
          done0 = true;
          s.tau = f2key(surv_min);
          s.count_above = survivors - surv_min_n;
          s.n_keep = static_cast<uint32_t>(kr) - s.count_above;
          s.capped = false;
          // ties: every rank's survivors equal to surv_min; recount from the lists
        }
      } else {
        s.list_mode = false;
        s.lo = f2key(row_min) - 1u;
        s.C_lo = static_cast<uint32_t>(V);
        const bool miss_with_t = trunc && survivors < static_cast<uint32_t>(kr);
        s.hi = miss_with_t ? f2key(t) - 1u : f2key(row_max);
        s.C_hi = miss_with_t ? survivors : 0u;
        if (warp == 0 && lane < static_cast<int>(c.C)) {
          const int64_t rl = static_cast<int64_t>(V) - static_cast<int64_t>(lane) * P.chunk;
          F.cnt_lo[lane] = static_cast<uint32_t>(rl <= 0 ? 0 : (rl < P.chunk ? rl : P.chunk));
          F.cnt_hi[lane] = miss_with_t ? vld(F.rank_surv[lane]) : 0u;
        }
      }
      if (done0) {
        // per-rank count of survivors equal to the boundary (one list scan)
        uint32_t mine = 0;
        for (uint32_t i = tid; i < s.list_len; i += kThreads) mine += (c.list_x[i] == surv_min) ? 1u : 0u;
        uint32_t tot;
        const uint32_t ex = block_excl_scan(F, mine, &tot);
        (void)ex;
        if (tid == 0) F.slots[c.ph & 1].u[0] = tot;
        cluster_sync_all();
        if (warp == 0 && lane < static_cast<int>(c.C))
          F.ties[lane] = ld_dsmem_u32(map_rank(smem_u32(&F.slots[c.ph & 1].u[0]), lane));
        __syncthreads();
        ++c.ph;
      } else {
        quaternary_search<DT, false>(c, s, static_cast<double>(kr), value_pivots);
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
    }

    // ---- A5 + A7: top-p search
    if (p_on && !sel_none) {
      const double pd = static_cast<double>(pr);
      if (k_on) {
        // Z_k = mass above tau_k + n_keep_k * w(tau_k): one mass scan with a
        // single pivot at tau_k over the list (if it covers (tau_k, max]) or
        // the chunk (compacting x > tau_k when it fits).
        const bool list_ok = s.list_mode && (path & QRITA_PATH_HIT);
        if (list_ok) {
          for (uint32_t i = tid; i < s.list_len; i += kThreads) c.list_w[i] = weight(c.list_x[i], c.m, c.m_neginf);
          __syncthreads();
        }
        float qf[3] = {pivot_f(tau_k), INFINITY, INFINITY};
        bool compact = false;
        if (!list_ok) {
          // compact x > tau_k while scanning; a CTA whose share does not fit
          // the list stays in chunk mode (the append never writes past cap)
          compact = true;
          if (tid == 0) F.list_n = 0;
          __syncthreads();
        }
        PAcc acc[3];
        // compaction range (tau_k, +inf]: keeps the exact top-k set minus ties
        scan_round<DT, true>(c, list_ok, s.list_len, qf, acc, compact, pivot_f(tau_k), INFINITY);
        reduce_merge_pivots<DT, true>(c, acc, 0u, 0.0);
        const double M_gt = vld(F.mg.pv[0].mass);
        const uint32_t C_gt = vld(F.mg.pv[0].cnt);
        const double w_tau = weight(key2f(tau_k), c.m, c.m_neginf);
        Z = M_gt + static_cast<double>(nk_k) * w_tau;
        const double target = pd * Z;
        z_used = Z;
        if (M_gt < target) {
          // the boundary is inside the tau_k tie group: keep fewer of them
          double nk = ceil((target - M_gt) / w_tau);
          nk = fmin(fmax(nk, 1.0), static_cast<double>(nk_k));
          tau = tau_k;
          n_keep = static_cast<uint32_t>(nk);
          count_above = C_gt;
          // F.ties still holds the per-rank tau_k counts from the top-k search
        } else {
          // search (tau_k, max] by mass
          Search sp;
          sp.lo = tau_k;
          sp.C_lo = C_gt;
          sp.M_lo = M_gt;
          sp.hi = f2key(row_max);
          sp.C_hi = 0;
          sp.M_hi = 0.0;
          sp.myM_hi = 0.0;
          if (list_ok) {
            sp.list_mode = true;
            sp.list_len = s.list_len;
          } else {
            const uint32_t ln = vld(F.list_n);
            sp.list_mode = ln <= c.cap && compact;
            // every CTA decides for itself: a CTA whose compaction overflowed
            // stays in chunk mode
            sp.list_len = ln;
          }
          sp.above_cnt = 0;
          sp.above_mass = 0.0;
          if (warp == 0 && lane < static_cast<int>(c.C)) {
            F.cnt_lo[lane] = vld(F.rank_cnt[0][lane]);
            F.cnt_hi[lane] = 0;
          }
          quaternary_search<DT, true>(c, sp, target, value_pivots);
          rounds_p = static_cast<uint32_t>(sp.rounds);
          if (sp.capped) {
            sel_none = true;
            row_status = QRITA_ROW_SEARCH_CAP;
          }
          tau = sp.tau;
          n_keep = sp.n_keep;
          count_above = sp.count_above;
        }
      } else {
        const double target = pd * Z;
        z_used = Z;
        const bool hit = trunc && !overflow && !force_fb && Mt >= target * (1.0 + 1e-5);
        path |= hit ? QRITA_PATH_HIT : QRITA_PATH_FALLBACK;
        Search sp;
        sp.myM_hi = 0.0;
        sp.above_cnt = 0;
        sp.above_mass = 0.0;
        if (hit) {
          for (uint32_t i = tid; i < my_surv; i += kThreads) c.list_w[i] = weight(c.list_x[i], c.m, c.m_neginf);
          sp.list_mode = true;
          sp.list_len = my_surv;
          sp.lo = f2key(t) - 1u;
          sp.C_lo = survivors;
          sp.M_lo = Mt;
          if (warp == 0 && lane < static_cast<int>(c.C)) F.cnt_lo[lane] = vld(F.rank_surv[lane]);
        } else {
          sp.list_mode = false;
          sp.list_len = 0;
          sp.lo = f2key(row_min) - 1u;
          sp.C_lo = static_cast<uint32_t>(V);
          sp.M_lo = Z;
          if (warp == 0 && lane < static_cast<int>(c.C)) {
            const int64_t rl = static_cast<int64_t>(V) - static_cast<int64_t>(lane) * P.chunk;
            F.cnt_lo[lane] = static_cast<uint32_t>(rl <= 0 ? 0 : (rl < P.chunk ? rl : P.chunk));
          }
        }
        sp.hi = f2key(row_max);
        sp.C_hi = 0;
        sp.M_hi = 0.0;
        if (warp == 0 && lane < static_cast<int>(c.C)) F.cnt_hi[lane] = 0;
        quaternary_search<DT, true>(c, sp, target, value_pivots);
        rounds_p = static_cast<uint32_t>(sp.rounds);
        if (sp.capped) {
          sel_none = true;
          row_status = QRITA_ROW_SEARCH_CAP;
        }
        tau = sp.tau;
        n_keep = sp.n_keep;
        count_above = sp.count_above;
      }
    }
  }

  // ---- A8 + A9: tie resolution and mask emission
  __syncthreads();
  uint32_t my_first = 0, my_ties = 0;
  if (!sel_all && !sel_none) {
    for (uint32_t l = 0; l < c.crank; ++l) my_first += vld(F.ties[l]);
    my_ties = vld(F.ties[c.crank]);
  }
  const float tau_f = key2f(tau);
  // 0: no ties kept, 1: all ties kept, 2: straddling (ordered pass)
  int tie_mode = 0;
  if (!sel_all && !sel_none && my_ties > 0) {
    if (my_first + my_ties <= n_keep) tie_mode = 1;
    else if (my_first < n_keep) tie_mode = 2;
  }
  const uint32_t keep_local = (tie_mode == 2) ? (n_keep - my_first) : 0u;
  const uintptr_t mask_body = reinterpret_cast<uintptr_t>(gmask + c.head_n);
  const bool vec_ok = (mask_body % E) == 0;
  {
    uint32_t running = 0;  // ties seen so far in index order (tie_mode 2)
    // head (index order first): thread 0 walks it sequentially
    if (tid == 0) {
      for (int i = 0; i < c.head_n; ++i) {
        const float x = head_elem(c, i);
        uint8_t b;
        if (sel_all) b = 1;
        else if (sel_none) b = 0;
        else if (x > tau_f) b = 1;
        else if (x == tau_f) {
          b = (tie_mode == 1) || (tie_mode == 2 && running < keep_local);
          ++running;
        } else b = 0;
        gmask[i] = b;
      }
    }
    if (tie_mode == 2) {
      // broadcast the head's tie count
      if (tid == 0) F.scan[0] = running;
      __syncthreads();
      running = vld(F.scan[0]);
      __syncthreads();
    }
    const int iters = (c.body_units + kThreads - 1) / kThreads;
    for (int it = 0; it < iters; ++it) {
      const int u = it * kThreads + tid;
      float xs[E];
      bool valid = u < c.body_units;
      if (valid) unpack<DT>(*reinterpret_cast<const uint4*>(sbody + 16 * u), xs);
      uint32_t rank0 = 0;
      if (tie_mode == 2) {
        uint32_t mine = 0;
        if (valid) {
#pragma unroll
          for (int e = 0; e < E; ++e) mine += (xs[e] == tau_f) ? 1u : 0u;
        }
        uint32_t tot;
        const uint32_t ex = block_excl_scan(F, mine, &tot);
        rank0 = running + ex;
        running += tot;
      }
      if (!valid) continue;
      uint8_t bytes[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const float x = xs[e];
        uint8_t b;
        if (sel_all) b = 1;
        else if (sel_none) b = 0;
        else if (x > tau_f) b = 1;
        else if (x == tau_f) {
          b = (tie_mode == 1) || (tie_mode == 2 && rank0 < keep_local);
          ++rank0;
        } else b = 0;
        bytes[e] = b;
      }
      uint8_t* dst = gmask + c.head_n + static_cast<size_t>(u) * E;
      if (vec_ok) {
        if constexpr (E == 4) {
          const uint32_t w = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (static_cast<uint32_t>(bytes[3]) << 24);
          *reinterpret_cast<uint32_t*>(dst) = w;
        } else {
          uint32_t w0 = bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (static_cast<uint32_t>(bytes[3]) << 24);
          uint32_t w1 = bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (static_cast<uint32_t>(bytes[7]) << 24);
          *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
        }
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = bytes[e];
      }
    }
    // tail: thread 0 sequentially, after every body tie was counted
    if (tid == 0) {
      uint8_t* tdst = gmask + c.head_n + static_cast<size_t>(c.body_units) * E;
      for (int j = 0; j < c.tail_n; ++j) {
        const float x = tail_elem(c, j);
        uint8_t b;
        if (sel_all) b = 1;
        else if (sel_none) b = 0;
        else if (x > tau_f) b = 1;
        else if (x == tau_f) {
          b = (tie_mode == 1) || (tie_mode == 2 && running < keep_local);
          ++running;
        } else b = 0;
        tdst[j] = b;
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
      info.n_boundary = sel_none ? 0u : (sel_all ? 0u : n_keep);
      info.kept = kept;
      info.status = row_status;
      info.z = z_used;
      info.reserved = 0.0;
      P.row_info[r] = info;
    }
  }

  // If a copy wait expired, give the copies one more bounded chance to land
  // before the CTA's shared memory is released.
  if (timed_out && tid == 0) {
    for (int pc = 0; pc < npieces; ++pc) (void)mbar_wait_bounded(smem_u32(&F.bars[pc]), 0, kWaitLimitNs);
  }
  // No CTA leaves while another may still read its shared memory.
  cluster_sync_all();
}

}  // namespace

size_t smem_bytes(int dtype, int chunk, int cap) {
  const int s = dtype == QRITA_DTYPE_F32 ? 4 : 2;
  size_t b = sizeof(Fixed);
  b += static_cast<size_t>(cap) * 8u;  // list values + weights
  b += 16u + static_cast<size_t>(chunk) * s + 32u;
  return (b + 127u) & ~static_cast<size_t>(127u);
}

int max_smem_per_block() {
  int dev = 0;
  cudaGetDevice(&dev);
  int v = 0;
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return v;
}

#ifdef QRITA_TRACE
extern "C" int qrita_debug_trace(double* out, int cap, int reset) {
  unsigned n = 0;
  cudaDeviceSynchronize();
  cudaMemcpyFromSymbol(&n, g_trace_n, sizeof(n));
  if (n > static_cast<unsigned>(cap)) n = cap;
  cudaMemcpyFromSymbol(out, g_trace, n * sizeof(double));
  if (reset) {
    unsigned z = 0;
    cudaMemcpyToSymbol(g_trace_n, &z, sizeof(z));
  }
  return static_cast<int>(n);
}
#endif

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
