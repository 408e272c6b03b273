// Fused exact top-k / top-p selection kernel for GB300 (sm_103a).
//
// Method: Qrita technical summary (gist.science, paper 2602.01518),
// "Methodology" parts 1-2 and "Implementation details" (pipeline).
//
// One thread-block cluster of C CTAs handles one row; CTA c owns a contiguous
// chunk of the row. The row is read from HBM once, through a shared-memory
// ring of 1-D bulk copies (TMA) whose first stages fly while A2 runs:
//
//   A2  mu, sigma (and a reference max) from one sample block of the row,
//       read identically by every CTA of the cluster (no exchange needed);
//       sigma is re-estimated without the sample's outliers;
//   A3  delta from the normal-quantile tables, t = mu + delta * sigma; a
//       top-k threshold the sample contradicts becomes an order statistic of
//       the sample; top-k rows get bracket pivots from the model;
//   A4  one streaming pass over the chunk keeps Z_t = {x >= t} (value and
//       index) in a shared-memory list, and tracks max / min / NaN / +inf
//       and, for top-p without top-k, the softmax mass of the row and of Z_t
//       (rows whose Z_t cannot fit the lists bin it by value instead);
//   --  one cluster merge through distributed shared memory;
//   A5  hit: the survivors stay in the CTAs' own lists; else a second
//       truncation at an order statistic of a larger sample (top-k), one
//       pass over the one-byte bin codes that lists the boundary's bin
//       (binned top-p rows), or distributed narrowing passes over the chunk (one 256-bin pass,
//       then two quaternary levels per cluster merge) until the range that
//       holds the boundary fits the own lists, from which it is extracted;
//   A6  the pivot search over the own lists of the cluster (64 bins a round,
//       merged through distributed shared memory), then the last candidates
//       are copied to every CTA, split again locally, and tested directly
//       (the z_mn / N_zmn test);
//   A7  the same search by softmax mass for top-p;
//   A8  boundary duplicates kept by lowest token id: per-rank counts from the
//       search, then an index cut inside the one straddling CTA;
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
constexpr float kClipSigmas = 4.0f;  // sample values beyond this many sigmas are outliers
// Second truncation (top-k rows whose first threshold missed or overflowed):
// the threshold is an order statistic of a larger sample of the row.
constexpr int kRetryBlocks = 64;
constexpr int kRetrySample = kRetryBlocks * 64;  // 4096 logits
constexpr int kRetryPer = kRetrySample / kThreads;
// Streaming ring: the chunk moves through shared memory in pieces of
// kPieceBytes by 1-D bulk copies (TMA), kStages pieces in flight.
constexpr int kStages = 2;
constexpr int kPieceBytes = 16384;
constexpr int kPieceUnits = kPieceBytes / 16;
constexpr int kRingBytes = kStages * kPieceBytes;
// Passes that leave (part of) the own list unused stream through a deeper
// ring: up to kMaxStages stages, the extra ones laid below the standard ring
// over the list's unused bytes.
constexpr int kMaxStages = 6;

static_assert(kPieceUnits % kThreads == 0, "a piece is whole rounds of the block");
// Bound of one wait for a bulk copy (a copy from valid global memory lands in
// microseconds; the bound only keeps a failing copy from hanging the kernel).
constexpr uint64_t kWaitLimitNs = 200ull * 1000ull * 1000ull;
constexpr int kBins = kNarrowPivots + 1;
// A chunk narrowing pass lays per-thread bins (counts, then fixed-point
// masses) over the start of the list region, clear of the streaming ring.
constexpr int kBinBytes = kBins * kThreads * (4 + 8);
#ifdef QRITA_TRACE_TIME
// Debug-only stage timestamps of every CTA (built with -DQRITA_TRACE_TIME):
// g_cta_stage[cta][i] = globaltimer at mark i (0 start, 15 end).
constexpr int kTraceCtas = 16384;
__device__ unsigned long long g_cta_stage[kTraceCtas][16];
__device__ long long g_cta_row[kTraceCtas];  // the row each CTA handled
#define QRITA_ROWID(r)                                                                          \
  do {                                                                                          \
    if (threadIdx.x == 0 && blockIdx.x < kTraceCtas) g_cta_row[blockIdx.x] = (r);               \
  } while (0)
#define QRITA_T(i)                                                                              \
  do {                                                                                          \
    if (threadIdx.x == 0 && blockIdx.x < kTraceCtas) g_cta_stage[blockIdx.x][i] = globaltimer_ns(); \
  } while (0)
#define QRITA_V(i, v)                                                                           \
  do {                                                                                          \
    if (threadIdx.x == 0 && blockIdx.x < kTraceCtas) g_cta_stage[blockIdx.x][i] = (v);         \
  } while (0)
#else
#define QRITA_ROWID(r) \
  do {                 \
  } while (0)
#define QRITA_T(i) \
  do {             \
  } while (0)
#define QRITA_V(i, v) \
  do {                \
  } while (0)
#endif

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


// Read of shared state another thread wrote before a barrier. Every such read
// goes through a volatile shared load so the compiler can neither reuse an
// earlier load of the same word nor move the load across the barrier.
template <typename T>
__device__ __forceinline__ T vld(const T& r) {
  return *reinterpret_cast<const volatile T*>(&r);
}

// exp(d) as 2^(d log2 e) by the hardware base-2 exponential (ex2.approx,
// subnormal results flushed to zero). d = x - s is formed first, so the
// argument's rounding error scales with |x - s| and not with the shift s:
// weights near the shift, which carry the mass, are within a few ulp of
// exp, and a row's weights all come from this one function.
constexpr float kLog2e = 1.4426950408889634f;
__device__ __forceinline__ float exp_shifted(float x, float s) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"((x - s) * kLog2e));
  return r;
}

// Softmax weight of x for row max m. A row whose max is -inf holds only
// -inf, and equal logits get equal weight 1.
__device__ __forceinline__ float weight(float x, float m, bool m_neginf) {
  return m_neginf ? 1.0f : exp_shifted(x, m);
}

// Fixed-point softmax weight: round(exp(x - m) * scale). Every place that
// weighs a value uses this one function, so sums and boundary weights agree.
__device__ __forceinline__ unsigned long long weight_fx(float x, float m, bool m_neginf, float scale) {
  return round_u64(weight(x, m, m_neginf) * scale);
}

// Bin of x among the increasing pivots (+inf padded): the number of pivots
// below x, by a 4-step branch-free search.
__device__ __forceinline__ int pivot_bin(const volatile float* qf, float x) {
  int b = 0;
  b += (x > qf[b + 7]) ? 8 : 0;
  b += (x > qf[b + 3]) ? 4 : 0;
  b += (x > qf[b + 1]) ? 2 : 0;
  b += (x > qf[b]) ? 1 : 0;
  return b;
}

// ---------------------------------------------------------------------------
// Shared-memory layout
// ---------------------------------------------------------------------------
struct alignas(16) Slot {  // what one CTA publishes for one cluster merge
  unsigned long long mass[kBins + 1];  // narrowing: per-bin fixed-point mass; [kBins] above hi
  uint32_t cnt[kBins + 1];             // narrowing: per-bin counts; [kBins] above hi
  float f[4];
  uint32_t u[4];
  float pr[4];  // float pairs (softmax sums of the streaming pass)
};

struct alignas(16) Bcast {  // written by one thread / warp 0 before a block barrier
  unsigned long long x[8];  // fixed-point masses (narrowing)
  float pr[16];             // float pairs: pair i is (pr[2i], pr[2i+1])
  float f[12];
  uint32_t u[28];
  uint32_t q[16];  // pivot keys, increasing
  float qf[16];    // pivot floats (+inf padding)
};


// Per-warp partial of one pivot of the local search.
struct alignas(16) LPart {
  unsigned long long mass;
  uint32_t cnt, zmin, nz, pad;
};

struct alignas(16) Fixed {
  Slot slots[2];
  Bcast bc;
  LPart lred[2][kWarps][3];  // quaternary search: per-warp partials, double-buffered
  float redf[kWarps][8];
  uint32_t redu[kWarps][kBins];
  uint32_t rank_bins[kMaxCluster][kBins + 1];  // latest narrowing merge, per rank
  uint32_t rank_n[kMaxCluster];   // per-rank own-list entries (survivors)
  uint32_t rank_lo[kMaxCluster];  // per-rank count above lo (narrowing: chunk; search: own list)
  uint32_t rank_hi[kMaxCluster];  // per-rank count above hi
  uint32_t ties[kMaxCluster];     // per-rank count of boundary-valued elements
  uint32_t pr_cnt[kMaxCluster][3];  // search round: per-rank counts above the pivots
  uint32_t pr_nz[kMaxCluster][3];   // search round: per-rank copies of the row's z_mn
  uint32_t dtot[3][3];              // search round: row count, z_mn, N_zmn per pivot
  unsigned long long dmass[3];      // search round: row mass above each pivot
  uint32_t scan[kWarps];
  uint32_t own_n;
  uint32_t seg_base[kWarps];  // own list: warp w's entries are [seg_base[w], + seg_cnt[w])
  uint32_t seg_cnt[kWarps];
  uint32_t col_mode;            // own list in per-thread columns instead:
  uint8_t col_n[kThreads];      // thread t's entries are t + j * kThreads, j < col_n[t]
  uint32_t tail_n;
  uint32_t tbin_c[64];               // search tail: counts and masses of its bins
  unsigned long long tbin_m[64];
  uint32_t tsel[2];                  // the bin holding the boundary, count above it
  unsigned long long tsel_m;         // and mass above it
  uint32_t tkey[2];                  // the smallest and largest key of its members
  float bp[16];                      // bracket pivots of the top-k search (+inf padded)
  uint32_t bp_bins[16];              // own-list survivors between consecutive bracket pivots
  uint32_t seg_n[kWarps];  // streaming pass: per-warp survivor counts
  uint32_t seg_ovf;        // a warp's survivors exceeded its segment
  uint32_t err;       // a bulk-copy wait of this CTA gave up
  uint32_t err_any;   // some CTA of the row reported err (written remotely)
  unsigned long long ring_bar[kMaxStages];  // one mbarrier per ring stage
};

// Bytes of the list region after Fixed: the own list (value + index), then
// the streaming ring.
__host__ __device__ constexpr size_t list_region_bytes(int ocap) {
  return static_cast<size_t>(ocap) * 8u + kRingBytes;
}

// Names of the broadcast slots
enum : int {
  // floats
  BF_MU = 0, BF_SIGMA, BF_MREF, BF_T, BF_MAX, BF_MIN, BF_LOF, BF_HIF, BF_PHAM,
  // uints
  BU_TRUNC = 0, BU_S, BU_OVF, BU_LO, BU_HI, BU_CLO, BU_CHI, BU_DONE, BU_TAU,
  BU_NKEEP, BU_CABOVE, BU_NP, BU_USED_VALUE, BU_VMODE, BU_MAXR, BU_BELOW, BU_FITS, BU_S2, BU_OVF2,
  BU_QKEY, BU_QWANT, BU_PHAC, BU_ROW, BU_SAMPLE_T, BU_KWCA, BU_KWCB, BU_SGE, BU_S2S,
  // fixed-point masses
  BX_TARGET = 0, BX_MLO, BX_MHI,
  // float pairs
  BP_ZR = 0, BP_MR, BP_MLO, BP_MHI, BP_TOTAL, BP_GAP, BP_PHA,
};
static_assert(BU_S2S < static_cast<int>(sizeof(Bcast::u) / sizeof(uint32_t)), "every uint slot fits the broadcast block");
static_assert(BP_PHA < static_cast<int>(sizeof(Bcast::pr) / sizeof(float) / 2), "every pair slot fits the broadcast block");

__device__ __forceinline__ void put_pair(Bcast& b, int i, F2 v) {
  b.pr[2 * i] = v.hi;
  b.pr[2 * i + 1] = v.lo;
}

__device__ __forceinline__ F2 get_pair(const Bcast& b, int i) {
  return f2_make(vld(b.pr[2 * i]), vld(b.pr[2 * i + 1]));
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

// Append the set bits' elements to this warp's segment of a list (no atomics):
// segment `seg` = entries [seg_base, seg_base + segcap); wn is the warp's
// running count (warp-uniform), which keeps counting past segcap.
template <int E>
__device__ __forceinline__ void seg_append(uint32_t& wn, float* vals, uint32_t* idxs, uint32_t seg_base,
                                           uint32_t segcap, const float (&xs)[E], uint32_t idx0,
                                           uint32_t bits) {
  if (__ballot_sync(kFull, bits != 0u) == 0u) return;
  const uint32_t lt = (1u << (threadIdx.x & 31)) - 1u;
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const bool mine = (bits >> e) & 1u;
    const uint32_t b = __ballot_sync(kFull, mine);
    if (mine) {
      const uint32_t pos = wn + __popc(b & lt);
      if (pos < segcap) {
        vals[seg_base + pos] = xs[e];
        idxs[seg_base + pos] = idx0 + e;
      }
    }
    wn += __popc(b);
  }
}

// ---------------------------------------------------------------------------
// Pivots: 25/50/75 % of a key range (lo, hi]
// ---------------------------------------------------------------------------
// Value-space quartiles (the pages' reading of "25/50/75 % of the search
// range") when value_ok and both ends are finite floats; otherwise quartiles
// of the 32-bit key range, which always shrink it fourfold. Writes up to 3
// strictly increasing keys inside (lo, hi) and returns how many.
__device__ __forceinline__ int quartile_pivots(uint32_t lo, uint32_t hi, bool value_ok, uint32_t& q0,
                                               uint32_t& q1, uint32_t& q2, bool& used_value) {
  const uint32_t span = hi - lo;
  used_value = false;
  q0 = q1 = q2 = hi;
  if (span <= 1u) return 0;
  if (span <= 4u) {
    q0 = lo + 1u;
    q1 = lo + 2u;
    q2 = lo + 3u;
    return static_cast<int>(span) - 1;
  }
  if (value_ok) {
    const float vlo = key2f(lo), vhi = key2f(hi);
    const float width = vhi - vlo;
    if (isfinite(vlo) && isfinite(vhi) && isfinite(width)) {
      const uint32_t a = f2key(fmaf(0.25f, width, vlo));
      const uint32_t b = f2key(fmaf(0.50f, width, vlo));
      const uint32_t c = f2key(fmaf(0.75f, width, vlo));
      if (lo < a && a < b && b < c && c < hi) {
        q0 = a;
        q1 = b;
        q2 = c;
        used_value = true;
        return 3;
      }
    }
  }
  q0 = lo + static_cast<uint32_t>((static_cast<uint64_t>(span) * 1u) >> 2);
  q1 = lo + static_cast<uint32_t>((static_cast<uint64_t>(span) * 2u) >> 2);
  q2 = lo + static_cast<uint32_t>((static_cast<uint64_t>(span) * 3u) >> 2);
  return 3;
}

// Two quaternary levels at once: the quartile pivots of (lo, hi] and of each
// of the four sub-ranges they cut, written in increasing order to the
// shared pivot arrays (keys and floats, +inf padded). Returns the count.
__device__ int two_level_pivots(uint32_t lo, uint32_t hi, bool value_ok, volatile uint32_t* q,
                                volatile float* qf, bool& used_value) {
  uint32_t a0, a1, a2;
  const int n1 = quartile_pivots(lo, hi, value_ok, a0, a1, a2, used_value);
  int n = 0;
  uint32_t a = lo;
#pragma unroll
  for (int s = 0; s <= 3; ++s) {
    if (s <= n1) {
      const uint32_t b = (s < n1) ? (s == 0 ? a0 : (s == 1 ? a1 : a2)) : hi;
      uint32_t b0, b1, b2;
      bool uv = false;
      const int n2 = quartile_pivots(a, b, value_ok, b0, b1, b2, uv);
      if (n2 > 0) q[n++] = b0;
      if (n2 > 1) q[n++] = b1;
      if (n2 > 2) q[n++] = b2;
      if (s < n1) q[n++] = b;
      a = b;
    }
  }
  for (int j = 0; j < 16; ++j) qf[j] = (j < n) ? pivot_f(q[j]) : INFINITY;
  for (int j = n; j < 16; ++j) q[j] = hi;
  return n;
}

// ---------------------------------------------------------------------------
// Per-CTA context
// ---------------------------------------------------------------------------
template <bool B>
struct BoolC {
  static constexpr bool value = B;
};

template <int DT>
struct Ctx {
  static constexpr int E = Elem<DT>::kPerUnit;
  static constexpr int S = Elem<DT>::kBytes;
  Fixed* F;
  unsigned char* lists;  // the list region (own list, then the ring)
  float* own_val;
  uint32_t* own_idx;
  uint32_t ocap;
  const unsigned char* gx;     // chunk start in global memory
  const unsigned char* gbody;  // first 16-byte aligned unit of the chunk
  uint8_t* gmask;              // chunk start in the mask
  int n, head_n, body_units, tail_n;
  uint32_t C, crank;
  uint32_t ring;        // shared address of the streaming ring
  const uint4* ring_ptr;  // the same ring, generic
  uint32_t ring_bar;    // shared address of F->ring_bar[0]
  uint32_t ring_phase;  // bit s: parity of stage s's next completion
  uint32_t ring_out;    // thread 0: stages with a copy not yet seen complete
  int ph;           // cluster merge counter (slot parity)
  float m;          // row max (softmax shift)
  bool m_neginf;
  float fix_scale;  // fixed-point scale of weights in [0, 1]
  bool zero_fill;       // the chunk's mask is to be zeroed early (by the search tail)
  bool zero_fill_done;  // and it was
  bool one_fill_done;   // a keep-all row's mask was filled with 1 by the streaming pass
  bool give_up_once;    // test flag: the next bounded copy wait reports that it gave up
  int split;            // bins of a list-search round and of a tail split (64; 4 or 2 by flag)
  int npiv;             // pivots of a narrowing pass (15; 3 or 1 by flag)
  bool wide_ok;         // the 256-bin first narrowing pass may run
};

// Fill the chunk's mask with one byte value (16-byte stores where aligned).
template <int DT>
__device__ __forceinline__ void fill_mask(Ctx<DT>& c, uint8_t fill) {
  const int tid = threadIdx.x;
  const uint32_t fill4 = fill ? 0x01010101u : 0u;
  const uintptr_t ma = reinterpret_cast<uintptr_t>(c.gmask);
  const int mh0 = static_cast<int>((16u - (ma & 15u)) & 15u);
  const int mh = mh0 < c.n ? mh0 : c.n;
  const int mb = (c.n - mh) / 16;
  const int mt = c.n - mh - mb * 16;
  if (tid < mh) c.gmask[tid] = fill;
  for (int i = tid; i < mb; i += kThreads)
    reinterpret_cast<uint4*>(c.gmask + mh)[i] = make_uint4(fill4, fill4, fill4, fill4);
  if (tid < mt) c.gmask[mh + mb * 16 + tid] = fill;
}

// Byte offset of ring stage st from the standard ring: stages 0 .. kStages-1
// are the standard ring; deeper rings add stages below it, stage kStages
// right below, the next below that, and so on.
__device__ __forceinline__ int stage_off(int st) {
  return st < kStages ? st * kPieceBytes : -(st - kStages + 1) * kPieceBytes;
}

// Issue the bulk copy of piece `piece` of the chunk body into ring stage `st`
// (thread 0 only).
template <int DT>
__device__ __forceinline__ void ring_issue(Ctx<DT>& c, int piece, int st) {
  const int u0 = piece * kPieceUnits;
  const int n = min(kPieceUnits, c.body_units - u0);
  const uint32_t bar = c.ring_bar + 8u * st;
  const uint32_t bytes = static_cast<uint32_t>(n) * 16u;
  mbar_expect_tx(bar, bytes);
  bulk_g2s(c.ring + static_cast<uint32_t>(stage_off(st)), c.gbody + 16 * static_cast<size_t>(u0), bytes, bar);
  c.ring_out |= 1u << st;
}

// Stages a pass may stream through when the first `used` bytes of the list
// region must stay intact (the ring grows down from the end of the region).
__host__ __device__ constexpr int ring_stages(size_t region, size_t used) {
  return region < used + static_cast<size_t>(kRingBytes)
             ? kStages
             : ((region - used) / kPieceBytes > static_cast<size_t>(kMaxStages)
                    ? kMaxStages
                    : static_cast<int>((region - used) / kPieceBytes));
}

// Units of one ring piece each thread holds: unit j of a piece starting at
// unit u0 is u0 + j * kThreads + threadIdx.x.
constexpr int kPieceThreadUnits = kPieceUnits / kThreads;

// Stream the chunk: the 16-byte aligned body through the shared-memory ring
// (kStages bulk copies in flight), then the head / tail elements (fewer than
// 2E, one per thread). piece_fn(v, u0, n) gets this thread's units of each
// piece (v[j] valid when j * kThreads + tid < n); scalar_fn(x, idx, valid)
// the head / tail element of this thread. Both are called by every thread
// the same number of times (convergent), valid or not. prefetched: the first
// min(kStages, pieces) copies were issued already (into the standard ring).
// nst: ring stages (kStages: the standard ring; more reach down into the own
// list, which the caller leaves unused there). Every copy issued here has
// landed when it returns, unless a wait gave up (F->err set; later calls then
// issue nothing).
template <int DT, typename PieceFn, typename ScalarFn>
__device__ __forceinline__ void stream_pieces(Ctx<DT>& c, PieceFn&& piece_fn, ScalarFn&& scalar_fn,
                                              bool prefetched, int nst = kStages) {
  constexpr int E = Ctx<DT>::E;
  constexpr int S = Ctx<DT>::S;
  Fixed& F = *c.F;
  const int tid = threadIdx.x;
  const int nb = c.body_units;
  const int npieces = (nb + kPieceUnits - 1) / kPieceUnits;
  // generic writes to these bytes before the async copies (a prefetched pass
  // still issues its stages below the standard ring here)
  if (!prefetched || nst > kStages) fence_proxy_async_smem();
  __syncthreads();  // earlier users of the ring's bytes are done
  if (tid == 0 && npieces > 0 && vld(F.err) == 0u) {
    for (int pc = prefetched ? kStages : 0; pc < npieces && pc < nst; ++pc) ring_issue(c, pc, pc);
  }
  int st = 0;
  for (int pc = 0; pc < npieces; ++pc, st = (st + 1 == nst) ? 0 : st + 1) {
    const uint32_t bar = c.ring_bar + 8u * st;
    bool ok = false;
    if (vld(F.err) == 0u) {
      if (c.give_up_once) {
        // QRITA_FLAG_TEST_GIVE_UP: this wait reports a timeout without waiting
        // (the copy itself still lands; the drain below waits for it)
        c.give_up_once = false;
      } else {
        ok = mbar_wait_bounded(bar, (c.ring_phase >> st) & 1u, kWaitLimitNs);
      }
    }
    if (ok) {
      c.ring_phase ^= 1u << st;
      if (tid == 0) c.ring_out &= ~(1u << st);
    } else {
      F.err = 1u;
    }
    const int u0 = pc * kPieceUnits;
    const int n = min(kPieceUnits, nb - u0);
    const uint4* sp = c.ring_ptr + stage_off(st) / 16;
    uint4 v[kPieceThreadUnits];
#pragma unroll
    for (int j = 0; j < kPieceThreadUnits; ++j) {
      const int u = j * kThreads + tid;
      v[j] = (u < n) ? sp[u] : make_uint4(0u, 0u, 0u, 0u);
    }
    __syncthreads();  // every thread holds its part of stage st: refill it now
    if (tid == 0 && pc + nst < npieces && vld(F.err) == 0u) ring_issue(c, pc + nst, st);
    piece_fn(v, u0, n);
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

// stream_pieces one unit at a time: unit_fn(xs, idx0, valid) per unit.
template <int DT, typename UnitFn, typename ScalarFn>
__device__ __forceinline__ void stream_chunk(Ctx<DT>& c, UnitFn&& unit_fn, ScalarFn&& scalar_fn,
                                             bool prefetched = false, int nst = kStages) {
  constexpr int E = Ctx<DT>::E;
  stream_pieces<DT>(
      c,
      [&](const uint4 (&v)[kPieceThreadUnits], int u0, int n) {
#pragma unroll
        for (int j = 0; j < kPieceThreadUnits; ++j) {
          const int u = j * kThreads + static_cast<int>(threadIdx.x);
          float xs[E];
          unpack<DT>(v[j], xs);
          unit_fn(xs, static_cast<uint32_t>(c.head_n + (u0 + u) * E), u < n);
        }
      },
      scalar_fn, prefetched, nst);
}

// The survivors of one ring piece (bits[j]: the elements of this thread's unit
// j that survive) to this warp's segment of the own list: positions from one
// warp scan of the per-thread counts. wn is the warp's running count
// (warp-uniform), which keeps counting past segcap.
template <int DT>
__device__ __forceinline__ void append_piece(Ctx<DT>& c, uint32_t& wn, uint32_t seg_base, uint32_t segcap,
                                             const float (&xs)[kPieceThreadUnits][Ctx<DT>::E],
                                             const uint32_t (&bits)[kPieceThreadUnits], int u0) {
  constexpr int E = Ctx<DT>::E;
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t cnt = 0;
#pragma unroll
  for (int j = 0; j < kPieceThreadUnits; ++j) cnt += __popc(bits[j]);
  if (__ballot_sync(kFull, cnt != 0u) == 0u) return;
  // warp prefix of the counts by bit planes: independent ballots instead of
  // a chain of shuffles (cnt < 2^kPlanes)
  constexpr int kPlanes = 32 - __builtin_clz(static_cast<unsigned>(kPieceThreadUnits * E));
  const uint32_t lt = (1u << lane) - 1u;
  uint32_t excl = 0, tot = 0;
#pragma unroll
  for (int b = 0; b < kPlanes; ++b) {
    const uint32_t plane = __ballot_sync(kFull, (cnt >> b) & 1u);
    excl += static_cast<uint32_t>(__popc(plane & lt)) << b;
    tot += static_cast<uint32_t>(__popc(plane)) << b;
  }
  uint32_t pos = wn + excl;
  wn += tot;
#pragma unroll
  for (int j = 0; j < kPieceThreadUnits; ++j) {
    uint32_t b = bits[j];
    const uint32_t idx0 = static_cast<uint32_t>(c.head_n + (u0 + j * kThreads + tid) * E);
    while (b != 0u) {
      const int e = __ffs(b) - 1;
      b &= b - 1u;
      float x = xs[j][0];
#pragma unroll
      for (int q = 1; q < E; ++q) x = (q == e) ? xs[j][q] : x;
      if (pos < segcap) {
        c.own_val[seg_base + pos] = x;
        c.own_idx[seg_base + pos] = idx0 + static_cast<uint32_t>(e);
      }
      ++pos;
    }
  }
}

// bf16 unit (8 elements, four packed words) survivor bits in the packed
// layout: bit i is element 2i (word i's low half), bit 16 + i element 2i + 1.
__device__ __forceinline__ uint32_t bf16_unit_bits(const uint4 v, uint32_t t2) {
  uint32_t b = bf2_ge_mask(v.x, t2) & 0x00010001u;
  b |= bf2_ge_mask(v.y, t2) & 0x00020002u;
  b |= bf2_ge_mask(v.z, t2) & 0x00040004u;
  b |= bf2_ge_mask(v.w, t2) & 0x00080008u;
  return b;
}

// Element (index within the unit) and value of packed bit p of a bf16 unit.
__device__ __forceinline__ int bf16_bit_elem(int p) { return ((p & 15) << 1) | (p >> 4); }
__device__ __forceinline__ float bf16_bit_value(const uint4 v, int p) {
  const int i = p & 15;
  const uint32_t w = i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
  return __uint_as_float((p >> 4) ? (w & 0xFFFF0000u) : (w << 16));
}

// append_piece for bf16 units in the packed bit layout: the values come
// straight from the raw units (only survivors are widened). A lane with
// survivors claims its slots of the warp's segment with one shared atomic on
// the warp's running count (F.seg_n[warp], zeroed before the pass): the
// segment is unordered, so no warp scan is needed. The four units' bits are
// folded into one 32-bit mask (unit j's low halves at bits 4j .. 4j + 3, its
// high halves at 16 + 4j ..), so a lane walks its survivors in one loop
// whose trip count is the warp's largest count of the piece; bit p names
// word p & 15 of the four units (a tree of selects) and its half p >> 4.
static_assert(kPieceThreadUnits == 4, "four units of 4 + 4 survivor bits fill one 32-bit mask");
template <int DT>
__device__ __forceinline__ void append_piece_bf16(Ctx<DT>& c, uint32_t seg_base, uint32_t segcap,
                                                  const uint4 (&v)[kPieceThreadUnits],
                                                  const uint32_t (&bits)[kPieceThreadUnits], int u0) {
  const int tid = threadIdx.x, warp = tid >> 5;
  uint32_t all = 0u;
#pragma unroll
  for (int j = 0; j < kPieceThreadUnits; ++j) all |= bits[j] << (4 * j);
  if (all == 0u) return;
  uint32_t pos = atomicAdd(&c.F->seg_n[warp], static_cast<uint32_t>(__popc(all)));
  const uint32_t idx_base = static_cast<uint32_t>(c.head_n + (u0 + tid) * 8);
  while (all != 0u) {
    const uint32_t p = static_cast<uint32_t>(__ffs(all) - 1);
    all &= all - 1u;
    const bool b0 = (p & 1u) != 0u, b1 = (p & 2u) != 0u, b2 = (p & 4u) != 0u, b3 = (p & 8u) != 0u;
    uint32_t wj[kPieceThreadUnits];
#pragma unroll
    for (int j = 0; j < kPieceThreadUnits; ++j)
      wj[j] = b1 ? (b0 ? v[j].w : v[j].z) : (b0 ? v[j].y : v[j].x);
    const uint32_t w = b3 ? (b2 ? wj[3] : wj[2]) : (b2 ? wj[1] : wj[0]);
    const uint32_t hi = p >> 4;
    // unit (p >> 2) & 3, element 2 (p & 3) + half
    const uint32_t idx = idx_base + ((p >> 2) & 3u) * (kThreads * 8u) + (((p & 3u) << 1) | hi);
    if (pos < segcap) {
      c.own_val[seg_base + pos] = __uint_as_float(hi ? (w & 0xFFFF0000u) : (w << 16));
      c.own_idx[seg_base + pos] = idx;
    }
    ++pos;
  }
}

// The values of this warp's segment entries [0, ns) read back from the row by
// their indices, eight loads a lane in flight (entries listed by index only;
// the warp's own index writes are visible after a barrier).
template <int DT>
__device__ __forceinline__ void gather_segment_values(Ctx<DT>& c, uint32_t seg_base, uint32_t ns) {
  constexpr int S = Ctx<DT>::S;
  constexpr int kG = 8;
  const int lane = threadIdx.x & 31;
  for (uint32_t k0 = 0; k0 < ns; k0 += 32u * kG) {
    uint32_t ix[kG];
    float x[kG];
#pragma unroll
    for (int q = 0; q < kG; ++q) {
      const uint32_t k = k0 + static_cast<uint32_t>(q * 32 + lane);
      ix[q] = k < ns ? c.own_idx[seg_base + k] : 0u;
    }
#pragma unroll
    for (int q = 0; q < kG; ++q) x[q] = load_elem<DT>(c.gx + static_cast<size_t>(ix[q]) * S);
#pragma unroll
    for (int q = 0; q < kG; ++q) {
      const uint32_t k = k0 + static_cast<uint32_t>(q * 32 + lane);
      if (k < ns) c.own_val[seg_base + k] = x[q];
    }
  }
}

// After a wait gave up: wait (bounded) for every copy still in flight into
// this CTA's ring, so that none lands after the CTA has exited (thread 0).
template <int DT>
__device__ void ring_drain(Ctx<DT>& c) {
  for (int st = 0; st < kMaxStages; ++st)
    if ((c.ring_out >> st) & 1u)
      (void)mbar_wait_bounded(c.ring_bar + 8u * st, (c.ring_phase >> st) & 1u, kWaitLimitNs);
}

// ---------------------------------------------------------------------------
// Distributed narrowing (fallback search over the lists or the chunk)
// ---------------------------------------------------------------------------
struct Range {
  uint32_t lo, hi;      // count/mass(> lo) >= target > count/mass(> hi)
  uint32_t c_lo, c_hi;  // row counts above lo / hi
  unsigned long long m_lo, m_hi;  // row masses above lo / hi (fixed point)
  unsigned long long target;      // fixed point (mass) or count
  bool target_from_total;  // the first pass sets target = p * (mass above lo + extra)
  float p_frac;
  unsigned long long extra;
  bool lo_all;          // lo lies below key(-inf): every element is above it
  bool pin_hi;          // extraction: keep everything above lo
  bool fits;            // every rank's part of the range fits its own list
  bool exact;           // hi - lo <= 1: the boundary value is hi
  bool below;           // the target exceeds everything above lo: the boundary is at lo
  int passes;
};

// One narrowing pass: up to 15 pivots (two quaternary levels) cut (lo, hi]
// into bins; every CTA bins its elements (from its list, or by streaming its
// chunk again), the bins merge across the cluster in rank order, and warp 0
// keeps the bin that holds the boundary. Counts are exact integers and
// masses exact sums of fixed-point weights, so the merge is deterministic.
// A chunk pass bins into per-thread columns of shared memory (no atomics)
// laid over the own list, which it leaves undefined.
template <int DT, bool MASS>
__device__ void narrow_pass(Ctx<DT>& c, Range& R, bool value_ok, bool* used_value_out) {
  constexpr int E = Ctx<DT>::E;
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    bool used_value = false;
    int np;
    if (c.npiv >= kNarrowPivots) {
      np = two_level_pivots(R.lo, R.hi, value_ok, F.bc.q, F.bc.qf, used_value);
    } else {
      // one quaternary level (3 pivots) or a binary split (the middle one)
      uint32_t q0, q1, q2;
      const int n1 = quartile_pivots(R.lo, R.hi, value_ok, q0, q1, q2, used_value);
      np = 0;
      if (c.npiv == 1) {
        if (n1 > 0) F.bc.q[np++] = n1 == 3 ? q1 : q0;
      } else {
        if (n1 > 0) F.bc.q[np++] = q0;
        if (n1 > 1) F.bc.q[np++] = q1;
        if (n1 > 2) F.bc.q[np++] = q2;
      }
      for (int j = 0; j < 16; ++j) F.bc.qf[j] = (j < np) ? pivot_f(F.bc.q[j]) : INFINITY;
      for (int j = np; j < 16; ++j) F.bc.q[j] = R.hi;
    }
    F.bc.u[BU_NP] = static_cast<uint32_t>(np);
    F.bc.u[BU_USED_VALUE] = used_value ? 1u : 0u;
    F.bc.f[BF_LOF] = R.lo_all ? -INFINITY : pivot_f(R.lo);
    F.bc.f[BF_HIF] = pivot_f(R.hi);
  }
  uint32_t* lcnt = reinterpret_cast<uint32_t*>(c.lists);  // [kBins][kThreads]
  unsigned long long* lmass =
      reinterpret_cast<unsigned long long*>(c.lists + kBins * kThreads * 4);  // [kBins][kThreads]
  __syncthreads();  // pivots published; earlier readers of the lists are done
  const volatile float* qf = F.bc.qf;
#pragma unroll
  for (int b = 0; b < kBins; ++b) {
    lcnt[b * kThreads + tid] = 0u;
    if (MASS) lmass[b * kThreads + tid] = 0ull;
  }
  const float lo_f = vld(F.bc.f[BF_LOF]);
  const float hi_f = vld(F.bc.f[BF_HIF]);
  const bool lo_all = R.lo_all;
  const float scale = c.fix_scale;
  uint32_t above_c = 0;
  unsigned long long above_m = 0ull;
  auto bin_one = [&](float x) {
    if (!(lo_all || x > lo_f)) return;
    unsigned long long wf = 0ull;
    if (MASS) wf = weight_fx(x, c.m, c.m_neginf, scale);
    if (x > hi_f) {
      ++above_c;
      above_m += wf;
      return;
    }
    const int b = pivot_bin(qf, x);
    lcnt[b * kThreads + tid] += 1u;
    if (MASS) lmass[b * kThreads + tid] += wf;
  };
  stream_chunk<DT>(
      c,
      [&](const float (&xs)[E], uint32_t, bool valid) {
        if (!valid) return;
#pragma unroll
        for (int e = 0; e < E; ++e) bin_one(xs[e]);
      },
      [&](float x, uint32_t, bool valid) {
        if (valid) bin_one(x);
      },
      false, ring_stages(list_region_bytes(static_cast<int>(c.ocap)), kBinBytes));
  above_c = warp_sum_u(above_c);
  above_m = warp_sum_u64(above_m);
  if (lane == 0) {
    F.redu[warp][0] = above_c;
    F.redu[warp][1] = static_cast<uint32_t>(above_m);
    F.redu[warp][2] = static_cast<uint32_t>(above_m >> 32);
  }
  __syncthreads();
  Slot& my = F.slots[c.ph & 1];
  {
    // warp w totals bins w and w + kWarps over the thread columns
    for (int b = warp; b < kBins; b += kWarps) {
      uint32_t s = 0;
      unsigned long long sm = 0ull;
      for (int i = lane; i < kThreads; i += 32) {
        s += vld(lcnt[b * kThreads + i]);
        if (MASS) sm += vld(lmass[b * kThreads + i]);
      }
      s = warp_sum_u(s);
      sm = warp_sum_u64(sm);
      if (lane == 0) {
        my.cnt[b] = s;
        my.mass[b] = sm;
      }
    }
  }
  if (tid == kThreads - 1) {
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
    // cumulative from the top: lane b gets the elements above pivot b-1
    // (lane 0: above lo), lane np+1 .. kBins: above hi
    uint32_t cc = (lane <= np || lane == kBins) ? tot_c : 0u;
    unsigned long long cm = (lane <= np || lane == kBins) ? tot_m : 0ull;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t c2 = __shfl_down_sync(kFull, cc, o);
      const unsigned long long m2 = __shfl_down_sync(kFull, cm, o);
      if (lane + o < 32) {
        cc += c2;
        cm += m2;
      }
    }
    __syncwarp();  // per-rank bins visible to the whole warp
    int lo_j = -1, hi_j = -1;
    const uint32_t above_hi_c = __shfl_sync(kFull, tot_c, kBins);
    const unsigned long long above_hi_m = __shfl_sync(kFull, tot_m, kBins);
    unsigned long long tgt = R.target;
    if (R.target_from_total) {
      const unsigned long long total = __shfl_sync(kFull, cm, 0) + R.extra;
      tgt = f2_to_u64(f2_mul(f2_from_u64(total), R.p_frac));
    }
    // walk the pivots upward (every lane, same values)
    for (int j = 0; j < np; ++j) {
      const uint32_t ac = __shfl_sync(kFull, cc, j + 1);
      const unsigned long long am = __shfl_sync(kFull, cm, j + 1);
      const bool reach = MASS ? (am >= tgt) : (static_cast<unsigned long long>(ac) >= tgt);
      if (hi_j < 0) {
        if (reach) lo_j = j;
        else hi_j = j;
      }
    }
    if (R.pin_hi) hi_j = -1;
    const uint32_t c0 = __shfl_sync(kFull, cc, 0);
    const unsigned long long m0 = __shfl_sync(kFull, cm, 0);
    const uint32_t clo = lo_j >= 0 ? __shfl_sync(kFull, cc, lo_j + 1) : c0;
    const unsigned long long mlo = lo_j >= 0 ? __shfl_sync(kFull, cm, lo_j + 1) : m0;
    const uint32_t chi = hi_j >= 0 ? __shfl_sync(kFull, cc, hi_j + 1) : above_hi_c;
    const unsigned long long mhi = hi_j >= 0 ? __shfl_sync(kFull, cm, hi_j + 1) : above_hi_m;
    if (lane == 0) {
      F.bc.x[BX_TARGET] = tgt;
      F.bc.u[BU_BELOW] = (MASS ? (m0 < tgt) : (static_cast<unsigned long long>(c0) < tgt)) ? 1u : 0u;
      F.bc.u[BU_LO] = lo_j >= 0 ? vld(F.bc.q[lo_j]) : R.lo;
      F.bc.u[BU_HI] = hi_j >= 0 ? vld(F.bc.q[hi_j]) : R.hi;
      F.bc.u[BU_CLO] = clo;
      F.bc.u[BU_CHI] = chi;
      F.bc.x[BX_MLO] = mlo;
      F.bc.x[BX_MHI] = mhi;
    }
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
  R.target = vld(F.bc.x[BX_TARGET]);
  R.target_from_total = false;
  R.lo = vld(F.bc.u[BU_LO]);
  R.hi = vld(F.bc.u[BU_HI]);
  R.c_lo = vld(F.bc.u[BU_CLO]);
  R.c_hi = vld(F.bc.u[BU_CHI]);
  R.m_lo = vld(F.bc.x[BX_MLO]);
  R.m_hi = vld(F.bc.x[BX_MHI]);
  R.lo_all = R.lo < kKeyNegInf;
  const uint32_t maxr = vld(F.bc.u[BU_MAXR]);
  R.fits = maxr <= c.ocap;
  R.exact = !R.pin_hi && (R.hi - R.lo <= 1u);
  R.below = vld(F.bc.u[BU_BELOW]) != 0u;
  ++R.passes;
  *used_value_out = vld(F.bc.u[BU_USED_VALUE]) != 0u;
}

// ---------------------------------------------------------------------------
// Wide narrowing pass: four quaternary levels at once. The range (lo, hi] is
// cut into 256 equal value bins (255 pivots); one pass over the chunk counts
// (and weighs) every bin with per-warp shared-memory histograms, one cluster
// merge totals them, and the bin holding the boundary becomes the range.
// List-region layout while it runs: per-warp counts and masses at 0 (24 KiB),
// the CTA's bin totals for the cluster at kWideTotOff, the ring above them.
// Remote CTAs read the totals between the pass's two cluster barriers.
// ---------------------------------------------------------------------------
constexpr int kWideBins = 256;
static_assert(kWideBins == kThreads, "one thread per wide bin");
constexpr int kWideTotOff = kWarps * kWideBins * 12;
// bytes of the list region the wide pass keeps: histograms, then the totals
constexpr int kWideUsed = kWideTotOff + 2048 + (kWideBins + 1) * 8;

// Exact 64-bit shared-memory accumulation by two 32-bit atomics: the low
// word's carry (seen in the value the first atomic returns) goes into the
// high word with the high half. Much cheaper than a 64-bit shared atomic.
__device__ __forceinline__ void add_u64_halves(unsigned long long* p, unsigned long long v) {
  uint32_t* w = reinterpret_cast<uint32_t*>(p);  // little-endian: w[0] low, w[1] high
  const uint32_t l = static_cast<uint32_t>(v);
  const uint32_t old = atomicAdd(w, l);
  const uint32_t h = static_cast<uint32_t>(v >> 32) + ((old + l) < old ? 1u : 0u);
  if (h != 0u) atomicAdd(w + 1, h);
}

// Block-wide inclusive suffix sum over the 256 bins (thread b holds bin b):
// returns the sum of bins b..255 (u64; counts fit, masses are below 2^63).
template <int DT>
__device__ __forceinline__ unsigned long long bin_suffix_sum(Ctx<DT>& c, unsigned long long v) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // reverse order: prefix over r = 255 - b; warp w' = kWarps-1-warp holds r's block
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_down_sync(kFull, incl, o);
    if (lane + o < 32) incl += y;
  }
  // incl = sum of lanes lane..31 of this warp; add the warps above
  if (lane == 0) {
    F.redu[warp][0] = static_cast<uint32_t>(incl);
    F.redu[warp][1] = static_cast<uint32_t>(incl >> 32);
  }
  __syncthreads();
  unsigned long long above = 0ull;
  for (int w = warp + 1; w < kWarps; ++w)
    above += static_cast<unsigned long long>(vld(F.redu[w][0])) |
             (static_cast<unsigned long long>(vld(F.redu[w][1])) << 32);
  __syncthreads();
  return incl + above;
}

template <int DT, bool MASS>
__device__ bool wide_pass(Ctx<DT>& c, Range& R) {
  constexpr int E = Ctx<DT>::E;
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (R.lo_all) return false;
  const float lo_v = pivot_f(R.lo);
  const float hi_v = pivot_f(R.hi);
  if (!isfinite(lo_v) || !isfinite(hi_v) || !(hi_v > lo_v)) return false;
  const float w = (hi_v - lo_v) * (1.0f / kWideBins);
  const float inv_w = 1.0f / w;
  if (!(w > 0.f) || !isfinite(inv_w)) return false;
  // pivots q_b = lo + (b + 1) w (b < 255), q_255 = hi: must increase strictly;
  // recomputed wherever needed (the same expression gives the same float)
  auto edge = [&](int b) -> float {
    return b >= kWideBins - 1 ? hi_v : fmaf(static_cast<float>(b + 1), w, lo_v);
  };
  const float q_prev = tid == 0 ? lo_v : edge(tid - 1);
  const float q_mine = edge(tid);
  if (__syncthreads_or(!(q_mine > q_prev)) != 0) return false;

  uint32_t* wcnt = reinterpret_cast<uint32_t*>(c.lists);  // [kWarps][256]
  unsigned long long* wmass =
      reinterpret_cast<unsigned long long*>(c.lists + kWarps * kWideBins * 4);  // [kWarps][256]
  uint32_t* tot_cnt = reinterpret_cast<uint32_t*>(c.lists + kWideTotOff);  // [257]
  unsigned long long* tot_mass =
      reinterpret_cast<unsigned long long*>(c.lists + kWideTotOff + 2048);  // [257]
  for (int wv = 0; wv < kWarps; ++wv) {
    wcnt[wv * kWideBins + tid] = 0u;
    if (MASS) wmass[wv * kWideBins + tid] = 0ull;
  }
  __syncthreads();
  const float scale = c.fix_scale;
  uint32_t above_c = 0;
  unsigned long long above_m = 0ull;
  auto bin_one = [&](float x) {
    if (!(x > lo_v)) return;
    unsigned long long wf = 0ull;
    if (MASS) wf = weight_fx(x, c.m, c.m_neginf, scale);
    if (x > hi_v) {
      ++above_c;
      above_m += wf;
      return;
    }
    int b = static_cast<int>((x - lo_v) * inv_w);
    b = b < 0 ? 0 : (b > kWideBins - 1 ? kWideBins - 1 : b);
    // the estimate is within a bin of the truth: settle it on the pivots
    if (b > 0 && x <= edge(b - 1)) --b;
    if (b > 0 && x <= edge(b - 1)) --b;
    if (b < kWideBins - 1 && x > edge(b)) ++b;
    if (b < kWideBins - 1 && x > edge(b)) ++b;
    atomicAdd(&wcnt[warp * kWideBins + b], 1u);
    if (MASS) add_u64_halves(&wmass[warp * kWideBins + b], wf);
  };
  stream_chunk<DT>(
      c,
      [&](const float (&xs)[E], uint32_t, bool valid) {
        if (!valid) return;
#pragma unroll
        for (int e = 0; e < E; ++e) bin_one(xs[e]);
      },
      [&](float x, uint32_t, bool valid) {
        if (valid) bin_one(x);
      },
      false, ring_stages(list_region_bytes(static_cast<int>(c.ocap)), kWideUsed));
  above_c = __reduce_add_sync(kFull, above_c);
  above_m = warp_sum_u64(above_m);
  if (lane == 0) {
    F.redu[warp][2] = above_c;
    F.redu[warp][3] = static_cast<uint32_t>(above_m);
    F.redu[warp][4] = static_cast<uint32_t>(above_m >> 32);
  }
  __syncthreads();
  {
    uint32_t cb = 0;
    unsigned long long mb = 0ull;
    for (int wv = 0; wv < kWarps; ++wv) {
      cb += vld(wcnt[wv * kWideBins + tid]);
      if (MASS) mb += vld(wmass[wv * kWideBins + tid]);
    }
    tot_cnt[tid] = cb;
    tot_mass[tid] = mb;
    if (tid == 0) {
      uint32_t ac = 0;
      unsigned long long am = 0ull;
      for (int wv = 0; wv < kWarps; ++wv) {
        ac += vld(F.redu[wv][2]);
        am += static_cast<unsigned long long>(vld(F.redu[wv][3])) |
              (static_cast<unsigned long long>(vld(F.redu[wv][4])) << 32);
      }
      tot_cnt[kWideBins] = ac;
      tot_mass[kWideBins] = am;
    }
  }
  cluster_sync_all();
  // row totals of bin tid, and above hi
  uint32_t rc = 0;
  unsigned long long rm = 0ull;
  for (uint32_t r = 0; r < c.C; ++r) {
    rc += ld_dsmem_u32(map_rank(smem_u32(&tot_cnt[tid]), r));
    if (MASS) {
      const uint32_t a = map_rank(smem_u32(&tot_mass[tid]), r);
      rm += static_cast<unsigned long long>(ld_dsmem_u32(a)) |
            (static_cast<unsigned long long>(ld_dsmem_u32(a + 4)) << 32);
    }
  }
  uint32_t ac = 0;
  unsigned long long am = 0ull;
  for (uint32_t r = 0; r < c.C; ++r) {
    ac += ld_dsmem_u32(map_rank(smem_u32(&tot_cnt[kWideBins]), r));
    if (MASS) {
      const uint32_t a = map_rank(smem_u32(&tot_mass[kWideBins]), r);
      am += static_cast<unsigned long long>(ld_dsmem_u32(a)) |
            (static_cast<unsigned long long>(ld_dsmem_u32(a + 4)) << 32);
    }
  }
  // count / mass above the lower edge of bin tid (bins tid..255, and above hi)
  const unsigned long long sc = bin_suffix_sum(c, rc) + ac;
  const unsigned long long sm = MASS ? bin_suffix_sum(c, rm) + am : 0ull;
  // the target (measured here when it is a share of this pass's total)
  unsigned long long tgt = R.target;
  if (R.target_from_total) {
    if (tid == 0) {
      F.bc.x[BX_TARGET] = f2_to_u64(f2_mul(f2_from_u64(sm + R.extra), R.p_frac));
    }
    __syncthreads();
    tgt = vld(F.bc.x[BX_TARGET]);
  }
  // bin b holds the boundary when above(lower edge of b) reaches the target
  // and above(upper edge) does not: the upper edge's "above" is bin b+1's
  const unsigned long long my_above = MASS ? sm : sc;
  const unsigned long long nxt = __shfl_down_sync(kFull, my_above, 1);
  // above(upper edge of bin b) for lane 31 comes from the next warp's lane 0
  if (lane == 0) {
    F.redu[warp][5] = static_cast<uint32_t>(my_above);
    F.redu[warp][6] = static_cast<uint32_t>(my_above >> 32);
    F.redu[warp][7] = static_cast<uint32_t>(sc);
  }
  __syncthreads();
  unsigned long long up = nxt;
  uint32_t up_c = __shfl_down_sync(kFull, static_cast<uint32_t>(sc), 1);
  if (lane == 31) {
    if (warp + 1 < kWarps) {
      up = static_cast<unsigned long long>(vld(F.redu[warp + 1][5])) |
           (static_cast<unsigned long long>(vld(F.redu[warp + 1][6])) << 32);
      up_c = vld(F.redu[warp + 1][7]);
    } else {
      up = MASS ? am : ac;
      up_c = ac;
    }
  }
  const bool below = tid == 0 && my_above < tgt;
  const bool here = my_above >= tgt && up < tgt;
  // (lo, hi] held the boundary on entry, so one bin claims it (or "below");
  // should none, the range stays and the next pass narrows it
  const bool claimed = __syncthreads_or(here || below) != 0;
  if (!claimed && tid == 0) {
    F.bc.u[BU_LO] = R.lo;
    F.bc.u[BU_HI] = R.hi;
    F.bc.u[BU_CLO] = R.c_lo;
    F.bc.u[BU_CHI] = R.c_hi;
    F.bc.x[BX_MLO] = R.m_lo;
    F.bc.x[BX_MHI] = R.m_hi;
    F.bc.u[BU_MAXR] = 0xFFFFFFFFu;
  }
  if (here) {
    F.bc.u[BU_LO] = tid == 0 ? R.lo : f2key(q_prev);
    F.bc.u[BU_HI] = tid == kWideBins - 1 ? R.hi : f2key(q_mine);
    F.bc.u[BU_CLO] = static_cast<uint32_t>(sc);
    F.bc.u[BU_CHI] = up_c;
    F.bc.x[BX_MLO] = MASS ? sm : 0ull;
    F.bc.x[BX_MHI] = MASS ? up : 0ull;
    // per-rank counts inside the bin (differences are what the callers use)
    uint32_t maxr = 0;
    for (uint32_t r = 0; r < c.C; ++r) {
      const uint32_t n = ld_dsmem_u32(map_rank(smem_u32(&tot_cnt[tid]), r));
      F.rank_lo[r] = n;
      F.rank_hi[r] = 0u;
      maxr = n > maxr ? n : maxr;
    }
    F.bc.u[BU_MAXR] = maxr;
  }
  if (tid == 0) {
    F.bc.u[BU_BELOW] = below ? 1u : 0u;
    F.bc.x[BX_TARGET] = tgt;
  }
  if (tid == 0 && below) {
    // nothing narrows: keep the range, report "below"
    F.bc.u[BU_LO] = R.lo;
    F.bc.u[BU_HI] = R.hi;
    F.bc.u[BU_CLO] = static_cast<uint32_t>(sc);
    F.bc.u[BU_CHI] = R.c_hi;
    F.bc.x[BX_MLO] = MASS ? sm : 0ull;
    F.bc.x[BX_MHI] = R.m_hi;
    F.bc.u[BU_MAXR] = 0xFFFFFFFFu;
  }
  __syncthreads();
  R.target = vld(F.bc.x[BX_TARGET]);
  R.target_from_total = false;
  R.lo = vld(F.bc.u[BU_LO]);
  R.hi = vld(F.bc.u[BU_HI]);
  R.c_lo = vld(F.bc.u[BU_CLO]);
  R.c_hi = vld(F.bc.u[BU_CHI]);
  R.m_lo = vld(F.bc.x[BX_MLO]);
  R.m_hi = vld(F.bc.x[BX_MHI]);
  R.lo_all = R.lo < kKeyNegInf;
  R.below = vld(F.bc.u[BU_BELOW]) != 0u;
  const uint32_t maxr = vld(F.bc.u[BU_MAXR]);
  R.fits = !R.below && maxr <= c.ocap;
  R.exact = !R.below && (R.hi - R.lo <= 1u);
  ++R.passes;
  cluster_sync_all();  // every CTA is done reading the others' bin totals
  return true;
}

template <int DT, bool MASS>
__device__ void narrow(Ctx<DT>& c, Range& R) {
  bool value_ok = true;
  R.passes = 0;
  R.fits = false;
  R.exact = false;
  R.below = false;
  bool wide_done = false;
  while (true) {
    const uint32_t span_before = R.hi - R.lo;
    bool used_value = false;
    if (!wide_done && c.wide_ok && wide_pass<DT, MASS>(c, R)) {
      wide_done = true;
      used_value = true;
      QRITA_T(11);
    } else {
      narrow_pass<DT, MASS>(c, R, value_ok, &used_value);
    }
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
  QRITA_T(12);
}

// ---------------------------------------------------------------------------
// Top-p rows binned by the streaming pass (top-p alone, far more survivors
// than the lists hold): the streaming pass also counts and weighs the
// survivors in kPhBins value bins of [t, ph_hi] (bin(x) = trunc((x - t) nb /
// (ph_hi - t)), a monotone function of x, so bins are value intervals; the
// survivors above ph_hi are totalled apart, in compensated fp32). A bin's
// weights are fp32 exp(x - m_ref) (at most 1 there) in fixed point, summed as
// two 32-bit halves per warp: exact integer sums, the same in any order. The
// pass also writes a code byte per logit in place of its mask byte: 0 below
// t, 1 + bin in the bins, kPhCodeAbove above ph_hi. After the merge the bin
// that holds the boundary is exact; one pass over the chunk's code bytes
// (code_pass: 1 byte a logit, from L2) then writes the final mask byte of
// every logit outside that bin and extracts the bin's logits to the own
// list, weighed exactly in the search's fixed point; the search runs on the
// list when the masses confirm the bracket.
// List-region layout while the streaming pass runs: the high halves of the
// per-warp masses at 0, the low halves after them (kWarps * kHistBins words
// each); the CTA's totals at kPhTotOff (64-bit masses, then the count above
// ph_hi and its compensated fp32 mass).
// ---------------------------------------------------------------------------
constexpr int kHistBins = 256;
static_assert(kHistBins == kThreads, "one thread per histogram bin");
constexpr int kPhBins = kHistBins - 2;      // bins of the first pass: codes 1 .. kPhBins
constexpr uint32_t kPhCodeAbove = 255u;     // code of a survivor above ph_hi (0: below t)
constexpr int kPhTotOff = 2 * kWarps * kHistBins * 4;
constexpr int kPhAboveOff = kPhTotOff + kHistBins * 8;

// Largest key k in [a, b] with bin(k) <= g, given bin(a) <= g; bin is
// monotone in the key. A 32-way search by each warp (every lane returns it).
template <typename BinFn>
__device__ __forceinline__ uint32_t last_key_in_bins(uint32_t a, uint32_t b, int g, BinFn&& bin) {
  const int lane = threadIdx.x & 31;
  if (bin(b) <= g) return b;
  uint32_t lo = a, hi = b;  // bin(lo) <= g < bin(hi)
  for (int it = 0; it < 40 && hi - lo > 1u; ++it) {
    const uint32_t span = hi - lo;
    const uint32_t probe = lo + static_cast<uint32_t>((static_cast<uint64_t>(span) * (lane + 1)) >> 5);
    const uint32_t bal = __ballot_sync(kFull, lane < 31 && bin(probe) <= g);
    const int L = __popc(bal);  // probes 0 .. L-1 are in, probe L (or hi) is out
    const uint32_t nlo = __shfl_sync(kFull, probe, L > 0 ? L - 1 : 0);
    const uint32_t nhi = __shfl_sync(kFull, probe, L < 31 ? L : 31);
    if (L > 0) lo = nlo;
    hi = L < 31 ? nhi : hi;
  }
  return lo;
}

template <int DT>
__device__ void own_segments_streamed(Ctx<DT>& c, uint32_t wn);

// The pass after the first-pass bins: one pass over the chunk's code bytes
// (the streaming pass wrote them in place of the mask bytes). A code above
// [c_lo, c_hi] becomes 1, one below it 0; a logit whose code lies in the
// range is reloaded from the row into this warp's segment of the own list,
// a lane claiming its slot with one shared atomic, and its byte becomes 0
// until the search decides. Publishes the own list's segments and returns
// this thread's count of logits above the range.
template <int DT>
__device__ uint32_t code_pass(Ctx<DT>& c, uint32_t c_lo, uint32_t c_hi) {
  constexpr int S = Ctx<DT>::S;
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t segcap = c.ocap / kWarps;
  const uint32_t seg_base = static_cast<uint32_t>(warp) * segcap;
  if (lane == 0) F.seg_n[warp] = 0u;
  __syncthreads();  // (also: every code byte of the chunk is written)
  uint8_t* m = c.gmask;
  const int n = c.n;
  // the final byte of logit i with code `code` (a logit in the range gets
  // its slot and index now, its value after the pass)
  auto one = [&](uint32_t code, int i) -> uint32_t {
    if (code >= c_lo && code <= c_hi) {
      const uint32_t pos = atomicAdd(&F.seg_n[warp], 1u);
      if (pos < segcap) c.own_idx[seg_base + pos] = static_cast<uint32_t>(i);
      return 0u;
    }
    return code > c_hi ? 1u : 0u;
  };
  // the four final bytes of a word of codes at byte offset i0. A word
  // without a code in the range (no byte equal to c_lo ... c_hi; this pass
  // runs with c_lo == c_hi) takes four byte compares at once: b > c_hi
  // exactly when b + (255 - c_hi) carries out of the byte, the carry being
  // the majority of the two top bits and the carry into bit 7
  const uint32_t cc4 = c_lo * 0x01010101u;
  const uint32_t d4 = (255u - c_hi) * 0x01010101u;
  const uint32_t d_low = d4 & 0x7F7F7F7Fu, d_top = d4 & 0x80808080u;
  auto word = [&](uint32_t v, int i0) -> uint32_t {
    const uint32_t t = v ^ cc4;
    if (c_lo != c_hi || ((t - 0x01010101u) & ~t & 0x80808080u) != 0u) {
      uint32_t out = 0u;
#pragma unroll
      for (int b = 0; b < 4; ++b) out |= one((v >> (8 * b)) & 0xFFu, i0 + b) << (8 * b);
      return out;
    }
    const uint32_t low = (v & 0x7F7F7F7Fu) + d_low;
    const uint32_t carry = (v & d_top) | ((v | d_top) & low);
    return (carry >> 7) & 0x01010101u;
  };
  // bytes to the first 16-byte boundary, then 16-byte vectors (four of them
  // a thread in flight: the loads do not wait on the stores before them),
  // then the last bytes
  const int head = min(static_cast<int>((16u - static_cast<uint32_t>(reinterpret_cast<uintptr_t>(m) & 15u)) & 15u), n);
  const int nv = (n - head) / 16;
  const int tail0 = head + 16 * nv;
  uint32_t above = 0;
  if (tid < head) {
    const uint32_t b = one(m[tid], tid);
    m[tid] = static_cast<uint8_t>(b);
    above += b;
  }
  uint4* mv = reinterpret_cast<uint4*>(m + head);
  constexpr int kV = 4;
  for (int vb = 0; vb < nv; vb += kV * kThreads) {
    uint4 v[kV];
#pragma unroll
    for (int q = 0; q < kV; ++q) {
      const int iv = vb + q * kThreads + tid;
      v[q] = iv < nv ? mv[iv] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int q = 0; q < kV; ++q) {
      const int iv = vb + q * kThreads + tid;
      if (iv < nv) {
        const int i0 = head + 16 * iv;
        const uint4 o = make_uint4(word(v[q].x, i0), word(v[q].y, i0 + 4), word(v[q].z, i0 + 8), word(v[q].w, i0 + 12));
        mv[iv] = o;
        above += __popc(o.x) + __popc(o.y) + __popc(o.z) + __popc(o.w);  // (bytes are 0 or 1)
      }
    }
  }
  if (tid < n - tail0) {
    const uint32_t b = one(m[tail0 + tid], tail0 + tid);
    m[tail0 + tid] = static_cast<uint8_t>(b);
    above += b;
  }
  __syncthreads();
  // the listed logits' values, loaded together
  const uint32_t wn = vld(F.seg_n[warp]);
  gather_segment_values<DT>(c, seg_base, min(wn, segcap));
  own_segments_streamed<DT>(c, wn);
  return above;
}

// Cluster merge after the pass that lists a range: F.rank_n[r] (list entries of rank r),
// F.bc.u[BU_S2] (row list entries), F.bc.u[BU_OVF2] (a list overflowed),
// F.bc.u[BU_CHI] (row count above hi), F.bc.x[BX_MHI] / [BX_MLO] (row mass
// above hi / of the lists).
template <int DT>
__device__ void merge_split(Ctx<DT>& c, uint32_t n, uint32_t ovf, uint32_t ca, unsigned long long ma,
                            unsigned long long mi) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Slot& my = F.slots[c.ph & 1];
  if (tid == 0) {
    my.u[0] = n;
    my.u[1] = ovf;
    my.u[2] = ca;
    my.mass[0] = ma;
    my.mass[1] = mi;
  }
  cluster_sync_all();
  if (warp == 0) {
    uint32_t rn = 0, ro = 0, rc = 0;
    unsigned long long rma = 0ull, rmi = 0ull;
    if (lane < static_cast<int>(c.C)) {
      const uint32_t ub = map_rank(smem_u32(&my.u[0]), static_cast<uint32_t>(lane));
      const uint32_t mb = map_rank(smem_u32(&my.mass[0]), static_cast<uint32_t>(lane));
      rn = ld_dsmem_u32(ub);
      ro = ld_dsmem_u32(ub + 4u);
      rc = ld_dsmem_u32(ub + 8u);
      rma = static_cast<unsigned long long>(ld_dsmem_u32(mb)) |
            (static_cast<unsigned long long>(ld_dsmem_u32(mb + 4u)) << 32);
      rmi = static_cast<unsigned long long>(ld_dsmem_u32(mb + 8u)) |
            (static_cast<unsigned long long>(ld_dsmem_u32(mb + 12u)) << 32);
      ro |= rn > c.ocap ? 1u : 0u;
      F.rank_n[lane] = rn;
    }
    const uint32_t tn = __reduce_add_sync(kFull, rn);
    const uint32_t to = __reduce_or_sync(kFull, ro);
    const uint32_t tcn = __reduce_add_sync(kFull, rc);
    const unsigned long long tma = warp_sum_u64(rma);
    const unsigned long long tmi = warp_sum_u64(rmi);
    if (lane == 0) {
      F.bc.u[BU_S2] = tn;
      F.bc.u[BU_OVF2] = to;
      F.bc.u[BU_CHI] = tcn;
      F.bc.x[BX_MHI] = tma;
      F.bc.x[BX_MLO] = tmi;
    }
  }
  __syncthreads();
  ++c.ph;
}

// The own list as kWarps segments: warp w owns entries [seg_base[w],
// seg_base[w] + seg_cnt[w]). After the streaming pass (and the second
// truncation) segment w holds warp w's survivors at w * segcap: publish the
// counts; F.own_n gets the exact survivor count and F.seg_ovf whether a
// warp's survivors exceeded its segment.
template <int DT>
__device__ void own_segments_streamed(Ctx<DT>& c, uint32_t wn) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t segcap = c.ocap / kWarps;
  if (lane == 0) {
    F.seg_n[warp] = wn;
    F.seg_base[warp] = static_cast<uint32_t>(warp) * segcap;
    F.seg_cnt[warp] = min(wn, segcap);
  }
  if (tid == 0) F.col_mode = 0u;
  __syncthreads();
  if (tid == 0) {
    uint32_t total = 0;
    bool ovf = false;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t n = vld(F.seg_n[w]);
      total += n;
      ovf = ovf || n > segcap;
    }
    F.own_n = total;
    F.seg_ovf = ovf ? 1u : 0u;
  }
  __syncthreads();
}

// After an extraction (entries [0, own_n) of the own list): eight equal
// slices, one per warp.
template <int DT>
__device__ void own_segments_contiguous(Ctx<DT>& c) {
  Fixed& F = *c.F;
  if (threadIdx.x == 0) {
    const uint32_t total = vld(F.own_n);
    const uint32_t n = min(total, c.ocap);
    const uint32_t slice = (n + kWarps - 1u) / kWarps;
    for (int w = 0; w < kWarps; ++w) {
      const uint32_t b = min(static_cast<uint32_t>(w) * slice, n);
      F.seg_base[w] = b;
      F.seg_cnt[w] = min(slice, n - b);
    }
    F.seg_ovf = total > c.ocap ? 1u : 0u;
    F.col_mode = 0u;
  }
  __syncthreads();
}

// After a streaming pass in column mode: thread t kept its survivors at
// t + j * kThreads (cn of them counted, at most ocap / kThreads stored).
template <int DT>
__device__ void own_columns_streamed(Ctx<DT>& c, uint32_t cn) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t colcap = c.ocap / kThreads;
  F.col_n[tid] = static_cast<uint8_t>(min(cn, colcap));
  const uint32_t ws = __reduce_add_sync(kFull, cn);
  if (lane == 0) F.seg_n[warp] = ws;
  const bool ovf = __syncthreads_or(cn > colcap) != 0;
  if (tid == 0) {
    uint32_t total = 0;
    for (int w = 0; w < kWarps; ++w) total += vld(F.seg_n[w]);
    F.own_n = total;
    F.seg_ovf = ovf ? 1u : 0u;
    F.col_mode = 1u;
  }
  __syncthreads();
}

// Columns to warp segments (the form the search and the emission scan
// fastest): each warp's column entries are staged densely in the ring's bytes
// (no stream is in flight) and copied back to the warp's segment. Left in
// columns when a warp holds more than the staging gives it.
template <int DT>
__device__ void own_columns_to_segments(Ctx<DT>& c) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr uint32_t kStage = kRingBytes / 8 / kWarps;  // entries per warp
  const uint32_t segcap = c.ocap / kWarps;
  const uint32_t n = vld(F.col_n[tid]);  // (at most the column capacity)
  uint32_t incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  const uint32_t tot = __shfl_sync(kFull, incl, 31);
  if (__syncthreads_or(tot > kStage || vld(F.seg_ovf) != 0u) != 0) return;
  float* sv = reinterpret_cast<float*>(const_cast<uint4*>(c.ring_ptr));
  uint32_t* si = reinterpret_cast<uint32_t*>(sv + kStage * kWarps);
  const uint32_t base = static_cast<uint32_t>(warp) * kStage + (incl - n);
  for (uint32_t j = 0; j < n; ++j) {
    sv[base + j] = c.own_val[j * kThreads + tid];
    si[base + j] = c.own_idx[j * kThreads + tid];
  }
  __syncthreads();  // every column is staged: the list region is free
  const uint32_t dst = static_cast<uint32_t>(warp) * segcap, src = static_cast<uint32_t>(warp) * kStage;
  for (uint32_t i = lane; i < tot; i += 32u) {
    c.own_val[dst + i] = sv[src + i];
    c.own_idx[dst + i] = si[src + i];
  }
  if (lane == 0) {
    F.seg_base[warp] = dst;
    F.seg_cnt[warp] = tot;
  }
  __syncthreads();
  if (tid == 0) F.col_mode = 0u;
  __syncthreads();
}

// fn(value, index) over this thread's share of the own list: its column, or
// its lane's stride of its warp's segment. Warp collectives inside fn must use
// the active mask (the lanes' trip counts differ).
template <int DT, typename Fn>
__device__ __forceinline__ void own_for(Ctx<DT>& c, Fn&& fn) {
  Fixed& F = *c.F;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (vld(F.col_mode) != 0u) {
    const uint32_t n = vld(F.col_n[threadIdx.x]);
    for (uint32_t j = 0; j < n; ++j) {
      const uint32_t i = j * kThreads + threadIdx.x;
      fn(c.own_val[i], c.own_idx[i]);
    }
    return;
  }
  const uint32_t base = vld(F.seg_base[warp]), n = vld(F.seg_cnt[warp]);
  for (uint32_t i = static_cast<uint32_t>(lane); i < n; i += 32u) fn(c.own_val[base + i], c.own_idx[base + i]);
}

// fn(value, index, valid) over this thread's share of the own list, like
// own_for, but every lane of a warp runs the same number of steps (a lane past
// its share passes valid = false), so fn may use full-warp collectives.
template <int DT, typename Fn>
__device__ __forceinline__ void own_for_warp(Ctx<DT>& c, Fn&& fn) {
  Fixed& F = *c.F;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (vld(F.col_mode) != 0u) {
    const uint32_t n = vld(F.col_n[threadIdx.x]);
    const uint32_t nmax = __reduce_max_sync(kFull, n);
    for (uint32_t j = 0; j < nmax; ++j) {
      const bool v = j < n;
      const uint32_t i = j * kThreads + threadIdx.x;
      fn(v ? c.own_val[i] : 0.f, v ? c.own_idx[i] : 0u, v);
    }
    return;
  }
  const uint32_t base = vld(F.seg_base[warp]), n = vld(F.seg_cnt[warp]);
  for (uint32_t i0 = 0; i0 < n; i0 += 32u) {
    const uint32_t i = i0 + static_cast<uint32_t>(lane);
    const bool v = i < n;
    fn(v ? c.own_val[base + i] : 0.f, v ? c.own_idx[base + i] : 0u, v);
  }
}

// Per-rank own-list counts above the search's lo and hi (F.rank_lo,
// F.rank_hi): n[r] entries of rank r lie above lo, none above hi.
template <int DT>
__device__ void rank_counts_from(Ctx<DT>& c, const uint32_t* n) {
  Fixed& F = *c.F;
  if (threadIdx.x < static_cast<int>(c.C)) {
    const uint32_t v = vld(n[threadIdx.x]);
    F.rank_lo[threadIdx.x] = v;
    F.rank_hi[threadIdx.x] = 0u;
  }
  __syncthreads();
}

// Position of sample element sidx of an n-element sample spread as blocks of
// 64 contiguous logits over the row (the whole row when V <= n).
__device__ __forceinline__ int64_t sample_pos(int sidx, int n, int V) {
  if (V <= n) return sidx;
  const int blocks = n / 64;
  return static_cast<int64_t>(sidx / 64) * (V / blocks) + (sidx % 64);
}

// The key of the j-th largest (j >= 1) of the keys the threads hold (have[q]
// marks the valid ones), by an MSB-first radix select with 8-bit digits over
// a 256-bin histogram in shared memory. Every thread returns the same key.
template <int DT, int N>
__device__ uint32_t radix_select(Ctx<DT>& c, const uint32_t (&key)[N], const bool (&have)[N], uint32_t j,
                                 uint32_t* hist) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t prefix = 0, mask = 0, want = j;
  __syncthreads();  // earlier users of the histogram's bytes are done
  for (int d = 3; d >= 0; --d) {
    hist[tid] = 0u;  // kThreads == 256 bins
    __syncthreads();
    const int sh = 8 * d;
#pragma unroll
    for (int q = 0; q < N; ++q)
      if (have[q] && (key[q] & mask) == prefix) atomicAdd(&hist[(key[q] >> sh) & 255u], 1u);
    __syncthreads();
    if (tid < 32) {
      // lane l holds bins 255 - 8l .. 248 - 8l (from the top)
      uint32_t b8[8], sum = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        b8[q] = vld(hist[255 - 8 * lane - q]);
        sum += b8[q];
      }
      uint32_t incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - sum;
      const bool here = excl < want && want <= incl;
      if (here) {
        uint32_t acc = excl;
        int bin = 255 - 8 * lane - 7;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (acc < want && want <= acc + b8[q]) {
            bin = 255 - 8 * lane - q;
            want -= acc;
          }
          acc += b8[q];
        }
        F.bc.u[BU_QKEY] = static_cast<uint32_t>(bin);
        F.bc.u[BU_QWANT] = want;
      }
    }
    __syncthreads();
    prefix |= vld(F.bc.u[BU_QKEY]) << sh;
    mask |= 255u << sh;
    want = vld(F.bc.u[BU_QWANT]);
    __syncthreads();
  }
  return prefix;
}

// The key of the j-th largest logit of a kRetrySample-logit sample of the
// row (of the whole row when V <= kRetrySample); the histogram lives in the
// ring's bytes (no stream is in flight).
template <int DT>
__device__ uint32_t sample_order_key(Ctx<DT>& c, const unsigned char* grow, int V, uint32_t j) {
  constexpr int S = Ctx<DT>::S;
  const int tid = threadIdx.x;
  uint32_t key[kRetryPer];
  bool have[kRetryPer];
#pragma unroll
  for (int q = 0; q < kRetryPer; ++q) {
    const int sidx = tid + q * kThreads;
    const int64_t pos = sample_pos(sidx, kRetrySample, V);
    have[q] = pos < V;
    key[q] = have[q] ? f2key(load_elem<DT>(grow + static_cast<size_t>(pos) * S)) : 0u;
  }
  return radix_select<DT, kRetryPer>(c, key, have, j, reinterpret_cast<uint32_t*>(const_cast<uint4*>(c.ring_ptr)));
}

// Survivors (x >= t2) of the chunk into the warps' segments of the own list,
// compacted; then one cluster merge of the counts: F.rank_n, F.bc.u[BU_S2]
// (row survivors) and F.bc.u[BU_OVF2] (some list overflowed).
template <int DT>
__device__ void retry_pass(Ctx<DT>& c, float t2) {
  constexpr int E = Ctx<DT>::E;
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t segcap = c.ocap / kWarps;
  const uint32_t seg_base = static_cast<uint32_t>(warp) * segcap;
  uint32_t wn = 0;
  stream_pieces<DT>(
      c,
      [&](const uint4 (&v)[kPieceThreadUnits], int u0, int n) {
        float xs[kPieceThreadUnits][E];
        uint32_t bits[kPieceThreadUnits];
#pragma unroll
        for (int j = 0; j < kPieceThreadUnits; ++j) {
          unpack<DT>(v[j], xs[j]);
          bits[j] = 0u;
          if (j * kThreads + tid < n) {
#pragma unroll
            for (int e = 0; e < E; ++e) bits[j] |= (xs[j][e] >= t2) ? (1u << e) : 0u;
          }
        }
        append_piece<DT>(c, wn, seg_base, segcap, xs, bits, u0);
      },
      [&](float x, uint32_t idx, bool valid) {
        const float xs[1] = {x};
        seg_append<1>(wn, c.own_val, c.own_idx, seg_base, segcap, xs, idx, (valid && x >= t2) ? 1u : 0u);
      },
      false);
  own_segments_streamed<DT>(c, wn);
  Slot& my = F.slots[c.ph & 1];
  if (tid == 0) {
    my.u[0] = vld(F.seg_ovf);
    my.u[1] = vld(F.own_n);
  }
  cluster_sync_all();
  if (warp == 0) {
    uint32_t n = 0, o = 0;
    if (lane < static_cast<int>(c.C)) {
      const uint32_t ub = map_rank(smem_u32(&my.u[0]), lane);
      o = ld_dsmem_u32(ub);
      n = ld_dsmem_u32(ub + 4);
      o |= n > c.ocap ? 1u : 0u;
      F.rank_n[lane] = n;
    }
    n = __reduce_add_sync(kFull, n);
    o = __reduce_or_sync(kFull, o);
    if (lane == 0) {
      F.bc.u[BU_S2] = n;
      F.bc.u[BU_OVF2] = o;
    }
  }
  __syncthreads();
  ++c.ph;
}

// ---------------------------------------------------------------------------
// Local quaternary search over the gathered set (block barriers only)
// ---------------------------------------------------------------------------
struct Local {
  uint32_t lo, hi, c_lo, c_hi;   // row counts above lo / hi
  unsigned long long m_lo, m_hi;  // row masses above lo / hi (fixed point, mass search)
  uint32_t c_above;               // row count above the gathered range
  unsigned long long m_above;     // row mass above the gathered range (fixed point)
  // result
  uint32_t tau, n_keep, count_above;
  int rounds;
  bool capped;
};

// Copies of a boundary value of fixed-point weight w needed when `need`
// mass is missing above it: ceil(need / w), clamped to [1, n].
__device__ __forceinline__ uint32_t copies_fx(unsigned long long need, unsigned long long w, uint32_t n) {
  unsigned long long k = w > 0ull ? (need + w - 1ull) / w : 1ull;
  k = k < 1ull ? 1ull : (k > n ? static_cast<unsigned long long>(n) : k);
  return static_cast<uint32_t>(k);
}


// Sum of a 64-bit value over the warp with 32-bit reductions: split into
// 21-bit parts, so no part's sum can wrap (values below 2^63).
__device__ __forceinline__ unsigned long long warp_sum_u64_redux(unsigned long long v) {
  const uint32_t p0 = static_cast<uint32_t>(v & 0x1FFFFFull);
  const uint32_t p1 = static_cast<uint32_t>((v >> 21) & 0x1FFFFFull);
  const uint32_t p2 = static_cast<uint32_t>(v >> 42);
  const unsigned long long s0 = __reduce_add_sync(kFull, p0);
  const unsigned long long s1 = __reduce_add_sync(kFull, p1);
  const unsigned long long s2 = __reduce_add_sync(kFull, p2);
  return s0 + (s1 << 21) + (s2 << 42);
}

// One cluster merge of a per-CTA count, mass and overflow flag (thread 0's
// arguments are what this CTA publishes): afterwards F.rank_n[r] is rank r's
// count, F.bc.u[BU_S2] the row total, F.bc.u[BU_MAXR] the largest count,
// F.bc.u[BU_OVF2] whether any rank flagged (or exceeded the list capacity)
// and F.bc.x[BX_MLO] the row's mass.
template <int DT>
__device__ void merge_count_mass(Ctx<DT>& c, uint32_t n, unsigned long long m, uint32_t ovf) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  Slot& my = F.slots[c.ph & 1];
  if (tid == 0) {
    my.u[0] = n;
    my.u[1] = ovf;
    my.mass[0] = m;
  }
  cluster_sync_all();
  if (warp == 0) {
    uint32_t rn = 0, ro = 0;
    unsigned long long rm = 0ull;
    if (lane < static_cast<int>(c.C)) {
      const uint32_t ub = map_rank(smem_u32(&my.u[0]), static_cast<uint32_t>(lane));
      rn = ld_dsmem_u32(ub);
      ro = ld_dsmem_u32(ub + 4u);
      const uint32_t mb = map_rank(smem_u32(&my.mass[0]), static_cast<uint32_t>(lane));
      rm = static_cast<unsigned long long>(ld_dsmem_u32(mb)) |
           (static_cast<unsigned long long>(ld_dsmem_u32(mb + 4u)) << 32);
      ro |= rn > c.ocap ? 1u : 0u;
      F.rank_n[lane] = rn;
    }
    const uint32_t tot = __reduce_add_sync(kFull, rn);
    const uint32_t mx = __reduce_max_sync(kFull, rn);
    const uint32_t o = __reduce_or_sync(kFull, ro);
    const unsigned long long tm = warp_sum_u64_redux(rm);
    if (lane == 0) {
      F.bc.u[BU_S2] = tot;
      F.bc.u[BU_MAXR] = mx;
      F.bc.u[BU_OVF2] = o;
      F.bc.x[BX_MLO] = tm;
    }
  }
  __syncthreads();
  ++c.ph;
}

// Tail of the search: once the range holds at most kTail elements (over the
// whole row) they are copied to every CTA, split into kTailBins value bins,
// and the elements of the bin holding the boundary each test themselves.
// Layout in the ring's bytes: values, weights, ranks, then the compacted
// candidates' values and weights.
constexpr int kTail = 1024;
// Bracket pivots: before the streaming pass, the Gaussian model places
// kBracket pivots where the count above is expected to be m_j k, m_j =
// 2^((7 - j) / 5) (2.6 k down to 0.38 k); each CTA counts its survivors
// above them and the first cluster merge totals the counts, so the top-k
// search starts from the bracket that holds the boundary.
constexpr int kBracket = 15;
constexpr int kTailBins = 64;
constexpr int kTailLevels = 3;   // bin splits of the tail at most
constexpr int kTailDirect = 64;  // sets this small are tested directly
constexpr int kTailValOff = 0;
constexpr int kTailWOff = kTailValOff + kTail * 4;
constexpr int kTailRankOff = kTailWOff + kTail * 8;
constexpr int kCandValOff = kTailRankOff + kTail;
constexpr int kCandWOff = kCandValOff + kTail * 4;
static_assert(kCandWOff + kTail * 8 <= kRingBytes, "the search tail exceeds the ring's bytes");
static_assert(kCandWOff % 8 == 0 && kTailWOff % 8 == 0, "tail weights are 8-byte aligned");
static_assert(kTailBins == 64, "the bin scan gives each lane of one warp two bins");

// Distributed search (A6 for counts, A7 for mass) over the own lists of the
// cluster: the pages' quaternary search, generalised to kSplit-way rounds.
// The search keeps count/mass(> lo) >= target > count/mass(> hi). Each round
// cuts (lo, hi] into kSplit bins by a monotone function of the value (equal
// value widths; equal key widths after a value split that kept more than half
// of the range), every CTA counts (and weighs) its own list into them, the
// bins merge through distributed shared memory, and every CTA keeps the bin
// where the count (mass) from the top reaches the target. Once the range
// holds at most kTail elements they are gathered and tested directly (the
// tail, where the pages' z_mn / N_zmn test decides). Masses are exact sums of
// fixed-point weights, so every decision is integer arithmetic.
// On entry F.rank_lo / F.rank_hi hold each rank's own-list counts above lo /
// hi, and s.c_hi / s.m_hi the row's count and mass above hi (including what
// lies above the lists' range). Each round scans only the lists' (lo, hi].
// On exit F.ties holds each rank's count of the boundary value.
// synced: a cluster barrier passed since any CTA of the row last used its
// ring (the tail is stored into the other CTAs' rings).
constexpr int kSplit = kTailBins;
struct RoundBin {  // one bin of one CTA's round, published for the cluster
  uint32_t cnt, above;  // elements in the bin, in the bins above it
  unsigned long long mass;
};
constexpr int kRoundPubOff = 26 * 1024;  // two alternating areas in the ring's bytes
static_assert(kRoundPubOff >= kCandWOff + kTail * 8, "round bins overlap the tail");
static_assert(kRoundPubOff + 2 * kSplit * static_cast<int>(sizeof(RoundBin)) <= kRingBytes,
              "round bins exceed the ring's bytes");

template <int DT, bool MASS>
__device__ void dsearch(Ctx<DT>& c, Local& s, unsigned long long target, bool value_pivots, bool synced = true) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float scale = c.fix_scale;
  const int C = static_cast<int>(c.C);
  // the search state is held, identical, by every thread of every CTA
  uint32_t lo = s.lo, hi = s.hi, c_lo = s.c_lo, c_hi = s.c_hi;
  unsigned long long m_lo = s.m_lo, m_hi = s.m_hi;
  uint32_t tau = 0, n_keep = 0, cabove = 0;
  int done = 0;  // 1: boundary found, 2: round cap
  bool collapsed = false;  // (lo, hi] holds one key: the boundary is hi
  // the boundary is the single key hi of (lo, hi]: keep the copies needed
  auto one_key = [&]() {
    tau = hi;
    cabove = c_hi;
    if (MASS) {
      const unsigned long long w = weight_fx(key2f(hi), c.m, c.m_neginf, scale);
      n_keep = copies_fx(target - m_hi, w, c_lo - c_hi);
    } else {
      n_keep = static_cast<uint32_t>(target) - c_hi;
    }
    done = 1;
    collapsed = true;
  };
  int rounds = 0;
  bool vmode = value_pivots;
  if (hi - lo <= 1u) one_key();
  RoundBin* pub = reinterpret_cast<RoundBin*>(reinterpret_cast<unsigned char*>(const_cast<uint4*>(c.ring_ptr)) +
                                              kRoundPubOff);
  // rounds over the own lists while the range is large
  while (done == 0 && c_lo - c_hi > static_cast<uint32_t>(kTail)) {
    if (rounds >= kMaxRounds) {
      done = 2;
      break;
    }
    const float lo_f = pivot_f(lo), hi_f = pivot_f(hi);
    const int ns = c.split;  // bins this round (kSplit unless a flag narrows it)
    const float inv = static_cast<float>(ns) / (hi_f - lo_f);
    const bool val = vmode && isfinite(lo_f) && isfinite(hi_f) && hi_f > lo_f && isfinite(inv) && inv > 0.f;
    const uint32_t span = hi - lo;
    // bin of a key in (lo, hi]: monotone in the key
    auto bin_of_key = [&](uint32_t k) -> int {
      if (val) {
        const int b = static_cast<int>((key2f(k) - lo_f) * inv);
        return b < 0 ? 0 : (b > ns - 1 ? ns - 1 : b);
      }
      return static_cast<int>((static_cast<uint64_t>(k - lo - 1u) * static_cast<uint64_t>(ns)) / span);
    };
    if (tid < kSplit) {
      F.tbin_c[tid] = 0u;
      F.tbin_m[tid] = 0ull;
    }
    __syncthreads();
    // only the range (lo, hi] is scanned: what lies above hi is counted in
    // c_hi / m_hi (and per rank in F.rank_hi) already
    own_for(c, [&](float x, uint32_t) {
      const uint32_t key = f2key(x);
      if (key <= lo || key > hi) return;
      const int b = bin_of_key(key);
      atomicAdd(&F.tbin_c[b], 1u);
      if (MASS) add_u64_halves(&F.tbin_m[b], weight_fx(x, c.m, c.m_neginf, scale));
    });
    __syncthreads();
    QRITA_T(8);
    RoundBin* my = pub + (rounds & 1) * kSplit;
    if (warp == 0) {
      // this CTA's bins, with the count above each, for the cluster (lane l:
      // bins 2l, 2l + 1)
      const uint32_t n0 = vld(F.tbin_c[2 * lane]), n1 = vld(F.tbin_c[2 * lane + 1]);
      uint32_t incl = n0 + n1;  // bins 2l .. 63 after the scan
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, incl, o);
        if (lane + o < 32) incl += y;
      }
      const uint32_t above1 = incl - n0 - n1;
      my[2 * lane] = RoundBin{n0, above1 + n1, MASS ? vld(F.tbin_m[2 * lane]) : 0ull};
      my[2 * lane + 1] = RoundBin{n1, above1, MASS ? vld(F.tbin_m[2 * lane + 1]) : 0ull};
    }
    cluster_sync_all();
    QRITA_T(9);
    if (tid < kSplit) {
      // the row's bin tid
      uint32_t rc = 0;
      unsigned long long rm = 0ull;
      for (int r = 0; r < C; ++r) {
        const uint32_t ab = map_rank(smem_u32(&my[tid]), static_cast<uint32_t>(r));
        rc += ld_dsmem_u32(ab);
        if (MASS)
          rm += static_cast<unsigned long long>(ld_dsmem_u32(ab + 8u)) |
                (static_cast<unsigned long long>(ld_dsmem_u32(ab + 12u)) << 32);
      }
      F.tbin_c[tid] = rc;
      F.tbin_m[tid] = rm;
    }
    __syncthreads();
    if (warp == 0) {
      // lane l holds bins 63 - 2l and 62 - 2l; prefix sums from the top find
      // the first bin whose cumulative total reaches the target
      const int b0 = kSplit - 1 - 2 * lane, b1 = b0 - 1;
      const uint32_t n0 = vld(F.tbin_c[b0]), n1 = vld(F.tbin_c[b1]);
      const unsigned long long v0w = MASS ? vld(F.tbin_m[b0]) : static_cast<unsigned long long>(n0);
      const unsigned long long v1w = MASS ? vld(F.tbin_m[b1]) : static_cast<unsigned long long>(n1);
      unsigned long long inc = v0w + v1w;
      uint32_t inc_n = n0 + n1;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(kFull, inc, o);
        const uint32_t yn = __shfl_up_sync(kFull, inc_n, o);
        if (lane >= o) {
          inc += y;
          inc_n += yn;
        }
      }
      const unsigned long long top = MASS ? m_hi : static_cast<unsigned long long>(c_hi);
      const unsigned long long ex = top + inc - (v0w + v1w);
      const uint32_t ex_n = c_hi + inc_n - (n0 + n1);
      const bool r0 = ex + v0w >= target, r1 = ex + v0w + v1w >= target;
      const uint32_t hit = __ballot_sync(kFull, r1);
      // (lo, hi] holds the boundary, so some bin reaches the target
      const int L = hit != 0u ? __ffs(hit) - 1 : 31;
      if (lane == L) {
        const bool first = r0;  // (no lane reached: lane 31 takes bin 0)
        const int bs = first ? b0 : b1;
        const uint32_t an = first ? ex_n : ex_n + n0;
        const unsigned long long am = first ? ex : ex + v0w;
        F.bc.u[BU_NP] = static_cast<uint32_t>(bs);
        F.bc.u[BU_CHI] = an;
        F.bc.u[BU_CLO] = an + (first ? n0 : n1);
        F.bc.x[BX_MHI] = MASS ? am : 0ull;
        F.bc.x[BX_MLO] = MASS ? am + (first ? v0w : v1w) : 0ull;
      }
    }
    __syncthreads();
    const int bs = static_cast<int>(vld(F.bc.u[BU_NP]));
    if (tid < C) {
      // rank tid's list counts above the new hi and lo
      const uint32_t ab = map_rank(smem_u32(&my[bs]), static_cast<uint32_t>(tid));
      const uint32_t in_bin = ld_dsmem_u32(ab), above = ld_dsmem_u32(ab + 4u);
      const uint32_t nh = vld(F.rank_hi[tid]) + above;
      F.rank_hi[tid] = nh;
      F.rank_lo[tid] = nh + in_bin;
    }
    const uint32_t old_n = c_lo - c_hi;
    c_hi = vld(F.bc.u[BU_CHI]);
    c_lo = vld(F.bc.u[BU_CLO]);
    m_hi = vld(F.bc.x[BX_MHI]);
    m_lo = vld(F.bc.x[BX_MLO]);
    const uint32_t nlo = bs == 0 ? lo : last_key_in_bins(lo + 1u, hi, bs - 1, bin_of_key);
    const uint32_t nhi = bs == ns - 1 ? hi : last_key_in_bins(lo + 1u, hi, bs, bin_of_key);
    lo = nlo;
    hi = nhi;
    ++rounds;
    // a value split that kept more than half of the range: key ranges next
    if (val && c_lo - c_hi > old_n / 2u) vmode = false;
    __syncthreads();  // F.rank_* and the broadcast read before the next round
    if (hi - lo <= 1u) one_key();
    QRITA_T(10);
  }
  if (done == 1 && collapsed) {
    // the range held one key: every copy of it is the boundary's
    if (tid < C) F.ties[tid] = vld(F.rank_lo[tid]) - vld(F.rank_hi[tid]);
    __syncthreads();
  }
  if (done == 0) {
    // tail: every CTA's (lo, hi] elements (rank_lo - rank_hi of them) are
    // stored into every CTA's tail buffer (the ring's bytes, idle during the
    // search) at the rank's offset. A CTA may still be streaming into its ring
    // unless a cluster barrier passed since: one is taken here if none did.
    if (!synced && rounds == 0) cluster_sync_all();
    unsigned char* rb = reinterpret_cast<unsigned char*>(const_cast<uint4*>(c.ring_ptr));
    float* tv = reinterpret_cast<float*>(rb + kTailValOff);
    unsigned long long* tw = reinterpret_cast<unsigned long long*>(rb + kTailWOff);
    uint8_t* tr = rb + kTailRankOff;
    float* cv = reinterpret_cast<float*>(rb + kCandValOff);
    unsigned long long* cw = reinterpret_cast<unsigned long long*>(rb + kCandWOff);
    uint32_t off = 0;
    for (int r = 0; r < static_cast<int>(c.crank); ++r) off += vld(F.rank_lo[r]) - vld(F.rank_hi[r]);
    uint32_t total = 0;
    for (int r = 0; r < C; ++r) total += vld(F.rank_lo[r]) - vld(F.rank_hi[r]);
    total = min(total, static_cast<uint32_t>(kTail));
    if (tid == 0) {
      F.tail_n = 0u;
      F.bc.u[BU_DONE] = 2u;  // unless a candidate answers (one always does)
    }
    __syncthreads();
    own_for(c, [&](float x, uint32_t) {
      const uint32_t key = f2key(x);  // keys: lo may lie below key(-inf)
      const bool in = key > lo && key <= hi;
      // positions: one shared atomic per warp step
      const uint32_t am = __activemask();
      const uint32_t bal = __ballot_sync(am, in);
      const int leader = __ffs(bal) - 1;
      uint32_t wbase = 0;
      if (lane == leader) wbase = atomicAdd(&F.tail_n, static_cast<uint32_t>(__popc(bal)));
      wbase = __shfl_sync(am, wbase, leader < 0 ? 0 : leader);
      if (in) {
        const uint32_t dst = off + wbase + static_cast<uint32_t>(__popc(bal & ((1u << lane) - 1u)));
        if (dst < static_cast<uint32_t>(kTail)) {
          const unsigned long long w = MASS ? weight_fx(x, c.m, c.m_neginf, scale) : 0ull;
          for (int r = 0; r < C; ++r) {
            const uint32_t rr = static_cast<uint32_t>(r);
            st_dsmem_u32(map_rank(smem_u32(&tv[dst]), rr), __float_as_uint(x));
            st_dsmem_u8(map_rank(smem_u32(&tr[dst]), rr), c.crank);
            if (MASS) {
              const uint32_t a = map_rank(smem_u32(&tw[dst]), rr);
              st_dsmem_u32(a, static_cast<uint32_t>(w));
              st_dsmem_u32(a + 4u, static_cast<uint32_t>(w >> 32));
            }
          }
        }
      }
    });
    QRITA_T(12);
    cluster_sync_all();  // every CTA's tail buffer is complete
    QRITA_T(13);
    if (c.zero_fill) {
      // the mask's zeros go out while the tail is tested (no cluster barrier
      // with release ordering follows before the emission)
      fill_mask<DT>(c, 0);
      c.zero_fill = false;
      c.zero_fill_done = true;
    }
    // the candidates: up to kTailLevels splits of the candidate set into
    // kTailBins bins by a monotone function of the value over the set's value
    // range [v0, v1], bin(x) = trunc((x - v0) nb / (v1 - v0)) (so bins are
    // value intervals in increasing order). The bin where the count (mass)
    // from the top reaches the target holds the boundary; its members become
    // the set. A set of one value is the boundary itself; a small set is
    // tested directly.
    if (tid < C) F.ties[tid] = 0u;
    uint32_t base_c = c_hi;  // count / mass above the set
    unsigned long long base_m = m_hi;
    const float* sv = tv;  // the set's values and weights
    const unsigned long long* sw = tw;
    uint32_t ns = total;
    float v0 = pivot_f(lo), v1 = pivot_f(hi);  // level 0: the range (lo, hi]
    bool one_value = false;
    for (int level = 0; level < kTailLevels && ns > static_cast<uint32_t>(kTailDirect); ++level) {
      const int tb = c.split;  // bins of this split
      const float inv_bw = static_cast<float>(tb) / (v1 - v0);
      if (!(isfinite(v0) && isfinite(v1) && v1 > v0 && isfinite(inv_bw) && inv_bw > 0.f)) break;
      // members satisfy x > v0 (level 0) or x >= v0 (later): never negative
      auto tbin = [&](float x) -> int {
        const int b = static_cast<int>((x - v0) * inv_bw);
        return b < 0 ? 0 : (b > tb - 1 ? tb - 1 : b);
      };
      if (tid < kTailBins) {
        F.tbin_c[tid] = 0u;
        F.tbin_m[tid] = 0ull;
      }
      __syncthreads();
      for (uint32_t i = tid; i < ns; i += kThreads) {
        const int b = tbin(sv[i]);
        atomicAdd(&F.tbin_c[b], 1u);
        if (MASS) add_u64_halves(&F.tbin_m[b], sw[i]);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l holds bins 63 - 2l and 62 - 2l; prefix sums from the top
        // find the first bin whose cumulative total reaches the target
        const int b0 = kTailBins - 1 - 2 * lane, b1 = b0 - 1;
        const uint32_t n0 = vld(F.tbin_c[b0]), n1 = vld(F.tbin_c[b1]);
        const unsigned long long v0w = MASS ? vld(F.tbin_m[b0]) : static_cast<unsigned long long>(n0);
        const unsigned long long v1w = MASS ? vld(F.tbin_m[b1]) : static_cast<unsigned long long>(n1);
        unsigned long long incl = v0w + v1w;
        uint32_t incl_n = n0 + n1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long y = __shfl_up_sync(kFull, incl, o);
          const uint32_t yn = __shfl_up_sync(kFull, incl_n, o);
          if (lane >= o) {
            incl += y;
            incl_n += yn;
          }
        }
        const unsigned long long top = MASS ? base_m : static_cast<unsigned long long>(base_c);
        const unsigned long long ex = top + incl - (v0w + v1w);
        const uint32_t ex_n = base_c + incl_n - (n0 + n1);
        const bool r0 = ex + v0w >= target, r1 = ex + v0w + v1w >= target;
        const uint32_t hit = __ballot_sync(kFull, r1);
        const int L = hit != 0u ? __ffs(hit) - 1 : -1;
        if (lane == (L < 0 ? 0 : L)) {
          F.tsel[0] = L < 0 ? 0xFFFFFFFFu : static_cast<uint32_t>(r0 ? b0 : b1);
          F.tsel[1] = r0 ? ex_n : ex_n + n0;
          F.tsel_m = MASS ? (r0 ? ex : ex + v0w) : 0ull;
          F.tkey[0] = 0xFFFFFFFFu;
          F.tkey[1] = 0u;
          F.tail_n = 0u;
        }
      }
      __syncthreads();
      const uint32_t sel = vld(F.tsel[0]);
      if (sel == 0xFFFFFFFFu) break;  // cannot happen while the set holds the boundary
      const int bs = static_cast<int>(sel);
      base_c = vld(F.tsel[1]);
      base_m = vld(F.tsel_m);
      // the members of bin bs become the set (compacted into cv / cw, in place
      // when the set is there already: every thread reads before any writes)
      float xr[kTail / kThreads];
      unsigned long long wr[kTail / kThreads];
      bool mem[kTail / kThreads];
#pragma unroll
      for (int j = 0; j < kTail / kThreads; ++j) {
        const uint32_t i = tid + static_cast<uint32_t>(j) * kThreads;
        mem[j] = false;
        xr[j] = 0.f;
        wr[j] = 0ull;
        if (i < ns) {
          xr[j] = sv[i];
          wr[j] = MASS ? sw[i] : 0ull;
          mem[j] = tbin(xr[j]) == bs;
        }
      }
      __syncthreads();
      uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
#pragma unroll
      for (int j = 0; j < kTail / kThreads; ++j) {
        if (mem[j]) {
          const uint32_t pos = atomicAdd(&F.tail_n, 1u);
          cv[pos] = xr[j];
          if (MASS) cw[pos] = wr[j];
          const uint32_t k = f2key(xr[j]);
          kmin = min(kmin, k);
          kmax = max(kmax, k);
        }
      }
      kmin = __reduce_min_sync(kFull, kmin);
      kmax = __reduce_max_sync(kFull, kmax);
      if (lane == 0) {
        atomicMin(&F.tkey[0], kmin);
        atomicMax(&F.tkey[1], kmax);
      }
      __syncthreads();
      ns = vld(F.tail_n);
      sv = cv;
      sw = cw;
      const uint32_t kmn = vld(F.tkey[0]), kmx = vld(F.tkey[1]);
      v0 = key2f(kmn);
      v1 = key2f(kmx);
      if (kmn == kmx) {
        one_value = true;
        break;
      }
    }
    if (one_value) {
      // every member equals v0: it is the boundary, with ns copies
      if (tid == 0) {
        const unsigned long long wv = MASS ? sw[0] : 1ull;
        F.bc.u[BU_TAU] = f2key(v0);
        F.bc.u[BU_CABOVE] = base_c;
        F.bc.u[BU_NKEEP] = MASS ? copies_fx(target - base_m, wv, ns) : static_cast<uint32_t>(target) - base_c;
        F.bc.u[BU_DONE] = 1u;
      }
    } else {
      // every member v tests itself: it is the boundary when count(> v) <
      // target <= count(>= v) (masses likewise), where further quaternary
      // rounds would stop (tau = v = z_mn, N_zmn = N(v))
      for (uint32_t ci = tid; ci < ns; ci += kThreads) {
        const float v = sv[ci];
        uint32_t gt = 0, eq = 0;
        unsigned long long mgt = 0ull;
        uint32_t i = 0;
        for (; i + 8u <= ns; i += 8u) {
          float xv[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) xv[u] = sv[i + u];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            gt += xv[u] > v ? 1u : 0u;
            eq += xv[u] == v ? 1u : 0u;
            if (MASS) mgt += xv[u] > v ? sw[i + u] : 0ull;
          }
        }
        for (; i < ns; ++i) {
          const float xv = sv[i];
          gt += xv > v ? 1u : 0u;
          eq += xv == v ? 1u : 0u;
          if (MASS) mgt += xv > v ? sw[i] : 0ull;
        }
        const unsigned long long above_gt = MASS ? mgt + base_m : static_cast<unsigned long long>(gt + base_c);
        const unsigned long long wv = MASS ? sw[ci] : 1ull;
        const unsigned long long above_ge = above_gt + static_cast<unsigned long long>(eq) * wv;
        // every copy of the boundary value answers, with the same values
        if (above_gt < target && target <= above_ge) {
          F.bc.u[BU_TAU] = f2key(v);
          const uint32_t ca = gt + base_c;
          F.bc.u[BU_CABOVE] = ca;
          F.bc.u[BU_NKEEP] = MASS ? copies_fx(target - above_gt, wv, eq) : static_cast<uint32_t>(target) - ca;
          F.bc.u[BU_DONE] = 1u;
        }
      }
    }
    __syncthreads();
    tau = vld(F.bc.u[BU_TAU]);
    n_keep = vld(F.bc.u[BU_NKEEP]);
    cabove = vld(F.bc.u[BU_CABOVE]);
    done = static_cast<int>(vld(F.bc.u[BU_DONE]));
    ++rounds;
    // per-rank copies of the boundary value
    const float tau_v = key2f(tau);
    for (uint32_t i = tid; i < total; i += kThreads) {
      if (tv[i] == tau_v) {
        const uint32_t rk = tr[i];
        if (rk < c.C) atomicAdd(&F.ties[rk], 1u);  // a rank index from shared memory: bounded
      }
    }
    __syncthreads();
  }
  (void)m_lo;
  QRITA_T(14);
  s.tau = tau;
  s.n_keep = n_keep;
  s.count_above = cabove;
  s.rounds = rounds;
  s.capped = done == 2;
}

// The index below which exactly `keep` of this CTA's own-list entries equal
// to tau lie (the own list holds every such element of the chunk). A group
// of at most kTieDirect radix-selects its keep-th smallest index; a larger
// one takes 16-way splits of the index range, invariant count(idx < lo) <
// keep <= count(idx < hi). mark_above: the scan over the own list also
// writes the mask's 1 for every entry above tau (the mask is filled already);
// the compacted group (F.tail_n indices in the ring's bytes, when they fit)
// stays for the emission.
constexpr uint32_t kTieDirect = 1024;
constexpr uint32_t kTieCap = kRingBytes / 4;

// The keep-th smallest of nt <= kThreads distinct indices tix[0 .. nt), plus
// one: thread i ranks index i by counting the smaller ones (every thread
// reads the same entry at each step, so the loads broadcast).
__device__ __forceinline__ uint32_t small_index_cut(Fixed& F, const uint32_t* tix, uint32_t nt, uint32_t keep) {
  const int tid = threadIdx.x;
  const uint32_t mine = static_cast<uint32_t>(tid) < nt ? tix[tid] : 0xFFFFFFFFu;
  uint32_t r = 0;
  for (uint32_t j = 0; j < nt; ++j) r += tix[j] < mine ? 1u : 0u;
  if (static_cast<uint32_t>(tid) < nt && r + 1u == keep) F.bc.u[BU_QKEY] = mine + 1u;
  __syncthreads();
  const uint32_t cut = vld(F.bc.u[BU_QKEY]);
  __syncthreads();
  return cut;
}
template <int DT>
__device__ uint32_t tie_index_cut(Ctx<DT>& c, float tau_f, uint32_t keep, bool mark_above) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the tie group's indices, compacted into the ring's bytes (no stream is in
  // flight); a group too large for them is scanned in the own list. Each
  // warp lists its own in a region of the ring's upper half, counting with
  // its ballots (no atomics); the regions are then packed in warp order.
  uint32_t* tix = reinterpret_cast<uint32_t*>(const_cast<uint4*>(c.ring_ptr));
  static_assert(kTieDirect + kThreads <= kTieCap / 2, "the index histogram fits after a small group");
  constexpr uint32_t kWarpTies = kTieCap / 2 / kWarps;
  uint32_t* wreg = tix + kTieCap / 2 + static_cast<uint32_t>(warp) * kWarpTies;
  __syncthreads();  // earlier users of the ring's bytes are done
  // wn: the warp's ties so far (warp-uniform: every lane takes every step)
  uint32_t wn = 0;
  own_for_warp(c, [&](float x, uint32_t ix, bool v) {
    if (v && mark_above && x > tau_f) c.gmask[ix] = 1;
    const bool eq = v && x == tau_f;
    const uint32_t bal = __ballot_sync(kFull, eq);
    if (eq) {
      const uint32_t pos = wn + static_cast<uint32_t>(__popc(bal & ((1u << lane) - 1u)));
      if (pos < kWarpTies) wreg[pos] = ix;
    }
    wn += static_cast<uint32_t>(__popc(bal));
  });
  if (lane == 0) F.redu[warp][0] = wn;
  __syncthreads();
  uint32_t wbase = 0, nt = 0;
  bool ovf = false;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const uint32_t n = vld(F.redu[w][0]);
    wbase += w < warp ? n : 0u;
    nt += n;
    ovf = ovf || n > kWarpTies;
  }
  if (!ovf)
    for (uint32_t k = static_cast<uint32_t>(lane); k < wn; k += 32u) tix[wbase + k] = wreg[k];
  // a warp's overflow leaves the group in the own list only (the count as a
  // group too large for the ring, for the emission too)
  if (tid == 0) F.tail_n = ovf ? kTieCap + 1u : nt;
  __syncthreads();
  if (ovf) nt = kTieCap + 1u;
  if (nt <= static_cast<uint32_t>(kThreads)) return small_index_cut(F, tix, nt, keep);
  if (nt <= kTieDirect) {
    // a small group: the keep-th smallest index (the (nt + 1 - keep)-th
    // largest) by a radix select over the indices, the histogram after them
    constexpr int kPerT = kTieDirect / kThreads;
    uint32_t key[kPerT];
    bool have[kPerT];
#pragma unroll
    for (int q = 0; q < kPerT; ++q) {
      const uint32_t i = static_cast<uint32_t>(tid + q * kThreads);
      have[q] = i < nt;
      key[q] = have[q] ? tix[i] : 0u;
    }
    const uint32_t kth = radix_select<DT, kPerT>(c, key, have, nt + 1u - keep, tix + kTieDirect);
    return kth + 1u;
  }
  const bool compact = nt <= kTieCap;
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
    auto count_one = [&](uint32_t ix) {
#pragma unroll
      for (int j = 0; j < 15; ++j) cnt[j] += (ix < piv[j]) ? 1u : 0u;
    };
    if (compact) {
      for (uint32_t i = tid; i < nt; i += kThreads) count_one(tix[i]);
    } else {
      own_for(c, [&](float x, uint32_t ix) {
        if (x == tau_f) count_one(ix);
      });
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

// ---------------------------------------------------------------------------
// Key histogram search (bf16 rows whose truncation hit): a bf16 logit has a
// 16-bit order key, and the survivors [t, max] of a row span few of them
// (a few hundred on Gaussian rows). One pass over the own lists counts every
// key; the row's counts (merged over the cluster through distributed shared
// memory) then give the top-k boundary directly: the bin where the count
// from the top reaches k is z_mn, its count N_zmn, and k - count(above) of
// its copies are kept. It is the quaternary search with a pivot at every
// key of the range, which ends in one round. Top-p over S_k follows from the
// same counts: a bin's mass is its count times the fixed-point weight of its
// one value (the boundary bin counts only the copies top-k keeps).
// Layout in the ring's bytes (idle after the streaming pass): this CTA's
// counts, then the row's counts (C > 1).
// ---------------------------------------------------------------------------
constexpr int kKeyHistBins = 2048;
static_assert(2 * kKeyHistBins * 4 <= kRingBytes, "the key histograms fit the ring's bytes");

// 16-bit order key of a logit widened from bf16 (the top half of its 32-bit
// key), and back to the value.
__device__ __forceinline__ uint32_t key16_of(float x) { return f2key(x) >> 16; }
__device__ __forceinline__ float value_of_key16(uint32_t k16) {
  const uint32_t b = (k16 & 0x8000u) ? (k16 ^ 0x8000u) : (~k16 & 0xFFFFu);
  return __uint_as_float(b << 16);
}

// Exclusive scan of a per-thread 64-bit value over the block, in thread order.
__device__ __forceinline__ unsigned long long block_excl_scan_u64(Fixed& F, unsigned long long v,
                                                                  unsigned long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) F.lred[1][warp][0].mass = incl;
  __syncthreads();
  unsigned long long wbase = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const unsigned long long s = vld(F.lred[1][w][0].mass);
    wbase += (w < warp) ? s : 0ull;
    tot += s;
  }
  __syncthreads();
  *total = tot;
  return wbase + incl - v;
}

struct KeyHist {
  uint32_t tau_k, nk_k, above_k;     // top-k boundary key, copies kept, count above
  uint32_t tau, n_keep, count_above;  // the final boundary (after top-p)
  unsigned long long z;               // Z_k (fixed point) when top-p ran
};

// base16: the 16-bit key of the smallest bf16 >= t (every own-list entry is
// at or above it); span: keys base16 .. key16(row max). Every thread of every
// CTA of the row returns the same result; F.ties holds each rank's count of
// the final boundary value.
template <int DT>
__device__ KeyHist keyhist_select(Ctx<DT>& c, uint32_t kk, bool p_on, float pr, uint32_t base16, uint32_t span) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x;
  uint32_t* lh = reinterpret_cast<uint32_t*>(const_cast<uint4*>(c.ring_ptr));
  uint32_t* rh = c.C > 1 ? lh + kKeyHistBins : lh;
  __syncthreads();  // earlier users of the ring's bytes are done
  for (uint32_t i = tid; i < span; i += kThreads) lh[i] = 0u;
  __syncthreads();
  const uint32_t lh_s = smem_u32(lh);
  own_for(c, [&](float x, uint32_t) {
    const uint32_t b = key16_of(x) - base16;
    red_inc_shared_at_if(lh_s + 4u * (b < span ? b : 0u), b < span);
  });
  if (c.C > 1) {
    cluster_sync_all();  // every CTA's counts are complete
    for (uint32_t i = tid; i < span; i += kThreads) {
      uint32_t sum = 0;
      for (uint32_t r = 0; r < c.C; ++r) sum += ld_dsmem_u32(map_rank(smem_u32(&lh[i]), r));
      rh[i] = sum;
    }
  }
  __syncthreads();
  // bins from the top: j = span - 1 - b; thread t holds j in [t P, t P + P)
  const uint32_t P = (span + kThreads - 1) / kThreads;
  const uint32_t j0 = min(static_cast<uint32_t>(tid) * P, span), j1 = min(j0 + P, span);
  uint32_t mine = 0;
  for (uint32_t j = j0; j < j1; ++j) mine += vld(rh[span - 1 - j]);
  uint32_t tot = 0;
  const uint32_t excl = block_excl_scan(F, mine, &tot);
  {
    uint32_t above = excl;
    for (uint32_t j = j0; j < j1; ++j) {
      const uint32_t n = vld(rh[span - 1 - j]);
      if (above < kk && kk <= above + n) {
        F.bc.u[BU_TAU] = j;
        F.bc.u[BU_CABOVE] = above;
      }
      above += n;
    }
  }
  __syncthreads();
  const uint32_t jk = vld(F.bc.u[BU_TAU]);
  KeyHist h;
  h.above_k = vld(F.bc.u[BU_CABOVE]);
  h.nk_k = kk - h.above_k;
  h.tau_k = f2key(value_of_key16(base16 + (span - 1 - jk)));
  h.tau = h.tau_k;
  h.n_keep = h.nk_k;
  h.count_above = h.above_k;
  h.z = 0ull;
  uint32_t jf = jk;  // the final boundary's bin (from the top)
  if (p_on) {
    // masses of the bins of S_k: count x weight of the bin's value
    const float scale = c.fix_scale;
    unsigned long long mm = 0ull;
    for (uint32_t j = j0; j < j1 && j <= jk; ++j) {
      const uint32_t n = j < jk ? vld(rh[span - 1 - j]) : h.nk_k;
      if (n != 0u) mm += static_cast<unsigned long long>(n) *
                         weight_fx(value_of_key16(base16 + (span - 1 - j)), c.m, c.m_neginf, scale);
    }
    unsigned long long zk = 0ull;
    const unsigned long long excl_m = block_excl_scan_u64(F, mm, &zk);
    const unsigned long long target = f2_to_u64(f2_mul(f2_from_u64(zk), pr));
    {
      unsigned long long am = excl_m;
      uint32_t ac = excl;
      for (uint32_t j = j0; j < j1 && j <= jk; ++j) {
        const uint32_t n = j < jk ? vld(rh[span - 1 - j]) : h.nk_k;
        if (n == 0u) continue;
        const unsigned long long w = weight_fx(value_of_key16(base16 + (span - 1 - j)), c.m, c.m_neginf, scale);
        const unsigned long long mj = static_cast<unsigned long long>(n) * w;
        if (am < target && target <= am + mj) {
          F.bc.u[BU_NP] = j;
          F.bc.u[BU_CHI] = ac;
          F.bc.u[BU_NKEEP] = copies_fx(target - am, w, n);
        }
        am += mj;
        ac += n;
      }
    }
    __syncthreads();
    jf = vld(F.bc.u[BU_NP]);
    h.tau = f2key(value_of_key16(base16 + (span - 1 - jf)));
    h.count_above = vld(F.bc.u[BU_CHI]);
    h.n_keep = vld(F.bc.u[BU_NKEEP]);
    h.z = zk;
  }
  // each rank's copies of the final boundary value
  const uint32_t bf = span - 1 - jf;
  if (tid < static_cast<int>(c.C)) {
    F.ties[tid] = c.C > 1 ? ld_dsmem_u32(map_rank(smem_u32(&lh[bf]), static_cast<uint32_t>(tid))) : vld(lh[bf]);
  }
  if (c.C > 1) cluster_sync_all();  // no CTA reuses its counts while another may read them
  else __syncthreads();
  return h;
}

// ---------------------------------------------------------------------------
// Key window for bf16 rows whose top-p runs alone over far more survivors than
// the lists hold. The streaming pass counts the logits of a window of 16-bit
// keys (from the bulk's top down to kKwBins keys, not below t) in a histogram
// of the CTA's own; a window bin holds one value, so its mass is its count
// times the fixed-point weight of that value, exact. The logits outside the
// window are weighed one by one (their sum, and apart the sum above the
// window, are constant offsets of the search). After the pass the bin where
// the mass from the top reaches p Z is the boundary (z_mn, its count N_zmn)
// with no extraction and no further search, and one emission pass writes the
// mask: everything above the boundary value, the boundary's copies
// provisionally, the ties beyond the lowest-index ones cleared afterwards.
// A boundary outside the window falls back to the narrowing passes.
// Layout in the list region while it runs: this CTA's counts, then (C > 1)
// the row's counts; during the emission the tie indices and a radix histogram.
// ---------------------------------------------------------------------------
constexpr int kKwBins = 4096;
constexpr uint32_t kKwHeadroom = 256;   // keys of the window above the bulk's top
constexpr uint32_t kKwTieCap = 4096;    // tie indices the emission collects
static_assert(2 * kKwBins * 4 <= kOwnCap * 8, "the key window's histograms fit the list region");
// |x| < 2^-8 holds most of the 16-bit keys (every small binade): a window
// that straddles zero leaves those keys out as a gap, weighed one by one
constexpr uint32_t kKeyPosGap = 0xBB80u;  // key of +2^-8
constexpr uint32_t kKeyNegGap = 0x447Fu;  // key of -2^-8

// The window: keys lo0 .. lo0 + bot_span - 1 (bottom part), a gap of
// blob_len keys, then top_span keys (top part). Bins hold the bottom part,
// then the top part, each in increasing key order.
struct KeyWindow {
  uint32_t lo0, bot_span, blob_len, top_span;
};

// The window below key k_hi: kKwBins keys down from it, leaving out the gap
// when it straddles zero; false when it cannot be placed (its top inside the
// gap). Logits below it are weighed one by one like those of the gap.
__device__ __forceinline__ bool key_window(uint32_t k_hi, KeyWindow& w) {
  const uint32_t nb = static_cast<uint32_t>(kKwBins);
  if (k_hi > kKeyNegGap && k_hi < kKeyPosGap) return false;
  w.bot_span = 0u;
  w.blob_len = 0u;
  if (k_hi <= kKeyNegGap) {
    w.lo0 = k_hi >= nb - 1u ? k_hi - (nb - 1u) : 0u;
    w.top_span = k_hi - w.lo0 + 1u;
    return true;
  }
  // the top part from +2^-8 (or less when the budget runs out), then below
  // the gap as many negative keys as the budget leaves
  const uint32_t top_lo = k_hi - kKeyPosGap >= nb ? k_hi - (nb - 1u) : kKeyPosGap;
  w.top_span = k_hi - top_lo + 1u;
  w.lo0 = top_lo;
  const uint32_t room = nb - w.top_span;
  if (room > 0u && top_lo == kKeyPosGap) {
    const uint32_t bot_lo = kKeyNegGap >= room - 1u ? kKeyNegGap - (room - 1u) : 0u;
    w.bot_span = kKeyNegGap - bot_lo + 1u;
    w.blob_len = top_lo - kKeyNegGap - 1u;
    w.lo0 = bot_lo;
  }
  return true;
}

// Key of bin b of the window.
__device__ __forceinline__ uint32_t window_key(const KeyWindow& w, uint32_t b) {
  return w.lo0 + (b < w.bot_span ? b : b + w.blob_len);
}

// Boundary of a top-p-alone bf16 row from the key window. Zo: softmax sum
// (shift m_ref) of the logits outside the window bins; Ma / ca: mass and count
// of those above the window; Mb / cb: of those in the gap; cf = exp(m_ref -
// m). Returns false (uniformly) when the boundary lies outside the bins. On
// success h holds the boundary and F.ties each rank's count of its value.
template <int DT>
__device__ bool kw_select(Ctx<DT>& c, float pr, const KeyWindow& kw, F2 Zo, F2 Ma, uint32_t ca, F2 Mb, uint32_t cb,
                          float cf, KeyHist& h) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x;
  const uint32_t nb = kw.bot_span + kw.top_span;
  uint32_t* lh = reinterpret_cast<uint32_t*>(c.lists);
  uint32_t* rh = c.C > 1 ? lh + kKwBins : lh;
  // -0 and +0 are one value: their keys (0x7FFF, 0x8000) share one bin
  // (both lie in one part only when that part spans zero without a gap)
  if (tid == 0 && kw.bot_span == 0u && kw.lo0 <= 0x7FFFu && 0x8000u - kw.lo0 < kw.top_span) {
    lh[0x8000u - kw.lo0] += lh[0x7FFFu - kw.lo0];
    lh[0x7FFFu - kw.lo0] = 0u;
  }
  if (c.C > 1) {
    cluster_sync_all();  // every CTA's counts are complete
    for (uint32_t i = tid; i < nb; i += kThreads) {
      uint32_t sum = 0;
      for (uint32_t r = 0; r < c.C; ++r) sum += ld_dsmem_u32(map_rank(smem_u32(&lh[i]), r));
      rh[i] = sum;
    }
  }
  __syncthreads();
  const float scale = c.fix_scale;
  const unsigned long long z_out = f2_to_u64(f2_mul(f2_mul(Zo, cf), scale));
  const unsigned long long m_top = f2_to_u64(f2_mul(f2_mul(Ma, cf), scale));
  const unsigned long long m_gap = f2_to_u64(f2_mul(f2_mul(Mb, cf), scale));
  // bins from the top: j = nb - 1 - b (the top part first, then past the gap
  // the bottom part); thread t holds j in [t P, t P + P)
  const uint32_t P = (nb + kThreads - 1) / kThreads;
  const uint32_t j0 = min(static_cast<uint32_t>(tid) * P, nb), j1 = min(j0 + P, nb);
  auto bin_w = [&](uint32_t j) -> unsigned long long {
    return weight_fx(value_of_key16(window_key(kw, nb - 1 - j)), c.m, c.m_neginf, scale);
  };
  unsigned long long mm = 0ull, mm_top = 0ull;
  uint32_t cc = 0;
  for (uint32_t j = j0; j < j1; ++j) {
    const uint32_t n = vld(rh[nb - 1 - j]);
    if (n != 0u) {
      const unsigned long long mj = static_cast<unsigned long long>(n) * bin_w(j);
      mm += mj;
      mm_top += j < kw.top_span ? mj : 0ull;
      cc += n;
    }
  }
  unsigned long long wtot = 0ull, wtop = 0ull;
  const unsigned long long excl_m = block_excl_scan_u64(F, mm, &wtot);
  (void)block_excl_scan_u64(F, mm_top, &wtop);
  uint32_t ctot = 0;
  const uint32_t excl_c = block_excl_scan(F, cc, &ctot);
  const unsigned long long target = f2_to_u64(f2_mul(f2_from_u64(z_out + wtot), pr));
  // the boundary must lie in the bins: above the window the mass stays below
  // the target; the top part, or past the gap the bottom part, reaches it
  const bool in_top = m_top < target && target <= m_top + wtop;
  const bool in_bot = kw.bot_span > 0u && m_top + wtop + m_gap < target && target <= m_top + wtot + m_gap;
  if (!(in_top || in_bot)) return false;
  {
    unsigned long long am = m_top + excl_m + (j0 >= kw.top_span ? m_gap : 0ull);
    uint32_t ac = ca + excl_c + (j0 >= kw.top_span ? cb : 0u);
    // only the thread whose bins hold the target walks them
    const unsigned long long end = am + mm + (j0 < kw.top_span && j1 > kw.top_span ? m_gap : 0ull);
    const uint32_t jend = (am < target && target <= end) ? j1 : j0;
    for (uint32_t j = j0; j < jend; ++j) {
      if (j == kw.top_span && j != j0) {  // crossing the gap inside this thread's bins
        am += m_gap;
        ac += cb;
      }
      const uint32_t n = vld(rh[nb - 1 - j]);
      if (n == 0u) continue;
      const unsigned long long w = bin_w(j);
      const unsigned long long mj = static_cast<unsigned long long>(n) * w;
      if (am < target && target <= am + mj) {
        F.bc.u[BU_NP] = j;
        F.bc.u[BU_CHI] = ac;
        F.bc.u[BU_NKEEP] = copies_fx(target - am, w, n);
      }
      am += mj;
      ac += n;
    }
  }
  __syncthreads();
  const uint32_t jf = vld(F.bc.u[BU_NP]);
  const uint32_t bf = nb - 1 - jf;
  h.tau = f2key(value_of_key16(window_key(kw, bf)));
  h.count_above = vld(F.bc.u[BU_CHI]);
  h.n_keep = vld(F.bc.u[BU_NKEEP]);
  h.z = z_out + wtot;
  h.tau_k = h.tau;
  h.nk_k = h.n_keep;
  h.above_k = h.count_above;
  if (tid < static_cast<int>(c.C)) {
    F.ties[tid] = c.C > 1 ? ld_dsmem_u32(map_rank(smem_u32(&lh[bf]), static_cast<uint32_t>(tid))) : vld(lh[bf]);
  }
  if (c.C > 1) cluster_sync_all();  // no CTA reuses its counts while another may read them
  else __syncthreads();
  return true;
}

// Mask emission of a key-window row (bf16): one pass over the chunk writes 1
// above tau and, when some of the boundary's copies are kept here, 1 for
// every copy while collecting their indices; then the copies from the
// keep_local-th lowest index on are cleared. Returns false (uniformly, and
// before any clearing) when the copies exceed what it can collect: the caller
// then writes the whole chunk again with the ties ranked in index order.
template <int DT>
__device__ bool kw_emit(Ctx<DT>& c, float tau_f, int tie_mode, uint32_t keep_local) {
  Fixed& F = *c.F;
  const int tid = threadIdx.x, lane = tid & 31;
  uint32_t* tix = reinterpret_cast<uint32_t*>(c.lists);
  uint32_t* rhist = tix + kKwTieCap;
  const uint32_t tb = __float_as_uint(tau_f) >> 16;  // tau is a bf16 value
  const uint32_t tau2 = tb | (tb << 16);
  const bool want_eq = tie_mode != 0, collect = tie_mode == 2;
  const uintptr_t mbp = reinterpret_cast<uintptr_t>(c.gmask + c.head_n);
  const bool vec_ok = (mbp % 8u) == 0u;
  if (tid == 0) F.tail_n = 0u;
  QRITA_T(11);
  // (stream_pieces opens with a block barrier: the reset is seen)
  auto push_ties = [&](uint32_t eqbits, uint32_t idx0) {
    // lanes with copies append their indices (rare: one value of the row)
    const uint32_t cnt = __popc(eqbits);
    const uint32_t am = __activemask();
    uint32_t incl = cnt;
    const uint32_t bal = __ballot_sync(am, cnt != 0u);
    if (bal == 0u) return;
    const int leader = __ffs(bal) - 1;
    // positions: an exclusive prefix over the active lanes by shuffles
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(am, incl, o);
      if (lane >= o && ((am >> (lane - o)) & 1u)) incl += y;
    }
    const uint32_t tot = __shfl_sync(am, incl, 31 - __clz(am));
    uint32_t base = 0;
    if (lane == leader) base = atomicAdd(&F.tail_n, tot);
    base = __shfl_sync(am, base, leader);
    uint32_t pos = base + incl - cnt;
    uint32_t b = eqbits;
    while (b != 0u) {
      const int q = __ffs(b) - 1;
      b &= b - 1u;
      if (pos < kKwTieCap) tix[pos] = idx0 + static_cast<uint32_t>(bf16_bit_elem(q));
      ++pos;
    }
  };
  stream_pieces<DT>(
      c,
      [&](const uint4 (&v)[kPieceThreadUnits], int u0, int n) {
#pragma unroll
        for (int j = 0; j < kPieceThreadUnits; ++j) {
          uint32_t eqbits = 0u;
          const uint32_t idx0 = static_cast<uint32_t>(c.head_n + (u0 + j * kThreads + tid) * 8);
          if (j * kThreads + tid < n) {
            const uint4 u = v[j];
            uint32_t e0 = 0u, e1 = 0u, e2 = 0u, e3 = 0u;
            if (want_eq) {
              e0 = bf2_eq_mask(u.x, tau2);
              e1 = bf2_eq_mask(u.y, tau2);
              e2 = bf2_eq_mask(u.z, tau2);
              e3 = bf2_eq_mask(u.w, tau2);
            }
            const uint32_t m0 = bf2_gt_mask(u.x, tau2) | e0, m1 = bf2_gt_mask(u.y, tau2) | e1;
            const uint32_t m2 = bf2_gt_mask(u.z, tau2) | e2, m3 = bf2_gt_mask(u.w, tau2) | e3;
            // element 2i is word i's low half, 2i + 1 its high half: bytes in order
            const uint32_t lo4 = __byte_perm(m0, m1, 0x6420) & 0x01010101u;
            const uint32_t hi4 = __byte_perm(m2, m3, 0x6420) & 0x01010101u;
            uint8_t* dst = c.gmask + idx0;
            if (vec_ok) {
              *reinterpret_cast<uint2*>(dst) = make_uint2(lo4, hi4);
            } else {
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                dst[e] = static_cast<uint8_t>((lo4 >> (8 * e)) & 1u);
                dst[4 + e] = static_cast<uint8_t>((hi4 >> (8 * e)) & 1u);
              }
            }
            if (collect)
              eqbits = (e0 & 0x00010001u) | (e1 & 0x00020002u) | (e2 & 0x00040004u) | (e3 & 0x00080008u);
          }
          if (collect) push_ties(eqbits, idx0);
        }
      },
      [&](float x, uint32_t idx, bool valid) {
        uint32_t eqb = 0u;
        if (valid) {
          c.gmask[idx] = (x > tau_f || (want_eq && x == tau_f)) ? 1 : 0;
          eqb = (collect && x == tau_f) ? 1u : 0u;
        }
        if (collect) push_ties(eqb, idx);  // bit 0 decodes to element 0: the index itself
      },
      false, ring_stages(list_region_bytes(static_cast<int>(c.ocap)), (kKwTieCap + kThreads) * 4));
  QRITA_T(12);
  if (!collect) return true;
  __syncthreads();
  const uint32_t nt = vld(F.tail_n);
  if (nt > kKwTieCap) return false;  // uniform: every thread read the same count
  if (keep_local >= nt) return true;
  if (nt <= static_cast<uint32_t>(kThreads)) {
    const uint32_t cut = small_index_cut(F, tix, nt, keep_local);
    if (static_cast<uint32_t>(tid) < nt && tix[tid] >= cut) c.gmask[tix[tid]] = 0;
    return true;
  }
  // the keep_local-th lowest index is the (nt + 1 - keep_local)-th largest
  constexpr int kPer = kKwTieCap / kThreads;
  uint32_t key[kPer];
  bool have[kPer];
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    const uint32_t i = static_cast<uint32_t>(tid + q * kThreads);
    have[q] = i < nt;
    key[q] = have[q] ? tix[i] : 0u;
  }
  const uint32_t kth = radix_select<DT, kPer>(c, key, have, nt + 1u - keep_local, rhist);
#pragma unroll
  for (int q = 0; q < kPer; ++q)
    if (have[q] && key[q] > kth) c.gmask[key[q]] = 0;
  return true;
}

// Row of cluster slot `slot` when the longest rows go first. Rows fall in
// four cost classes, taken in this order, each in row order:
//   3  top-p alone (the streaming pass weighs every logit; most take a
//      second pass);
//   2  top-k expecting more survivors than per-thread columns hold (every
//      warp appends survivors piece by piece);
//   1  the other top-k rows;
//   0  rows that keep everything (one pass that writes ones).
// So the longest rows start in the first wave and the shortest fill the
// last. Every thread returns the row.
__device__ int64_t heavy_first_row(const Params& P, Fixed& F, int64_t slot) {
  const int tid = threadIdx.x;
  const int64_t B = P.B;
  const int64_t per = (B + kThreads - 1) / kThreads;
  const int64_t r0 = min(B, static_cast<int64_t>(tid) * per), r1 = min(B, r0 + per);
  const float col_rows = static_cast<float>(P.ocap / 8) * static_cast<float>(P.C);
  auto cost_class = [&](int64_t r) -> int {
    int32_t k = P.k ? P.k[r] : 0;
    const float p = P.p ? P.p[r] : 1.0f;
    bool k_on = k >= 1 && k < P.V;
    bool p_on = p < 1.0f;  // NaN: off
    if (p_on && !(p > 0.0f)) {  // p <= 0 keeps one token, as k = 1
      p_on = false;
      k_on = P.V > 1;
      k = 1;
    }
    if (!k_on && !p_on) return 0;
    if (!k_on) return 3;
    return 2.4f * static_cast<float>(k) > col_rows ? 2 : 1;
  };
  // per-class counts, four 16-bit fields (B <= 65535 rows reorder)
  unsigned long long mine = 0ull;
  for (int64_t r = r0; r < r1; ++r) mine += 1ull << (16 * cost_class(r));
  unsigned long long tot = 0ull;
  const unsigned long long before = block_excl_scan_u64(F, mine, &tot);
  auto field = [](unsigned long long v, int c) -> int64_t { return static_cast<int64_t>((v >> (16 * c)) & 0xFFFFull); };
  // the slot's class and its rank within the class
  int want_c = 0;
  int64_t want = slot;
  for (int c = 3; c >= 0; --c) {
    if (want < field(tot, c)) {
      want_c = c;
      break;
    }
    want -= field(tot, c);
  }
  if (tid == 0) F.bc.u[BU_ROW] = static_cast<uint32_t>(slot);  // unless a block holds it
  __syncthreads();
  const int64_t have_before = field(before, want_c), have = field(mine, want_c);
  if (want >= have_before && want < have_before + have) {
    int64_t seen = have_before;
    for (int64_t r = r0; r < r1; ++r) {
      if (cost_class(r) == want_c) {
        if (seen == want) F.bc.u[BU_ROW] = static_cast<uint32_t>(r);
        ++seen;
      }
    }
  }
  __syncthreads();
  const int64_t row = vld(F.bc.u[BU_ROW]);
  __syncthreads();
  return row;
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 2) select_kernel(const __grid_constant__ Params P) {
  constexpr int E = Ctx<DT>::E;
  constexpr int S = Ctx<DT>::S;
  extern __shared__ __align__(128) unsigned char smem[];
  Fixed& F = *reinterpret_cast<Fixed*>(smem);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // the previous kernel of the stream (which may have written the logits,
  // k or p) has completed and its writes are visible past this point; the
  // next kernel may be scheduled from now on (it waits the same way)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  Ctx<DT> c;
  c.F = &F;
  c.ocap = static_cast<uint32_t>(P.ocap);
  c.lists = smem + sizeof(Fixed);
  {
    unsigned char* ring = c.lists + (list_region_bytes(P.ocap) - kRingBytes);
    c.ring = smem_u32(ring);
    c.ring_ptr = reinterpret_cast<const uint4*>(ring);
    c.ring_bar = smem_u32(&c.F->ring_bar[0]);
    c.ring_phase = 0u;
    c.ring_out = 0u;
  }
  c.own_val = reinterpret_cast<float*>(c.lists);
  c.own_idx = reinterpret_cast<uint32_t*>(c.own_val + P.ocap);
  c.C = static_cast<uint32_t>(P.C);
  c.crank = cluster_rank();
  c.ph = 0;
  c.m = 0.f;
  c.m_neginf = false;
  c.fix_scale = 0.f;
  c.zero_fill = false;
  c.zero_fill_done = false;
  c.one_fill_done = false;

  const int64_t r = P.heavy_first ? heavy_first_row(P, F, blockIdx.x / P.C) : blockIdx.x / P.C;
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
  // the test flag voids row 0 from its first CTA: uniform over that CTA
  c.give_up_once = (P.flags & QRITA_FLAG_TEST_GIVE_UP) != 0u && r == 0 && c.crank == 0u;
  // search width: the pages' quaternary form (3 pivots) or a binary split
  // for ablations; by default 64-bin rounds and two quaternary levels a pass
  c.split = (P.flags & QRITA_FLAG_SEARCH_BINARY) ? 2 : ((P.flags & QRITA_FLAG_SEARCH_QUATERNARY) ? 4 : kSplit);
  c.npiv = (P.flags & QRITA_FLAG_SEARCH_BINARY) ? 1 : ((P.flags & QRITA_FLAG_SEARCH_QUATERNARY) ? 3 : kNarrowPivots);
  c.wide_ok = (P.flags & (QRITA_FLAG_SEARCH_BINARY | QRITA_FLAG_SEARCH_QUATERNARY)) == 0u;
  QRITA_T(0);
  QRITA_ROWID(r);

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
    constexpr int kPer = (kSampleBlocks * kSampleBlock) / kThreads;
    float sv[kPer];  // this thread's sample values (NaN: none)
    float sn = 0.f, sx = 0.f, sxx = 0.f, smax = -INFINITY;
    float raw[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int sidx = tid + j * kThreads;
      int64_t pos;
      if (V <= kSampleBlocks * kSampleBlock) {
        pos = sidx;
      } else {
        pos = static_cast<int64_t>(sidx / kSampleBlock) * (V / kSampleBlocks) + (sidx % kSampleBlock);
      }
      raw[j] = pos < V ? load_elem<DT>(grow + static_cast<size_t>(pos) * S) : NAN;
    }
    // the ring's first copies of the streaming pass fly while the sample
    // statistics are taken (the chunk does not depend on them); issued after
    // the sample loads, so these are not queued behind them
    if (tid == 0) {
      F.own_n = 0;
      F.err = 0u;
      F.err_any = 0u;
      for (int st = 0; st < kMaxStages; ++st) mbar_init(c.ring_bar + 8u * st, 1u);
      fence_mbar_init();
      const int npieces = (c.body_units + kPieceUnits - 1) / kPieceUnits;
      for (int pc = 0; pc < npieces && pc < kStages; ++pc) ring_issue(c, pc, pc);
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      sv[j] = NAN;
      {
        const float x = raw[j];
        if (isfinite(x)) {
          sv[j] = x;
          sn += 1.f;
          sx += x;
          sxx = fmaf(x, x, sxx);
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
    __syncthreads();
    // first estimate, then the same moments over the values within
    // kClipSigmas of it: a rare outlier in the sample would otherwise
    // inflate sigma and push the threshold above the k-th logit
    float a = 0.f, b = 0.f, d = 0.f, mx = -INFINITY;
    for (int w = 0; w < kWarps; ++w) {
      a += vld(F.redf[w][0]);
      b += vld(F.redf[w][1]);
      d += vld(F.redf[w][2]);
      mx = fmaxf(mx, vld(F.redf[w][3]));
    }
    {
      const float mean0 = a > 0.f ? b / a : 0.f;
      const float sd0 = a > 0.f ? sqrtf(fmaxf(d / a - mean0 * mean0, 0.f)) : 0.f;
      const float lim = kClipSigmas * sd0;
      float cn = 0.f, cx = 0.f, cxx = 0.f;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const float x = sv[j];
        if (fabsf(x - mean0) <= lim) {  // false for NaN
          cn += 1.f;
          cx += x;
          cxx = fmaf(x, x, cxx);
        }
      }
      cn = warp_sum_f(cn);
      cx = warp_sum_f(cx);
      cxx = warp_sum_f(cxx);
      if (lane == 0) {  // (slots apart from the first partials)
        F.redf[warp][4] = cn;
        F.redf[warp][5] = cx;
        F.redf[warp][6] = cxx;
      }
      __syncthreads();
    }
    if (tid == 0) {
      float ca = 0.f, cb = 0.f, cd = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        ca += vld(F.redf[w][4]);
        cb += vld(F.redf[w][5]);
        cd += vld(F.redf[w][6]);
      }
      if (ca > 0.f) {  // else keep the first estimate
        a = ca;
        b = cb;
        d = cd;
      }
      const float mean = a > 0.f ? b / a : 0.f;
      const float var = a > 0.f ? fmaxf(d / a - mean * mean, 0.f) : 0.f;
      const float mu = mean;
      const float sigma = sqrtf(var);
      F.bc.f[BF_MU] = mu;
      F.bc.f[BF_SIGMA] = sigma;
      F.bc.f[BF_MREF] = mx > -INFINITY ? mx : 0.f;
      // ---- A3: delta from the normal-quantile tables, threshold t
      bool trunc = false;
      float t = -INFINITY;
      if (!(P.flags & QRITA_FLAG_NO_TRUNCATION) && a > 0.f && !keep_all) {
        if (k_on) {
          // alpha * k expected survivors (up to 2^(1/4) more from the table's
          // rounding) should fit 80 % of the row's own lists
          const float room = 0.8f * static_cast<float>(P.ocap) * static_cast<float>(P.C) /
                             (1.19f * static_cast<float>(kr));
          const float alpha = fmaxf(fminf(P.alpha_k, room), P.alpha_min_k);
          const float u = alpha * static_cast<float>(kr) / static_cast<float>(V);
          if (u <= P.u_max_k) {
            int i = static_cast<int>(floorf(-4.0f * log2f(u)));
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
      F.bc.u[BU_SAMPLE_T] = 0u;
      F.bc.u[BU_SGE] = 0u;
      F.bc.u[BU_S2S] = 0u;
    }
    __syncthreads();
    // A top-k threshold the sample contradicts (a quarter or less of the
    // sample values expected above the k-th logit lie above it, as on rows
    // bounded below the Gaussian tail): an order statistic of the sample with
    // a margin is the threshold instead, when its expected survivors fit.
    // When fewer than two sample values are expected above the k-th logit,
    // the sample cannot test t itself; there a tail much lighter than the
    // Gaussian's (a quarter or less of the sample values it puts above
    // mu + 2 sigma) and no sample value at or above t decide instead.
    if (k_on && vld(F.bc.u[BU_TRUNC]) != 0u &&
        (P.flags & (QRITA_FLAG_FORCE_FALLBACK | QRITA_FLAG_FORCE_RETRY)) == 0u) {
      const float tt = vld(F.bc.f[BF_T]);
      const float t2s = fmaf(2.0f, vld(F.bc.f[BF_SIGMA]), vld(F.bc.f[BF_MU]));
      // the sample's count at or above t (high half) and of finite values
      // (low half; at most kSampleBlocks * kSampleBlock), and its count at or
      // above mu + 2 sigma, one block reduction
      uint32_t ge_f = 0, ge_2s = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        ge_f += (sv[j] >= tt ? 0x10000u : 0u) + (isnan(sv[j]) ? 0u : 1u);
        ge_2s += sv[j] >= t2s ? 1u : 0u;
      }
      ge_f = __reduce_add_sync(kFull, ge_f);
      ge_2s = __reduce_add_sync(kFull, ge_2s);
      if (lane == 0) {
        atomicAdd(&F.bc.u[BU_SGE], ge_f);
        atomicAdd(&F.bc.u[BU_S2S], ge_2s);
      }
      __syncthreads();
      const uint32_t tot_ge_f = vld(F.bc.u[BU_SGE]);
      const int n_ge = static_cast<int>(tot_ge_f >> 16), n_f = static_cast<int>(tot_ge_f & 0xFFFFu);
      const int n_2s = static_cast<int>(vld(F.bc.u[BU_S2S]));
      const float lam = static_cast<float>(kr) * static_cast<float>(n_f) / static_cast<float>(V);
      const int jq = static_cast<int>(ceilf(lam + 3.0f * sqrtf(lam) + 3.0f));
      const float expect = static_cast<float>(jq) * static_cast<float>(V) / static_cast<float>(n_f > 0 ? n_f : 1);
      // (P(X >= mu + 2 sigma) = 0.02275 for a Gaussian)
      const bool light = 4.0f * static_cast<float>(n_2s) < 0.02275f * static_cast<float>(n_f);
      if (n_f >= 256 && (lam >= 2.0f || light) && 4.0f * static_cast<float>(n_ge) < lam && jq <= n_f &&
          expect <= 0.85f * static_cast<float>(P.ocap) * static_cast<float>(P.C)) {
        // the jq-th largest sample value (histogram in the list region, free
        // here: the ring's first copies are in flight)
        uint32_t key[kPer];
        bool have[kPer];
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
          have[j] = !isnan(sv[j]);
          key[j] = have[j] ? f2key(sv[j]) : 0u;
        }
        const uint32_t kq = radix_select<DT, kPer>(c, key, have, static_cast<uint32_t>(jq),
                                                   reinterpret_cast<uint32_t*>(c.lists));
        if (tid == 0) {
          F.bc.f[BF_T] = key2f(kq);
          F.bc.u[BU_SAMPLE_T] = 1u;
        }
        __syncthreads();
      }
    }
  }
  const float mu = vld(F.bc.f[BF_MU]);
  const float sigma = vld(F.bc.f[BF_SIGMA]);
  const float m_ref = vld(F.bc.f[BF_MREF]);
  const float t = vld(F.bc.f[BF_T]);
  const bool trunc = vld(F.bc.u[BU_TRUNC]) != 0u;
  QRITA_T(1);
  const bool value_pivots = (P.flags & QRITA_FLAG_KEY_PIVOTS) == 0u;
  // bracket pivots for a top-k search over the survivors (identical in every
  // CTA of the row: they come from the shared sample); never below t, so the
  // own lists' counts above them are the row's
  // (a threshold the sample chose: the pivots split [t, m_ref] evenly, the
  // Gaussian model having failed for the row)
  const bool sample_t = vld(F.bc.u[BU_SAMPLE_T]) != 0u;
  // (bf16 rows place the boundary with the key histogram instead)
  const bool bracket = trunc && k_on && !p_only && value_pivots && sigma > 0.f && isfinite(sigma) &&
                       isfinite(mu) && isfinite(m_ref) && (P.flags & QRITA_FLAG_FORCE_FALLBACK) == 0u &&
                       !(DT == QRITA_DTYPE_BF16 && (P.flags & QRITA_FLAG_NO_KEY_HIST) == 0u);
  if (bracket && tid < 16) {
    float q = INFINITY;
    if (tid < kBracket) {
      if (sample_t) {
        q = fmaxf(fmaf(static_cast<float>(tid + 1) * (1.0f / 16.0f), m_ref - t, t), t);
      } else {
        const float mj = exp2f(static_cast<float>(7 - tid) * 0.2f);
        const float u = fminf(mj * static_cast<float>(kr) / static_cast<float>(V), 0.5f);
        q = fmaxf(mu - sigma * normcdfinvf(u), t);
      }
    }
    F.bp[tid] = q;  // published by the streaming pass's first block barrier
    F.bp_bins[tid] = 0u;
  }
  // top-p alone with far more expected survivors than the lists hold: the
  // streaming pass also bins the survivors in [t, ph_hi] (see code_pass)
  // (ph_hi = min(m_ref, mu + 4 sigma), so an outlier in the sample does not
  // widen them; weights there are at most 1)
  float ph_inv_w = 0.f, ph_hi = 0.f, ph_sc = 0.f, ph_lsc = 0.f, ph_ilsc = 0.f;
  int ph_sbits = 0, ph_lbits = 0;
  bool ph = false;
  if (p_only && trunc && sigma > 0.f && isfinite(m_ref) && (P.flags & QRITA_FLAG_FORCE_FALLBACK) == 0u) {
    const float expect = static_cast<float>(V) * normcdff((mu - t) / sigma);
    ph_hi = fminf(m_ref, fmaf(kClipSigmas, sigma, mu));
    ph_inv_w = static_cast<float>(kPhBins) / (ph_hi - t);
    ph = ph_hi > t && expect > 0.9f * static_cast<float>(c.ocap) * static_cast<float>(c.C) && isfinite(ph_inv_w) &&
         ph_inv_w > 0.f;
    // fixed-point bin masses per warp, in two 32-bit halves: a warp bins at
    // most chunk / kWarps + 32 logits (2^pw at most), so a low half of
    // 31 - pw bits and a high half of ph_sbits - (31 - pw) bits both sum
    // without overflow when ph_sbits <= 63 - 2 pw (the same scale in every
    // CTA of the row)
    const uint32_t per_warp = static_cast<uint32_t>(P.chunk) / kWarps + 32u;
    const int pw = 32 - __clz(per_warp);
    ph_lbits = 31 - pw;
    ph_sbits = min(36, 63 - 2 * pw);
    ph_sc = exp2f(static_cast<float>(ph_sbits));
    ph_lsc = exp2f(static_cast<float>(ph_lbits));
    ph_ilsc = exp2f(static_cast<float>(-ph_lbits));
    ph = ph && ph_sbits >= 20;  // (chunks of millions of logits narrow instead)
  }
  // bf16 rows of that kind count a window of 16-bit keys instead (exact
  // bins: see kw_select); the window reaches kKwHeadroom keys above the
  // bulk's top and at most kKwBins keys down, never below t
  bool kw = false;
  KeyWindow kwin = {0u, 0u, 0u, 0u};
  if (DT == QRITA_DTYPE_BF16 && ph && c.C <= 4u && (P.flags & QRITA_FLAG_NO_KEY_HIST) == 0u) {
    const uint32_t k_hi = min(key16_of(__uint_as_float(bf16_ceil_bits(ph_hi) << 16)) + kKwHeadroom, 0xFF7Fu);
    if (key_window(k_hi, kwin)) {
      kw = true;
      ph = false;
    }
  }
  const uint32_t kw_nb = kwin.bot_span + kwin.top_span;
  if (ph) {
    uint32_t* h = reinterpret_cast<uint32_t*>(c.lists);
    for (int i = tid; i < 2 * kWarps * kHistBins; i += kThreads) h[i] = 0u;
    // published by the streaming pass's first block barrier
  }
  if (kw) {
    uint32_t* h = reinterpret_cast<uint32_t*>(c.lists);
    for (uint32_t i = tid; i < kw_nb; i += kThreads) h[i] = 0u;
  }

  // ---- A4: the streaming pass (the one HBM read of the row)
  {
    float vmax = -INFINITY, vmin = INFINITY;
    // bf16 rows without top-p alone: packed running max / min (-inf, +inf
    // pairs) and the threshold as the smallest bf16 >= t, in both halves
    uint32_t vmax2 = 0xFF80FF80u, vmin2 = 0x7F807F80u, t2 = 0u;
    if (DT == QRITA_DTYPE_BF16 && trunc) {
      const uint32_t tb = bf16_ceil_bits(t);
      t2 = tb | (tb << 16);
    }
    uint32_t wn = 0;  // this warp's survivors (its segment of the own list)
    if (lane == 0) F.seg_n[warp] = 0u;  // (the bf16 pieces count there; stream_pieces opens with a barrier)
    const uint32_t segcap = c.ocap / kWarps;
    const uint32_t seg_base = static_cast<uint32_t>(warp) * segcap;
    F2 zs = {0.f, 0.f}, ms = {0.f, 0.f};
    // two instances: the softmax sums (one exponential per element) only where
    // top-p runs alone
    // top-k rows expecting few survivors per CTA keep them in per-thread
    // columns of the own list (no warp communication per piece)
    uint32_t cn = 0;
    const uint32_t colcap = c.ocap / kThreads;
    const bool col = !p_only && trunc && k_on &&
                     2.4f * static_cast<float>(kr) <= static_cast<float>(c.ocap / 8u) * static_cast<float>(c.C);
    const int stream_nst = kStages;  // (deeper rings here measured no gain)
    // top-k rows with truncation on one CTA write their mask's zeros during
    // the pass (a lone CTA's stream is latency-bound, so the stores cost
    // nothing there; rows split over a cluster stream at full bandwidth and
    // zero the mask later): the emission then only scatters the kept ids from
    // the lists; a row that ends on another path rewrites every byte
    const bool zfill = !p_only && trunc && k_on && c.C == 1u;
    // keep-all rows on one CTA write their 1s the same way (a row found
    // non-finite is rewritten by the emission)
    const bool ofill = keep_all && c.C == 1u;
    const uint32_t fill_w = ofill ? 0x01010101u : 0u;
    const uint8_t fill_b = ofill ? 1 : 0;
    const bool zvec = (reinterpret_cast<uintptr_t>(c.gmask + c.head_n) % E) == 0u;
    auto fill_unit = [&](int u) {
      uint8_t* dst = c.gmask + c.head_n + static_cast<size_t>(u) * E;
      if (zvec) {
        if constexpr (E == 4) *reinterpret_cast<uint32_t*>(dst) = fill_w;
        else *reinterpret_cast<uint2*>(dst) = make_uint2(fill_w, fill_w);
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[e] = fill_b;
      }
    };
    auto col_put = [&](float x, uint32_t idx) {
      if (cn < colcap) {
        c.own_val[cn * kThreads + tid] = x;
        c.own_idx[cn * kThreads + tid] = idx;
      }
      ++cn;
    };
    const uint32_t ph_hi_s = smem_u32(reinterpret_cast<uint32_t*>(c.lists) + warp * kHistBins);
    const uint32_t ph_lo_s = ph_hi_s + kWarps * kHistBins * 4;
    uint32_t ph_n = 0, ph_ac = 0;  // survivors; those above ph_hi
    F2 ph_am = {0.f, 0.f};         // and the latter's weight (shift m_ref)
    // a survivor's bin (its weight w <= 1 as round(w 2^sbits), in a high and
    // a low half) and its code byte
    auto ph_bin = [&](float x, float w) -> uint32_t {
      ++ph_n;
      if (x <= ph_hi) {
        int b = static_cast<int>((x - t) * ph_inv_w);
        b = b > kPhBins - 1 ? kPhBins - 1 : b;
        const float v = w * ph_sc;                 // exact scaling
        const float hf = truncf(v * ph_ilsc);       // v / 2^L, rounded down
        const uint32_t hi = static_cast<uint32_t>(hf);
        const uint32_t lo = __float2uint_rn(fmaf(-hf, ph_lsc, v));  // exact remainder, rounded
        const uint32_t off = 4u * static_cast<uint32_t>(b);
        red_add_shared_at(ph_hi_s + off, hi);
        red_add_shared_at(ph_lo_s + off, lo);
        return 1u + static_cast<uint32_t>(b);
      }
      ++ph_ac;
      f2_add(ph_am, w);
      return kPhCodeAbove;
    };
    auto streaming_pass = [&](auto po, auto cm, auto hc, auto zf) {
      constexpr bool PO = decltype(po)::value;
      constexpr bool COL = decltype(cm)::value;
      constexpr bool PH = decltype(hc)::value;
      constexpr bool ZF = decltype(zf)::value;  // fill the mask while streaming (zeros; 1s on keep-all rows)
      stream_pieces<DT>(
          c,
          [&](const uint4 (&v)[kPieceThreadUnits], int u0, int n) {
            if constexpr (DT == QRITA_DTYPE_BF16 && !PO) {
              // packed bf16: max / min and the survivor test on pairs; only
              // survivors are widened
              uint32_t bits[kPieceThreadUnits];
#pragma unroll
              for (int j = 0; j < kPieceThreadUnits; ++j) {
                bits[j] = 0u;
                if (j * kThreads + tid < n) {
                  const uint4 u = v[j];
                  vmax2 = bf2_max_nan(vmax2, bf2_max_nan(bf2_max_nan(u.x, u.y), bf2_max_nan(u.z, u.w)));
                  vmin2 = bf2_min(vmin2, bf2_min(bf2_min(u.x, u.y), bf2_min(u.z, u.w)));
                  if (trunc) bits[j] = bf16_unit_bits(u, t2);
                  if constexpr (ZF) fill_unit(u0 + j * kThreads + tid);
                }
              }
              if constexpr (COL) {
#pragma unroll
                for (int j = 0; j < kPieceThreadUnits; ++j) {
                  uint32_t b = bits[j];
                  const uint32_t idx0 = static_cast<uint32_t>(c.head_n + (u0 + j * kThreads + tid) * E);
                  while (b != 0u) {
                    const int q = __ffs(b) - 1;
                    b &= b - 1u;
                    col_put(bf16_bit_value(v[j], q), idx0 + static_cast<uint32_t>(bf16_bit_elem(q)));
                  }
                }
              } else {
                append_piece_bf16<DT>(c, seg_base, segcap, v, bits, u0);
              }
              return;
            }
            float xs[kPieceThreadUnits][E];
            uint32_t bits[kPieceThreadUnits];
            float zu = 0.f, mu_ = 0.f;  // this piece's softmax partials (shift m_ref)
#pragma unroll
            for (int j = 0; j < kPieceThreadUnits; ++j) {
              unpack<DT>(v[j], xs[j]);
              bits[j] = 0u;
              if (j * kThreads + tid < n) {
                if constexpr (!PO && ZF) fill_unit(u0 + j * kThreads + tid);
                uint32_t cw[E / 4] = {};  // code bytes (PH)
#pragma unroll
                for (int e = 0; e < E; ++e) {
                  const float x = xs[j][e];
                  vmax = fmax_nan(vmax, x);
                  vmin = fminf(vmin, x);
                  const bool surv = trunc && x >= t;
                  bits[j] |= surv ? (1u << e) : 0u;
                  if constexpr (PO) {
                    const float w = exp_shifted(x, m_ref);
                    zu += w;
                    mu_ += surv ? w : 0.f;
                    if constexpr (PH) {
                      const uint32_t code = surv ? ph_bin(x, w) : 0u;
                      cw[e >> 2] |= code << (8 * (e & 3));
                    }
                  }
                }
                if constexpr (PH) {
                  // the unit's code bytes in place of its mask bytes (read
                  // back by code_pass, which writes the final bytes)
                  uint8_t* dst = c.gmask + c.head_n + static_cast<size_t>(u0 + j * kThreads + tid) * E;
                  if (zvec) {
                    if constexpr (E == 4) *reinterpret_cast<uint32_t*>(dst) = cw[0];
                    else *reinterpret_cast<uint2*>(dst) = make_uint2(cw[0], cw[E / 4 - 1]);
                  } else {
#pragma unroll
                    for (int e = 0; e < E; ++e) dst[e] = static_cast<uint8_t>(cw[e >> 2] >> (8 * (e & 3)));
                  }
                }
              }
            }
            if constexpr (PO) {
              f2_add(zs, zu);
              f2_add(ms, mu_);
            }
            if constexpr (COL) {
#pragma unroll
              for (int j = 0; j < kPieceThreadUnits; ++j) {
                uint32_t b = bits[j];
                const uint32_t idx0 = static_cast<uint32_t>(c.head_n + (u0 + j * kThreads + tid) * E);
                while (b != 0u) {
                  const int e = __ffs(b) - 1;
                  b &= b - 1u;
                  float x = xs[j][0];
#pragma unroll
                  for (int q = 1; q < E; ++q) x = (q == e) ? xs[j][q] : x;
                  col_put(x, idx0 + static_cast<uint32_t>(e));
                }
              }
            } else if constexpr (!PH) {
              append_piece<DT>(c, wn, seg_base, segcap, xs, bits, u0);
            }
          },
          [&](float x, uint32_t idx, bool valid) {
            if constexpr (DT == QRITA_DTYPE_BF16 && !PO && !COL) {
              // the pieces counted this warp's survivors in F.seg_n[warp]
              __syncwarp();
              wn = vld(F.seg_n[warp]);
              __syncwarp();
            }
            uint32_t bits = 0;
            if (valid) {
              vmax = fmax_nan(vmax, x);
              vmin = fminf(vmin, x);
              const bool surv = trunc && x >= t;
              bits = surv ? 1u : 0u;
              if constexpr (!PO && ZF) c.gmask[idx] = fill_b;
              if constexpr (PO) {
                const float w = exp_shifted(x, m_ref);
                f2_add(zs, w);
                f2_add(ms, surv ? w : 0.f);
                if constexpr (PH) c.gmask[idx] = static_cast<uint8_t>(surv ? ph_bin(x, w) : 0u);
              }
            }
            const float xs[1] = {x};
            if constexpr (COL) {
              if (bits) col_put(x, idx);
            } else if constexpr (!PH) {
              if (trunc) seg_append<1>(wn, c.own_val, c.own_idx, seg_base, segcap, xs, idx, bits);
            }
          },
          true, stream_nst);
    };
    // key-window rows: counts of the window's keys; every other logit weighed
    // (shift m_ref) into the sum outside the window, and apart above it
    F2 kw_out = {0.f, 0.f}, kw_top = {0.f, 0.f}, kw_gap = {0.f, 0.f};
    // (kw_ge_t: this thread's survivors x >= t among the rare logits; the
    // window's are read off its bins after the pass)
    uint32_t kw_ca = 0, kw_cb = 0, kw_ge_t = 0, kw_kt = 0;
    if constexpr (DT == QRITA_DTYPE_BF16) {
      if (kw) {
        uint32_t* kwh = reinterpret_cast<uint32_t*>(c.lists);
        const uint32_t top_off = kwin.bot_span + kwin.blob_len;
        const uint32_t top_end = top_off + kwin.top_span;
        float po = 0.f, pa = 0.f, pg = 0.f;  // partials of the current piece
        // order keys of both halves of a packed word: x ^ 0xFFFF for negative
        // halves, x ^ 0x8000 for the others (-0 keeps its own key; zeros lie
        // in the gap)
        auto keys2 = [](uint32_t w) -> uint32_t {
          const uint32_t sgn = (w >> 15) & 0x00010001u;
          return w ^ ((sgn * 0x7FFFu) | 0x80008000u);
        };
        // x >= t exactly when key(x) >= the key of the smallest bf16 >= t
        kw_kt = keys2(t2 & 0xFFFFu) & 0xFFFFu;
        // logits outside the bins (below the window, in the gap, above it:
        // rare) are weighed one by one; k: the 16-bit order key of raw h
        auto kw_rare = [&](uint32_t k, uint32_t h) {
          const uint32_t d = k - kwin.lo0;  // wraps for keys below the window
          const float w = exp_shifted(__uint_as_float(h << 16), m_ref);
          po += w;
          kw_ge_t += k >= kw_kt ? 1u : 0u;
          if (k >= kwin.lo0) {
            if (d >= top_end) {
              pa += w;
              ++kw_ca;
            } else {
              pg += w;
              ++kw_cb;
            }
          }
        };
        // one key: counted in its bin (predicated, no branch), or marked rare
        const uint32_t kwh_s = smem_u32(kwh);
        auto kw_key = [&](uint32_t k) -> bool {
          const uint32_t d = k - kwin.lo0;
          const uint32_t dt = d - top_off;
          const bool ib = d < kwin.bot_span, it = dt < kwin.top_span;
          const bool in = ib | it;
          red_inc_shared_at_if(kwh_s + 4u * (ib ? d : dt + kwin.bot_span), in);
          return in;
        };
        auto kw_unit = [&](const uint4 u) {
          const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
          uint32_t rare = 0u;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const uint32_t k2 = keys2(wv[i]);
            rare |= kw_key(k2 & 0xFFFFu) ? 0u : (1u << (2 * i));
            rare |= kw_key(k2 >> 16) ? 0u : (2u << (2 * i));
          }
          while (rare != 0u) {
            const int e = __ffs(rare) - 1;
            rare &= rare - 1u;
            const uint32_t w = e < 2 ? u.x : (e < 4 ? u.y : (e < 6 ? u.z : u.w));
            const uint32_t h = (e & 1) ? (w >> 16) : (w & 0xFFFFu);
            kw_rare(keys2(h) & 0xFFFFu, h);
          }
        };
        stream_pieces<DT>(
            c,
            [&](const uint4 (&v)[kPieceThreadUnits], int u0, int n) {
              po = pa = pg = 0.f;
#pragma unroll
              for (int j = 0; j < kPieceThreadUnits; ++j) {
                if (j * kThreads + tid < n) {
                  const uint4 u = v[j];
                  vmax2 = bf2_max_nan(vmax2, bf2_max_nan(bf2_max_nan(u.x, u.y), bf2_max_nan(u.z, u.w)));
                  vmin2 = bf2_min(vmin2, bf2_min(bf2_min(u.x, u.y), bf2_min(u.z, u.w)));
                  kw_unit(u);
                }
              }
              f2_add(kw_out, po);
              f2_add(kw_top, pa);
              f2_add(kw_gap, pg);
            },
            [&](float x, uint32_t, bool valid) {
              po = pa = pg = 0.f;
              if (valid) {
                vmax = fmax_nan(vmax, x);
                vmin = fminf(vmin, x);
                const uint32_t h = __float_as_uint(x) >> 16;
                const uint32_t k = keys2(h) & 0xFFFFu;
                if (!kw_key(k)) kw_rare(k, h);
              }
              f2_add(kw_out, po);
              f2_add(kw_top, pa);
              f2_add(kw_gap, pg);
            },
            true, stream_nst);
        zs = kw_out;
        ms = kw_top;
      }
    }
    if (kw) {
      // handled above
    } else if (ph) streaming_pass(BoolC<true>{}, BoolC<false>{}, BoolC<true>{}, BoolC<false>{});
    else if (p_only) streaming_pass(BoolC<true>{}, BoolC<false>{}, BoolC<false>{}, BoolC<false>{});
    else if (col && zfill) streaming_pass(BoolC<false>{}, BoolC<true>{}, BoolC<false>{}, BoolC<true>{});
    else if (col) streaming_pass(BoolC<false>{}, BoolC<true>{}, BoolC<false>{}, BoolC<false>{});
    else if (zfill || ofill) streaming_pass(BoolC<false>{}, BoolC<false>{}, BoolC<false>{}, BoolC<true>{});
    else streaming_pass(BoolC<false>{}, BoolC<false>{}, BoolC<false>{}, BoolC<false>{});
    QRITA_T(2);
    c.zero_fill_done = zfill;
    c.one_fill_done = ofill;
    if (col) {
      own_columns_streamed<DT>(c, cn);
      // bf16 rows place their boundaries with the key histogram, which reads
      // the columns as they are; the others (or a histogram that gives way)
      // convert them for the search
      if (!(DT == QRITA_DTYPE_BF16 && (P.flags & QRITA_FLAG_NO_KEY_HIST) == 0u)) own_columns_to_segments<DT>(c);
    } else {
      own_segments_streamed<DT>(c, trunc ? wn : 0u);
    }
    if (bracket) {
      // survivors between consecutive bracket pivots (bin b: b pivots below)
      const volatile float* bq = F.bp;
      own_for(c, [&](float x, uint32_t) { atomicAdd(&F.bp_bins[pivot_bin(bq, x)], 1u); });
      __syncthreads();
    }
    if (bracket && warp == 0) {
      // this CTA's count above each bracket pivot (the bins above it), for
      // the merge
      uint32_t v = lane < 16 ? vld(F.bp_bins[lane]) : 0u;
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) {
        const uint32_t y = __shfl_down_sync(kFull, v, o);
        if (lane + o < 16) v += y;
      }
      const uint32_t above = __shfl_down_sync(kFull, v, 1);  // bins lane + 1 .. 15
      if (lane < kBracket) F.slots[c.ph & 1].cnt[lane] = above;
    }
    uint32_t kw_ca_cta = 0, kw_cb_cta = 0;
    if (kw) {
      // survivors (x >= t) are counted, none is in the own list (the merge
      // sees an overflow); the count above the window goes to the merge.
      // The window's survivors: its bins at or above t's key (a bin is one
      // key; the bins are complete: a block barrier has passed)
      {
        const uint32_t* kwh = reinterpret_cast<const uint32_t*>(c.lists);
        for (uint32_t b = tid; b < kw_nb; b += kThreads)
          if (window_key(kwin, b) >= kw_kt) kw_ge_t += kwh[b];
      }
      const uint32_t wg = __reduce_add_sync(kFull, kw_ge_t), wa = __reduce_add_sync(kFull, kw_ca);
      const uint32_t wb = __reduce_add_sync(kFull, kw_cb);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        kw_gap = f2_merge(kw_gap, f2_make(__shfl_xor_sync(kFull, kw_gap.hi, o), __shfl_xor_sync(kFull, kw_gap.lo, o)));
      if (lane == 0) {
        F.redu[warp][0] = wg;
        F.redu[warp][1] = wa;
        F.redu[warp][2] = wb;
        F.redf[warp][6] = kw_gap.hi;
        F.redf[warp][7] = kw_gap.lo;
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t a = 0, b = 0, g = 0;
        F2 mg = {0.f, 0.f};
        for (int w = 0; w < kWarps; ++w) {
          a += vld(F.redu[w][0]);
          b += vld(F.redu[w][1]);
          g += vld(F.redu[w][2]);
          mg = f2_merge(mg, f2_make(vld(F.redf[w][6]), vld(F.redf[w][7])));
        }
        F.own_n = a;
        F.seg_ovf = 1u;
        kw_ca_cta = b;
        kw_cb_cta = g;
        kw_gap = mg;
      }
      __syncthreads();
    }
    if (ph) {
      // this CTA's bin totals and its survivors above m_ref, read by the
      // other CTAs of the row after the merge; the survivors are counted
      // (none is in the own list: the merge sees an overflow)
      unsigned long long* tm = reinterpret_cast<unsigned long long*>(c.lists + kPhTotOff);
      uint32_t* ta = reinterpret_cast<uint32_t*>(c.lists + kPhAboveOff);
      const uint32_t* h = reinterpret_cast<const uint32_t*>(c.lists);
      // bin tid: the fixed-point mass hi 2^L + lo summed over the warps (exact)
      unsigned long long sh = 0ull, sl = 0ull;
      for (int w = 0; w < kWarps; ++w) {
        sh += vld(h[w * kHistBins + tid]);
        sl += vld(h[(kWarps + w) * kHistBins + tid]);
      }
      tm[tid] = (sh << ph_lbits) + sl;
      const uint32_t wnn = __reduce_add_sync(kFull, ph_n), wac = __reduce_add_sync(kFull, ph_ac);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1)
        ph_am = f2_merge(ph_am, f2_make(__shfl_xor_sync(kFull, ph_am.hi, o), __shfl_xor_sync(kFull, ph_am.lo, o)));
      if (lane == 0) {
        F.redu[warp][0] = wnn;
        F.redu[warp][1] = wac;
        F.redf[warp][6] = ph_am.hi;
        F.redf[warp][7] = ph_am.lo;
      }
      __syncthreads();
      if (tid == 0) {
        uint32_t a = 0, b = 0;
        F2 m2 = {0.f, 0.f};
        for (int w = 0; w < kWarps; ++w) {
          a += vld(F.redu[w][0]);
          b += vld(F.redu[w][1]);
          m2 = f2_merge(m2, f2_make(vld(F.redf[w][6]), vld(F.redf[w][7])));
        }
        F.own_n = a;
        F.seg_ovf = 1u;
        ta[0] = b;
        ta[1] = __float_as_uint(m2.hi);
        ta[2] = __float_as_uint(m2.lo);
      }
      __syncthreads();
    }
    if (DT == QRITA_DTYPE_BF16 && (!p_only || kw)) {
      vmax = fmax_nan(vmax, fmax_nan(__uint_as_float(vmax2 << 16), __uint_as_float(vmax2 & 0xFFFF0000u)));
      vmin = fminf(vmin, fminf(__uint_as_float(vmin2 << 16), __uint_as_float(vmin2 & 0xFFFF0000u)));
    }
    // block reduce
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      vmax = fmax_nan(vmax, __shfl_xor_sync(kFull, vmax, o));
      vmin = fminf(vmin, __shfl_xor_sync(kFull, vmin, o));
      if (p_only) {
        const F2 a = f2_make(__shfl_xor_sync(kFull, zs.hi, o), __shfl_xor_sync(kFull, zs.lo, o));
        const F2 b = f2_make(__shfl_xor_sync(kFull, ms.hi, o), __shfl_xor_sync(kFull, ms.lo, o));
        zs = f2_merge(zs, a);
        ms = f2_merge(ms, b);
      }
    }
    if (lane == 0) {
      F.redf[warp][0] = vmax;
      F.redf[warp][1] = vmin;
      F.redf[warp][3] = zs.hi;
      F.redf[warp][4] = zs.lo;
      F.redf[warp][5] = ms.hi;
      F.redf[warp][6] = ms.lo;
    }
    __syncthreads();
    Slot& my = F.slots[c.ph & 1];
    if (tid == 0) {
      float a = -INFINITY, b = INFINITY;
      F2 z = {0.f, 0.f}, mm = {0.f, 0.f};
      for (int w = 0; w < kWarps; ++w) {
        a = fmax_nan(a, vld(F.redf[w][0]));
        b = fminf(b, vld(F.redf[w][1]));
        z = f2_merge(z, f2_make(vld(F.redf[w][3]), vld(F.redf[w][4])));
        mm = f2_merge(mm, f2_make(vld(F.redf[w][5]), vld(F.redf[w][6])));
      }
      my.f[0] = a;
      my.f[1] = b;
      my.u[0] = trunc ? vld(F.seg_ovf) : 0u;
      my.u[1] = trunc ? vld(F.own_n) : 0u;
      my.u[2] = kw_ca_cta;
      my.u[3] = kw_cb_cta;
      my.f[2] = kw_gap.hi;  // (thread 0 holds the CTA's gap mass)
      my.f[3] = kw_gap.lo;
      my.pr[0] = z.hi;
      my.pr[1] = z.lo;
      my.pr[2] = mm.hi;
      my.pr[3] = mm.lo;
    }
    cluster_sync_all();
    if (bracket) {
      // rank r's count above bracket pivot j (thread 16 r + j)
      const uint32_t r = static_cast<uint32_t>(tid) >> 4, j = static_cast<uint32_t>(tid) & 15u;
      if (r < c.C && j < static_cast<uint32_t>(kBracket))
        F.rank_bins[r][j] = ld_dsmem_u32(map_rank(smem_u32(&my.cnt[j]), r));
    }
    if (warp == 0) {
      float a = -INFINITY, b = INFINITY;
      uint32_t surv = 0, ovf = 0, kwc = 0, kwb = 0;
      F2 z = {0.f, 0.f}, mm = {0.f, 0.f}, mg = {0.f, 0.f};
      if (lane < static_cast<int>(c.C)) {
        const uint32_t fb = map_rank(smem_u32(&my.f[0]), lane);
        a = ld_dsmem_f32(fb);
        b = ld_dsmem_f32(fb + 4);
        const uint32_t ub = map_rank(smem_u32(&my.u[0]), lane);
        ovf = ld_dsmem_u32(ub);
        surv = ld_dsmem_u32(ub + 4);
        kwc = ld_dsmem_u32(ub + 8);
        kwb = ld_dsmem_u32(ub + 12);
        mg = f2_make(ld_dsmem_f32(fb + 8), ld_dsmem_f32(fb + 12));
        const uint32_t pb = map_rank(smem_u32(&my.pr[0]), lane);
        z = f2_make(ld_dsmem_f32(pb), ld_dsmem_f32(pb + 4));
        mm = f2_make(ld_dsmem_f32(pb + 8), ld_dsmem_f32(pb + 12));
        ovf |= surv > c.ocap ? 1u : 0u;
        F.rank_n[lane] = surv;
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        a = fmax_nan(a, __shfl_xor_sync(kFull, a, o));
        b = fminf(b, __shfl_xor_sync(kFull, b, o));
        surv += __shfl_xor_sync(kFull, surv, o);
        kwc += __shfl_xor_sync(kFull, kwc, o);
        kwb += __shfl_xor_sync(kFull, kwb, o);
        mg = f2_merge(mg, f2_make(__shfl_xor_sync(kFull, mg.hi, o), __shfl_xor_sync(kFull, mg.lo, o)));
        ovf |= __shfl_xor_sync(kFull, ovf, o);
        z = f2_merge(z, f2_make(__shfl_xor_sync(kFull, z.hi, o), __shfl_xor_sync(kFull, z.lo, o)));
        mm = f2_merge(mm, f2_make(__shfl_xor_sync(kFull, mm.hi, o), __shfl_xor_sync(kFull, mm.lo, o)));
      }
      if (lane == 0) {
        F.bc.f[BF_MAX] = a;
        F.bc.f[BF_MIN] = b;
        F.bc.u[BU_S] = surv;
        F.bc.u[BU_KWCA] = kwc;
        F.bc.u[BU_KWCB] = kwb;
        put_pair(F.bc, BP_GAP, mg);
        F.bc.u[BU_OVF] = ovf;
        put_pair(F.bc, BP_ZR, z);
        put_pair(F.bc, BP_MR, mm);
      }
    }
    __syncthreads();
    ++c.ph;
  }
  QRITA_T(3);
  const float row_max = vld(F.bc.f[BF_MAX]);
  const float row_min = vld(F.bc.f[BF_MIN]);
  const uint32_t survivors = vld(F.bc.u[BU_S]);
  const bool overflow = vld(F.bc.u[BU_OVF]) != 0u;
  const bool invalid = isnan(row_max) || row_max == INFINITY;
  const F2 Zr = get_pair(F.bc, BP_ZR);
  const F2 Mr = get_pair(F.bc, BP_MR);
  c.m = row_max;
  c.m_neginf = (row_max == -INFINITY);
  // weights exp(x - m) lie in [0, 1]: fixed point with headroom for V terms
  c.fix_scale = exp2f(static_cast<float>(62 - (32 - __clz(static_cast<uint32_t>(V)))));
  const float inv_scale = 1.0f / c.fix_scale;  // a power of two: exact

  uint32_t path = (k_on ? QRITA_PATH_TOPK : 0u) | (p_on ? QRITA_PATH_TOPP : 0u) |
                  (trunc ? QRITA_PATH_TRUNC : 0u) | (overflow ? QRITA_PATH_OVERFLOW : 0u) |
                  (keep_all ? QRITA_PATH_KEEP_ALL : 0u) |
                  (vld(F.bc.u[BU_SAMPLE_T]) != 0u ? QRITA_PATH_SAMPLE_T : 0u);
  const bool force_fb = (P.flags & QRITA_FLAG_FORCE_FALLBACK) != 0u;
  const bool force_retry = (P.flags & QRITA_FLAG_FORCE_RETRY) != 0u;

  // Selection: keep key > tau, plus the n_keep lowest-id elements equal to
  // tau; F.ties[rank] counts the elements equal to tau in each rank's chunk.
  uint32_t tau = 0, n_keep = 0, count_above = 0;
  uint32_t rounds_k = 0, rounds_p = 0, passes = 0;
  uint32_t row_status = invalid ? QRITA_ROW_NONFINITE : QRITA_ROW_OK;
  unsigned long long z_used = 0ull;  // softmax denominator top-p used (fixed point)
  bool sel_all = keep_all && !invalid;
  bool sel_none = invalid;
  bool list_emit = false;     // every kept element is in this CTA's own list
  bool ties_in_list = false;  // every element equal to tau is in this CTA's own list
  bool ties_known = false;    // F.ties holds the per-rank tie counts
  bool ph_mask = false;       // the mask holds 1 above the own lists' range, 0 elsewhere
  bool kw_done = false;       // the key window placed the top-p boundary (kw_emit writes the mask)

  if (!invalid && !keep_all) {
    // the streaming pass summed exp(x - m_ref); shift m is a factor exp(m_ref - m) away
    const bool ref_ok = !c.m_neginf && isfinite(Zr.hi) && isfinite(Mr.hi) && Zr.hi > 0.f &&
                        row_max - m_ref < 80.0f;
    const float cf = ref_ok ? expf(m_ref - row_max) : 0.f;
    const F2 Zm = f2_mul(Zr, cf), Mm = f2_mul(Mr, cf);

    bool k_full = false;  // the own lists hold every element of S_k above tau_k
    uint32_t tau_k = 0, nk_k = 0, above_k = 0;
    bool kh_done = false;  // the key histogram placed both boundaries
    kw_done = false;
    uint32_t kh_final_tau = 0, kh_final_keep = 0, kh_final_above = 0;
    if (k_on) {
      const uint32_t target = static_cast<uint32_t>(kr);
      const bool hit = trunc && !overflow && !force_fb && !force_retry && survivors >= target;
      if (hit) path |= QRITA_PATH_HIT;
      Local s;
      s.c_above = 0;
      s.m_above = 0ull;
      s.m_lo = s.m_hi = 0ull;
      bool have_exact = false;
      bool searched = false;  // the search ran on the own lists' survivors
      uint32_t qk = 0, S2 = 0;
      bool ovf2 = true;
      // bf16 rows whose survivors span at most kKeyHistBins keys: one
      // histogram of the keys replaces the pivot rounds (and top-p over S_k)
      const uint32_t kh_base = DT == QRITA_DTYPE_BF16 && trunc ? key16_of(__uint_as_float(bf16_ceil_bits(t) << 16)) : 0u;
      const uint32_t kh_top = DT == QRITA_DTYPE_BF16 ? key16_of(row_max) : 0u;
      const bool kh = DT == QRITA_DTYPE_BF16 && hit && (P.flags & QRITA_FLAG_NO_KEY_HIST) == 0u &&
                      kh_top >= kh_base && kh_top - kh_base < static_cast<uint32_t>(kKeyHistBins);
      // columns left for the key histogram become segments for a search
      if (!kh && vld(F.col_mode) != 0u) own_columns_to_segments<DT>(c);
      if (kh) {
        const KeyHist h = keyhist_select<DT>(c, target, p_on, pr, kh_base, kh_top - kh_base + 1u);
        path |= QRITA_PATH_KEYHIST;
        s.tau = h.tau_k;
        s.n_keep = h.nk_k;
        s.count_above = h.above_k;
        s.rounds = 1;
        s.capped = false;
        kh_final_tau = h.tau;
        kh_final_keep = h.n_keep;
        kh_final_above = h.count_above;
        z_used = h.z;
        kh_done = true;
        searched = true;
      } else if (hit && bracket) {
        // Z_t is in the own lists, and the merged bracket counts place the
        // boundary: lane j totals pivot j over the ranks; the largest j whose
        // count reaches k is lo, the next pivot hi (counts fall with j)
        uint32_t tj = 0;
        if (lane < kBracket)
          for (uint32_t r = 0; r < c.C; ++r) tj += vld(F.rank_bins[r][lane]);
        const uint32_t reach = __ballot_sync(kFull, lane < kBracket && tj >= target);
        const int js = reach != 0u ? 31 - __clz(reach) : -1;
        const uint32_t t_lo = __shfl_sync(kFull, tj, js < 0 ? 0 : js);
        const bool hi_piv = js + 1 < kBracket;
        const uint32_t t_hi = __shfl_sync(kFull, tj, hi_piv ? js + 1 : 0);
        s.lo = js >= 0 ? f2key(vld(F.bp[js])) : f2key(t) - 1u;
        s.c_lo = js >= 0 ? t_lo : survivors;
        s.hi = hi_piv ? f2key(vld(F.bp[js + 1])) : f2key(row_max);
        s.c_hi = hi_piv ? t_hi : 0u;
        if (tid < static_cast<int>(c.C)) {
          F.rank_lo[tid] = js >= 0 ? vld(F.rank_bins[tid][js]) : vld(F.rank_n[tid]);
          F.rank_hi[tid] = hi_piv ? vld(F.rank_bins[tid][js + 1]) : 0u;
        }
        __syncthreads();
        c.zero_fill = !c.zero_fill_done;  // the mask is all zeros but for the scattered kept ids
        dsearch<DT, false>(c, s, target, value_pivots);
        searched = true;
      } else if (hit) {
        // Z_t is in the own lists: the candidates are (key(t) - 1, max]
        rank_counts_from<DT>(c, F.rank_n);
        s.lo = f2key(t) - 1u;
        s.c_lo = survivors;
        s.hi = f2key(row_max);
        s.c_hi = 0;
        dsearch<DT, false>(c, s, target, value_pivots);
        searched = true;
      } else if (!force_fb) {
        // second truncation: when the first threshold missed (or left too many
        // candidates), an order statistic of a larger sample of the row whose
        // expected survivors fit the own lists
        const int n_s = V < kRetrySample ? V : kRetrySample;
        uint32_t jq;
        if (V <= kRetrySample) {
          jq = target;  // the sample is the row: t2 is the k-th logit itself
        } else {
          const float lam = static_cast<float>(target) * static_cast<float>(n_s) / static_cast<float>(V);
          jq = static_cast<uint32_t>(ceilf(lam + 4.0f * sqrtf(lam) + 4.0f));
        }
        const float expect = static_cast<float>(jq) * static_cast<float>(V) / static_cast<float>(n_s);
        if (jq <= static_cast<uint32_t>(n_s) &&
            expect <= 0.75f * static_cast<float>(c.ocap) * static_cast<float>(c.C)) {
          path |= QRITA_PATH_RETRY;
          qk = sample_order_key<DT>(c, grow, V, jq);
          retry_pass<DT>(c, key2f(qk));
          S2 = vld(F.bc.u[BU_S2]);
          ovf2 = vld(F.bc.u[BU_OVF2]) != 0u;
          if (!ovf2 && S2 >= target) {
            // Z_t2 is in the own lists: the candidates are (key(t2) - 1, max]
            rank_counts_from<DT>(c, F.rank_n);
            s.lo = qk - 1u;
            s.c_lo = S2;
            s.hi = f2key(row_max);
            s.c_hi = 0;
            dsearch<DT, false>(c, s, target, value_pivots);
            searched = true;
          }
        }
      }
      if (searched) {
        k_full = true;
        list_emit = true;
        ties_in_list = true;
      } else {
        // narrow over the chunk, then search the extracted range
        path |= QRITA_PATH_FALLBACK;
        Range R;
        R.pin_hi = false;
        R.m_lo = R.m_hi = 0ull;
        R.target = target;
        R.target_from_total = false;
        R.p_frac = 0.f;
        R.extra = 0ull;
        R.lo = f2key(row_min) - 1u;
        R.c_lo = static_cast<uint32_t>(V);
        const bool miss_t = trunc && !overflow && survivors < target;
        const bool miss_t2 = !ovf2 && S2 < target;  // the second threshold missed too
        R.hi = f2key(row_max);
        R.c_hi = 0u;
        if (miss_t) {
          R.hi = f2key(t) - 1u;
          R.c_hi = survivors;
        }
        if (miss_t2 && S2 >= R.c_hi) {
          R.hi = qk - 1u;
          R.c_hi = S2;
        }
        R.lo_all = R.lo < kKeyNegInf;
        narrow<DT, false>(c, R);
        passes += static_cast<uint32_t>(R.passes);
        if (R.exact) {
          s.tau = R.hi;
          s.count_above = R.c_hi;
          s.n_keep = target - R.c_hi;
          s.rounds = 0;
          s.capped = false;
          have_exact = true;
          if (tid < static_cast<int>(c.C)) F.ties[tid] = vld(F.rank_lo[tid]) - vld(F.rank_hi[tid]);
          __syncthreads();
        } else if (!R.fits) {
          s.capped = true;
          s.rounds = 0;
        } else {
          extract_range<DT>(c, R);
          own_segments_contiguous<DT>(c);
          // each rank's list holds exactly its part of the range
          if (tid < static_cast<int>(c.C)) {
            F.rank_lo[tid] = vld(F.rank_lo[tid]) - vld(F.rank_hi[tid]);
            F.rank_hi[tid] = 0u;
          }
          __syncthreads();
          s.lo = R.lo;
          s.c_lo = R.c_lo;
          s.hi = R.hi;
          s.c_hi = R.c_hi;
          s.c_above = R.c_hi;  // elements above hi exceed every pivot
          dsearch<DT, false>(c, s, target, value_pivots, false);
          k_full = R.c_hi == 0u;  // nothing lies above the extracted range
          list_emit = false;
          ties_in_list = true;
        }
      }
      (void)have_exact;
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
      ties_known = !sel_none;
      if (kh_done) {
        tau = kh_final_tau;
        n_keep = kh_final_keep;
        count_above = kh_final_above;
        if (p_on) rounds_p = 1u;
      }
    }

    QRITA_T(4);
    bool extracted_above_k = false;  // the own lists hold exactly {x > tau_k}
    if (p_on && k_on && !k_full && !sel_none) {
      // S_k without its boundary copies is {x > tau_k}: extract it
      Range Rx;
      Rx.lo = tau_k;
      Rx.hi = kKeyPosInf;
      Rx.lo_all = false;
      Rx.pin_hi = true;
      extract_range<DT>(c, Rx);
      own_segments_contiguous<DT>(c);
      merge_count_mass<DT>(c, vld(F.own_n), 0ull, vld(F.seg_ovf));
      if (vld(F.bc.u[BU_OVF2]) == 0u) {
        k_full = true;
        extracted_above_k = true;
      }
    }
    if (p_on && !sel_none && !kh_done) {
      const float scale = c.fix_scale;
      if (k_on && k_full) {
        // top-p over S_k, all of it in the own lists:
        // Z_k = mass(> tau_k) + n_keep_k w(tau_k)
        const float tk = key2f(tau_k);
        uint32_t cnt = 0;
        unsigned long long acc = 0ull;
        own_for(c, [&](float x, uint32_t) {
          if (x > tk) {
            ++cnt;
            acc += weight_fx(x, c.m, c.m_neginf, scale);
          }
        });
        cnt = __reduce_add_sync(kFull, cnt);
        acc = warp_sum_u64_redux(acc);
        if (lane == 0) {
          F.lred[0][warp][0].mass = acc;
          F.lred[0][warp][0].cnt = cnt;
        }
        __syncthreads();
        uint32_t cta_n = 0;
        unsigned long long cta_m = 0ull;
        if (tid == 0) {
          for (int w = 0; w < kWarps; ++w) {
            cta_n += vld(F.lred[0][w][0].cnt);
            cta_m += vld(F.lred[0][w][0].mass);
          }
        }
        merge_count_mass<DT>(c, cta_n, cta_m, 0u);
        const unsigned long long M_gt = vld(F.bc.x[BX_MLO]);
        const unsigned long long w_tau = weight_fx(tk, c.m, c.m_neginf, scale);
        const unsigned long long Zk = M_gt + static_cast<unsigned long long>(nk_k) * w_tau;
        const unsigned long long target = f2_to_u64(f2_mul(f2_from_u64(Zk), pr));
        z_used = Zk;
        if (M_gt < target) {
          // the boundary lies in the tau_k tie group: keep fewer of them
          n_keep = copies_fx(target - M_gt, w_tau, nk_k);
          count_above = above_k;
          if (extracted_above_k) {
            // the lists hold {x > tau_k} only: the tie group is not in them
            list_emit = false;
            ties_in_list = false;
          }
        } else {
          rank_counts_from<DT>(c, F.rank_n);
          Local s;
          s.lo = tau_k;
          s.c_lo = above_k;
          s.m_lo = M_gt;
          s.hi = f2key(row_max);
          s.c_hi = 0;
          s.m_hi = 0ull;
          s.c_above = 0;
          s.m_above = 0ull;
          dsearch<DT, true>(c, s, target, value_pivots);
          rounds_p = static_cast<uint32_t>(s.rounds);
          if (s.capped) {
            sel_none = true;
            row_status = QRITA_ROW_SEARCH_CAP;
          }
          tau = s.tau;
          n_keep = s.n_keep;
          count_above = s.count_above;
          if (extracted_above_k) {
            // tau > tau_k: the kept set and the tie group are in the lists
            list_emit = true;
            ties_in_list = true;
          }
        }
      } else {
        // top-p only, or top-p over an S_k too large for the lists
        // (key-window rows first: see kw_select)
        if (kw && !k_on && ref_ok) {
          KeyHist h;
          if (kw_select<DT>(c, pr, kwin, Zr, Mr, vld(F.bc.u[BU_KWCA]), get_pair(F.bc, BP_GAP),
                            vld(F.bc.u[BU_KWCB]), cf, h)) {
            path |= QRITA_PATH_KEYHIST | QRITA_PATH_HIT;
            tau = h.tau;
            n_keep = h.n_keep;
            count_above = h.count_above;
            z_used = h.z;
            rounds_p = 1u;
            passes = 1u;  // the emission pass
            ties_known = true;
            kw_done = true;
          }
        }
      }
      if (!kw_done && !(k_on && k_full)) {
        // top-p only, or top-p over an S_k too large for the lists
        const bool hit = !k_on && trunc && !overflow && !force_fb && ref_ok && !kw &&
                         f2_ge(Mm, f2_mul(f2_mul(Zm, pr), 1.0f + 1e-5f));
        if (!k_on) path |= hit ? QRITA_PATH_HIT : QRITA_PATH_FALLBACK;
        Local s;
        s.c_above = 0;
        s.m_above = 0ull;
        bool have_exact = false;
        if (hit) {
          // Z_t is in the own lists: the candidates are (key(t) - 1, max]
          rank_counts_from<DT>(c, F.rank_n);
          z_used = f2_to_u64(f2_mul(Zm, scale));
          s.lo = f2key(t) - 1u;
          s.c_lo = survivors;
          s.m_lo = f2_to_u64(f2_mul(Mm, scale));
          s.hi = f2key(row_max);
          s.c_hi = 0;
          s.m_hi = 0ull;
          list_emit = true;
          ties_in_list = true;
          dsearch<DT, true>(c, s, f2_to_u64(f2_mul(f2_mul(Zm, pr), scale)), value_pivots);
        } else {
          // narrow by mass in fixed point (shift m); a pass over the chunk
          // measures the denominator (Z, or mass(> tau_k) for S_k) itself
          Range R;
          R.pin_hi = false;
          R.p_frac = pr;
          R.extra = 0ull;
          R.target_from_total = true;
          R.target = 0ull;
          R.m_lo = R.m_hi = 0ull;
          // top-p alone, truncation hit by mass but too many survivors: the
          // boundary lies above t, and the target is p Z from the streaming pass
          // (key-window rows summed other quantities: narrow from the whole row)
          const bool mass_hit = !k_on && trunc && !force_fb && ref_ok && !kw &&
                                f2_ge(Mm, f2_mul(f2_mul(Zm, pr), 1.0f + 1e-5f));
          bool ph_done = false;
          if (ph && mass_hit) {
            // the first pass's bins, read from every CTA of the row: thread
            // tid holds bin b = kPhBins - 1 - tid (from the top), its count
            // and its exact mass moved to the search's fixed point (shift m:
            // times cf 2^(S - sbits), cf = exp(m_ref - m))
            const unsigned long long* tm = reinterpret_cast<const unsigned long long*>(c.lists + kPhTotOff);
            const uint32_t* ta = reinterpret_cast<const uint32_t*>(c.lists + kPhAboveOff);
            const int b_t = kPhBins - 1 - tid;
            unsigned long long rb = 0ull;
            if (b_t >= 0) {
              for (uint32_t r = 0; r < c.C; ++r) {
                const uint32_t ab = map_rank(smem_u32(&tm[b_t]), r);
                rb += static_cast<unsigned long long>(ld_dsmem_u32(ab)) |
                      (static_cast<unsigned long long>(ld_dsmem_u32(ab + 4u)) << 32);
              }
            }
            const float conv = cf * (scale / ph_sc);  // (a power of two times cf)
            const unsigned long long rm = rb != 0ull ? f2_to_u64(f2_mul(f2_from_u64(rb), conv)) : 0ull;
            if (warp == 0) {
              // the survivors above ph_hi: compensated mass (shift m_ref)
              F2 am = {0.f, 0.f};
              if (lane < static_cast<int>(c.C)) {
                am = f2_make(__uint_as_float(ld_dsmem_u32(map_rank(smem_u32(&ta[1]), static_cast<uint32_t>(lane)))),
                             __uint_as_float(ld_dsmem_u32(map_rank(smem_u32(&ta[2]), static_cast<uint32_t>(lane)))));
              }
#pragma unroll
              for (int o = 16; o > 0; o >>= 1)
                am = f2_merge(am, f2_make(__shfl_xor_sync(kFull, am.hi, o), __shfl_xor_sync(kFull, am.lo, o)));
              if (lane == 0) {
                put_pair(F.bc, BP_PHA, am);
                F.bc.u[BU_NP] = 0xFFFFFFFFu;  // the bin that holds the boundary: none yet
              }
            }
            unsigned long long m_bins = 0ull;
            // mass of the bins above thread tid's (barriers inside)
            const unsigned long long m_above_b = block_excl_scan_u64(F, rm, &m_bins);
            const unsigned long long a_row = f2_to_u64(f2_mul(f2_mul(get_pair(F.bc, BP_PHA), cf), scale));
            const unsigned long long target = f2_to_u64(f2_mul(f2_mul(Zm, pr), scale));
            // the boundary: among the survivors above ph_hi (code
            // kPhCodeAbove), or in the one bin where the mass from the top
            // reaches the target
            if (tid == 0 && target <= a_row) {
              F.bc.u[BU_NP] = kPhCodeAbove;
              F.bc.x[BX_MHI] = 0ull;
            }
            if (b_t >= 0 && target > a_row) {
              const unsigned long long above = a_row + m_above_b;
              if (above < target && target <= above + rm) {
                F.bc.u[BU_NP] = 1u + static_cast<uint32_t>(b_t);
                F.bc.x[BX_MHI] = above;
              }
            }
            __syncthreads();
            const uint32_t code = vld(F.bc.u[BU_NP]);
            const bool found = code != 0xFFFFFFFFu;
            const unsigned long long m_above = vld(F.bc.x[BX_MHI]);
            cluster_sync_all();  // every CTA has read the others' totals
            if (found) {
              // the code's key range: bin(x) as the streaming pass computed it
              auto bfun = [&](uint32_t k) -> int {
                const float x = key2f(k);
                if (!(x >= t)) return -1;
                if (x > ph_hi) return kPhBins;
                const int b = static_cast<int>((x - t) * ph_inv_w);
                return b > kPhBins - 1 ? kPhBins - 1 : b;
              };
              const uint32_t kt = f2key(t), km = f2key(ph_hi);
              const bool to_top = code == kPhCodeAbove;
              const int bb = static_cast<int>(code) - 1;
              const uint32_t lo_key = to_top ? km : (bb == 0 ? kt - 1u : last_key_in_bins(kt, km, bb - 1, bfun));
              const uint32_t hi_key = to_top ? f2key(row_max) : last_key_in_bins(kt, km, bb, bfun);
              const uint32_t ca = code_pass<DT>(c, code, code);
              passes += 1u;
              // the list's exact mass (entries past a full segment are lost:
              // the list then overflowed and is not used)
              unsigned long long mi = 0ull;
              own_for(c, [&](float x, uint32_t) { mi += weight_fx(x, c.m, c.m_neginf, scale); });
              mi = warp_sum_u64(mi);
              const uint32_t wca = __reduce_add_sync(kFull, ca);
              if (lane == 0) {
                F.lred[0][warp][1].mass = mi;
                F.lred[0][warp][0].cnt = wca;
              }
              __syncthreads();
              unsigned long long tmi = 0ull;
              uint32_t tca = 0;
              for (int w = 0; w < kWarps; ++w) {
                tmi += vld(F.lred[0][w][1].mass);
                tca += vld(F.lred[0][w][0].cnt);
              }
              __syncthreads();
              merge_split<DT>(c, vld(F.own_n), vld(F.seg_ovf), tca, 0ull, tmi);
              const uint32_t c_above = vld(F.bc.u[BU_CHI]);
              const uint32_t n_in = vld(F.bc.u[BU_S2]);
              const bool ovf_in = vld(F.bc.u[BU_OVF2]) != 0u;
              const unsigned long long m_in = vld(F.bc.x[BX_MLO]);
              // the exact masses confirm the bracket: search the lists (a
              // test flag treats the bracket as missed)
              if (!ovf_in && m_above < target && target <= m_above + m_in &&
                  (P.flags & QRITA_FLAG_HIST_MISS) == 0u) {
                rank_counts_from<DT>(c, F.rank_n);
                s.lo = lo_key;
                s.hi = hi_key;
                s.c_lo = c_above + n_in;
                s.c_hi = c_above;
                s.m_lo = m_above + m_in;
                s.m_hi = m_above;
                s.c_above = c_above;
                s.m_above = m_above;
                z_used = f2_to_u64(f2_mul(Zm, scale));
                list_emit = true;
                ties_in_list = true;
                ph_mask = true;
                path |= QRITA_PATH_HIST;
                dsearch<DT, true>(c, s, target, value_pivots);
                ph_done = true;
              }
            }
          }
          if (!ph_done) {
            if (k_on) {
              R.lo = tau_k;
              R.c_lo = above_k;
              R.extra = static_cast<unsigned long long>(nk_k) * weight_fx(key2f(tau_k), c.m, c.m_neginf, scale);
            } else if (mass_hit) {
              R.lo = f2key(t) - 1u;
              R.c_lo = survivors;
              R.target_from_total = false;
              R.target = f2_to_u64(f2_mul(f2_mul(Zm, pr), scale));
              R.m_lo = f2_to_u64(f2_mul(Mm, scale));
            } else {
              R.lo = f2key(row_min) - 1u;
              R.c_lo = static_cast<uint32_t>(V);
            }
            R.lo_all = R.lo < kKeyNegInf;
            R.hi = f2key(row_max);
            R.c_hi = 0;
            narrow<DT, true>(c, R);
            passes += static_cast<uint32_t>(R.passes);
            const unsigned long long target = R.target;
            z_used = f2_to_u64(f2_mul(f2_from_u64(target), 1.0f / pr));
            // the chunk passes overwrote the lists: the emission streams the
            // chunk unless an extraction below refills them
            list_emit = false;
            ties_in_list = false;
            if (R.below) {
              // only after top-k: mass(> tau_k) < p Z_k, so the boundary lies in
              // the tau_k tie group (whose per-rank counts F.ties still holds)
              s.tau = tau_k;
              s.n_keep = copies_fx(target - R.m_lo, weight_fx(key2f(tau_k), c.m, c.m_neginf, scale), nk_k);
              s.count_above = above_k;
              s.rounds = 0;
              s.capped = false;
              have_exact = true;
            } else if (R.exact) {
              s.tau = R.hi;
              s.n_keep = copies_fx(target - R.m_hi, weight_fx(key2f(R.hi), c.m, c.m_neginf, scale), R.c_lo - R.c_hi);
              s.count_above = R.c_hi;
              s.rounds = 0;
              s.capped = false;
              have_exact = true;
              if (tid < static_cast<int>(c.C)) F.ties[tid] = vld(F.rank_lo[tid]) - vld(F.rank_hi[tid]);
              __syncthreads();
              ties_known = true;
            } else if (!R.fits) {
              s.capped = true;
              s.rounds = 0;
            } else {
              extract_range<DT>(c, R);
              own_segments_contiguous<DT>(c);
              if (tid < static_cast<int>(c.C)) {
                F.rank_lo[tid] = vld(F.rank_lo[tid]) - vld(F.rank_hi[tid]);
                F.rank_hi[tid] = 0u;
              }
              __syncthreads();
              s.lo = R.lo;
              s.hi = R.hi;
              s.c_lo = R.c_lo;
              s.c_hi = R.c_hi;
              s.c_above = R.c_hi;
              s.m_lo = R.m_lo;
              s.m_hi = R.m_hi;
              s.m_above = R.m_hi;
              ties_in_list = true;
              dsearch<DT, true>(c, s, target, value_pivots, false);
            }
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
        if (!sel_none && !have_exact) ties_known = true;
      }
    }
  }
  QRITA_T(5);

  // The last cluster barrier (see the end of the row) is entered here when
  // nothing below touches another CTA's memory or streams the chunk: its
  // arrive now, its wait at the end. A bulk-copy wait that gave up is
  // reported to every CTA before the arrive.
  const bool early_arrive = c.C > 1 && (sel_all || sel_none || list_emit);
  const bool zero_filled = c.zero_fill_done;
  if (early_arrive) {
    if (__syncthreads_or(vld(F.err) != 0u) != 0) {
      if (tid == 0) {
        ring_drain<DT>(c);
        for (uint32_t rr = 0; rr < c.C; ++rr) st_dsmem_u32(map_rank(smem_u32(&F.err_any), rr), 1u);
      }
      __syncthreads();
      cluster_arrive();  // release: the flags are seen after the wait
    } else {
      // this CTA's accesses to other CTAs' memory were loads already used
      cluster_arrive_relaxed();
    }
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
  // the cut's scan over the own list also writes the kept entries above tau
  // when the mask is filled already (the emission then writes only the ties)
  const bool fused_ties = tie_mode == 2 && ties_in_list && list_emit && (zero_filled || ph_mask);
  if (tie_mode == 2) {
    if (ties_in_list) {
      idx_cut = tie_index_cut<DT>(c, tau_f, keep_local, fused_ties);
    } else {
      ordered_ties = true;
    }
  }
  QRITA_T(6);

  // ---- A9: mask emission
  bool kw_emitted = false;
  if constexpr (DT == QRITA_DTYPE_BF16) {
    if (kw_done && !sel_all && !sel_none) kw_emitted = kw_emit<DT>(c, tau_f, tie_mode, keep_local);
  }
  if (kw_emitted) {
    // written
  } else if (sel_all || sel_none || list_emit) {
    // fill the chunk's mask (unless the streaming pass or the search tail
    // filled it already), then scatter the kept ids of the own list
    if (sel_all ? !c.one_fill_done : (sel_none || !(zero_filled || ph_mask))) fill_mask<DT>(c, sel_all ? 1 : 0);
    if (list_emit && !sel_all && !sel_none) {
      __syncthreads();  // the fill is ordered before the scatter
      if (fused_ties) {
        // the entries above tau are written: the ties below the cut remain
        const uint32_t nt = vld(F.tail_n);
        if (nt <= kTieCap) {
          const uint32_t* tix = reinterpret_cast<const uint32_t*>(c.ring_ptr);
          for (uint32_t i = tid; i < nt; i += kThreads) {
            const uint32_t ix = tix[i];
            if (ix < idx_cut) c.gmask[ix] = 1;
          }
        } else {
          own_for(c, [&](float x, uint32_t ix) {
            if (x == tau_f && ix < idx_cut) c.gmask[ix] = 1;
          });
        }
      } else {
        own_for(c, [&](float x, uint32_t ix) {
          bool keep = x > tau_f;
          if (x == tau_f) keep = (tie_mode == 1) || (tie_mode == 2 && ix < idx_cut);
          if (keep) c.gmask[ix] = 1;
        });
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
    stream_chunk<DT>(
        c,
        [&](const float (&xs)[E], uint32_t idx0, bool valid) {
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
          if (!valid) return;
          uint8_t bytes[E];
#pragma unroll
          for (int e = 0; e < E; ++e) bytes[e] = byte_of(xs[e], idx0 + e, rank);
          uint8_t* dst = c.gmask + idx0;
          if (vec_ok) {
            if constexpr (E == 4) {
              *reinterpret_cast<uint32_t*>(dst) =
                  bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (static_cast<uint32_t>(bytes[3]) << 24);
            } else {
              const uint32_t w0 =
                  bytes[0] | (bytes[1] << 8) | (bytes[2] << 16) | (static_cast<uint32_t>(bytes[3]) << 24);
              const uint32_t w1 =
                  bytes[4] | (bytes[5] << 8) | (bytes[6] << 16) | (static_cast<uint32_t>(bytes[7]) << 24);
              *reinterpret_cast<uint2*>(dst) = make_uint2(w0, w1);
            }
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) dst[e] = bytes[e];
          }
        },
        [&](float x, uint32_t idx, bool valid) {
          // the head was emitted above: only tail elements remain (index order = thread order)
          const bool tail = valid && idx >= static_cast<uint32_t>(c.head_n);
          uint32_t rank = 0;
          if (ordered_ties) {
            uint32_t tot;
            rank = running + block_excl_scan(F, (tail && x == tau_f) ? 1u : 0u, &tot);
            running += tot;
          }
          if (tail) c.gmask[idx] = byte_of(x, idx, rank);
        },
        false, ring_stages(list_region_bytes(static_cast<int>(c.ocap)), 0));
  }
  QRITA_T(7);

  // ---- a bulk-copy wait that gave up anywhere in the row voids the row.
  // The last cluster barrier: no CTA leaves while another may still access
  // its memory, and every CTA learns whether any CTA of the row failed.
  __syncthreads();
  if (early_arrive) {
    cluster_wait();
  } else {
    if (tid == 0 && vld(F.err) != 0u) {
      ring_drain<DT>(c);
      for (uint32_t rr = 0; rr < c.C; ++rr) st_dsmem_u32(map_rank(smem_u32(&F.err_any), rr), 1u);
    }
    if (c.C > 1) cluster_sync_all();
    else __syncthreads();
  }
  if (vld(F.err_any) != 0u) {
    for (int i = tid; i < c.n; i += kThreads) c.gmask[i] = 0;
    row_status = QRITA_ROW_TIMEOUT;
    sel_none = true;
    sel_all = false;
  }
  QRITA_T(15);

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
      info.z = static_cast<double>(z_used) / static_cast<double>(c.fix_scale);
      info.passes = passes;
      info.reserved = 0u;
      P.row_info[r] = info;
    }
  }
}

}  // namespace

static_assert(2 * (sizeof(Fixed) + list_region_bytes(kOwnCap) + 128 + kSmemReservedPerCta) <=
                  static_cast<size_t>(kSmemPerSm),
              "two CTAs must fit one SM");

size_t smem_bytes(int ocap) {
  const size_t lists = list_region_bytes(ocap);
  // the ring must clear the own list and the narrowing bins laid over the region
  const size_t ring_off = lists - kRingBytes;
  if (ring_off < static_cast<size_t>(kBinBytes) || ring_off < static_cast<size_t>(kWideTotOff) + 4096u) return 0;
  return (sizeof(Fixed) + lists + 127u) & ~static_cast<size_t>(127u);
}

int max_smem_per_block() {
  int dev = 0;
  cudaGetDevice(&dev);
  int v = 0;
  cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  return v;
}

#ifdef QRITA_TRACE_TIME
extern "C" int qrita_debug_stages(unsigned long long* out, int n) {
  cudaDeviceSynchronize();
  if (n > kTraceCtas) n = kTraceCtas;
  return static_cast<int>(cudaMemcpyFromSymbol(out, g_cta_stage, sizeof(unsigned long long) * 16 * n));
}
extern "C" int qrita_debug_rows(long long* out, int n) {
  cudaDeviceSynchronize();
  if (n > kTraceCtas) n = kTraceCtas;
  return static_cast<int>(cudaMemcpyFromSymbol(out, g_cta_row, sizeof(long long) * n));
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
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(prm.C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: the CTAs may be scheduled while the
  // previous kernel of the stream drains; they wait for it (griddepcontrol)
  // before touching memory
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (dtype == QRITA_DTYPE_F32) {
    e = cudaLaunchKernelEx(&cfg, select_kernel<QRITA_DTYPE_F32>, prm);
  } else {
    e = cudaLaunchKernelEx(&cfg, select_kernel<QRITA_DTYPE_BF16>, prm);
  }
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaGetLastError());
}

}  // namespace qrita
