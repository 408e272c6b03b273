// Internal interface between the C ABI (qrita_api.cpp) and the kernel
// translation unit (qrita_kernel.cu). Not installed; not part of the ABI.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "qrita.h"

namespace qrita {

// delta tables (Qrita technical summary, "Methodology", part 1: precomputed
// tables from the normal quantile function, keyed on the target k or p).
//   lut_k[i] = Phi^-1(1 - 2^(-i/4)),  i = 0..127  (keyed on u = alpha*k/V;
//              the kernel takes i = floor(-4 log2 u), so 2^(-i/4) >= u)
//   lut_p[i] = Phi^-1(2^(-i/4)),      i = 0..63   (keyed on q = 1 - p;
//              the kernel takes i = ceil(-4 log2 q), so 2^(-i/4) <= q)
// Rounding the key toward the larger u / smaller q lowers the threshold, so
// the table never makes truncation less likely to hit than the exact value.
constexpr int kLutK = 128;
constexpr int kLutP = 64;

// Threads per CTA of the selection kernel.
constexpr int kThreads = 256;
// 16-byte units each thread keeps in flight while streaming a chunk.
constexpr int kUnroll = 8;
// Largest cluster the launcher uses (16 needs the non-portable opt-in).
constexpr int kMaxCluster = 16;
// Pivots one distributed narrowing pass evaluates: two quaternary levels,
// the 3 quartile pivots of the range and the 3 of each of its 4 quarters.
constexpr int kNarrowPivots = 15;
// Upper bound on quaternary rounds of one local search and on narrowing
// passes (guards; the pivot rule at least halves the key range every round
// on average, so 32-bit keys need at most about 34 rounds).
constexpr int kMaxRounds = 64;

// Capacity of a CTA's own candidate list (entries of value + index): 72 KiB,
// plus the 32 KiB streaming ring: two CTAs per SM.
constexpr int kOwnCap = 9216;
// Shared memory of one SM on GB300 and what the runtime reserves per CTA: two
// CTAs must fit.
constexpr int kSmemPerSm = 228 * 1024;
constexpr int kSmemReservedPerCta = 1024;

struct Params {
  const void* logits;
  uint8_t* mask;
  const int32_t* k;
  const float* p;
  int32_t* row_status;
  qrita_row_info_t* row_info;
  int64_t B;
  int32_t V;
  int32_t C;        // CTAs per row (cluster size)
  int32_t chunk;    // elements per CTA (multiple of 16)
  int32_t ocap;     // own candidate list capacity per CTA (entries)
  uint32_t flags;   // QRITA_FLAG_*
  int32_t heavy_first;  // more CTAs than fit at once: the rows expected to run longest start first
  float alpha_k;    // top-k truncation safety factor (u = alpha_k * k / V)
  float alpha_min_k;  // the smallest factor used to keep the survivors within the lists
  float margin_p;   // subtracted from the top-p delta
  float u_max_k;    // no truncation when alpha_k * k / V exceeds this
  float lut_k[kLutK];
  float lut_p[kLutP];
};


// Bytes of dynamic shared memory the kernel needs for an own-list capacity
// (0: the capacity leaves no room for the streaming ring).
size_t smem_bytes(int ocap);

// Launch the selection kernel (grid B*C, cluster C). Returns a cudaError_t.
int launch_select(const Params& prm, int dtype, size_t smem, qrita_stream_t stream);

// Largest dynamic shared memory per block on the current device.
int max_smem_per_block();

// Outputs beyond the mask (qrita_outputs.cu). Both return a cudaError_t.
constexpr int32_t kMaxIds = 8192;  // largest kmax of qrita_topk_ids
size_t ids_smem_bytes(int32_t kmax);
int launch_ids(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k, int32_t kmax,
               const uint8_t* mask, int32_t* out_ids, qrita_stream_t stream);
int launch_candidates(const void* logits, int dtype, int64_t B, int64_t V, const uint8_t* mask, int32_t cap,
                      int32_t* out_ids, float* out_probs, int32_t* out_count, const float* u, int32_t* out_sample,
                      qrita_stream_t stream);

}  // namespace qrita
