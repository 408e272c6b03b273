// C ABI of the selection library: argument checks, the delta tables, the
// launch shape, and the host-buffer entry point. See include/qrita.h.

#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>

#include <cuda_runtime.h>

#include "qrita.h"
#include "qrita_internal.h"

namespace qrita {
namespace {

// ---------------------------------------------------------------------------
// delta tables (Qrita technical summary, "Methodology", part 1: delta comes
// from precomputed tables derived from the normal quantile function, adapted
// to the target k or p). Phi^-1 is found by bisection on the C library's
// erfc, Phi(z) = erfc(-z / sqrt 2) / 2, to a bracket of 1e-13.
// ---------------------------------------------------------------------------
double normal_cdf(double z) { return 0.5 * std::erfc(-z / std::sqrt(2.0)); }

double normal_quantile(double prob) {
  if (prob <= 0.0) return -std::numeric_limits<double>::infinity();
  if (prob >= 1.0) return std::numeric_limits<double>::infinity();
  double lo = -40.0, hi = 40.0;
  for (int it = 0; it < 200 && hi - lo > 1e-13; ++it) {
    const double mid = 0.5 * (lo + hi);
    if (normal_cdf(mid) < prob) lo = mid;
    else hi = mid;
  }
  return 0.5 * (lo + hi);
}

struct Tables {
  float lut_k[kLutK];
  float lut_p[kLutP];
};

Tables build_tables() {
  Tables t;
  for (int i = 0; i < kLutK; ++i) {
    // Phi^-1(1 - u) = -Phi^-1(u), evaluated in the accurate lower tail
    const double u = std::exp2(-0.25 * i);
    t.lut_k[i] = static_cast<float>(-normal_quantile(u));
  }
  for (int i = 0; i < kLutP; ++i) {
    const double q = std::exp2(-0.25 * i);
    t.lut_p[i] = static_cast<float>(normal_quantile(q));
  }
  return t;
}

const Tables& tables() {
  static const Tables t = build_tables();
  return t;
}

// Truncation tuning (the pages give no constants; these only move speed,
// never the result): u = alpha_k * k / V, truncation skipped above u_max;
// alpha shrinks toward kAlphaMinK when alpha * k survivors would not fit the
// own lists.
constexpr float kAlphaK = 2.0f;
constexpr float kAlphaMinK = 1.25f;
constexpr float kUMaxK = 0.25f;
constexpr float kMarginP = 0.25f;

constexpr int kCtasPerSm = 2;
// Rows shorter than this per CTA are not split further.
constexpr int64_t kMinChunk = 3072;
// Chunk indices must fit below the rank bits of a gathered tag.
constexpr int64_t kMaxChunk = int64_t(1) << 27;

int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int n = 0;
  cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
  if (dev >= 0 && dev < 64 && n > 0) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

int smem_optin() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) {
    int v = cached[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  const int n = max_smem_per_block();
  if (dev >= 0 && dev < 64 && n > 0) cached[dev].store(n, std::memory_order_relaxed);
  return n;
}

int elem_bytes(int dtype) { return dtype == QRITA_DTYPE_F32 ? 4 : 2; }

struct Shape {
  int C;
  int chunk;
  int ocap;
  size_t smem;
  bool multi_wave;  // more CTAs than the device holds at once
};

// Rows are reordered (heavy first) only for batches this small: every CTA
// reads all k and p to find its row.
constexpr int64_t kMaxReorderRows = 8192;

// Launch shape: the row is split into C contiguous chunks (one CTA each, one
// cluster per row). C is the largest power of two that keeps the whole batch
// in one wave of resident CTAs, so small batches spread over every SM while
// large batches keep one CTA per row and stream it whole.
int choose_shape(int64_t B, int64_t V, uint32_t flags, Shape* out) {
  const int optin = smem_optin();
  if (optin <= 0) return QRITA_ECUDA;
  int C = 1;
  if (flags & QRITA_FLAG_CLUSTER_SET) {
    const int shift = static_cast<int>((flags >> QRITA_FLAG_CLUSTER_SHIFT) & 7u);
    if (shift > 4) return QRITA_EINVAL;
    C = 1 << shift;
  } else {
    const int64_t slots = static_cast<int64_t>(sm_count()) * kCtasPerSm;
    while (C < kMaxCluster && B * (2 * C) <= slots && (V + 2 * C - 1) / (2 * C) >= kMinChunk) C *= 2;
  }
  while ((V + C - 1) / C > kMaxChunk) {
    if (C >= kMaxCluster) return QRITA_EUNSUPPORTED;
    C *= 2;
  }
  int64_t chunk = (V + C - 1) / C;
  chunk = (chunk + 15) / 16 * 16;
  if (B * C > static_cast<int64_t>(std::numeric_limits<int32_t>::max())) return QRITA_EUNSUPPORTED;
  const int ocap = kOwnCap;
  const size_t smem = smem_bytes(ocap);
  if (smem == 0 || smem > static_cast<size_t>(optin)) return QRITA_EUNSUPPORTED;
  out->multi_wave = B * C > static_cast<int64_t>(sm_count()) * kCtasPerSm;
  out->C = C;
  out->chunk = static_cast<int>(chunk);
  out->ocap = ocap;
  out->smem = smem;
  return QRITA_OK;
}

int check_args(const void* logits, int dtype, int64_t B, int64_t V, const uint8_t* out_mask,
               uint32_t flags) {
  if (dtype != QRITA_DTYPE_F32 && dtype != QRITA_DTYPE_BF16) return QRITA_EINVAL;
  if (B < 0 || V < 1 || V > std::numeric_limits<int32_t>::max()) return QRITA_EINVAL;
  if (flags & ~QRITA_FLAG_KNOWN_MASK) return QRITA_EINVAL;
  if (B == 0) return QRITA_OK;
  if (logits == nullptr || out_mask == nullptr) return QRITA_EINVAL;
  if (reinterpret_cast<uintptr_t>(logits) % static_cast<uintptr_t>(elem_bytes(dtype)) != 0)
    return QRITA_EINVAL;
  return QRITA_OK;
}

int select_impl(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k,
                const float* p, uint8_t* out_mask, qrita_stream_t stream, uint32_t flags,
                int32_t* row_status, qrita_row_info_t* row_info) {
  int rc = check_args(logits, dtype, B, V, out_mask, flags);
  if (rc != QRITA_OK || B == 0) return rc;
  Shape sh;
  rc = choose_shape(B, V, flags, &sh);
  if (rc != QRITA_OK) return rc;
  Params prm;
  std::memset(&prm, 0, sizeof(prm));
  prm.logits = logits;
  prm.mask = out_mask;
  prm.k = k;
  prm.p = p;
  prm.row_status = row_status;
  prm.row_info = row_info;
  prm.B = B;
  prm.V = static_cast<int32_t>(V);
  prm.C = sh.C;
  prm.chunk = sh.chunk;
  prm.ocap = sh.ocap;
  prm.flags = flags;
  prm.heavy_first = (sh.multi_wave && B <= kMaxReorderRows && (p != nullptr || k != nullptr)) ? 1 : 0;
  prm.alpha_k = kAlphaK;
  prm.alpha_min_k = kAlphaMinK;
  prm.margin_p = kMarginP;
  prm.u_max_k = kUMaxK;
  const Tables& t = tables();
  std::memcpy(prm.lut_k, t.lut_k, sizeof(prm.lut_k));
  std::memcpy(prm.lut_p, t.lut_p, sizeof(prm.lut_p));
  const int e = launch_select(prm, dtype, sh.smem, stream);
  return e == 0 ? QRITA_OK : QRITA_ECUDA;
}

size_t align256(size_t x) { return (x + 255u) & ~static_cast<size_t>(255u); }

}  // namespace
}  // namespace qrita

extern "C" {

int qrita_select(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k,
                 const float* p, uint8_t* out_mask, qrita_stream_t stream) {
  return qrita::select_impl(logits, dtype, B, V, k, p, out_mask, stream, 0u, nullptr, nullptr);
}

int qrita_select_ex(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k,
                    const float* p, uint8_t* out_mask, qrita_stream_t stream, uint32_t flags,
                    int32_t* row_status, qrita_row_info_t* row_info) {
  return qrita::select_impl(logits, dtype, B, V, k, p, out_mask, stream, flags, row_status,
                            row_info);
}

size_t qrita_host_staging_bytes(int dtype, int64_t B, int64_t V) {
  if ((dtype != QRITA_DTYPE_F32 && dtype != QRITA_DTYPE_BF16) || B < 0 || V < 1 ||
      V > std::numeric_limits<int32_t>::max())
    return 0;
  // every section and the sum must fit size_t (0 = invalid, as above)
  constexpr size_t kMax = std::numeric_limits<size_t>::max();
  const size_t b = static_cast<size_t>(B), v = static_cast<size_t>(V);
  const size_t eb = static_cast<size_t>(qrita::elem_bytes(dtype));
  if (b != 0 && v > (kMax / 8u) / b) return 0;  // B*V*eb and the 256-byte roundings stay far below kMax
  const size_t n = b * v;
  return qrita::align256(n * eb) + qrita::align256(b * 4) + qrita::align256(b * 4) + qrita::align256(n);
}

int qrita_select_host(const void* h_logits, int dtype, int64_t B, int64_t V, const int32_t* h_k,
                      const float* h_p, uint8_t* h_mask, void* d_staging, size_t staging_bytes,
                      qrita_stream_t stream) {
  int rc = qrita::check_args(h_logits, dtype, B, V, h_mask, 0u);
  if (rc != QRITA_OK || B == 0) return rc;
  const size_t need = qrita_host_staging_bytes(dtype, B, V);
  if (d_staging == nullptr || staging_bytes < need) return QRITA_EINVAL;
  const size_t n = static_cast<size_t>(B) * static_cast<size_t>(V);
  const size_t lb = n * qrita::elem_bytes(dtype);
  unsigned char* base = static_cast<unsigned char*>(d_staging);
  void* d_logits = base;
  int32_t* d_k = reinterpret_cast<int32_t*>(base + qrita::align256(lb));
  float* d_p = reinterpret_cast<float*>(base + qrita::align256(lb) + qrita::align256(B * 4));
  uint8_t* d_mask = base + qrita::align256(lb) + 2 * qrita::align256(B * 4);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  // once a copy is enqueued, every return waits for the stream first: the
  // caller may free or reuse its host buffers as soon as the call returns
  auto fail_after_enqueue = [st](int code) {
    (void)cudaStreamSynchronize(st);
    return code;
  };
  if (cudaMemcpyAsync(d_logits, h_logits, lb, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return fail_after_enqueue(QRITA_ECUDA);
  if (h_k && cudaMemcpyAsync(d_k, h_k, B * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return fail_after_enqueue(QRITA_ECUDA);
  if (h_p && cudaMemcpyAsync(d_p, h_p, B * 4, cudaMemcpyHostToDevice, st) != cudaSuccess)
    return fail_after_enqueue(QRITA_ECUDA);
  rc = qrita::select_impl(d_logits, dtype, B, V, h_k ? d_k : nullptr, h_p ? d_p : nullptr, d_mask,
                          stream, 0u, nullptr, nullptr);
  if (rc != QRITA_OK) return fail_after_enqueue(rc);
  if (cudaMemcpyAsync(h_mask, d_mask, n, cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return fail_after_enqueue(QRITA_ECUDA);
  if (cudaStreamSynchronize(st) != cudaSuccess) return QRITA_ECUDA;
  return QRITA_OK;
}

int qrita_topk_ids(const void* logits, int dtype, int64_t B, int64_t V, const int32_t* k, int32_t kmax,
                   uint8_t* out_mask, int32_t* out_ids, qrita_stream_t stream) {
  int rc = qrita::check_args(logits, dtype, B, V, out_mask, 0u);
  if (rc != QRITA_OK || B == 0) return rc;
  if (k == nullptr || out_ids == nullptr || kmax < 1 || kmax > qrita::kMaxIds) return QRITA_EINVAL;
  if (B > static_cast<int64_t>(std::numeric_limits<int32_t>::max())) return QRITA_EUNSUPPORTED;
  rc = qrita::select_impl(logits, dtype, B, V, k, nullptr, out_mask, stream, 0u, nullptr, nullptr);
  if (rc != QRITA_OK) return rc;
  return qrita::launch_ids(logits, dtype, B, V, k, kmax, out_mask, out_ids, stream) == 0 ? QRITA_OK : QRITA_ECUDA;
}

int qrita_candidates(const void* logits, int dtype, int64_t B, int64_t V, const uint8_t* mask, int32_t cap,
                     int32_t* out_ids, float* out_probs, int32_t* out_count, const float* u, int32_t* out_sample,
                     qrita_stream_t stream) {
  int rc = qrita::check_args(logits, dtype, B, V, mask, 0u);
  if (rc != QRITA_OK || B == 0) return rc;
  if (cap < 1 || out_ids == nullptr || out_probs == nullptr || out_count == nullptr) return QRITA_EINVAL;
  if ((u == nullptr) != (out_sample == nullptr)) return QRITA_EINVAL;
  if (B > static_cast<int64_t>(std::numeric_limits<int32_t>::max())) return QRITA_EUNSUPPORTED;
  return qrita::launch_candidates(logits, dtype, B, V, mask, cap, out_ids, out_probs, out_count, u, out_sample,
                                  stream) == 0
             ? QRITA_OK
             : QRITA_ECUDA;
}

int qrita_delta_table(int which, float* out, int n) {
  const qrita::Tables& t = qrita::tables();
  const float* src = nullptr;
  int len = 0;
  if (which == 0) {
    src = t.lut_k;
    len = qrita::kLutK;
  } else if (which == 1) {
    src = t.lut_p;
    len = qrita::kLutP;
  } else {
    return -1;
  }
  if (out != nullptr && n > 0) std::memcpy(out, src, sizeof(float) * static_cast<size_t>(n < len ? n : len));
  return len;
}

const char* qrita_strerror(int code) {
  switch (code) {
    case QRITA_OK:
      return "success";
    case QRITA_EINVAL:
      return "invalid argument";
    case QRITA_EUNSUPPORTED:
      return "unsupported size: a row does not fit the shared memory of one cluster";
    case QRITA_ECUDA:
      return "CUDA runtime or launch error";
    default:
      return "unknown error code";
  }
}

int qrita_version(void) { return 100; }

}  // extern "C"
