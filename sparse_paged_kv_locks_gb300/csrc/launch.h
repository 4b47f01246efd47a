// Internal launchers of the LOCKS kernels (called by the C ABI in api.cu).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>

#include "locks.h"

namespace locks {

// Launch facts cached per CUDA device: function attributes are set per
// device, and SM counts and occupancy are properties of the device, so a
// process that launches on several GPUs keeps one entry for each.  The
// caches are function-level statics (zero-initialised); concurrent first
// calls compute the same value, so relaxed atomics suffice.
constexpr int kMaxCachedDevices = 64;
using DeviceFlags = std::atomic<int>[kMaxCachedDevices];

inline int cached_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev >= 0 && dev < kMaxCachedDevices ? dev : -1;
}

// Runs `step` (returning cudaError_t, e.g. a cudaFuncSetAttribute) until it
// has succeeded once on the current device.
template <class F>
cudaError_t once_per_device(DeviceFlags &done, F step) {
  const int dev = cached_device();
  if (dev >= 0 && done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = step();
  if (e == cudaSuccess && dev >= 0) done[dev].store(1, std::memory_order_relaxed);
  return e;
}

// A positive per-device value (SM count, resident blocks per SM) computed by
// `make` on the first call on each device; a `make` result below 1 is
// returned as 1 and not cached.
template <class F>
int per_device_value(DeviceFlags &cache, F make) {
  const int dev = cached_device();
  int v = dev >= 0 ? cache[dev].load(std::memory_order_relaxed) : 0;
  if (v > 0) return v;
  v = make();
  if (v < 1) return 1;
  if (dev >= 0) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

// Streaming multiprocessors of the current device (1 if the query fails).
inline int device_sm_count() {
  static DeviceFlags cache;
  return per_device_value(cache, [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
            cudaSuccess)
      return 0;
    return n;
  });
}

// locks_score_select on a cudaStream_t, with the scoring kernel optionally
// launched after_query (see launch_score).
locks_status_t score_select(const void *q, const void *summaries,
                            const int32_t *seq_lens, int batch, int h_q,
                            int h_kv, int max_pages, int k, int32_t *idx_out,
                            void *workspace, size_t workspace_bytes,
                            cudaStream_t stream, bool after_query);

cudaError_t launch_build(const void *k_cache, int64_t num_phys, int h_kv,
                         const int32_t *pt, int batch, int max_pages,
                         const int32_t *seq_ids, const int32_t *page_ids,
                         int n_pairs, void *summaries, float *tau_out,
                         float *unq_out, int flags, int32_t *status,
                         cudaStream_t stream);

cudaError_t launch_pack(const float *mu, const float *basis,
                        const float *coeffs, int n, void *records, int flags,
                        cudaStream_t stream);

cudaError_t launch_append(const void *k_new, const void *v_new, void *k_cache,
                          void *v_cache, int64_t num_phys, int h_kv,
                          const int32_t *pt, int batch, int max_pages,
                          int32_t *seq_lens, void *summaries, float *tau_out,
                          int flags, int32_t *status, cudaStream_t stream);

// after_query: launch as a programmatic dependent of the preceding kernel,
// which may write only the query (the kernel reads seq_lens and the
// summaries and starts its first copies before waiting on it).
cudaError_t launch_score(const void *q, const void *summaries,
                         const int32_t *seq_lens, int batch, int h_kv, int G,
                         int max_pages, float *s_hat, int32_t *status,
                         cudaStream_t stream, bool after_query = false);

// Single-launch score and select (share-average rule) for units with short
// page lists: one cluster of `cluster` CTAs per (sequence, KV head).
// fused_cluster_size: the cluster size for these sizes on the current
// device, 0 when the fused form does not apply (G > 8, more than 8192
// pages, more units than SMs, or the clusters cannot all be resident).
int fused_cluster_size(int batch, int h_kv, int G, int max_pages);
cudaError_t launch_score_select_fused(const void *q, const void *summaries,
                                      const int32_t *seq_lens, int batch,
                                      int h_kv, int G, int max_pages, int k,
                                      int cluster, float *s_hat, int32_t *idx,
                                      int32_t *status, cudaStream_t stream,
                                      bool after_query);

cudaError_t launch_select(const float *scores, const int32_t *seq_lens,
                          int batch, int h_kv, int G, int max_pages, int k,
                          int rule, int32_t *idx, uint32_t *keybuf,
                          int32_t *status, cudaStream_t stream);

cudaError_t launch_decode(const void *q, const void *k_cache,
                          const void *v_cache, int64_t num_phys,
                          const int32_t *pt, const int32_t *seq_lens,
                          const int32_t *idx, int k, int batch, int h_kv,
                          int G, int max_pages, int max_warps, void *o_out,
                          float *lse_out, float *o_part, float *lse_part,
                          int *meta, int32_t *status, cudaStream_t stream,
                          int32_t *status_mirror = nullptr);

// locks_sparse_decode on a cudaStream_t; status_mirror (optional): where
// the merge kernel copies the device status word at the end of the step
// (a mapped host word, for instance).
locks_status_t sparse_decode(const void *q, const void *k_cache,
                             const void *v_cache, int64_t num_phys_pages,
                             const int32_t *page_table,
                             const int32_t *seq_lens, const int32_t *idx,
                             int k, int batch, int h_q, int h_kv,
                             int max_pages, void *o_out, float *lse_out,
                             void *workspace, size_t workspace_bytes,
                             cudaStream_t stream, int32_t *status_mirror);

cudaError_t launch_exact(const void *q, const void *k_cache, int64_t num_phys,
                         const int32_t *pt, const int32_t *seq_lens,
                         int batch, int h_kv, int G, int max_pages,
                         float *scores, int32_t *status, cudaStream_t stream);

cudaError_t launch_build_variant(const void *k_cache, int64_t num_phys,
                                 int h_kv, const int32_t *pt, int batch,
                                 int max_pages, const int32_t *seq_ids,
                                 const int32_t *page_ids, int n_pairs,
                                 int rank, int vbits, void *records,
                                 float *tau_out, int32_t *status,
                                 cudaStream_t stream);

cudaError_t launch_score_variant(const void *q, const void *records,
                                 int rank, int vbits,
                                 const int32_t *seq_lens, int batch, int h_kv,
                                 int G, int max_pages, float *scores,
                                 int32_t *status, cudaStream_t stream);

// the scorer of one basis width (variant_b2.cu, variant_b4.cu, variant_b8.cu)
template <int VB>
cudaError_t launch_variant_bits(int rank, const void *q, const void *records,
                                const int32_t *seq_lens, int batch, int h_kv,
                                int G, int max_pages, float *scores,
                                int32_t *status, cudaStream_t stream);

size_t variant_record_bytes(int rank, int vbits);
// largest batch whose per-sequence tables fit beside the variant's ring
int variant_max_batch(int rank, int vbits);

int score_max_batch();
int exact_max_batch();
int decode_max_batch();

}  // namespace locks
