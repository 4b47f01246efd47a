// C ABI of liblocks.so: argument validation, workspace carving and launches
// on the caller's stream.  No allocation, no synchronisation (except
// locks_read_status, which documents it).
#include <stdio.h>

#include "common.cuh"
#include "launch.h"

using namespace locks;

namespace locks {
std::atomic<long long> g_kernel_launches{0};
}

static thread_local int g_last_cuda = 0;

static locks_status_t fail_cuda(cudaError_t e) {
  g_last_cuda = (int)e;
  return LOCKS_ERR_CUDA;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// bytes of the scoring region: s_hat [batch][h_kv][G][max_pages] float and
// selection keys [batch][h_kv][max_pages] u32
static size_t score_region(int batch, int h_q, int h_kv, int max_pages) {
  const size_t G = (size_t)(h_q / h_kv);
  return round_up((size_t)batch * h_kv * G * max_pages * 4, 256) +
         round_up((size_t)batch * h_kv * max_pages * 4, 256);
}

// Decode partials: one slot per (unit, warp) piece, slot index unit + warp,
// so units + (warps launched) slots suffice.  The grid never has more warps
// than list positions nor more than kDecMaxWarps.
constexpr long long kDecMaxWarps = 8192;

static long long decode_warps_cap(int batch, int h_kv, int list_len) {
  long long w = (long long)batch * h_kv * list_len;
  if (w > kDecMaxWarps) w = kDecMaxWarps;
  return w < 1 ? 1 : w;
}

// bytes of the decode region: the unit layout written by the decode kernel
// (int meta[batch + 2]), o_part [slots][G][128] float and lse_part
// [slots][G] float
static size_t decode_meta_bytes(int batch) {
  return round_up(((size_t)batch + 2) * 4, 256);
}
static size_t decode_slots(int batch, int h_kv, int list_len) {
  return (size_t)batch * h_kv + (size_t)decode_warps_cap(batch, h_kv, list_len);
}
static size_t decode_region(int batch, int h_q, int h_kv, int list_len) {
  const size_t rows = decode_slots(batch, h_kv, list_len) * (size_t)(h_q / h_kv);
  return decode_meta_bytes(batch) + round_up(rows * kDim * 4, 256) +
         round_up(rows * 4, 256);
}

static bool heads_ok(int h_q, int h_kv) {
  return h_kv >= 1 && h_q >= h_kv && h_q % h_kv == 0;
}

static locks_status_t check_select_args(int batch, int h_q, int h_kv,
                                        int max_pages, int k,
                                        const int32_t *seq_lens,
                                        int32_t *idx_out, void *workspace) {
  if (batch < 0 || max_pages < 1 || k < 2 || !heads_ok(h_q, h_kv))
    return LOCKS_ERR_INVALID_ARG;
  if (h_q / h_kv > kMaxGroup) return LOCKS_ERR_UNSUPPORTED;
  if (batch > 65535 || h_kv > 65535) return LOCKS_ERR_UNSUPPORTED;
  if ((long long)max_pages * kPage > 0x7fffffffLL) return LOCKS_ERR_UNSUPPORTED;
  if (batch > 0 && (!seq_lens || !idx_out || !workspace))
    return LOCKS_ERR_INVALID_ARG;
  return LOCKS_OK;
}

locks_status_t locks::score_select(const void *q, const void *summaries,
                                   const int32_t *seq_lens, int batch, int h_q,
                                   int h_kv, int max_pages, int k,
                                   int32_t *idx_out, void *workspace,
                                   size_t workspace_bytes, cudaStream_t stream,
                                   bool after_query) {
  locks_status_t st = check_select_args(batch, h_q, h_kv, max_pages, k,
                                        seq_lens, idx_out, workspace);
  if (st != LOCKS_OK) return st;
  if (batch == 0) return LOCKS_OK;
  if (!q || !summaries) return LOCKS_ERR_INVALID_ARG;
  if (batch > score_max_batch()) return LOCKS_ERR_UNSUPPORTED;
  if (workspace_bytes < kWsHeader + score_region(batch, h_q, h_kv, max_pages))
    return LOCKS_ERR_WORKSPACE;
  const int G = h_q / h_kv;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *status = reinterpret_cast<int32_t *>(ws);
  float *s_hat = reinterpret_cast<float *>(ws + kWsHeader);
  uint32_t *keys = reinterpret_cast<uint32_t *>(
      ws + kWsHeader + round_up((size_t)batch * h_kv * G * max_pages * 4, 256));
  // short page lists on fewer units than SMs: one launch, the selection
  // done by the cluster that scored the unit
  const int cluster = fused_cluster_size(batch, h_kv, G, max_pages);
  if (cluster > 0) {
    const cudaError_t e = launch_score_select_fused(
        q, summaries, seq_lens, batch, h_kv, G, max_pages, k, cluster, s_hat,
        idx_out, status, stream, after_query);
    return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
  }
  cudaError_t e = launch_score(q, summaries, seq_lens, batch, h_kv, G,
                               max_pages, s_hat, status, stream, after_query);
  if (e != cudaSuccess) return fail_cuda(e);
  e = launch_select(s_hat, seq_lens, batch, h_kv, G, max_pages, k,
                    LOCKS_MERGE_SHARE_AVERAGE, idx_out, keys, status, stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks::sparse_decode(
    const void *q, const void *k_cache, const void *v_cache,
    int64_t num_phys_pages, const int32_t *page_table,
    const int32_t *seq_lens, const int32_t *idx, int k, int batch, int h_q,
    int h_kv, int max_pages, void *o_out, float *lse_out, void *workspace,
    size_t workspace_bytes, cudaStream_t stream, int32_t *status_mirror) {
  if (batch < 0 || max_pages < 1 || num_phys_pages < 1 || !heads_ok(h_q, h_kv))
    return LOCKS_ERR_INVALID_ARG;
  if (idx && k < 1) return LOCKS_ERR_INVALID_ARG;
  if (h_q / h_kv > kMaxGroup) return LOCKS_ERR_UNSUPPORTED;
  if (batch > 65535 || h_kv > 65535) return LOCKS_ERR_UNSUPPORTED;
  if ((long long)max_pages * kPage > 0x7fffffffLL) return LOCKS_ERR_UNSUPPORTED;
  if (batch == 0) return LOCKS_OK;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || !o_out ||
      !lse_out || !workspace)
    return LOCKS_ERR_INVALID_ARG;
  const int list_len = idx ? k : max_pages;
  // every list entry of every (sequence, KV head) is one int32 position
  if ((long long)batch * h_kv * list_len > 0x7fffffffLL)
    return LOCKS_ERR_UNSUPPORTED;
  if (batch > decode_max_batch()) return LOCKS_ERR_UNSUPPORTED;
  if (workspace_bytes < kWsHeader + decode_region(batch, h_q, h_kv, list_len))
    return LOCKS_ERR_WORKSPACE;
  const int G = h_q / h_kv;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *status = reinterpret_cast<int32_t *>(ws);
  const size_t rows = decode_slots(batch, h_kv, list_len) * (size_t)G;
  int *meta = reinterpret_cast<int *>(ws + kWsHeader);
  float *o_part =
      reinterpret_cast<float *>(ws + kWsHeader + decode_meta_bytes(batch));
  float *lse_part = reinterpret_cast<float *>(
      ws + kWsHeader + decode_meta_bytes(batch) + round_up(rows * kDim * 4, 256));
  const int max_warps = (int)decode_warps_cap(batch, h_kv, list_len);
  cudaError_t e = launch_decode(
      q, k_cache, v_cache, num_phys_pages, page_table, seq_lens, idx, k, batch,
      h_kv, G, max_pages, max_warps, o_out, lse_out, o_part, lse_part, meta,
      status, stream, status_mirror);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

extern "C" {

const char *locks_status_string(locks_status_t s) {
  switch (s) {
    case LOCKS_OK: return "ok";
    case LOCKS_ERR_INVALID_ARG: return "invalid argument";
    case LOCKS_ERR_UNSUPPORTED: return "unsupported size";
    case LOCKS_ERR_WORKSPACE: return "workspace too small";
    case LOCKS_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

int locks_last_cuda_error(void) { return g_last_cuda; }

long long locks_kernel_launches(void) {
  return g_kernel_launches.load(std::memory_order_relaxed);
}

size_t locks_summary_record_bytes(void) { return (size_t)kRec; }

locks_status_t locks_workspace_size(int batch, int h_q, int h_kv,
                                    int max_pages, int k, size_t *bytes) {
  if (!bytes || batch < 0 || max_pages < 1 || k < 1 || !heads_ok(h_q, h_kv))
    return LOCKS_ERR_INVALID_ARG;
  if (h_q / h_kv > kMaxGroup) return LOCKS_ERR_UNSUPPORTED;
  const size_t a = score_region(batch, h_q, h_kv, max_pages);
  const size_t b = decode_region(batch, h_q, h_kv, k);
  *bytes = kWsHeader + (a > b ? a : b);
  return LOCKS_OK;
}

static bool build_flags_ok(int flags) {
  return (flags & ~LOCKS_BUILD_VSCALE_PER_PAGE) == 0;
}

locks_status_t locks_build_summaries(
    const void *k_cache, int64_t num_phys_pages, int h_kv,
    const int32_t *page_table, int batch, int max_pages,
    const int32_t *seq_ids, const int32_t *page_ids, int n_pairs,
    void *summaries, float *tau_out, float *unquantised_out, int32_t *status,
    locks_stream_t stream) {
  return locks_build_summaries_ex(k_cache, num_phys_pages, h_kv, page_table,
                                  batch, max_pages, seq_ids, page_ids, n_pairs,
                                  summaries, tau_out, unquantised_out, 0,
                                  status, stream);
}

locks_status_t locks_build_summaries_ex(
    const void *k_cache, int64_t num_phys_pages, int h_kv,
    const int32_t *page_table, int batch, int max_pages,
    const int32_t *seq_ids, const int32_t *page_ids, int n_pairs,
    void *summaries, float *tau_out, float *unquantised_out, int flags,
    int32_t *status, locks_stream_t stream) {
  if (n_pairs < 0 || h_kv < 1 || batch < 1 || max_pages < 1 ||
      num_phys_pages < 1 || !build_flags_ok(flags))
    return LOCKS_ERR_INVALID_ARG;
  if (n_pairs == 0) return LOCKS_OK;
  if (!k_cache || !page_table || !seq_ids || !page_ids || !summaries)
    return LOCKS_ERR_INVALID_ARG;
  cudaError_t e = launch_build(k_cache, num_phys_pages, h_kv, page_table,
                               batch, max_pages, seq_ids, page_ids, n_pairs,
                               summaries, tau_out, unquantised_out, flags,
                               status, (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

static bool variant_ok(int rank, int vbits) {
  return (rank == 4 || rank == 8 || rank == 12 || rank == 15) &&
         (vbits == 2 || vbits == 4 || vbits == 8);
}

size_t locks_variant_record_bytes(int rank, int vbits) {
  return variant_ok(rank, vbits) ? variant_record_bytes(rank, vbits) : 0;
}

locks_status_t locks_build_variant(
    const void *k_cache, int64_t num_phys_pages, int h_kv,
    const int32_t *page_table, int batch, int max_pages,
    const int32_t *seq_ids, const int32_t *page_ids, int n_pairs, int rank,
    int vbits, void *records, float *tau_out, int32_t *status,
    locks_stream_t stream) {
  if (!variant_ok(rank, vbits)) return LOCKS_ERR_INVALID_ARG;
  if (n_pairs < 0 || h_kv < 1 || batch < 1 || max_pages < 1 ||
      num_phys_pages < 1)
    return LOCKS_ERR_INVALID_ARG;
  if (n_pairs == 0) return LOCKS_OK;
  if (!k_cache || !page_table || !seq_ids || !page_ids || !records)
    return LOCKS_ERR_INVALID_ARG;
  cudaError_t e = launch_build_variant(
      k_cache, num_phys_pages, h_kv, page_table, batch, max_pages, seq_ids,
      page_ids, n_pairs, rank, vbits, records, tau_out, status,
      (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_score_variant(const void *q, const void *records,
                                   int rank, int vbits,
                                   const int32_t *seq_lens, int batch,
                                   int h_q, int h_kv, int max_pages,
                                   float *scores_out, int32_t *status,
                                   locks_stream_t stream) {
  if (!variant_ok(rank, vbits)) return LOCKS_ERR_INVALID_ARG;
  if (batch < 0 || max_pages < 1 || !heads_ok(h_q, h_kv))
    return LOCKS_ERR_INVALID_ARG;
  if (h_q / h_kv > kMaxGroup) return LOCKS_ERR_UNSUPPORTED;
  if (batch > variant_max_batch(rank, vbits) || h_kv > 65535 ||
      (long long)max_pages * kPage > 0x7fffffffLL)
    return LOCKS_ERR_UNSUPPORTED;
  if (batch == 0) return LOCKS_OK;
  if (!q || !records || !seq_lens || !scores_out) return LOCKS_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(records) & 15u) return LOCKS_ERR_INVALID_ARG;
  cudaError_t e = launch_score_variant(q, records, rank, vbits, seq_lens,
                                       batch, h_kv, h_q / h_kv, max_pages,
                                       scores_out, status,
                                       (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_pack_summaries(const float *mu, const float *basis,
                                    const float *coeffs, int n, void *records,
                                    locks_stream_t stream) {
  return locks_pack_summaries_ex(mu, basis, coeffs, n, records, 0, stream);
}

locks_status_t locks_pack_summaries_ex(const float *mu, const float *basis,
                                       const float *coeffs, int n,
                                       void *records, int flags,
                                       locks_stream_t stream) {
  if (n < 0 || !build_flags_ok(flags)) return LOCKS_ERR_INVALID_ARG;
  if (n == 0) return LOCKS_OK;
  if (!mu || !basis || !coeffs || !records) return LOCKS_ERR_INVALID_ARG;
  cudaError_t e = launch_pack(mu, basis, coeffs, n, records, flags,
                              (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_score_select(const void *q, const void *summaries,
                                  const int32_t *seq_lens, int batch, int h_q,
                                  int h_kv, int max_pages, int k,
                                  int32_t *idx_out, void *workspace,
                                  size_t workspace_bytes,
                                  locks_stream_t stream) {
  return locks::score_select(q, summaries, seq_lens, batch, h_q, h_kv,
                             max_pages, k, idx_out, workspace, workspace_bytes,
                             (cudaStream_t)stream, false);
}

locks_status_t locks_score_pages(const void *q, const void *summaries,
                                 const int32_t *seq_lens, int batch, int h_q,
                                 int h_kv, int max_pages, float *scores_out,
                                 int32_t *status, locks_stream_t stream) {
  if (batch < 0 || max_pages < 1 || !heads_ok(h_q, h_kv))
    return LOCKS_ERR_INVALID_ARG;
  if (h_q / h_kv > kMaxGroup) return LOCKS_ERR_UNSUPPORTED;
  if ((long long)max_pages * kPage > 0x7fffffffLL) return LOCKS_ERR_UNSUPPORTED;
  if (batch == 0) return LOCKS_OK;
  if (!q || !summaries || !seq_lens || !scores_out)
    return LOCKS_ERR_INVALID_ARG;
  if (batch > score_max_batch()) return LOCKS_ERR_UNSUPPORTED;
  cudaError_t e = launch_score(q, summaries, seq_lens, batch, h_kv,
                               h_q / h_kv, max_pages, scores_out, status,
                               (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_exact_page_scores(
    const void *q, const void *k_cache, int64_t num_phys_pages,
    const int32_t *page_table, const int32_t *seq_lens, int batch, int h_q,
    int h_kv, int max_pages, float *scores_out, int32_t *status,
    locks_stream_t stream) {
  if (batch < 0 || max_pages < 1 || num_phys_pages < 1 || !heads_ok(h_q, h_kv))
    return LOCKS_ERR_INVALID_ARG;
  if (h_q / h_kv > kMaxGroup) return LOCKS_ERR_UNSUPPORTED;
  if ((long long)max_pages * kPage > 0x7fffffffLL ||
      (long long)batch * h_kv * max_pages > 0x7fffffffLL)
    return LOCKS_ERR_UNSUPPORTED;
  if (batch == 0) return LOCKS_OK;
  if (!q || !k_cache || !page_table || !seq_lens || !scores_out)
    return LOCKS_ERR_INVALID_ARG;
  if (batch > exact_max_batch()) return LOCKS_ERR_UNSUPPORTED;
  cudaError_t e = launch_exact(q, k_cache, num_phys_pages, page_table,
                               seq_lens, batch, h_kv, h_q / h_kv, max_pages,
                               scores_out, status, (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_select_pages_merge(const float *scores,
                                        const int32_t *seq_lens, int batch,
                                        int h_q, int h_kv, int max_pages,
                                        int k, int rule, int32_t *idx_out,
                                        void *workspace,
                                        size_t workspace_bytes,
                                        locks_stream_t stream) {
  if (rule != LOCKS_MERGE_SHARE_AVERAGE && rule != LOCKS_MERGE_GROUP_MAX &&
      rule != LOCKS_MERGE_GROUP_MASS)
    return LOCKS_ERR_INVALID_ARG;
  locks_status_t st = check_select_args(batch, h_q, h_kv, max_pages, k,
                                        seq_lens, idx_out, workspace);
  if (st != LOCKS_OK) return st;
  if (batch == 0) return LOCKS_OK;
  if (!scores) return LOCKS_ERR_INVALID_ARG;
  if (workspace_bytes < kWsHeader + score_region(batch, h_q, h_kv, max_pages))
    return LOCKS_ERR_WORKSPACE;
  const int G = h_q / h_kv;
  uint8_t *ws = static_cast<uint8_t *>(workspace);
  int32_t *status = reinterpret_cast<int32_t *>(ws);
  uint32_t *keys = reinterpret_cast<uint32_t *>(
      ws + kWsHeader + round_up((size_t)batch * h_kv * G * max_pages * 4, 256));
  cudaError_t e =
      launch_select(scores, seq_lens, batch, h_kv, G, max_pages, k, rule,
                    idx_out, keys, status, (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_select_pages(const float *scores, const int32_t *seq_lens,
                                  int batch, int h_q, int h_kv, int max_pages,
                                  int k, int32_t *idx_out, void *workspace,
                                  size_t workspace_bytes,
                                  locks_stream_t stream) {
  return locks_select_pages_merge(scores, seq_lens, batch, h_q, h_kv,
                                  max_pages, k, LOCKS_MERGE_SHARE_AVERAGE,
                                  idx_out, workspace, workspace_bytes, stream);
}

locks_status_t locks_sparse_decode(
    const void *q, const void *k_cache, const void *v_cache,
    int64_t num_phys_pages, const int32_t *page_table,
    const int32_t *seq_lens, const int32_t *idx, int k, int batch, int h_q,
    int h_kv, int max_pages, void *o_out, float *lse_out, void *workspace,
    size_t workspace_bytes, locks_stream_t stream) {
  return locks::sparse_decode(q, k_cache, v_cache, num_phys_pages, page_table,
                              seq_lens, idx, k, batch, h_q, h_kv, max_pages,
                              o_out, lse_out, workspace, workspace_bytes,
                              (cudaStream_t)stream, nullptr);
}

locks_status_t locks_append_kv(const void *k_new, const void *v_new,
                               void *k_cache, void *v_cache,
                               int64_t num_phys_pages, int h_kv,
                               const int32_t *page_table, int batch,
                               int max_pages, int32_t *seq_lens,
                               void *summaries, float *tau_out,
                               int32_t *status, locks_stream_t stream) {
  return locks_append_kv_ex(k_new, v_new, k_cache, v_cache, num_phys_pages,
                            h_kv, page_table, batch, max_pages, seq_lens,
                            summaries, tau_out, 0, status, stream);
}

locks_status_t locks_append_kv_ex(const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache,
                                  int64_t num_phys_pages, int h_kv,
                                  const int32_t *page_table, int batch,
                                  int max_pages, int32_t *seq_lens,
                                  void *summaries, float *tau_out, int flags,
                                  int32_t *status, locks_stream_t stream) {
  if (batch < 0 || h_kv < 1 || max_pages < 1 || num_phys_pages < 1 ||
      !build_flags_ok(flags))
    return LOCKS_ERR_INVALID_ARG;
  if (h_kv > 32) return LOCKS_ERR_UNSUPPORTED;
  if (batch == 0) return LOCKS_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !page_table || !seq_lens ||
      !summaries)
    return LOCKS_ERR_INVALID_ARG;
  cudaError_t e = launch_append(k_new, v_new, k_cache, v_cache, num_phys_pages,
                                h_kv, page_table, batch, max_pages, seq_lens,
                                summaries, tau_out, flags, status,
                                (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_clear_status(void *status_word, locks_stream_t stream) {
  if (!status_word) return LOCKS_ERR_INVALID_ARG;
  cudaError_t e =
      cudaMemsetAsync(status_word, 0, sizeof(int32_t), (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

locks_status_t locks_read_status(const void *status_word, int32_t *host_out,
                                 locks_stream_t stream) {
  if (!status_word || !host_out) return LOCKS_ERR_INVALID_ARG;
  cudaError_t e = cudaMemcpyAsync(host_out, status_word, sizeof(int32_t),
                                  cudaMemcpyDeviceToHost, (cudaStream_t)stream);
  if (e != cudaSuccess) return fail_cuda(e);
  e = cudaStreamSynchronize((cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : fail_cuda(e);
}

}  // extern "C"
