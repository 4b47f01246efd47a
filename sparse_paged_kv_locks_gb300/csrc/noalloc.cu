// Score-and-select for callers that cannot allocate device memory.
//
// Some callers may not allocate on the decode path at all: a serving engine
// whose device memory plan is frozen once it has started, a plugin that is
// handed only its input and output buffers, or code that must not touch the
// allocator while it runs.  locks_score_select_static gives them the same
// computation as locks_score_select with the scratch (page scores and
// selection keys) taken from a fixed array compiled into this library
// instead of a caller workspace.
//
// The array is a file-scope __device__ symbol, so every GPU that loads the
// library holds it until the process exits.  Host code must not hand the
// symbol itself to a kernel: on the host it names a host-side stand-in, not
// a device address.  The device address is looked up once per device with
// cudaGetSymbolAddress, with that device current, on the first call made on
// that device (so that first call should happen before any stream capture),
// and cached for the life of the process; a cudaDeviceReset of that device
// afterwards is not supported (the array may be placed elsewhere).
#include <mutex>

#include "common.cuh"
#include "launch.h"

namespace locks {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

static void *g_scratch_ptr[kMaxDevices];
static std::mutex g_scratch_mutex;

static size_t scratch_round(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace locks

using namespace locks;

extern "C" locks_status_t locks_score_select_static(
    const void *q, const void *summaries, const int32_t *seq_lens, int batch,
    int h_q, int h_kv, int max_pages, int k, int32_t *idx_out, int32_t *status,
    locks_stream_t stream) {
  if (batch < 0 || max_pages < 1 || k < 2 || h_kv < 1 || h_q < h_kv ||
      h_q % h_kv != 0)
    return LOCKS_ERR_INVALID_ARG;
  const int G = h_q / h_kv;
  if (G > kMaxGroup || batch > 65535 || h_kv > 65535 ||
      (long long)max_pages * kPage > 0x7fffffffLL)
    return LOCKS_ERR_UNSUPPORTED;
  if (batch == 0) return LOCKS_OK;
  if (!q || !summaries || !seq_lens || !idx_out) return LOCKS_ERR_INVALID_ARG;
  if (batch > score_max_batch()) return LOCKS_ERR_UNSUPPORTED;
  // scores [batch][h_kv][G][max_pages] float, then keys [batch][h_kv]
  // [max_pages] u32, each region rounded to 256 bytes
  const size_t score_bytes =
      scratch_round((size_t)batch * h_kv * G * max_pages * 4);
  const size_t key_bytes = scratch_round((size_t)batch * h_kv * max_pages * 4);
  if (score_bytes + key_bytes > kStaticScratchBytes)
    return LOCKS_ERR_UNSUPPORTED;  // beyond the built-in scratch

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return LOCKS_ERR_CUDA;
  void *base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
      void *p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
      if (e != cudaSuccess || p == nullptr) return LOCKS_ERR_CUDA;
      g_scratch_ptr[dev] = p;
    }
    base = g_scratch_ptr[dev];
  }
  // Nothing in the scratch has to start at zero: the scores of every full
  // page and every key are written before they are read within this call.
  float *s_hat = static_cast<float *>(base);
  uint32_t *keys = reinterpret_cast<uint32_t *>(
      static_cast<unsigned char *>(base) + score_bytes);
  cudaError_t e = launch_score(q, summaries, seq_lens, batch, h_kv, G,
                               max_pages, s_hat, status, (cudaStream_t)stream);
  if (e != cudaSuccess) return LOCKS_ERR_CUDA;
  e = launch_select(s_hat, seq_lens, batch, h_kv, G, max_pages, k,
                    LOCKS_MERGE_SHARE_AVERAGE, idx_out, keys, status,
                    (cudaStream_t)stream);
  return e == cudaSuccess ? LOCKS_OK : LOCKS_ERR_CUDA;
}
