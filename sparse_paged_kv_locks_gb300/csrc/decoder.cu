// Decoder object of the C ABI: one layer's decode step (LOCKS reading notes
// §2 Fig. 1 decode path: score the page summaries, select k pages, attend
// over them) driven from host buffers.  The first step records, on a
// private capture stream, a kernel that pulls the query from page-locked
// host memory into the device staging buffer and the four kernels of
// locks_score_select + locks_sparse_decode, the attention kernels writing
// o and lse straight into the caller's page-locked output buffers and the
// merge kernel copying the device status word out, as one CUDA graph;
// every later step is one graph launch on the caller's stream and one
// stream synchronisation.  The host buffers are reached through their
// mapped device addresses (page-locked memory is mapped into the GPU's
// address space under unified addressing; on Grace-Blackwell the accesses
// cross NVLink-C2C), which costs a few microseconds less per step than
// copy-engine transfers of these few hundred kilobytes.  Another query
// buffer is patched into the copy kernel's graph node; other output
// buffers make the next step record the graph again.
#include <stdint.h>

#include <new>

#include <cuda_runtime.h>

#include "common.cuh"
#include "launch.h"
#include "locks.h"

struct locks_decoder {
  // caller-owned device buffers and shape
  const void *k_cache, *v_cache;
  int64_t num_phys;
  const int32_t *page_table;
  const void *summaries;
  const int32_t *seq_lens;
  int batch, h_q, h_kv, max_pages, k;
  void *q_dev;
  int32_t *idx;
  void *workspace;
  size_t ws_bytes;
  size_t q_bytes;
  // runtime objects owned by the decoder
  cudaStream_t cap = nullptr;
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  cudaGraphNode_t n_in = nullptr;
  int graph_kernels = 0;  // kernel nodes of the instantiated step
  int32_t *st_host = nullptr;  // page-locked, one int32
  int32_t *st_map = nullptr;   // its mapped device address
  // host buffers the instantiated graph copies from / to, and their mapped
  // device addresses
  const void *q_host = nullptr;
  void *o_host = nullptr;
  float *lse_host = nullptr;
  const void *q_map = nullptr;
  void *o_map = nullptr;
  float *lse_map = nullptr;
  int last_cuda = 0;
};

namespace {

locks_status_t fail(locks_decoder *d, cudaError_t e) {
  d->last_cuda = (int)e;
  return LOCKS_ERR_CUDA;
}

// Mapped device address of page-locked (cudaHostAlloc or cudaHostRegister)
// host memory, 16-byte aligned; NULL for anything else.
const void *mapped(const void *p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || !a.devicePointer) return nullptr;
  if (reinterpret_cast<uintptr_t>(a.devicePointer) % 16 != 0) return nullptr;
  return a.devicePointer;
}

constexpr int kCopyThreads = 256;
constexpr int kCopyMaxCtas = 4 * 152;

int copy_grid(size_t n16) {
  size_t g = (n16 + kCopyThreads - 1) / kCopyThreads;
  if (g > (size_t)kCopyMaxCtas) g = kCopyMaxCtas;
  return g < 1 ? 1 : (int)g;
}

// query in: host (mapped) -> device staging buffer, 16 bytes per thread
__global__ void __launch_bounds__(kCopyThreads)
    host_in_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                   long long n16) {
  locks::pdl_trigger();  // scoring may start its summary stream meanwhile
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n16;
       i += (long long)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

// One step's work on `s`: query in, score + select, sparse attention with
// (o, lse, status word) out.  q_map / o_map / lse_map are mapped device
// addresses of the caller's host buffers.
locks_status_t enqueue_step(locks_decoder *d, cudaStream_t s,
                            const void *q_map, void *o_map, float *lse_map) {
  const long long n16 = (long long)(d->q_bytes / 16);
  host_in_kernel<<<copy_grid(n16), kCopyThreads, 0, s>>>(
      static_cast<const uint4 *>(q_map), static_cast<uint4 *>(d->q_dev), n16);
  cudaError_t e = locks::launched();
  if (e != cudaSuccess) return fail(d, e);
  locks_status_t st = locks::score_select(
      d->q_dev, d->summaries, d->seq_lens, d->batch, d->h_q, d->h_kv,
      d->max_pages, d->k, d->idx, d->workspace, d->ws_bytes, s, true);
  if (st != LOCKS_OK) return st;
  return locks::sparse_decode(d->q_dev, d->k_cache, d->v_cache, d->num_phys,
                              d->page_table, d->seq_lens, d->idx, d->k,
                              d->batch, d->h_q, d->h_kv, d->max_pages, o_map,
                              lse_map, d->workspace, d->ws_bytes, s,
                              d->st_map);
}

void drop_graph(locks_decoder *d) {
  if (d->exec) cudaGraphExecDestroy(d->exec);
  if (d->graph) cudaGraphDestroy(d->graph);
  d->exec = nullptr;
  d->graph = nullptr;
  d->n_in = nullptr;
  d->graph_kernels = 0;
}

// Warm-up run ordered after the caller's stream (first launches set kernel
// attributes), then capture and instantiate; finds the query copy kernel's
// node by its function.
locks_status_t record(locks_decoder *d, cudaStream_t caller,
                      const void *q_map, void *o_map, float *lse_map) {
  cudaEvent_t ev;
  cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
  if (e != cudaSuccess) return fail(d, e);
  e = cudaEventRecord(ev, caller);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(d->cap, ev, 0);
  cudaEventDestroy(ev);
  if (e != cudaSuccess) return fail(d, e);
  locks_status_t st = enqueue_step(d, d->cap, q_map, o_map, lse_map);
  if (st != LOCKS_OK) return st;
  e = cudaStreamSynchronize(d->cap);
  if (e != cudaSuccess) return fail(d, e);
  e = cudaStreamBeginCapture(d->cap, cudaStreamCaptureModeThreadLocal);
  if (e != cudaSuccess) return fail(d, e);
  st = enqueue_step(d, d->cap, q_map, o_map, lse_map);
  cudaGraph_t g = nullptr;
  e = cudaStreamEndCapture(d->cap, &g);
  if (st != LOCKS_OK || e != cudaSuccess) {
    if (g) cudaGraphDestroy(g);
    return st != LOCKS_OK ? st : fail(d, e);
  }
  d->graph = g;
  e = cudaGraphInstantiate(&d->exec, g, 0);
  if (e != cudaSuccess) {
    drop_graph(d);
    return fail(d, e);
  }
  size_t n = 0;
  e = cudaGraphGetNodes(g, nullptr, &n);
  cudaGraphNode_t nodes[64];
  if (e != cudaSuccess || n > 64) {
    drop_graph(d);
    return e != cudaSuccess ? fail(d, e) : LOCKS_ERR_UNSUPPORTED;
  }
  e = cudaGraphGetNodes(g, nodes, &n);
  if (e != cudaSuccess) {
    drop_graph(d);
    return fail(d, e);
  }
  for (size_t i = 0; i < n; ++i) {
    cudaGraphNodeType t;
    if (cudaGraphNodeGetType(nodes[i], &t) != cudaSuccess ||
        t != cudaGraphNodeTypeKernel)
      continue;
    ++d->graph_kernels;
    cudaKernelNodeParams p;
    if (cudaGraphKernelNodeGetParams(nodes[i], &p) != cudaSuccess) continue;
    if (p.func == reinterpret_cast<void *>(host_in_kernel)) d->n_in = nodes[i];
  }
  if (!d->n_in) {
    drop_graph(d);
    return LOCKS_ERR_UNSUPPORTED;
  }
  return LOCKS_OK;
}

locks_status_t retarget_query(locks_decoder *d, const void *q_map) {
  const long long n16 = (long long)(d->q_bytes / 16);
  const void *src = q_map;
  long long n = n16;
  void *args[3] = {const_cast<void **>(&src), &d->q_dev, &n};
  cudaKernelNodeParams p = {};
  p.func = reinterpret_cast<void *>(host_in_kernel);
  p.gridDim = dim3(copy_grid(n16));
  p.blockDim = dim3(kCopyThreads);
  p.kernelParams = args;
  cudaError_t e = cudaGraphExecKernelNodeSetParams(d->exec, d->n_in, &p);
  return e == cudaSuccess ? LOCKS_OK : fail(d, e);
}

}  // namespace

extern "C" {

locks_status_t locks_decoder_create(
    const void *k_cache, const void *v_cache, int64_t num_phys_pages,
    const int32_t *page_table, const void *summaries, const int32_t *seq_lens,
    int batch, int h_q, int h_kv, int max_pages, int k, void *q_dev,
    int32_t *idx, void *workspace, size_t workspace_bytes,
    locks_decoder_t **out) {
  if (!out) return LOCKS_ERR_INVALID_ARG;
  *out = nullptr;
  if (batch < 1 || k < 2 || max_pages < 1 || num_phys_pages < 1 ||
      h_kv < 1 || h_q < h_kv || h_q % h_kv != 0)
    return LOCKS_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || !page_table || !summaries || !seq_lens ||
      !q_dev || !idx || !workspace)
    return LOCKS_ERR_INVALID_ARG;
  size_t need = 0;
  locks_status_t st =
      locks_workspace_size(batch, h_q, h_kv, max_pages, k, &need);
  if (st != LOCKS_OK) return st;
  if (workspace_bytes < need) return LOCKS_ERR_WORKSPACE;
  locks_decoder *d = new (std::nothrow) locks_decoder;
  if (!d) return LOCKS_ERR_UNSUPPORTED;
  d->k_cache = k_cache;
  d->v_cache = v_cache;
  d->num_phys = num_phys_pages;
  d->page_table = page_table;
  d->summaries = summaries;
  d->seq_lens = seq_lens;
  d->batch = batch;
  d->h_q = h_q;
  d->h_kv = h_kv;
  d->max_pages = max_pages;
  d->k = k;
  d->q_dev = q_dev;
  d->idx = idx;
  d->workspace = workspace;
  d->ws_bytes = workspace_bytes;
  d->q_bytes = (size_t)batch * h_q * LOCKS_HEAD_DIM * 2;
  cudaError_t e = cudaStreamCreateWithFlags(&d->cap, cudaStreamNonBlocking);
  if (e == cudaSuccess)
    e = cudaHostAlloc(reinterpret_cast<void **>(&d->st_host), sizeof(int32_t),
                      cudaHostAllocMapped);
  if (e == cudaSuccess)
    e = cudaHostGetDevicePointer(reinterpret_cast<void **>(&d->st_map),
                                 d->st_host, 0);
  if (e != cudaSuccess) {
    locks_decoder_destroy(d);
    return LOCKS_ERR_CUDA;
  }
  *d->st_host = 0;
  *out = d;
  return LOCKS_OK;
}

locks_status_t locks_decoder_step_host(locks_decoder_t *d,
                                       const void *q_host, void *o_host,
                                       float *lse_host, int32_t *status_out,
                                       locks_stream_t stream) {
  if (!d || !q_host || !o_host || !lse_host) return LOCKS_ERR_INVALID_ARG;
  const void *q_map = q_host == d->q_host ? d->q_map : mapped(q_host);
  void *o_map =
      o_host == d->o_host ? d->o_map : const_cast<void *>(mapped(o_host));
  float *lse_map = lse_host == d->lse_host
                       ? d->lse_map
                       : static_cast<float *>(const_cast<void *>(
                             mapped(lse_host)));
  if (!q_map || !o_map || !lse_map) return LOCKS_ERR_INVALID_ARG;
  // the graph writes o and lse into the recorded output buffers: others
  // need a new recording; another query buffer is patched in place
  if (d->exec && (o_map != d->o_map || lse_map != d->lse_map)) drop_graph(d);
  locks_status_t st = LOCKS_OK;
  if (!d->exec)
    st = record(d, (cudaStream_t)stream, q_map, o_map, lse_map);
  else if (q_map != d->q_map)
    st = retarget_query(d, q_map);
  if (st != LOCKS_OK) return st;
  d->q_host = q_host;
  d->o_host = o_host;
  d->lse_host = lse_host;
  d->q_map = q_map;
  d->o_map = o_map;
  d->lse_map = lse_map;
  cudaError_t e = cudaGraphLaunch(d->exec, (cudaStream_t)stream);
  if (e == cudaSuccess) {
    locks::note_launches(d->graph_kernels);
    e = cudaStreamSynchronize((cudaStream_t)stream);
  }
  if (e != cudaSuccess) return fail(d, e);
  if (status_out) *status_out = *d->st_host;
  return LOCKS_OK;
}

int locks_decoder_last_cuda_error(const locks_decoder_t *d) {
  return d ? d->last_cuda : 0;
}

void locks_decoder_destroy(locks_decoder_t *d) {
  if (!d) return;
  drop_graph(d);
  if (d->cap) cudaStreamDestroy(d->cap);
  if (d->st_host) cudaFreeHost(d->st_host);
  delete d;
}

}  // extern "C"
