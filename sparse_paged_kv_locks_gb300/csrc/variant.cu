// Rank / precision variants (LOCKS reading notes §6 ablation): record size,
// batch limit and the scorer's dispatch by basis width (the kernels live in
// variant_score.cuh, instantiated by variant_b2.cu, variant_b4.cu and
// variant_b8.cu).
#include "launch.h"
#include "variant_layout.cuh"

namespace locks {

size_t variant_record_bytes(int rank, int vbits) {
  return (size_t)var_stride(rank, vbits);
}

template <int R>
static int max_batch_rank(int vbits) {
  const size_t fixed = vbits == 2   ? variant_smem_bytes<R, 2>(0)
                       : vbits == 4 ? variant_smem_bytes<R, 4>(0)
                                    : variant_smem_bytes<R, 8>(0);
  return (int)((227 * 1024 - fixed) / (3 * sizeof(int)));
}

int variant_max_batch(int rank, int vbits) {
  switch (rank) {
    case 4: return max_batch_rank<4>(vbits);
    case 8: return max_batch_rank<8>(vbits);
    case 12: return max_batch_rank<12>(vbits);
    default: return max_batch_rank<15>(vbits);
  }
}

cudaError_t launch_score_variant(const void *q, const void *records,
                                 int rank, int vbits,
                                 const int32_t *seq_lens, int batch, int h_kv,
                                 int G, int max_pages, float *scores,
                                 int32_t *status, cudaStream_t stream) {
  switch (vbits) {
    case 2:
      return launch_variant_bits<2>(rank, q, records, seq_lens, batch, h_kv,
                                    G, max_pages, scores, status, stream);
    case 4:
      return launch_variant_bits<4>(rank, q, records, seq_lens, batch, h_kv,
                                    G, max_pages, scores, status, stream);
    case 8:
      return launch_variant_bits<8>(rank, q, records, seq_lens, batch, h_kv,
                                    G, max_pages, scores, status, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace locks
