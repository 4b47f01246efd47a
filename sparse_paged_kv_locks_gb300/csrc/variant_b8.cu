// Variant scorers with a 8-bit basis, ranks 4, 8, 12 and 15
// (variant_score.cuh); one translation unit per basis width so the
// instantiations compile in parallel.
#include "variant_score.cuh"

namespace locks {

template cudaError_t launch_variant_bits<8>(int, const void *, const void *,
                                              const int32_t *, int, int, int,
                                              int, float *, int32_t *,
                                              cudaStream_t);

}  // namespace locks
